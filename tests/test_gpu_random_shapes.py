"""A seeded sweep of shapes against the oracle: T from 1 to 700 (ragged against every tile), d and the shard
width F/N from the smallest the ABI takes (multiples of 8) upward, N from 1 to 16.  Forward of the block,
and the sequence-parallel forward + backward (T a multiple of N)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bf16_close, dev, f64
from tensor_transformer_mlp_tp_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def _shapes(seed, n, sp):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        N = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
        d = 8 * int(rng.integers(1, 49))             # 8 .. 384
        fw = 8 * int(rng.integers(1, 33))            # shard width 8 .. 256
        T = int(rng.integers(1, 701))
        if sp:
            T = N * max(1, T // N)
        out.append((T, d, fw * N, N))
    return out


@pytest.mark.parametrize("T,d,F,N", _shapes(20261202, 40, sp=False))
def test_forward_random_shape(T, d, F, N):
    w = inputs.small_workload(T, d, N, F=F, name=f"rand_{T}_{d}_{F}_{N}")
    X, A, B, b = (inputs.draw(w, n) for n in ("X", "A", "B", "bias"))
    Y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_forward(dev(X[0]), dev(A[0]), dev(B[0]), dev(b[0]), N, Y)
    torch.cuda.synchronize()
    assert_bf16_close("Y", f64(Y), oracle.mlp_tp(X[1], A[1], B[1], b[1], N))


@pytest.mark.parametrize("T,d,F,N", _shapes(20261203, 15, sp=True))
def test_sp_forward_backward_random_shape(T, d, F, N):
    w = inputs.small_workload(T, d, N, F=F, sp=True, backward=True, bias=None, name=f"rsp_{T}_{d}_{F}_{N}")
    X, g, be, A, B, dY = (inputs.draw(w, n) for n in ("X", "gamma", "beta", "A", "B", "dY"))
    rows = T // N
    xs = list(dev(X[0]).split(rows))
    Y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    Hpre = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
    H = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_sp_forward(xs, dev(g[0]), dev(be[0]), dev(A[0]), dev(B[0]), N, list(Y.split(rows)), Hpre_out=Hpre,
                             H_out=H)
    dX = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    dA = torch.empty(d, F, dtype=torch.bfloat16, device="cuda")
    dB = torch.empty(F, d, dtype=torch.bfloat16, device="cuda")
    dgam = torch.empty(d, dtype=torch.float32, device="cuda")
    dbet = torch.empty(d, dtype=torch.float32, device="cuda")
    binding.tpmlp_sp_backward(xs, dev(g[0]), dev(be[0]), dev(A[0]), dev(B[0]), Hpre, list(dev(dY[0]).split(rows)), N,
                              list(dX.split(rows)), dA, dB, dgam, dbet, H=H)
    torch.cuda.synchronize()
    st, site = binding.tpmlp_get_device_status()
    assert st == binding.OK, f"device status {binding.status_string(st)} (site {site})"
    Xc = [X[1][j * rows:(j + 1) * rows] for j in range(N)]
    dYc = [dY[1][j * rows:(j + 1) * rows] for j in range(N)]
    assert_bf16_close("Y", f64(Y), np.concatenate(oracle.sp_forward(Xc, g[1], be[1], 1e-5, A[1], B[1], None, N)))
    ref = oracle.sp_backward(Xc, g[1], be[1], 1e-5, A[1], B[1], None, dYc, N)
    assert_bf16_close("dX", f64(dX), np.concatenate(ref["dX_chunks"]))
    assert_bf16_close("dA", f64(dA), ref["dA"])
    assert_bf16_close("dB", f64(dB), ref["dB"])
    assert_bf16_close("dgamma", dgam.double().cpu().numpy(), ref["dgamma"])
    assert_bf16_close("dbeta", dbet.double().cpu().numpy(), ref["dbeta"])
