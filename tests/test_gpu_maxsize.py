"""Sizes whose flattened element offsets pass 2^31 - 1: a row index times the row length no longer fits a
signed 32-bit integer, so every global offset the kernels form has to be 64-bit.  The MLP cases draw the
workloads' own seeded normal inputs; the LayerNorm case (2^31 elements, too many to draw on the host in a
test) uses a hashed integer pattern, x[r, c] = (((a r + b c) mod 2^32) >> 8) mod 251 - 125, divided by 128
(exact in bf16, no row repeating), built on the device in row blocks; the oracle recomputes the same values
for a sample of rows that includes the first and the last row of the tensor and of each chunk.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bf16_close, dev, f64
from tensor_transformer_mlp_tp_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def _pattern_device(T, d, mr=2654435761, mc=40503, block=16384):
    x = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    cols = torch.arange(d, device="cuda", dtype=torch.int64)[None, :] * mc
    for r0 in range(0, T, block):
        r = torch.arange(r0, min(T, r0 + block), device="cuda", dtype=torch.int64)[:, None] * mr
        h = torch.bitwise_right_shift(torch.bitwise_and(r + cols, 0xFFFFFFFF), 8)
        x[r0:r0 + r.shape[0]] = ((h % 251 - 125).to(torch.float32) / 128.0).to(torch.bfloat16)
    return x


def _pattern_rows(rows, d, mr=2654435761, mc=40503):
    r = np.asarray(rows, dtype=np.int64)[:, None] * mr
    c = np.arange(d, dtype=np.int64)[None, :] * mc
    return ((((r + c) & 0xFFFFFFFF) >> 8) % 251 - 125).astype(np.float64) / 128.0


def _sample(T, N, k, seed):
    per = T // N
    edges = [j * per for j in range(N)] + [(j + 1) * per - 1 for j in range(N)]
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([edges, rng.choice(T, k, replace=False), [0, T - 1]]))


def test_layernorm_gather_past_2_31_elements():
    """T = 2^19 + 256 rows of d = 4096 (offsets past 2^31) in 8 chunks: LayerNorm and the gather into row slots."""
    T, d, N = (1 << 19) + 256, 4096, 8
    X = _pattern_device(T, d)
    c = np.arange(d)
    g = 1.0 + ((c * 31) % 17 - 8) / 64.0
    be = ((c * 13) % 11 - 5) / 64.0
    gd = dev(inputs.f32_to_bf16_bits(g.astype(np.float32)))
    bd = dev(inputs.f32_to_bf16_bits(be.astype(np.float32)))
    Xg = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_layernorm_gather(list(X.split(T // N)), gd, bd, N, Xg)
    torch.cuda.synchronize()
    st, site = binding.tpmlp_get_device_status()
    assert st == binding.OK, f"device status {binding.status_string(st)} (site {site})"
    rows = _sample(T, N, 48, 1)
    got = f64(Xg[torch.from_numpy(rows).cuda()])
    assert_bf16_close("Xg[rows]", got, oracle.layer_norm(_pattern_rows(rows, d), g, be, 1e-5))


def test_mlp_forward_hidden_past_2_31_elements():
    """T = 131328 tokens, d = 1024, F = 16384, N = 8: the hidden activation H has more than 2^31 elements."""
    T, d, F, N = (1 << 17) + 256, 1024, 16384, 8
    w = inputs.small_workload(T, d, N, F=F, bias=None, name=f"maxsize_T{T}_d{d}_F{F}")
    A, B, Xh = inputs.draw(w, "A"), inputs.draw(w, "B"), inputs.draw(w, "X")
    X = dev(Xh[0])
    Y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_forward(X, dev(A[0]), dev(B[0]), None, N, Y)
    torch.cuda.synchronize()
    st, site = binding.tpmlp_get_device_status()
    assert st == binding.OK, f"device status {binding.status_string(st)} (site {site})"
    rows = _sample(T, N, 48, 2)
    got = f64(Y[torch.from_numpy(rows).cuda()])
    assert_bf16_close("Y[rows]", got, oracle.mlp_tp(Xh[1][rows], A[1], B[1], None, N))


def test_mlp_backward_past_2_31_elements():
    """The backward at T = 131328, d = 1024, F = 16384, N = 8 (dHpre, H and Hpre past 2^31 elements; the weight
    gradients reduce over K = T = 131328): dX on sampled rows, dA[:, C] and dB[C, :] over all tokens for a
    sample C of hidden units."""
    T, d, F, N = (1 << 17) + 256, 1024, 16384, 8
    w = inputs.small_workload(T, d, N, F=F, bias=None, backward=True, name=f"maxsize_T{T}_d{d}_F{F}")
    A, B = inputs.draw(w, "A"), inputs.draw(w, "B")
    Xh, dYh = inputs.draw(w, "X"), inputs.draw(w, "dY")
    Ad, Bd = dev(A[0]), dev(B[0])
    X, dY = dev(Xh[0]), dev(dYh[0])
    Y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    Hpre = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
    H = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_forward(X, Ad, Bd, None, N, Y, Hpre, H)
    del Y
    dX = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    dA = torch.empty(d, F, dtype=torch.bfloat16, device="cuda")
    dB = torch.empty(F, d, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_backward(X, Ad, Bd, None, Hpre, dY, N, dX, dA, dB, H=H)
    torch.cuda.synchronize()
    st, site = binding.tpmlp_get_device_status()
    assert st == binding.OK, f"device status {binding.status_string(st)} (site {site})"
    del Hpre, H
    rows = _sample(T, N, 32, 3)
    ref = oracle.mlp_backward(Xh[1][rows], A[1], B[1], None, dYh[1][rows])
    assert_bf16_close("dX[rows]", f64(dX[torch.from_numpy(rows).cuda()]), ref["dX"])
    C = np.unique(np.concatenate([np.random.default_rng(4).choice(F, 14, replace=False), [0, F - 1]]))
    gu = oracle.mlp_backward(Xh[1], A[1][:, C], B[1][C, :], None, dYh[1])
    Ct = torch.from_numpy(C).cuda()
    assert_bf16_close("dA[:, C]", f64(dA[:, Ct]), gu["dA"])
    assert_bf16_close("dB[C, :]", f64(dB[Ct, :]), gu["dB"])


def test_reduce_scatter_past_2_31_elements():
    """The explicit reduce-scatter of N = 8 partials of T = 65600 rows x d = 4096 (offsets into the partials
    past 2^31): chunk j's rows are the fixed-order sum of the partials' rows, on sampled rows of every chunk."""
    T, d, N = 65600, 4096, 8
    P = torch.empty(N, T, d, dtype=torch.bfloat16, device="cuda")
    for i in range(N):
        P[i] = _pattern_device(T, d, 2654435761 + 7 * i, 40503 + 11 * i)
    Yc = [torch.empty(T // N, d, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    binding.tpmlp_reduce_scatter(P, N, Yc)
    torch.cuda.synchronize()
    st, site = binding.tpmlp_get_device_status()
    assert st == binding.OK, f"device status {binding.status_string(st)} (site {site})"
    rows = _sample(T, N, 48, 5)
    per = T // N
    got = np.stack([f64(Yc[r // per][r % per]) for r in rows])
    ref = oracle.all_reduce([_pattern_rows(rows, d, 2654435761 + 7 * i, 40503 + 11 * i) for i in range(N)])
    assert_bf16_close("Y[rows]", got, ref)
