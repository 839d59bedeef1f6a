"""The workspace-free LayerNorm backward (tpmlp_layernorm_backward_noalloc).

It exists for callers that cannot allocate device memory where they run the
backward (a framework whose pool owns the device memory, latency-critical code
that must not enter the CUDA allocator).  Its scratch is a fixed array inside
the library, shared by every call on the device.  This file is named so that
pytest collects it last; it must pass on its own in a fresh process and after
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bf16_close, dev, f64
from tensor_transformer_mlp_tp_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,d,N", [(1024, 4096, 8), (300, 136, 4), (256, 8192, 8)])
def test_noalloc_matches_workspace_entry_point_twice(T, d, N):
    w = inputs.small_workload(T, d, N, sp=True, backward=True, name=f"noalloc_{T}_{d}_{N}")
    X = dev(inputs.draw(w, "X")[0])
    g = dev(inputs.draw(w, "gamma")[0])
    dXg = dev(inputs.draw(w, "dY")[0])
    rows = T // N
    xs = list(X.split(rows))
    ref_dx = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    ref_dg = torch.empty(d, dtype=torch.float32, device="cuda")
    ref_db = torch.empty(d, dtype=torch.float32, device="cuda")
    binding.tpmlp_layernorm_backward(xs, g, dXg, N, list(ref_dx.split(rows)), ref_dg, ref_db)
    # the oracle's LayerNorm backward on the same chunks, the ground truth for both entry points
    Xo, go, dXo = inputs.draw(w, "X")[1], inputs.draw(w, "gamma")[1], inputs.draw(w, "dY")[1]
    refs = [oracle.layer_norm_backward(Xo[lo:hi], go, 1e-5, dXo[lo:hi]) for lo, hi in oracle.chunk_ranges(T, N)]
    o_dx = np.concatenate([r[0] for r in refs])
    o_dg, o_db = sum(r[1] for r in refs), sum(r[2] for r in refs)
    for call in range(2):  # the shared scratch keeps the previous call's contents
        dx = torch.full((T, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        dg = torch.full((d,), float("nan"), dtype=torch.float32, device="cuda")
        db = torch.full((d,), float("nan"), dtype=torch.float32, device="cuda")
        binding.tpmlp_layernorm_backward_noalloc(xs, g, dXg, N, list(dx.split(rows)), dg, db)
        torch.cuda.synchronize()
        assert_bf16_close(f"dX (call {call})", f64(dx), f64(ref_dx))
        assert_bf16_close(f"dgamma (call {call})", f64(dg), f64(ref_dg))
        assert_bf16_close(f"dbeta (call {call})", f64(db), f64(ref_db))
        assert_bf16_close(f"dX vs oracle (call {call})", f64(dx), o_dx)
        assert_bf16_close(f"dgamma vs oracle (call {call})", f64(dg), o_dg)
        assert_bf16_close(f"dbeta vs oracle (call {call})", f64(db), o_db)
    st, site = binding.tpmlp_get_device_status()
    assert st == binding.OK, (st, site)


def test_noalloc_rejects_rows_wider_than_its_scratch():
    N, rows, d = 2, 4, 8200
    xs = [torch.zeros(rows, d, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    with pytest.raises(binding.TpMlpError) as e:
        binding.tpmlp_layernorm_backward_noalloc(xs, torch.ones(d, dtype=torch.bfloat16, device="cuda"),
                                                 torch.zeros(N * rows, d, dtype=torch.bfloat16, device="cuda"), N,
                                                 [torch.empty_like(x) for x in xs],
                                                 torch.empty(d, device="cuda"), torch.empty(d, device="cuda"))
    assert e.value.status == binding.ERR_UNSUPPORTED
