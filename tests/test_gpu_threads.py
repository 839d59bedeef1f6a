"""Concurrent calls from two host threads, each on its own CUDA stream with its own workspace (the C ABI is
thread-compatible: its per-device state sits behind a lock, and ctypes releases the interpreter lock for the
length of each call, so the two threads' host code really runs at the same time)."""
import threading

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bf16_close, dev, f64
from tensor_transformer_mlp_tp_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def _case(T, d, N, seed):
    w = inputs.small_workload(T, d, N, name=f"threads_{T}_{d}_{N}")
    X, A, B, b = (inputs.draw(w, n, seed=seed) for n in ("X", "A", "B", "bias"))
    ref = oracle.mlp_tp(X[1], A[1], B[1], b[1], N)
    return (dev(X[0]), dev(A[0]), dev(B[0]), dev(b[0])), ref


def test_forward_from_two_threads_on_two_streams():
    cases = [(512, 256, 4, 1), (384, 128, 8, 2)]
    prepared = [_case(*c) for c in cases]
    results, errors = [None, None], []
    barrier = threading.Barrier(2)

    def worker(k):
        try:
            (X, A, B, b), _ = prepared[k]
            T, d, N, _ = cases[k]
            s = torch.cuda.Stream()
            ws = binding.workspace(binding.make_shape(T, d, 4 * d, N), binding.OP_FWD)
            outs = [torch.empty(T, d, dtype=torch.bfloat16, device="cuda") for _ in range(20)]
            torch.cuda.current_stream().synchronize()
            barrier.wait()
            for Y in outs:
                binding.tpmlp_forward(X, A, B, b, N, Y, ws=ws, stream=s)
            s.synchronize()
            results[k] = outs
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    st, site = binding.tpmlp_get_device_status()
    assert st == binding.OK, f"device status {binding.status_string(st)} (site {site})"
    for k, outs in enumerate(results):
        ref = prepared[k][1]
        assert_bf16_close(f"Y thread {k}", f64(outs[-1]), ref)
        first = outs[0].clone()
        assert all(torch.equal(first, y) for y in outs[1:]), f"thread {k}: repeated calls differ"
