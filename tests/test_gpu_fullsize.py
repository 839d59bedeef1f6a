"""Parity at the full workload sizes, in the exact launch sequence ``bench.py`` times.

Forward rows are independent, so the oracle recomputes a seeded sample of
rows (for the sequence-parallel block: a sample of rows of every chunk).
Backward: input-gradient rows are independent too; dA columns and dB rows
belong to single hidden units, so the oracle recomputes the block restricted
to a sample of hidden units over all T tokens.  dgamma/dbeta sum over every
row: at the full size they are checked by the oracle's LayerNorm backward
applied to the GPU's own gathered gradient dXg, whose sampled rows are
checked first; independently of the GPU, the same launch sequence at the
full width (d = 4096, F = 16384) on T = 1024 tokens is checked in full,
dgamma and dbeta included.  The smallest workload (GPT-2-medium shape) is
checked in full.
"""
import numpy as np
import pytest
import torch

import oracle
from bench import Step
from gpu_util import assert_bf16_close, f64
from tensor_transformer_mlp_tp_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def _run(name):
    w = inputs.WORKLOADS[name]
    step = Step(w, torch, binding)
    step.run()
    torch.cuda.synchronize()
    st, site = binding.tpmlp_get_device_status()
    assert st == binding.OK, f"device status {binding.status_string(st)} (site {site})"
    return w, step


def test_gpt2_medium_forward_full():
    w, step = _run("gpt2_medium_fwd")
    X, A, B, b = (inputs.draw(w, n)[1] for n in ("X", "A", "B", "bias"))
    assert_bf16_close("Y", f64(step.Y), oracle.mlp_tp(X, A, B, b, w.N))


def test_mlp7b_forward_sampled_rows():
    w, step = _run("mlp7b_fwd")
    rows = np.sort(np.random.default_rng(7).choice(w.T, 256, replace=False))
    X = inputs.draw(w, "X", rows=rows)[1]
    A, B = inputs.draw(w, "A")[1], inputs.draw(w, "B")[1]
    b = inputs.draw(w, "bias")[1]
    assert_bf16_close("Y[rows]", f64(step.Y)[rows], oracle.mlp_tp(X, A, B, b, w.N))


def _chunk_rows(w, per_chunk, seed):
    rng = np.random.default_rng(seed)
    return [np.sort(rng.choice(w.rows_per_chunk, per_chunk, replace=False)) + j * w.rows_per_chunk
            for j in range(w.N)]


def test_sp_large_forward_sampled_rows():
    w, step = _run("sp_large_fwd")
    sel = _chunk_rows(w, 16, 5)
    Xs = [inputs.draw(w, "X", rows=r)[1] for r in sel]
    g, be = inputs.draw(w, "gamma")[1], inputs.draw(w, "beta")[1]
    A, B = inputs.draw(w, "A")[1], inputs.draw(w, "B")[1]
    ref = oracle.sp_forward(Xs, g, be, 1e-5, A, B, None, w.N)
    Y = f64(step.Y)
    assert_bf16_close("Y[rows]", np.concatenate([Y[r] for r in sel]), np.concatenate(ref))


def test_sp_block_forward_backward_sampled():
    w, step = _run("sp_block_fwd_bwd")
    N = w.N
    g, be = inputs.draw(w, "gamma")[1], inputs.draw(w, "beta")[1]
    A, B = inputs.draw(w, "A")[1], inputs.draw(w, "B")[1]
    # rows: forward output, input gradient and the gathered gradient dXg
    sel = _chunk_rows(w, 16, 11)
    Xs = [inputs.draw(w, "X", rows=r)[1] for r in sel]
    dYs = [inputs.draw(w, "dY", rows=r)[1] for r in sel]
    ref_y = oracle.sp_forward(Xs, g, be, 1e-5, A, B, None, N)
    Y = f64(step.Y)
    assert_bf16_close("Y[rows]", np.concatenate([Y[r] for r in sel]), np.concatenate(ref_y))
    ref_b = oracle.sp_backward(Xs, g, be, 1e-5, A, B, None, dYs, N)
    dX, dXg = f64(step.dX), f64(step.dXg)
    assert_bf16_close("dX[rows]", np.concatenate([dX[r] for r in sel]), np.concatenate(ref_b["dX_chunks"]))
    assert_bf16_close("dXg[rows]", np.concatenate([dXg[r] for r in sel]), np.concatenate(ref_b["dXg_chunks"]))
    # hidden units: dA[:, C] and dB[C, :] over all tokens
    X = inputs.draw(w, "X")[1]
    dY = inputs.draw(w, "dY")[1]
    Xg = oracle.all_gather([oracle.layer_norm(X[lo:hi], g, be, 1e-5) for lo, hi in oracle.chunk_ranges(w.T, N)])
    C = np.sort(np.random.default_rng(3).choice(w.F, 128, replace=False))
    gu = oracle.mlp_backward(Xg, A[:, C], B[C, :], None, dY)
    assert_bf16_close("dA[:, C]", f64(step.dA)[:, C], gu["dA"])
    assert_bf16_close("dB[C, :]", f64(step.dB)[C, :], gu["dB"])
    # dgamma, dbeta: the oracle's LayerNorm backward of every chunk, fed the GPU's dXg
    dga, dbe = 0.0, 0.0
    for lo, hi in oracle.chunk_ranges(w.T, N):
        _, a, c = oracle.layer_norm_backward(X[lo:hi], g, 1e-5, dXg[lo:hi])
        dga, dbe = dga + a, dbe + c
    assert_bf16_close("dgamma", step.dgamma.double().cpu().numpy(), dga)
    assert_bf16_close("dbeta", step.dbeta.double().cpu().numpy(), dbe)


def test_sp_block_full_width_checked_in_full():
    """The SP step's launch sequence at d = 4096, F = 16384, N = 8 on 1024 tokens (128-row chunks): every
    output against the oracle's own forward and backward, so dgamma and dbeta (sums over all rows) rest on
    the oracle's gathered gradient, not the GPU's."""
    w = inputs.small_workload(1024, 4096, 8, F=16384, sp=True, backward=True, bias=None, name="sp_full_width_t1024")
    step = Step(w, torch, binding)
    step.run()
    torch.cuda.synchronize()
    st, site = binding.tpmlp_get_device_status()
    assert st == binding.OK, f"device status {binding.status_string(st)} (site {site})"
    X, g, be, A, B, dY = (inputs.draw(w, n)[1] for n in ("X", "gamma", "beta", "A", "B", "dY"))
    cr = oracle.chunk_ranges(w.T, w.N)
    Xc, dYc = [X[lo:hi] for lo, hi in cr], [dY[lo:hi] for lo, hi in cr]
    assert_bf16_close("Y", f64(step.Y), np.concatenate(oracle.sp_forward(Xc, g, be, 1e-5, A, B, None, w.N)))
    ref = oracle.sp_backward(Xc, g, be, 1e-5, A, B, None, dYc, w.N)
    assert_bf16_close("dX", f64(step.dX), np.concatenate(ref["dX_chunks"]))
    assert_bf16_close("dXg", f64(step.dXg), np.concatenate(ref["dXg_chunks"]))
    assert_bf16_close("dA", f64(step.dA), ref["dA"])
    assert_bf16_close("dB", f64(step.dB), ref["dB"])
    assert_bf16_close("dgamma", step.dgamma.double().cpu().numpy(), ref["dgamma"])
    assert_bf16_close("dbeta", step.dbeta.double().cpu().numpy(), ref["dbeta"])


def test_sp_step_is_deterministic():
    """Two runs of the SP step's launch sequence at the full width (d = 4096, F = 16384, N = 8, 1024 tokens) on
    the same inputs agree bit for bit: the shard sums run in K order inside one accumulator, and the
    dgamma/dbeta column sums and every other reduction have a fixed order."""
    w = inputs.small_workload(1024, 4096, 8, F=16384, sp=True, backward=True, bias=None, name="sp_full_width_t1024")
    step = Step(w, torch, binding)
    outs = []
    for _ in range(2):
        step.run()
        torch.cuda.synchronize()
        outs.append([t.clone() for t in (step.Y, step.dX, step.dXg, step.dA, step.dB, step.dgamma, step.dbeta)])
    st, site = binding.tpmlp_get_device_status()
    assert st == binding.OK, f"device status {binding.status_string(st)} (site {site})"
    for name, a, b in zip(("Y", "dX", "dXg", "dA", "dB", "dgamma", "dbeta"), *outs):
        assert torch.equal(a, b), name
