"""GPU parity of the rest of the sequence-parallel region: the row layer's bias, Dropout and the residual
(``Y_j = X_j + dropout(Z_j + b2)``) fused into the row-parallel GEMM's chunked store or into the explicit
reduce-scatter, and their backward (dropout backward with the row-bias gradient, the residual's gradient
added in the LayerNorm backward), against the CPU oracle.

The keep mask is integer work and is compared bit for bit: without a residual a dropped element is an
exact zero and a kept one is not, and with a residual a dropped element equals the residual exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import Guarded, assert_bf16_close, dev, f64
from tensor_transformer_mlp_tp_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

SEED, OFFSET = 0x5EED_0F_D40, 3


@pytest.fixture(autouse=True)
def _device_status_clean():
    yield
    st, site = binding.tpmlp_get_device_status()
    assert st == binding.OK, f"device status {binding.status_string(st)} (wait site {site})"


def _chunks(x, N):
    return [x[lo:hi] for lo, hi in oracle.chunk_ranges(x.shape[0], N)]


def _bias2(w, d):
    return inputs.draw(w, "bias2", shape=(d,), dist=(0.0, 0.5))


def _keep(T, d, p, seed=SEED, offset=OFFSET):
    return oracle.dropout_keep(T, d, 0, p, seed, offset)


# (T, d, F, N): several 256-row pair tiles and 256-wide column tiles, ragged against both
SHAPES = [(512, 384, 1536, 4), (320, 256, 1024, 8), (96, 136, 544, 2), (1024, 512, 2048, 8)]


@pytest.mark.parametrize("T,d,F,N", SHAPES)
@pytest.mark.parametrize("p", [0.0, 0.1, 0.5])
def test_gemm2_bias_dropout_add(T, d, F, N, p):
    w = inputs.small_workload(T, d, N, F=F, sp=True, name=f"g2tail_{T}_{d}_{N}")
    H = inputs.draw(w, "H", shape=(T, F), dist=(0.0, 1.0))
    B = inputs.draw(w, "B")
    b2 = _bias2(w, d)
    R = inputs.draw(w, "X")
    rows = T // N
    Z = oracle.all_reduce([oracle.row_parallel_partial(H[1][:, lo:hi], B[1][lo:hi]) for lo, hi in oracle.shard_ranges(F, N)])
    keep = _keep(T, d, p)
    scale = 1.0 / (1.0 - float(np.float32(p)))
    ref = R[1] + np.where(keep, (Z + b2[1]) * scale, 0.0)
    Y = [Guarded((rows, d)) for _ in range(N)]
    Rc = list(dev(R[0]).split(rows))
    binding.tpmlp_gemm2_bias_dropout_add(dev(H[0]), dev(B[0]), N, [y.t for y in Y], bias2=dev(b2[0]), p=p,
                                         seed=SEED, offset=OFFSET, R_chunks=Rc)
    torch.cuda.synchronize()
    got = np.concatenate([f64(y.t) for y in Y])
    assert_bf16_close("Y", got, ref)
    assert np.array_equal(got[~keep], R[1][~keep]), "a dropped element differs from its residual"
    assert all(y.intact() for y in Y)
    # without the residual the mask shows directly: dropped elements are exact zeros, kept ones are not
    Y0 = [Guarded((rows, d)) for _ in range(N)]
    binding.tpmlp_gemm2_bias_dropout_add(dev(H[0]), dev(B[0]), N, [y.t for y in Y0], bias2=dev(b2[0]), p=p,
                                         seed=SEED, offset=OFFSET)
    torch.cuda.synchronize()
    got0 = np.concatenate([f64(y.t) for y in Y0])
    assert np.array_equal(got0 != 0.0, keep)
    assert_bf16_close("Y without residual", got0, np.where(keep, (Z + b2[1]) * scale, 0.0))


@pytest.mark.parametrize("N,p", [(2, 0.0), (4, 0.25), (8, 0.5)])
def test_reduce_scatter_bias_dropout_add(N, p):
    T, d = 64 * N, 200
    rng = np.random.default_rng(N)
    Pb = inputs.f32_to_bf16_bits(rng.normal(size=(N, T, d)).astype(np.float32)).reshape(N, T, d)
    Pv = inputs.bf16_bits_to_f64(Pb).reshape(N, T, d)
    w = inputs.small_workload(T, d, N, sp=True, name=f"rstail_{N}")
    b2 = _bias2(w, d)
    R = inputs.draw(w, "X")
    rows = T // N
    keep = _keep(T, d, p)
    scale = 1.0 / (1.0 - float(np.float32(p)))
    Z = np.concatenate(oracle.reduce_scatter(list(Pv), N))
    ref = R[1] + np.where(keep, (Z + b2[1]) * scale, 0.0)
    Y = [Guarded((rows, d)) for _ in range(N)]
    binding.tpmlp_reduce_scatter_bias_dropout_add(dev(Pb), N, [y.t for y in Y], bias2=dev(b2[0]), p=p, seed=SEED,
                                                  offset=OFFSET, R_chunks=list(dev(R[0]).split(rows)))
    torch.cuda.synchronize()
    got = np.concatenate([f64(y.t) for y in Y])
    assert_bf16_close("Y", got, ref)
    assert np.array_equal(got[~keep], R[1][~keep])
    assert all(y.intact() for y in Y)


@pytest.mark.parametrize("T,d,N,p", [(1000, 1024, 8, 0.1), (96, 136, 3, 0.5), (64, 4096, 4, 0.0), (48, 8, 2, 0.3)])
def test_dropout_backward(T, d, N, p):
    w = inputs.small_workload(T, d, N, sp=True, backward=True, name=f"dropbwd_{T}_{d}_{N}")
    dY = inputs.draw(w, "dY")
    rows = T // N
    keep = _keep(T, d, p)
    scale = 1.0 / (1.0 - float(np.float32(p)))
    dZ = Guarded((T, d))
    db2 = Guarded((d,))
    binding.tpmlp_dropout_backward(list(dev(dY[0]).split(rows)), N, dZ.t, dbias2=db2.t, p=p, seed=SEED,
                                   offset=OFFSET)
    torch.cuda.synchronize()
    ref = np.where(keep, dY[1] * scale, 0.0)
    got = f64(dZ.t)
    assert np.array_equal(got != 0.0, keep & (dY[1] != 0.0))
    assert_bf16_close("dZ", got, ref)
    assert_bf16_close("dbias2", f64(db2.t), ref.sum(axis=0))
    assert dZ.intact() and db2.intact()


@pytest.mark.parametrize("T,d,N", [(1000, 1024, 8), (96, 2048, 4), (200, 4096, 8), (2400, 4096, 8), (24, 136, 3),
                                   (64, 8192, 2)])
def test_layernorm_backward_add(T, d, N):
    """The streamed and the generic LayerNorm backward with the residual's gradient added to dx."""
    w = inputs.small_workload(T, d, N, sp=True, backward=True, name=f"lnadd_{T}_{d}_{N}")
    X, g = inputs.draw(w, "X"), inputs.draw(w, "gamma")
    dXg = inputs.draw(w, "dY")
    Rg = inputs.draw(w, "dY", seed=1)
    rows = T // N
    dX = [Guarded((rows, d)) for _ in range(N)]
    dga, dbe = Guarded((d,), torch.float32), Guarded((d,), torch.float32)
    binding.tpmlp_layernorm_backward_add(list(dev(X[0]).split(rows)), dev(g[0]), dev(dXg[0]),
                                         list(dev(Rg[0]).split(rows)), N, [x.t for x in dX], dga.t, dbe.t)
    torch.cuda.synchronize()
    refs = [oracle.layer_norm_backward(X[1][lo:hi], g[1], 1e-5, dXg[1][lo:hi]) for lo, hi in oracle.chunk_ranges(T, N)]
    assert_bf16_close("dX", np.concatenate([f64(x.t) for x in dX]), np.concatenate([r[0] for r in refs]) + Rg[1])
    assert_bf16_close("dgamma", f64(dga.t), sum(r[1] for r in refs))
    assert_bf16_close("dbeta", f64(dbe.t), sum(r[2] for r in refs))
    assert all(x.intact() for x in dX + [dga, dbe])


@pytest.mark.parametrize("T,d,N,rs_mode,p", [(512, 256, 4, binding.RS_FUSED, 0.1),
                                              (256, 128, 8, binding.RS_PARTIALS, 0.25),
                                              (96, 136, 2, binding.RS_FUSED, 0.0),
                                              (320, 192, 8, binding.RS_FUSED, 0.5)])
def test_sp_block_forward_backward(T, d, N, rs_mode, p):
    """The whole region, forward and backward, through the block calls with saved activations."""
    w = inputs.small_workload(T, d, N, sp=True, backward=True, bias=(0.0, 0.2), name=f"spblock_{T}_{d}_{N}")
    X, A, B, b, g, be, dY = [inputs.draw(w, n) for n in ("X", "A", "B", "bias", "gamma", "beta", "dY")]
    b2 = _bias2(w, d)
    F = w.F
    rows = T // N
    Xc = list(dev(X[0]).split(rows))
    Y = [Guarded((rows, d)) for _ in range(N)]
    Hpre = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
    H = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
    Xg = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    Ad, Bd, bd, gd, bed = dev(A[0]), dev(B[0]), dev(b[0]), dev(g[0]), dev(be[0])
    binding.tpmlp_sp_block_forward(Xc, gd, bed, Ad, Bd, N, [y.t for y in Y], bias=bd, bias2=dev(b2[0]), p=p,
                                   seed=SEED, offset=OFFSET, rs_mode=rs_mode, Hpre_out=Hpre, H_out=H, Xg_out=Xg)
    dX = [Guarded((rows, d)) for _ in range(N)]
    dA, dB = Guarded((d, F)), Guarded((F, d))
    dbias, db2 = Guarded((F,)), Guarded((d,))
    dga, dbe = Guarded((d,), torch.float32), Guarded((d,), torch.float32)
    binding.tpmlp_sp_block_backward(Xc, gd, bed, Ad, Bd, Hpre, list(dev(dY[0]).split(rows)), N, [x.t for x in dX],
                                    dA.t, dB.t, dga.t, dbe.t, bias=bd, dbias=dbias.t, dbias2=db2.t, p=p, seed=SEED,
                                    offset=OFFSET, H=H, Xg=Xg)
    torch.cuda.synchronize()
    Xo = _chunks(X[1], N)
    refY = oracle.sp_block_forward(Xo, g[1], be[1], 1e-5, A[1], B[1], b[1], b2[1], p, SEED, OFFSET, N)
    gotY = np.concatenate([f64(y.t) for y in Y])
    assert_bf16_close("Y", gotY, np.concatenate(refY))
    keep = _keep(T, d, p)
    assert np.array_equal(gotY[~keep], X[1][~keep])
    ref = oracle.sp_block_backward(Xo, g[1], be[1], 1e-5, A[1], B[1], b[1], p, SEED, OFFSET, _chunks(dY[1], N), N)
    assert_bf16_close("dX", np.concatenate([f64(x.t) for x in dX]), np.concatenate(ref["dX_chunks"]))
    for name, t, r in (("dA", dA, ref["dA"]), ("dB", dB, ref["dB"]), ("db", dbias, ref["db"]),
                       ("db2", db2, ref["db2"]), ("dgamma", dga, ref["dgamma"]), ("dbeta", dbe, ref["dbeta"])):
        assert_bf16_close(name, f64(t.t), r)
    assert all(t.intact() for t in Y + dX + [dA, dB, dbias, db2, dga, dbe])


def test_sp_block_without_tail_equals_sp_forward_plus_residual():
    """p = 0, no row bias: the block output is the residual plus tpmlp_sp_forward's output, bit for bit
    apart from the one rounding of the sum."""
    T, d, N = 256, 256, 4
    w = inputs.small_workload(T, d, N, sp=True, name="spblock_plain")
    X, A, B, b, g, be = [inputs.draw(w, n) for n in ("X", "A", "B", "bias", "gamma", "beta")]
    rows = T // N
    Xc = list(dev(X[0]).split(rows))
    args = (Xc, dev(g[0]), dev(be[0]), dev(A[0]), dev(B[0]), N)
    Yb = [torch.empty(rows, d, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    Ys = [torch.empty(rows, d, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    binding.tpmlp_sp_block_forward(*args, Yb, bias=dev(b[0]))
    binding.tpmlp_sp_forward(*args, Ys, bias=dev(b[0]))
    torch.cuda.synchronize()
    # Ys is the bf16-rounded Z; the block rounds X + Z once, so compare against X + Ys within one rounding
    got = np.concatenate([f64(y) for y in Yb])
    near = X[1] + np.concatenate([f64(y) for y in Ys])
    assert np.all(np.abs(got - near) <= np.abs(near) * 2.0 ** -8 + np.abs(np.concatenate([f64(y) for y in Ys])) * 2.0 ** -8)


def test_dropout_mask_changes_with_offset_and_seed():
    T, d, N = 128, 256, 2
    rows = T // N
    ones = torch.ones(T, d, dtype=torch.bfloat16, device="cuda")
    outs = []
    for seed, offset in ((1, 0), (1, 1), (2, 0), (1, 0)):
        dZ = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
        binding.tpmlp_dropout_backward(list(ones.split(rows)), N, dZ, p=0.5, seed=seed, offset=offset)
        outs.append(f64(dZ) != 0)
    torch.cuda.synchronize()
    assert np.array_equal(outs[0], outs[3])
    assert np.array_equal(outs[0], oracle.dropout_keep(T, d, 0, 0.5, 1, 0))
    for other in outs[1:3]:
        assert 0.4 < (outs[0] == other).mean() < 0.6


# ----------------------------------------------------------------------------- saved keep mask

def _packed_keep(T, d, p):
    """The oracle's keep mask as the bit layout the calls write: bit e % 8 of byte e / 8."""
    return np.packbits(_keep(T, d, p).reshape(-1), bitorder="little")


def _mask_buffer(T, d):
    return Guarded((binding.keep_mask_bytes(T, d),), torch.uint8)


@pytest.mark.parametrize("T,d,F,N", [(512, 384, 1536, 4), (96, 136, 544, 2)])
def test_keep_mask_written_by_the_row_parallel_gemm(T, d, F, N):
    """The fused store writes the keep bits it applies (bit for bit the oracle's mask; d = 136 has a
    ragged 32-column group at each row's end)."""
    p = 0.3
    w = inputs.small_workload(T, d, N, F=F, sp=True, name=f"g2mask_{T}_{d}_{N}")
    H, B = inputs.draw(w, "H", shape=(T, F), dist=(0.0, 1.0)), inputs.draw(w, "B")
    rows = T // N
    mask = _mask_buffer(T, d)
    Y = [torch.empty(rows, d, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    binding.tpmlp_gemm2_bias_dropout_add(dev(H[0]), dev(B[0]), N, Y, p=p, seed=SEED, offset=OFFSET,
                                         keep_mask=mask.t)
    torch.cuda.synchronize()
    assert np.array_equal(mask.t.cpu().numpy(), _packed_keep(T, d, p))
    assert mask.intact()


def test_keep_mask_written_by_the_reduce_scatter():
    N, p = 4, 0.25
    T, d = 64 * N, 200
    rng = np.random.default_rng(7)
    Pb = inputs.f32_to_bf16_bits(rng.normal(size=(N, T, d)).astype(np.float32)).reshape(N, T, d)
    rows = T // N
    mask = _mask_buffer(T, d)
    Y = [torch.empty(rows, d, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    binding.tpmlp_reduce_scatter_bias_dropout_add(dev(Pb), N, Y, p=p, seed=SEED, offset=OFFSET, keep_mask=mask.t)
    torch.cuda.synchronize()
    assert np.array_equal(mask.t.cpu().numpy(), _packed_keep(T, d, p))
    assert mask.intact()


@pytest.mark.parametrize("T,d,N,p", [(1000, 1024, 8, 0.1), (96, 136, 3, 0.5)])
def test_dropout_backward_reads_the_keep_mask(T, d, N, p):
    """With the saved mask the backward gives the same bits as regenerating it; a mask that differs from
    the generator's (all ones) is what the backward then applies."""
    w = inputs.small_workload(T, d, N, sp=True, backward=True, name=f"dropbwd_{T}_{d}_{N}")
    dY = inputs.draw(w, "dY")
    rows = T // N
    dYc = list(dev(dY[0]).split(rows))
    mask = torch.from_numpy(_packed_keep(T, d, p)).cuda()
    outs = []
    for m in (None, mask):
        dZ = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
        db2 = torch.empty(d, dtype=torch.bfloat16, device="cuda")
        binding.tpmlp_dropout_backward(dYc, N, dZ, dbias2=db2, p=p, seed=SEED, offset=OFFSET, keep_mask=m)
        outs.append((dZ, db2))
    ones = torch.full((binding.keep_mask_bytes(T, d),), 255, dtype=torch.uint8, device="cuda")
    dZ1 = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_dropout_backward(dYc, N, dZ1, p=p, seed=SEED, offset=OFFSET, keep_mask=ones)
    torch.cuda.synchronize()
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    scale = 1.0 / (1.0 - float(np.float32(p)))
    assert_bf16_close("dZ (mask of ones)", f64(dZ1), dY[1] * scale)


def test_sp_block_keep_mask_forward_to_backward():
    """The block forward saves the mask; the block backward given it matches the one that regenerates it."""
    T, d, N, p = 256, 256, 4, 0.2
    w = inputs.small_workload(T, d, N, sp=True, backward=True, bias=(0.0, 0.2), name="spblock_mask")
    X, A, B, b, g, be, dY = [inputs.draw(w, n) for n in ("X", "A", "B", "bias", "gamma", "beta", "dY")]
    F = w.F
    rows = T // N
    Xc = list(dev(X[0]).split(rows))
    Ad, Bd, bd, gd, bed = dev(A[0]), dev(B[0]), dev(b[0]), dev(g[0]), dev(be[0])
    mask = _mask_buffer(T, d)
    Hpre = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
    Y = [torch.empty(rows, d, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    binding.tpmlp_sp_block_forward(Xc, gd, bed, Ad, Bd, N, Y, bias=bd, p=p, seed=SEED, offset=OFFSET,
                                   Hpre_out=Hpre, keep_mask=mask.t)
    grads = []
    for m in (None, mask.t):
        dX = [torch.empty(rows, d, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
        dA, dB = torch.empty(d, F, dtype=torch.bfloat16, device="cuda"), torch.empty(F, d, dtype=torch.bfloat16, device="cuda")
        dga, dbe = torch.empty(d, device="cuda"), torch.empty(d, device="cuda")
        binding.tpmlp_sp_block_backward(Xc, gd, bed, Ad, Bd, Hpre, list(dev(dY[0]).split(rows)), N, dX, dA, dB, dga,
                                        dbe, bias=bd, p=p, seed=SEED, offset=OFFSET, keep_mask=m)
        grads.append(dX + [dA, dB, dga, dbe])
    torch.cuda.synchronize()
    assert np.array_equal(mask.t.cpu().numpy(), _packed_keep(T, d, p))
    for a, b in zip(*grads):
        assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16),
                           b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16))
