"""GPU parity: every step and block call of the C ABI against the CPU oracle.

Shapes span several 128 x 256 output tiles and several 64-deep k-blocks, with
ragged tails in every GEMM dimension, N in {1, 2, 4, 8}.  Integer-valued
inputs make the shard reduction exact, so those cases compare bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import Guarded, assert_bf16_close, assert_fp32_close, dev, f64
from tensor_transformer_mlp_tp_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

# (T, d, N): T ragged against 128-row tiles, d against 64-deep k-blocks / 256-wide n-tiles
SHAPES = [(300, 192, 4), (128, 256, 8), (257, 136, 2), (64, 64, 1), (513, 320, 8), (1, 64, 2)]


@pytest.fixture(autouse=True)
def _device_status_clean():
    yield
    st, site = binding.tpmlp_get_device_status()
    assert st == binding.OK, f"device status {binding.status_string(st)} (wait site {site})"


def _draw(w, *names):
    return [inputs.draw(w, n) for n in names]


def _chunks(x, N):
    return [x[lo:hi] for lo, hi in oracle.chunk_ranges(x.shape[0], N)]


@pytest.mark.parametrize("T,d,N", SHAPES)
@pytest.mark.parametrize("with_bias", [True, False])
def test_gemm1_bias_gelu(T, d, N, with_bias):
    w = inputs.small_workload(T, d, N, bias=(0.0, 0.5) if with_bias else None)
    X, A, b = _draw(w, "X", "A", "bias")
    F = 4 * d
    H = Guarded((T, F))
    Hp = Guarded((T, F))
    binding.tpmlp_gemm1_bias_gelu(dev(X[0]), dev(A[0]), dev(b[0]) if b else None, N, H.t, Hp.t)
    torch.cuda.synchronize()
    pre = oracle.mlp_backward(X[1], A[1], np.zeros((F, d)), b[1] if b else None, np.zeros((T, d)))["Hpre"]
    # the shard view: H's column block i is the column-parallel output of shard i
    ref = np.concatenate([oracle.column_parallel(X[1], A[1][:, lo:hi], (b[1] if b else np.zeros(F))[lo:hi])
                          for lo, hi in oracle.shard_ranges(F, N)], axis=1)
    assert_bf16_close("H", f64(H.t), ref)
    assert_bf16_close("Hpre", f64(Hp.t), pre)
    assert H.intact() and Hp.intact()


@pytest.mark.parametrize("T,d,N", SHAPES)
def test_gemm2_shard_accum(T, d, N):
    w = inputs.small_workload(T, d, N)
    F = 4 * d
    Hb, _ = inputs.draw(w, "X", shape=(T, F), dist=(0.0, 0.5))
    B = inputs.draw(w, "B")
    Hv = inputs.bf16_bits_to_f64(Hb).reshape(T, F)
    Y = Guarded((T, d))
    binding.tpmlp_gemm2_shard_accum(dev(Hb), dev(B[0]), N, Y=Y.t)
    torch.cuda.synchronize()
    parts = [oracle.row_parallel_partial(Hv[:, lo:hi], B[1][lo:hi]) for lo, hi in oracle.shard_ranges(F, N)]
    assert_bf16_close("Y", f64(Y.t), oracle.all_reduce(parts))
    assert Y.intact()


@pytest.mark.parametrize("T,d,F,N", [(600, 128, 4096, 8), (1000, 320, 2560, 4), (2050, 256, 8192, 8)])
def test_gemm2_long_k_few_tiles(T, d, F, N):
    """Long K (40 to 128 k-blocks, the shards' rows walked into one accumulator) against few output tiles,
    ragged in T; two launches back to back (the second one's set-up overlaps the first one's tail)."""
    w = inputs.small_workload(T, d, N, F=F)
    Hb, _ = inputs.draw(w, "X", shape=(T, F), dist=(0.0, 0.5))
    B = inputs.draw(w, "B")
    Hv = inputs.bf16_bits_to_f64(Hb).reshape(T, F)
    Hd, Bd = dev(Hb), dev(B[0])
    Ys = [Guarded((T, d)) for _ in range(2)]
    for Y in Ys:
        binding.tpmlp_gemm2_shard_accum(Hd, Bd, N, Y=Y.t)
    torch.cuda.synchronize()
    ref = oracle.all_reduce([oracle.row_parallel_partial(Hv[:, lo:hi], B[1][lo:hi])
                             for lo, hi in oracle.shard_ranges(F, N)])
    for Y in Ys:
        assert_bf16_close("Y", f64(Y.t), ref)
        assert Y.intact()
    assert torch.equal(Ys[0].t, Ys[1].t)


def _int_matrix(rng, shape):
    return inputs.f32_to_bf16_bits(rng.integers(-1, 2, shape).astype(np.float32)).reshape(shape)


@pytest.mark.parametrize("N", [1, 2, 4, 8])
def test_shard_reduction_bit_exact_integers(N):
    """With entries in {-1, 0, 1} every partial and sum is an integer |v| <= 256: exact in bf16 and fp32."""
    rng = np.random.default_rng(100 + N)
    T, d, F = 384, 192, 512
    Hb = _int_matrix(rng, (T, F))
    Bb = _int_matrix(rng, (F, d))
    Hv = inputs.bf16_bits_to_f64(Hb).reshape(T, F)
    Bv = inputs.bf16_bits_to_f64(Bb).reshape(F, d)
    parts = [oracle.row_parallel_partial(Hv[:, lo:hi], Bv[lo:hi]) for lo, hi in oracle.shard_ranges(F, N)]
    ref = oracle.all_reduce(parts)
    assert np.max(np.abs(ref)) <= 256
    H_d, B_d = dev(Hb), dev(Bb)
    Y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_gemm2_shard_accum(H_d, B_d, N, Y=Y)
    # fused reduce-scatter store
    Yc = [torch.empty(T // N, d, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    binding.tpmlp_gemm2_shard_accum(H_d, B_d, N, Y_chunks=Yc)
    # explicit partials, then the reduce-scatter kernel
    P = torch.empty(N, T, d, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_gemm2_partials(H_d, B_d, N, P)
    Yr = [torch.empty(T // N, d, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    binding.tpmlp_reduce_scatter(P, N, Yr)
    torch.cuda.synchronize()
    assert np.array_equal(f64(Y), ref)
    for i in range(N):
        assert np.array_equal(f64(P[i]), parts[i])
    rs = oracle.reduce_scatter(parts, N)
    for j in range(N):
        assert np.array_equal(f64(Yc[j]), rs[j])
        assert np.array_equal(f64(Yr[j]), rs[j])
    # AllReduce = AllGather(ReduceScatter)
    assert np.array_equal(np.concatenate([f64(c) for c in Yr]), f64(Y))


@pytest.mark.parametrize("T,d,N", SHAPES)
@pytest.mark.parametrize("with_bias", [True, False])
def test_forward(T, d, N, with_bias):
    w = inputs.small_workload(T, d, N, bias=(0.0, 0.02) if with_bias else None)
    X, A, B, b = _draw(w, "X", "A", "B", "bias")
    Y = Guarded((T, d))
    binding.tpmlp_forward(dev(X[0]), dev(A[0]), dev(B[0]), dev(b[0]) if b else None, N, Y.t)
    torch.cuda.synchronize()
    assert_bf16_close("Y", f64(Y.t), oracle.mlp_tp(X[1], A[1], B[1], b[1] if b else None, N))
    assert Y.intact()


@pytest.mark.parametrize("T,d,N", [(256, 256, 4), (1024, 512, 8), (96, 136, 8), (512, 64, 2)])
def test_layernorm_gather(T, d, N):
    w = inputs.small_workload(T, d, N, sp=True)
    X, g, b = _draw(w, "X", "gamma", "beta")
    Xd = dev(X[0])
    Xg = Guarded((T, d))
    binding.tpmlp_layernorm_gather(list(Xd.split(T // N)), dev(g[0]), dev(b[0]), N, Xg.t)
    torch.cuda.synchronize()
    ref = oracle.all_gather([oracle.layer_norm(c, g[1], b[1], 1e-5) for c in _chunks(X[1], N)])
    assert_bf16_close("Xg", f64(Xg.t), ref)
    assert Xg.intact()


def test_layernorm_wide_rows():
    """d = 8192 (two warps per row) and d = 4096 (one warp per row in registers)."""
    for d in (4096, 8192):
        T, N = 64, 8
        w = inputs.small_workload(T, d, N, sp=True, name=f"lnwide{d}")
        X, g, b = _draw(w, "X", "gamma", "beta")
        Xg = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
        binding.tpmlp_layernorm_gather(list(dev(X[0]).split(T // N)), dev(g[0]), dev(b[0]), N, Xg)
        torch.cuda.synchronize()
        ref = oracle.all_gather([oracle.layer_norm(c, g[1], b[1], 1e-5) for c in _chunks(X[1], N)])
        assert_bf16_close(f"Xg d={d}", f64(Xg), ref)


@pytest.mark.parametrize("T,d,N", [(8200, 4096, 8), (2056, 8192, 8), (4104, 2048, 4), (3000, 1024, 8),
                                   (1216, 512, 8), (1000, 256, 8), (152, 4096, 8), (153, 8192, 9)])
def test_layernorm_gather_streamed(T, d, N):
    """The streamed forward: many passes around each CTA's slot ring (rows well above the SM count, ragged
    against it), one row per CTA and more CTAs than rows, every width it covers; checked in full."""
    w = inputs.small_workload(T, d, N, sp=True, name=f"lnstream_{T}_{d}")
    X, g, b = _draw(w, "X", "gamma", "beta")
    Xg = Guarded((T, d))
    binding.tpmlp_layernorm_gather(list(dev(X[0]).split(T // N)), dev(g[0]), dev(b[0]), N, Xg.t)
    torch.cuda.synchronize()
    ref = oracle.all_gather([oracle.layer_norm(c, g[1], b[1], 1e-5) for c in _chunks(X[1], N)])
    assert_bf16_close("Xg", f64(Xg.t), ref)
    assert Xg.intact()


@pytest.mark.parametrize("N", [2, 4, 8])
def test_reduce_scatter_random(N):
    T, d = 64 * N, 200
    rng = np.random.default_rng(N)
    Pb = inputs.f32_to_bf16_bits(rng.normal(size=(N, T, d)).astype(np.float32)).reshape(N, T, d)
    Pv = inputs.bf16_bits_to_f64(Pb).reshape(N, T, d)
    Y = [Guarded((T // N, d)) for _ in range(N)]
    binding.tpmlp_reduce_scatter(dev(Pb), N, [y.t for y in Y])
    torch.cuda.synchronize()
    ref = oracle.reduce_scatter(list(Pv), N)
    for j in range(N):
        assert_bf16_close(f"chunk {j}", f64(Y[j].t), ref[j])
        assert Y[j].intact()


@pytest.mark.parametrize("T,d,N", [(256, 128, 4), (384, 192, 8), (128, 256, 2), (384, 128, 8), (1024, 128, 64)])
@pytest.mark.parametrize("rs_mode", [binding.RS_FUSED, binding.RS_PARTIALS])
def test_sp_forward(T, d, N, rs_mode):
    w = inputs.small_workload(T, d, N, sp=True, bias=(0.0, 0.02))
    X, g, b, A, B, bias = _draw(w, "X", "gamma", "beta", "A", "B", "bias")
    Yc = [Guarded((T // N, d)) for _ in range(N)]
    if rs_mode == binding.RS_PARTIALS and (4 * d // N) % 64:
        with pytest.raises(binding.TpMlpError) as e:   # partials need 64-column shard widths
            binding.tpmlp_sp_forward(list(dev(X[0]).split(T // N)), dev(g[0]), dev(b[0]), dev(A[0]), dev(B[0]), N,
                                     [y.t for y in Yc], bias=dev(bias[0]), rs_mode=rs_mode)
        assert e.value.status == binding.ERR_UNSUPPORTED
        return
    binding.tpmlp_sp_forward(list(dev(X[0]).split(T // N)), dev(g[0]), dev(b[0]), dev(A[0]), dev(B[0]), N,
                             [y.t for y in Yc], bias=dev(bias[0]), rs_mode=rs_mode)
    torch.cuda.synchronize()
    ref = oracle.sp_forward(_chunks(X[1], N), g[1], b[1], 1e-5, A[1], B[1], bias[1], N)
    assert_bf16_close("Y", np.concatenate([f64(y.t) for y in Yc]), np.concatenate(ref))
    assert all(y.intact() for y in Yc)


@pytest.mark.parametrize("T,d,N", [(300, 192, 4), (256, 128, 8), (130, 64, 2), (200, 128, 64)])
@pytest.mark.parametrize("saved", ["none", "hpre", "hpre_h"])
def test_backward(T, d, N, saved):
    w = inputs.small_workload(T, d, N, backward=True, bias=(0.0, 0.2))
    X, A, B, b, dY = _draw(w, "X", "A", "B", "bias", "dY")
    F = 4 * d
    Xd, Ad, Bd, bd = dev(X[0]), dev(A[0]), dev(B[0]), dev(b[0])
    Hpre = H = None
    if saved != "none":
        Hpre = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
        Hs = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
        binding.tpmlp_forward(Xd, Ad, Bd, bd, N, torch.empty(T, d, dtype=torch.bfloat16, device="cuda"), Hpre, Hs)
        H = Hs if saved == "hpre_h" else None
    dX, dA, dB, db = Guarded((T, d)), Guarded((d, F)), Guarded((F, d)), Guarded((F,))
    binding.tpmlp_backward(Xd, Ad, Bd, bd, Hpre, dev(dY[0]), N, dX.t, dA.t, dB.t, db.t, H=H)
    torch.cuda.synchronize()
    ref = oracle.mlp_backward_tp(X[1], A[1], B[1], b[1], dY[1], N)
    for name, got, r in [("dX", dX, ref["dX"]), ("dA", dA, ref["dA"]), ("dB", dB, ref["dB"]), ("db", db, ref["db"])]:
        assert_bf16_close(name, f64(got.t), r)
        assert got.intact()


@pytest.mark.parametrize("T,d,N", [(256, 128, 4), (384, 192, 8), (64, 256, 2), (1024, 128, 64)])
@pytest.mark.parametrize("save_xg", [False, True])
def test_sp_backward(T, d, N, save_xg):
    w = inputs.small_workload(T, d, N, sp=True, backward=True, bias=None)
    X, g, b, A, B, dY = _draw(w, "X", "gamma", "beta", "A", "B", "dY")
    F = 4 * d
    rows = T // N
    xs = list(dev(X[0]).split(rows))
    # dY chunks as separate allocations: exercises the gather of non-contiguous chunks
    dys = [dev(c) for c in _chunks(dY[0], N)]
    Hpre = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
    Hs = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    Xg = torch.empty(T, d, dtype=torch.bfloat16, device="cuda") if save_xg else None
    binding.tpmlp_sp_forward(xs, dev(g[0]), dev(b[0]), dev(A[0]), dev(B[0]), N, list(Y.split(rows)), Hpre_out=Hpre,
                             H_out=Hs, Xg_out=Xg)
    dX = [Guarded((rows, d)) for _ in range(N)]
    dA, dB = Guarded((d, F)), Guarded((F, d))
    dgam, dbet = Guarded((d,), torch.float32), Guarded((d,), torch.float32)
    binding.tpmlp_sp_backward(xs, dev(g[0]), dev(b[0]), dev(A[0]), dev(B[0]), Hpre, dys, N, [x.t for x in dX], dA.t,
                              dB.t, dgam.t, dbet.t, H=Hs, Xg=Xg)
    torch.cuda.synchronize()
    ref = oracle.sp_backward(_chunks(X[1], N), g[1], b[1], 1e-5, A[1], B[1], None, _chunks(dY[1], N), N)
    assert_bf16_close("dX", np.concatenate([f64(x.t) for x in dX]), np.concatenate(ref["dX_chunks"]))
    assert_bf16_close("dA", f64(dA.t), ref["dA"])
    assert_bf16_close("dB", f64(dB.t), ref["dB"])
    assert_bf16_close("dgamma", f64(dgam.t), ref["dgamma"])
    assert_bf16_close("dbeta", f64(dbet.t), ref["dbeta"])
    assert all(x.intact() for x in dX + [dA, dB, dgam, dbet])


@pytest.mark.parametrize("d,N,rows", [(8, 1, 1), (8, 4, 3), (8, 2, 17), (16, 8, 2), (16, 4, 5)])
def test_degenerate_small_shapes(d, N, rows):
    """The smallest widths the ABI takes (d = 8, shards of 8 columns of F = 4 d, down to one row per chunk):
    K below one 64-deep k-block everywhere, a single partial tile; forward, SP forward and SP backward."""
    T, F = N * rows, 4 * d
    w = inputs.small_workload(T, d, N, sp=True, backward=True, bias=(0.0, 0.02), name=f"tiny_{d}_{N}_{rows}")
    X, g, be, A, B, b, dY = _draw(w, "X", "gamma", "beta", "A", "B", "bias", "dY")
    Y = Guarded((T, d))
    binding.tpmlp_forward(dev(X[0]), dev(A[0]), dev(B[0]), dev(b[0]), N, Y.t)
    torch.cuda.synchronize()
    assert_bf16_close("Y", f64(Y.t), oracle.mlp_tp(X[1], A[1], B[1], b[1], N))
    xs = list(dev(X[0]).split(rows))
    Yc = [Guarded((rows, d)) for _ in range(N)]
    Hpre = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
    Hs = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_sp_forward(xs, dev(g[0]), dev(be[0]), dev(A[0]), dev(B[0]), N, [y.t for y in Yc], bias=dev(b[0]),
                             Hpre_out=Hpre, H_out=Hs)
    dX = [Guarded((rows, d)) for _ in range(N)]
    dA, dB, db = Guarded((d, F)), Guarded((F, d)), Guarded((F,))
    dgam, dbet = Guarded((d,), torch.float32), Guarded((d,), torch.float32)
    binding.tpmlp_sp_backward(xs, dev(g[0]), dev(be[0]), dev(A[0]), dev(B[0]), Hpre, list(dev(dY[0]).split(rows)), N,
                              [x.t for x in dX], dA.t, dB.t, dgam.t, dbet.t, bias=dev(b[0]), dbias=db.t, H=Hs)
    torch.cuda.synchronize()
    Xc, dYc = _chunks(X[1], N), _chunks(dY[1], N)
    assert_bf16_close("Y chunks", np.concatenate([f64(y.t) for y in Yc]),
                      np.concatenate(oracle.sp_forward(Xc, g[1], be[1], 1e-5, A[1], B[1], b[1], N)))
    ref = oracle.sp_backward(Xc, g[1], be[1], 1e-5, A[1], B[1], b[1], dYc, N)
    assert_bf16_close("dX", np.concatenate([f64(x.t) for x in dX]), np.concatenate(ref["dX_chunks"]))
    for name, t, r in (("dA", dA, ref["dA"]), ("dB", dB, ref["dB"]), ("db", db, ref["db"]),
                       ("dgamma", dgam, ref["dgamma"]), ("dbeta", dbet, ref["dbeta"])):
        assert_bf16_close(name, f64(t.t), r)
    assert all(t.intact() for t in [Y, dA, dB, db, dgam, dbet] + Yc + dX)


def test_fp32_tiny_config_full():
    """The tiny fp32 workload (T=128, d=64, F=256, N=2) in full, to 1e-5 relative."""
    w = inputs.WORKLOADS["tiny_fp32_fwd"]
    X, A, B, b = _draw(w, "X", "A", "B", "bias")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    Y = torch.empty(w.T, w.d, dtype=torch.float32, device="cuda")
    binding.tpmlp_forward(t(X[0]), t(A[0]), t(B[0]), t(b[0]), w.N, Y)
    torch.cuda.synchronize()
    assert_fp32_close("Y", f64(Y), oracle.mlp_tp(X[1], A[1], B[1], b[1], w.N))


def test_empty_tokens_is_noop():
    d, N = 64, 2
    X = torch.empty(0, d, dtype=torch.bfloat16, device="cuda")
    A = torch.zeros(d, 4 * d, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(4 * d, d, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(0, d, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    binding.tpmlp_forward(X, A, B, None, N, Y, ws=ws)


def test_invalid_arguments_rejected_before_launch():
    d = 64
    X = torch.zeros(32, d, dtype=torch.bfloat16, device="cuda")
    A = torch.zeros(d, 4 * d, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(4 * d, d, dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros(32, d, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.TpMlpError) as e:
        binding.tpmlp_forward(X, A, B, None, 3, Y)          # 256 % 3 != 0
    assert e.value.status == binding.ERR_INVALID_ARG
    with pytest.raises(binding.TpMlpError) as e:
        binding.tpmlp_forward(X, A, B, None, 2, Y, ws=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == binding.ERR_WORKSPACE
    flat = torch.zeros(32 * d + 1, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.TpMlpError) as e:
        binding.tpmlp_forward(flat[1:].view(32, d), A, B, None, 2, Y)  # 2-byte aligned X
    assert e.value.status == binding.ERR_INVALID_ARG
    Yc = [torch.zeros(10, d, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    with pytest.raises(binding.TpMlpError):
        binding.tpmlp_reduce_scatter(torch.zeros(3, 31, d, dtype=torch.bfloat16, device="cuda"), 3, Yc)  # 31 % 3


def test_wait_timeout_selftest_reports_and_clears():
    binding.tpmlp_selftest_wait_timeout(2000)
    st, site = binding.tpmlp_get_device_status()
    assert st == binding.ERR_TIMEOUT and site == 99
    st, _ = binding.tpmlp_get_device_status()
    assert st == binding.OK
    # the context stays usable
    test_forward(128, 64, 2, False)


def _exact_gelu(x):
    return 0.5 * x * (1.0 + np.vectorize(math.erf)(x / math.sqrt(2.0)))


def _exact_gelu_prime(x):
    return 0.5 * (1.0 + np.vectorize(math.erf)(x / math.sqrt(2.0))) + x * np.exp(-0.5 * x * x) / math.sqrt(2 * math.pi)


def test_device_gelu_and_gelu_prime_pointwise():
    """Pre-activations set exactly (one nonzero input column, unit weights), so H = GeLU(x) and
    dHpre = GeLU'(x) can be compared point by point with the closed forms: within half a bf16 ulp of the
    result plus 1e-6 absolute."""
    T, d, N = 512, 64, 2
    F = 256
    xs = np.linspace(-8.0, 8.0, T).astype(np.float32)
    xb = inputs.f32_to_bf16_bits(xs)
    xv = inputs.bf16_bits_to_f64(xb)
    X = np.zeros((T, d), dtype=np.uint16)
    X[:, 0] = xb
    A = np.zeros((d, F), dtype=np.uint16)
    A[0, :] = inputs.f32_to_bf16_bits(np.ones(F, dtype=np.float32))
    H = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
    Hp = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_gemm1_bias_gelu(dev(X), dev(A), None, N, H, Hp)
    # dH = dY B^T = 1: dY = e_0 rows, B[:, 0] = 1
    dY = np.zeros((T, d), dtype=np.uint16)
    dY[:, 0] = inputs.f32_to_bf16_bits(np.ones(T, dtype=np.float32))
    B = np.zeros((F, d), dtype=np.uint16)
    B[:, 0] = inputs.f32_to_bf16_bits(np.ones(F, dtype=np.float32))
    dHp = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_gemm_dh_geluprime(dev(dY), dev(B), Hp, N, dHp)
    torch.cuda.synchronize()
    assert np.array_equal(f64(Hp)[:, 0], xv)
    for got, ref in [(f64(H), _exact_gelu(xv)), (f64(dHp), _exact_gelu_prime(xv))]:
        err = np.abs(got - ref[:, None])
        bound = np.abs(ref[:, None]) * 2.0 ** -8 + 1e-6
        assert np.all(err <= bound), float(np.max(err - bound))


@pytest.mark.parametrize("T,d,N", [(1000, 1024, 8), (96, 2048, 4), (64, 512, 2), (200, 4096, 8), (24, 136, 3)])
def test_layernorm_backward_step(T, d, N):
    """The LayerNorm backward step alone (streamed row kernel + column partials, or the generic kernel)."""
    w = inputs.small_workload(T, d, N, sp=True, backward=True, name=f"lnbwd_{T}_{d}_{N}")
    X, g = inputs.draw(w, "X"), inputs.draw(w, "gamma")
    dXg = inputs.draw(w, "dY")
    rows = T // N
    dX = [Guarded((rows, d)) for _ in range(N)]
    dga, dbe = Guarded((d,), torch.float32), Guarded((d,), torch.float32)
    binding.tpmlp_layernorm_backward(list(dev(X[0]).split(rows)), dev(g[0]), dev(dXg[0]), N, [x.t for x in dX],
                                     dga.t, dbe.t)
    torch.cuda.synchronize()
    refs = [oracle.layer_norm_backward(X[1][lo:hi], g[1], 1e-5, dXg[1][lo:hi]) for lo, hi in oracle.chunk_ranges(T, N)]
    assert_bf16_close("dX", np.concatenate([f64(x.t) for x in dX]), np.concatenate([r[0] for r in refs]))
    assert_bf16_close("dgamma", f64(dga.t), sum(r[1] for r in refs))
    assert_bf16_close("dbeta", f64(dbe.t), sum(r[2] for r in refs))
    assert all(x.intact() for x in dX + [dga, dbe])


@pytest.mark.parametrize("T,d,N,max_blocks", [(1024, 8192, 8, 1), (1024, 8192, 8, 37), (600, 4096, 4, 5),
                                                (600, 4096, 4, 7), (300, 136, 4, 2), (256, 2048, 8, 300)])
def test_layernorm_backward_capped_blocks(T, d, N, max_blocks):
    """The LayerNorm backward with its dgamma/dbeta partials capped below the SM count (the grid a small
    scratch gives), down to one CTA, in the fused kernels (d = 2048, 4096, 8192) and the generic one
    (d = 136); a cap above the rows changes nothing.  At d = 4096 with 7 CTAs each CTA's 85 or 86 rows
    are not a multiple of its three consumer teams and wrap the 12-slot ring seven times."""
    w = inputs.small_workload(T, d, N, sp=True, backward=True, name=f"lnbwd_cap_{T}_{d}_{max_blocks}")
    X, g = inputs.draw(w, "X"), inputs.draw(w, "gamma")
    dXg = inputs.draw(w, "dY")
    rows = T // N
    dX = [Guarded((rows, d)) for _ in range(N)]
    dga, dbe = Guarded((d,), torch.float32), Guarded((d,), torch.float32)
    ws = Guarded((max_blocks * 2 * d,), torch.float32)
    binding.tpmlp_layernorm_backward_blocks(list(dev(X[0]).split(rows)), dev(g[0]), dev(dXg[0]), N,
                                            [x.t for x in dX], dga.t, dbe.t, max_blocks, ws=ws.t.view(torch.uint8))
    torch.cuda.synchronize()
    refs = [oracle.layer_norm_backward(X[1][lo:hi], g[1], 1e-5, dXg[1][lo:hi]) for lo, hi in oracle.chunk_ranges(T, N)]
    assert_bf16_close("dX", np.concatenate([f64(x.t) for x in dX]), np.concatenate([r[0] for r in refs]))
    assert_bf16_close("dgamma", f64(dga.t), sum(r[1] for r in refs))
    assert_bf16_close("dbeta", f64(dbe.t), sum(r[2] for r in refs))
    assert all(x.intact() for x in dX + [dga, dbe, ws])


def test_layernorm_backward_blocks_rejects_a_short_workspace():
    N, rows, d = 2, 8, 1024
    xs = [torch.zeros(rows, d, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    args = (xs, torch.ones(d, dtype=torch.bfloat16, device="cuda"),
            torch.zeros(N * rows, d, dtype=torch.bfloat16, device="cuda"), N, [torch.empty_like(x) for x in xs],
            torch.empty(d, device="cuda"), torch.empty(d, device="cuda"))
    with pytest.raises(binding.TpMlpError) as e:
        binding.tpmlp_layernorm_backward_blocks(*args, 4, ws=torch.empty(4 * 2 * d * 4 - 16, dtype=torch.uint8,
                                                                         device="cuda"))
    assert e.value.status == binding.ERR_WORKSPACE
    with pytest.raises(binding.TpMlpError) as e:
        binding.tpmlp_layernorm_backward_blocks(*args, 0, ws=torch.empty(1024, dtype=torch.uint8, device="cuda"))
    assert e.value.status == binding.ERR_INVALID_ARG


@pytest.mark.parametrize("T,d,N", [(256, 4096, 8), (96, 8192, 4), (200, 1024, 8), (24, 136, 3)])
def test_rmsnorm_gather(T, d, N):
    """The listing's RMS norm, with its bf16 rounding of x * rstd before the weight."""
    w = inputs.small_workload(T, d, N, sp=True, name=f"rms_{T}_{d}_{N}")
    X, g = inputs.draw(w, "X"), inputs.draw(w, "gamma")
    Xg = Guarded((T, d))
    binding.tpmlp_rmsnorm_gather(list(dev(X[0]).split(T // N)), dev(g[0]), N, Xg.t)
    torch.cuda.synchronize()
    ref = oracle.all_gather([oracle.rms_norm(c, g[1], 1e-5) for c in _chunks(X[1], N)])
    assert_bf16_close("Xg", f64(Xg.t), ref)
    # both sides round x * rstd to bf16: elementwise within one output rounding plus a rare one-ulp flip
    err = np.abs(f64(Xg.t) - ref)
    assert np.mean(err <= np.abs(ref) * 2.0 ** -8 + 1e-30) > 0.999
    assert Xg.intact()


@pytest.mark.parametrize("T,d,N", [(32768, 4096, 8), (49152, 2048, 8), (81920, 1024, 8)])
def test_layernorm_gather_long_sequences(T, d, N):
    """Enough rows per warp that the persistent, software-pipelined LayerNorm runs; a seeded sample of
    rows (including the first and last of every chunk) is checked against the oracle."""
    w = inputs.small_workload(T, d, N, sp=True, name=f"lnlong_{T}_{d}")
    X, g, b = _draw(w, "X", "gamma", "beta")
    Xg = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_layernorm_gather(list(dev(X[0]).split(T // N)), dev(g[0]), dev(b[0]), N, Xg)
    torch.cuda.synchronize()
    rng = np.random.default_rng(T)
    rows = np.unique(np.concatenate([rng.integers(0, T, 384), np.arange(0, T, T // N), np.arange(T // N - 1, T, T // N)]))
    ref = oracle.layer_norm(X[1][rows], g[1], b[1], 1e-5)
    assert_bf16_close("Xg sample", f64(Xg[torch.from_numpy(rows).cuda()]), ref)


@pytest.mark.parametrize("d", [1024, 4096, 8192])
def test_layernorm_backward_large_mean(d):
    """Rows whose mean is large against their spread (x = 3000 + 50 N(0, 1) in bf16, steps of 16): the
    streamed backward's shifted sums keep the variance, where E[x^2] - mean^2 in fp32 (about 9e6, in
    steps of 0.5 to 1) would lose a few per cent of it."""
    T, N = 64, 4
    w = inputs.small_workload(T, d, N, sp=True, backward=True, name=f"lnbwd_mean_{d}")
    g, dXg = inputs.draw(w, "gamma"), inputs.draw(w, "dY")
    X = inputs.draw(w, "X", dist=(3000.0, 50.0))
    rows = T // N
    dX = [torch.empty(rows, d, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    dga, dbe = torch.empty(d, device="cuda"), torch.empty(d, device="cuda")
    binding.tpmlp_layernorm_backward(list(dev(X[0]).split(rows)), dev(g[0]), dev(dXg[0]), N, dX, dga, dbe)
    torch.cuda.synchronize()
    refs = [oracle.layer_norm_backward(X[1][lo:hi], g[1], 1e-5, dXg[1][lo:hi]) for lo, hi in oracle.chunk_ranges(T, N)]
    assert_bf16_close("dX", np.concatenate([f64(x) for x in dX]), np.concatenate([r[0] for r in refs]))
    assert_bf16_close("dgamma", f64(dga), sum(r[1] for r in refs))


@pytest.mark.parametrize("d", [1024, 4096, 8192])
def test_layernorm_forward_large_mean(d):
    """The gathered LayerNorm on rows whose mean is 60 times their spread (shifted one-round statistics)."""
    T, N = 64, 4
    w = inputs.small_workload(T, d, N, sp=True, name=f"lnfwd_mean_{d}")
    g, b = inputs.draw(w, "gamma"), inputs.draw(w, "beta")
    X = inputs.draw(w, "X", dist=(3000.0, 50.0))
    Xg = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_layernorm_gather(list(dev(X[0]).split(T // N)), dev(g[0]), dev(b[0]), N, Xg)
    torch.cuda.synchronize()
    ref = oracle.all_gather([oracle.layer_norm(c, g[1], b[1], 1e-5) for c in _chunks(X[1], N)])
    assert_bf16_close("Xg", f64(Xg), ref)
