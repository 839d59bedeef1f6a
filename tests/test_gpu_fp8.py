"""GPU parity of the FP8 (E4M3) forward with delayed scaling against the CPU oracle.

The E4M3 codes are integer results: where both sides quantise the same float32 product (bf16 weights
times a scale) they must agree bit for bit; where the value being quantised is itself a float32
computation on the GPU and a float64 one in the oracle (the norm output, the GeLU output), the two may
round to neighbouring codes on values within rounding error of a midpoint, so those are checked for
agreement on all but a tiny fraction and for at most one code step apart.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import Guarded, assert_bf16_close, dev, f64
from tensor_transformer_mlp_tp_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _device_status_clean():
    yield
    st, site = binding.tpmlp_get_device_status()
    assert st == binding.OK, f"device status {binding.status_string(st)} (wait site {site})"


def _chunks(x, N):
    return [x[lo:hi] for lo, hi in oracle.chunk_ranges(x.shape[0], N)]


def e4m3_values(t):
    """E4M3 byte tensor (uint8, CUDA) -> float64 numpy values."""
    return t.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()


def e4m3_bytes(values):
    """Exactly representable float64 values -> E4M3 byte tensor on the GPU (torch's cast, exact here)."""
    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32)).to(torch.float8_e4m3fn)
    assert np.array_equal(t.to(torch.float64).numpy(), values)
    return t.view(torch.uint8).cuda()


def f32dev(x):
    return torch.tensor(np.asarray(x, dtype=np.float32).reshape(-1), device="cuda")


def _code_step_agreement(got, ref, min_equal=0.999, mant_bits=3, min_quantum=2.0 ** -9):
    """Codes equal on all but a tiny fraction; the rest one format step apart (neighbouring values).
    E4M3: 3 mantissa bits, smallest quantum 2**-9; E5M2: 2 bits, 2**-16."""
    eq = got == ref
    assert eq.mean() >= min_equal, eq.mean()
    if not eq.all():
        g, r = got[~eq], ref[~eq]
        hi = np.maximum(np.abs(g), np.abs(r))
        # one step is at most 2**-mant_bits of the larger magnitude (the subnormal quantum below that)
        assert np.all(np.abs(g - r) <= np.maximum(hi * 2.0 ** -mant_bits, min_quantum) + 1e-30)
        assert np.all(np.sign(g) * np.sign(r) >= 0)


def e5m2_values(t):
    return t.cpu().view(torch.float8_e5m2).to(torch.float64).numpy()


def e5m2_bytes(values):
    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32)).to(torch.float8_e5m2)
    assert np.array_equal(t.to(torch.float64).numpy(), values)
    return t.view(torch.uint8).cuda()


def assert_fp8_close(name, got, ref, maxrel=0.1, frob=2e-2):
    """Block-level FP8 tolerance against the oracle's own casts: where the GPU's fp32 value and the oracle's
    fp64 value of a tensor fall on two sides of a rounding midpoint the two casts differ by one format step
    (up to 2**-3 of the element for E4M3, 2**-2 for E5M2); a fraction of a percent of such flips moves the
    GEMM results by about 1%.  The FP8 block tests also check every gradient at the bf16 band with the
    oracle fed this run's own saved codes, which removes the flips; this looser check is the second one."""
    from gpu_util import errors
    m, f = errors(got, ref)
    assert np.all(np.isfinite(got)) and m <= maxrel and f <= frob, f"{name}: max {m:.3e} frob {f:.3e}"


@pytest.mark.parametrize("rows,cols,transpose", [(256, 1024, True), (4096, 320, True), (48, 80, True),
                                                 (256, 1024, False), (48, 80, False)])
def test_cast_e4m3_codes_are_bit_exact(rows, cols, transpose):
    w = inputs.small_workload(64, 64, 2, name=f"cast_{rows}_{cols}")
    W = inputs.draw(w, "W", shape=(rows, cols), dist=(0.0, 0.02))
    S = 448.0 / np.max(np.abs(W[1])) * 0.9
    scale, amax = f32dev([S]), torch.zeros(1, device="cuda")
    out = torch.empty((cols, rows) if transpose else (rows, cols), dtype=torch.uint8, device="cuda")
    binding.tpmlp_cast_e4m3(dev(W[0]), scale, out, amax, transpose=transpose)
    torch.cuda.synchronize()
    ref = oracle.quantize_e4m3(W[1], S)
    got = e4m3_values(out)
    assert np.array_equal(got, ref.T if transpose else ref)
    assert float(amax.item()) == np.max(np.abs(W[1]))


@pytest.mark.parametrize("T,d,N", [(256, 1024, 8), (96, 4096, 4), (64, 8192, 2), (40, 256, 4)])
def test_layernorm_gather_e4m3(T, d, N):
    w = inputs.small_workload(T, d, N, sp=True, name=f"lnq_{T}_{d}_{N}")
    X, g, b = (inputs.draw(w, n) for n in ("X", "gamma", "beta"))
    Xg = oracle.all_gather([oracle.layer_norm(c, g[1], b[1], 1e-5) for c in _chunks(X[1], N)])
    S = 448.0 / np.max(np.abs(Xg))
    scale, amax = f32dev([S]), torch.zeros(1, device="cuda")
    Xq = torch.empty(T, d, dtype=torch.uint8, device="cuda")
    binding.tpmlp_layernorm_gather_e4m3(list(dev(X[0]).split(T // N)), dev(g[0]), dev(b[0]), N, scale, Xq, amax)
    torch.cuda.synchronize()
    _code_step_agreement(e4m3_values(Xq), oracle.quantize_e4m3(Xg, S))
    assert abs(float(amax.item()) / np.max(np.abs(Xg)) - 1) < 1e-5


# (T, d, F, N): a lone 64-row block (the odd CTA all zero fill), ragged F against 256-wide tiles and
# 128-deep k-blocks, several pair tiles
GEMM_SHAPES = [(512, 256, 1024, 4), (256, 512, 1056, 4), (64, 1024, 4096, 2), (320, 512, 2048, 8)]


def _fp8_problem(T, d, F, N, name):
    w = inputs.small_workload(T, d, N, F=F, bias=(0.0, 0.5), name=name)
    X, A, B, b = (inputs.draw(w, n) for n in ("X", "A", "B", "bias"))
    sx, sa, sb = (448.0 / np.max(np.abs(v[1])) for v in (X, A, B))
    return X, A, B, b, sx, sa, sb


@pytest.mark.parametrize("T,d,F,N", GEMM_SHAPES)
def test_gemm1_e4m3(T, d, F, N):
    X, A, B, b, sx, sa, _ = _fp8_problem(T, d, F, N, f"g1q_{T}_{d}_{F}")
    qx, qa = oracle.quantize_e4m3(X[1], sx), oracle.quantize_e4m3(A[1], sa)
    H = oracle.gelu(qx @ qa / (float(np.float32(sx)) * float(np.float32(sa))) + b[1])
    sh = 448.0 / np.max(np.abs(H))
    Hq = Guarded((T, F), torch.uint8)
    Hpre = Guarded((T, F))
    amax = torch.zeros(1, device="cuda")
    binding.tpmlp_gemm1_e4m3(e4m3_bytes(qx), e4m3_bytes(qa.T), dev(b[0]), N, f32dev([sx]), f32dev([sa]),
                             f32dev([sh]), Hq.t, amax, Hpre=Hpre.t)
    torch.cuda.synchronize()
    _code_step_agreement(e4m3_values(Hq.t), oracle.quantize_e4m3(H, sh))
    assert_bf16_close("Hpre", f64(Hpre.t), qx @ qa / (float(np.float32(sx)) * float(np.float32(sa))) + b[1])
    assert abs(float(amax.item()) / np.max(np.abs(H)) - 1) < 1e-5
    assert Hq.intact() and Hpre.intact()


@pytest.mark.parametrize("T,d,F,N", GEMM_SHAPES)
@pytest.mark.parametrize("chunked", [True, False])
def test_gemm2_e4m3(T, d, F, N, chunked):
    w = inputs.small_workload(T, d, N, F=F, name=f"g2q_{T}_{d}_{F}")
    Hv = oracle.gelu(inputs.draw(w, "H", shape=(T, F), dist=(0.0, 1.0))[1])
    B = inputs.draw(w, "B")
    sh, sb = 448.0 / np.max(np.abs(Hv)), 448.0 / np.max(np.abs(B[1]))
    qh, qb = oracle.quantize_e4m3(Hv, sh), oracle.quantize_e4m3(B[1], sb)
    ref = oracle.all_reduce([qh[:, lo:hi] @ qb[lo:hi] for lo, hi in oracle.shard_ranges(F, N)]) / (
        float(np.float32(sh)) * float(np.float32(sb)))
    args = (e4m3_bytes(qh), e4m3_bytes(qb.T), N, f32dev([sh]), f32dev([sb]))
    if chunked:
        Y = [Guarded((T // N, d)) for _ in range(N)]
        binding.tpmlp_gemm2_e4m3(*args, Y_chunks=[y.t for y in Y])
        torch.cuda.synchronize()
        got = np.concatenate([f64(y.t) for y in Y])
    else:
        Y = [Guarded((T, d))]
        binding.tpmlp_gemm2_e4m3(*args, Y=Y[0].t)
        torch.cuda.synchronize()
        got = f64(Y[0].t)
    assert_bf16_close("Y", got, ref)
    assert all(y.intact() for y in Y)


def test_fp8_update_scales():
    L = 16
    rng = np.random.default_rng(3)
    hist = rng.uniform(0.5, 4.0, size=(4, L))
    hist[3] = 0.0                      # a tensor with no history yet keeps scale 1 until it has one
    am = np.array([3.0, 0.25, 7.5, 0.0])
    scale = torch.zeros(4, device="cuda")
    amax = f32dev(am)
    history = torch.tensor(hist.astype(np.float32), device="cuda")
    binding.tpmlp_fp8_update_scales(binding.fp8_state(scale, amax, history, margin=1))
    torch.cuda.synchronize()
    h32 = hist.astype(np.float32).astype(np.float64)
    for i in range(4):
        rolled = oracle.roll_amax_history(h32[i], np.float32(am[i]))
        assert np.array_equal(history[i].cpu().double().numpy(), rolled)
        assert abs(float(scale[i].item()) / oracle.fp8_scale(rolled, margin=1) - 1) < 1e-6
    assert float(amax.abs().sum().item()) == 0.0


@pytest.mark.parametrize("T,d,F,N", [(512, 256, 1024, 4), (256, 1024, 4096, 8), (64, 512, 1056, 2)])
def test_sp_forward_fp8_block(T, d, F, N):
    """The whole FP8 block: weight casts, E4M3 LayerNorm, both E4M3 GEMMs, the delayed-scale update."""
    w = inputs.small_workload(T, d, N, F=F, sp=True, bias=(0.0, 0.2), name=f"spq_{T}_{d}_{F}")
    X, A, B, b, g, be = (inputs.draw(w, n) for n in ("X", "A", "B", "bias", "gamma", "beta"))
    Xo = _chunks(X[1], N)
    # scales as delayed scaling would give them after steady amaxes: 448 / amax of each tensor (H's amax
    # depends on the other three scales, so it comes from a second pass)
    first = oracle.sp_forward_fp8(Xo, g[1], be[1], 1e-5, A[1], B[1], b[1], N, (1.0, 1.0, 1.0, 1.0))["amax"]
    s3 = [float(np.float32(448.0 / first[k])) for k in ("X", "A", "B")]
    am = oracle.sp_forward_fp8(Xo, g[1], be[1], 1e-5, A[1], B[1], b[1], N, (*s3, 1.0))["amax"]
    scales = (*s3, float(np.float32(448.0 / am["H"])))
    ref = oracle.sp_forward_fp8(Xo, g[1], be[1], 1e-5, A[1], B[1], b[1], N, scales)
    L = 8
    hist = np.tile(np.array([[am["X"]], [am["A"]], [am["B"]], [am["H"]]]), (1, L)).astype(np.float32)
    scale, amax = f32dev(scales), torch.zeros(4, device="cuda")
    history = torch.tensor(hist, device="cuda")
    state = binding.fp8_state(scale, amax, history)
    Y = [Guarded((T // N, d)) for _ in range(N)]
    binding.tpmlp_sp_forward_fp8(list(dev(X[0]).split(T // N)), dev(g[0]), dev(be[0]), dev(A[0]), dev(B[0]), N,
                                 [y.t for y in Y], state, bias=dev(b[0]))
    binding.tpmlp_fp8_update_scales(state)          # the step is over: delayed-scale update
    torch.cuda.synchronize()
    got = np.concatenate([f64(y.t) for y in Y])
    assert_bf16_close("Y (fp8)", got, np.concatenate(ref["Y_chunks"]))
    # the quantisation error itself is of E4M3's size against the unquantised block
    full = np.concatenate(oracle.sp_forward(Xo, g[1], be[1], 1e-5, A[1], B[1], b[1], N))
    err = np.linalg.norm(got - full) / np.linalg.norm(full)
    assert err < 0.08, err
    # the step recorded its amaxes into the history and derived the next scales from it
    new_hist = history.cpu().double().numpy()
    for i, k in enumerate(("X", "A", "B", "H")):
        assert abs(new_hist[i, -1] / ref["amax"][k] - 1) < 1e-5, k
        assert np.array_equal(new_hist[i, :-1], hist[i, 1:].astype(np.float64))
        expect = oracle.fp8_scale(oracle.roll_amax_history(hist[i].astype(np.float64), ref["amax"][k]))
        assert abs(float(scale[i].item()) / expect - 1) < 1e-5, k
    assert float(amax.abs().sum().item()) == 0.0
    assert all(y.intact() for y in Y)



# ----------------------------------------------------------------------------- FP8 backward (E5M2 gradients)

@pytest.mark.parametrize("rows,cols,transpose", [(256, 1024, True), (48, 80, True), (256, 1024, False)])
def test_cast_e5m2_codes_are_bit_exact(rows, cols, transpose):
    w = inputs.small_workload(64, 64, 2, name=f"cast5_{rows}_{cols}")
    G = inputs.draw(w, "G", shape=(rows, cols), dist=(0.0, 3.0))
    S = 57344.0 / np.max(np.abs(G[1])) * 0.5
    scale, amax = f32dev([S]), torch.zeros(1, device="cuda")
    out = torch.empty((cols, rows) if transpose else (rows, cols), dtype=torch.uint8, device="cuda")
    binding.tpmlp_cast_e5m2(dev(G[0]), scale, out, amax, transpose=transpose)
    torch.cuda.synchronize()
    ref = oracle.quantize_e5m2(G[1], S)
    assert np.array_equal(e5m2_values(out), ref.T if transpose else ref)
    assert float(amax.item()) == np.max(np.abs(G[1]))


@pytest.mark.parametrize("rows,cols", [(256, 1024), (4096, 48), (80, 16)])
def test_transpose_bytes(rows, cols):
    src = torch.randint(0, 256, (rows, cols), dtype=torch.uint8, device="cuda")
    dst = torch.empty(cols, rows, dtype=torch.uint8, device="cuda")
    binding.tpmlp_transpose_bytes(src, dst)
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), src.cpu().t().contiguous())


@pytest.mark.parametrize("a_fmt,b_fmt", [(binding.E4M3, binding.E5M2), (binding.E5M2, binding.E4M3),
                                         (binding.E4M3, binding.E4M3), (binding.E5M2, binding.E5M2)])
@pytest.mark.parametrize("M,N,K", [(512, 256, 1024), (320, 1056, 512), (64, 512, 2048)])
def test_gemm_fp8_mixed_formats(a_fmt, b_fmt, M, N, K):
    """Operands given as exact codes: the product of the codes divided by the scales, fp32 accumulation."""
    w = inputs.small_workload(64, 64, 2, name=f"gq_{M}_{N}_{K}_{a_fmt}{b_fmt}")
    Av = inputs.draw(w, "A8", shape=(M, K), dist=(0.0, 1.0))[1]
    Bv = inputs.draw(w, "B8", shape=(N, K), dist=(0.0, 1.0))[1]
    sa, sb = 64.0, 2048.0 / 3
    q = {binding.E4M3: oracle.quantize_e4m3, binding.E5M2: oracle.quantize_e5m2}
    enc = {binding.E4M3: e4m3_bytes, binding.E5M2: e5m2_bytes}
    qa, qb = q[a_fmt](Av, sa), q[b_fmt](Bv, sb)
    C = Guarded((M, N))
    binding.tpmlp_gemm_fp8(enc[a_fmt](qa), a_fmt, enc[b_fmt](qb), b_fmt, f32dev([sa]), f32dev([sb]), C.t)
    torch.cuda.synchronize()
    ref = qa @ qb.T / (float(np.float32(sa)) * float(np.float32(sb)))
    assert_bf16_close("C", f64(C.t), ref)
    assert C.intact()


@pytest.mark.parametrize("T,d,F,N", [(512, 256, 1024, 4), (320, 512, 1056, 4), (64, 1024, 2048, 2)])
def test_gemm_dh_geluprime_e5m2(T, d, F, N):
    w = inputs.small_workload(T, d, N, F=F, backward=True, name=f"dhq_{T}_{d}_{F}")
    dY, B = inputs.draw(w, "dY"), inputs.draw(w, "B")
    Hpre = inputs.draw(w, "Hpre", shape=(T, F), dist=(0.0, 2.0))
    sdy, sb = 57344.0 / np.max(np.abs(dY[1])) / 2, 448.0 / np.max(np.abs(B[1]))
    qdy, qb = oracle.quantize_e5m2(dY[1], sdy), oracle.quantize_e4m3(B[1], sb)
    g = qdy @ qb.T / (float(np.float32(sdy)) * float(np.float32(sb))) * oracle.gelu_prime(Hpre[1])
    sg = 57344.0 / np.max(np.abs(g)) / 2
    dHq = Guarded((T, F), torch.uint8)
    db = Guarded((F,))
    amax = torch.zeros(1, device="cuda")
    binding.tpmlp_gemm_dh_geluprime_e5m2(e5m2_bytes(qdy), e4m3_bytes(qb), dev(Hpre[0]), N, f32dev([sdy]),
                                         f32dev([sb]), f32dev([sg]), dHq.t, amax, dbias=db.t)
    torch.cuda.synchronize()
    _code_step_agreement(e5m2_values(dHq.t), oracle.quantize_e5m2(g, sg), mant_bits=2, min_quantum=2.0 ** -16)
    assert_bf16_close("db", f64(db.t), g.sum(axis=0))
    assert abs(float(amax.item()) / np.max(np.abs(g)) - 1) < 1e-5
    assert dHq.intact() and db.intact()


@pytest.mark.parametrize("T,d,F,N", [(512, 256, 1024, 4), (256, 1024, 4096, 8), (64, 512, 1056, 2)])
def test_sp_forward_backward_fp8_block(T, d, F, N):
    """FP8 forward with saved Hpre / Xq / Hq, FP8 backward with E5M2 gradients, then both updates."""
    w = inputs.small_workload(T, d, N, F=F, sp=True, backward=True, bias=(0.0, 0.2), name=f"spqb_{T}_{d}_{F}")
    X, A, B, b, g, be, dY = (inputs.draw(w, n) for n in ("X", "A", "B", "bias", "gamma", "beta", "dY"))
    Xo, dYo = _chunks(X[1], N), _chunks(dY[1], N)
    first = oracle.sp_forward_fp8(Xo, g[1], be[1], 1e-5, A[1], B[1], b[1], N, (1.0, 1.0, 1.0, 1.0))["amax"]
    s3 = [float(np.float32(448.0 / first[k])) for k in ("X", "A", "B")]
    am = oracle.sp_forward_fp8(Xo, g[1], be[1], 1e-5, A[1], B[1], b[1], N, (*s3, 1.0))["amax"]
    scales = (*s3, float(np.float32(448.0 / am["H"])))
    gam = oracle.sp_backward_fp8(Xo, g[1], be[1], 1e-5, A[1], B[1], b[1], dYo, N, scales, (1.0, 1.0))["amax"]
    gscales = (float(np.float32(57344.0 / gam["dY"] / 2)), float(np.float32(57344.0 / gam["dHpre"] / 2)))
    ref = oracle.sp_backward_fp8(Xo, g[1], be[1], 1e-5, A[1], B[1], b[1], dYo, N, scales, gscales)

    L = 4
    fwd = binding.fp8_state(f32dev(scales), torch.zeros(4, device="cuda"), torch.ones(4, L, device="cuda"))
    grad_scale, grad_amax = f32dev(gscales), torch.zeros(2, device="cuda")
    grad_hist = torch.ones(2, L, device="cuda")
    grad = binding.fp8_state(grad_scale, grad_amax, grad_hist)
    rows = T // N
    Xc = list(dev(X[0]).split(rows))
    Ad, Bd, gd = dev(A[0]), dev(B[0]), dev(g[0])
    Y = [torch.empty(rows, d, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    Hpre = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
    Xq = torch.empty(T, d, dtype=torch.uint8, device="cuda")
    Hq = torch.empty(T, F, dtype=torch.uint8, device="cuda")
    binding.tpmlp_sp_forward_fp8(Xc, gd, dev(be[0]), Ad, Bd, N, Y, fwd, bias=dev(b[0]), Hpre_out=Hpre, Xq_out=Xq,
                                 Hq_out=Hq)
    dX = [Guarded((rows, d)) for _ in range(N)]
    dA, dB, db = Guarded((d, F)), Guarded((F, d)), Guarded((F,))
    dga, dbe = Guarded((d,), torch.float32), Guarded((d,), torch.float32)
    dHq = Guarded((T, F), torch.uint8)
    binding.tpmlp_sp_backward_fp8(Xc, gd, Ad, Bd, Hpre, Xq, Hq, list(dev(dY[0]).split(rows)), N, fwd, grad,
                                  [x.t for x in dX], dA.t, dB.t, dga.t, dbe.t, dbias=db.t, dHq_out=dHq.t)
    torch.cuda.synchronize()
    # (1) the E5M2 dHpre codes the block formed, against the oracle's from the same saved forward (Xq, Hq
    # and the bf16 Hpre): equal up to one-step flips where a value lies within rounding of a midpoint
    fwd_saved = {"qX": e4m3_values(Xq), "qH": e4m3_values(Hq), "Hpre": f64(Hpre)}
    mid = oracle.sp_backward_fp8(Xo, g[1], be[1], 1e-5, A[1], B[1], b[1], dYo, N, scales, gscales, saved=fwd_saved)
    _code_step_agreement(e5m2_values(dHq.t), mid["qdHpre"], mant_bits=2, min_quantum=2.0 ** -16)
    # (2) the rest of the chain from the codes this GPU run saved (the forward's and the block's E5M2
    # dHpre): every gradient at the bf16 band, so a wrong tile or operand of any backward GEMM shows
    saved = dict(fwd_saved, qdHpre=e5m2_values(dHq.t))
    same = oracle.sp_backward_fp8(Xo, g[1], be[1], 1e-5, A[1], B[1], b[1], dYo, N, scales, gscales, saved=saved)
    assert_bf16_close("dX (fp8, saved codes)", np.concatenate([f64(x.t) for x in dX]),
                      np.concatenate(same["dX_chunks"]))
    for name, t, r in (("dA", dA, same["dA"]), ("dB", dB, same["dB"]), ("db", db, same["db"]),
                       ("dgamma", dga, same["dgamma"]), ("dbeta", dbe, same["dbeta"])):
        assert_bf16_close(name + " (fp8, saved codes)", f64(t.t), r)
    # (3) against the oracle's own codes: the one-step flips of (1) move the GEMM results by about 1%
    assert_fp8_close("dX", np.concatenate([f64(x.t) for x in dX]), np.concatenate(ref["dX_chunks"]))
    for name, t, r in (("dA", dA, ref["dA"]), ("dB", dB, ref["dB"]), ("db", db, ref["db"]),
                       ("dgamma", dga, ref["dgamma"]), ("dbeta", dbe, ref["dbeta"])):
        assert_fp8_close(name, f64(t.t), r)
    # against the unquantised backward the error is the formats' size
    exact = oracle.sp_backward(Xo, g[1], be[1], 1e-5, A[1], B[1], b[1], dYo, N)
    for name, got in (("dA", f64(dA.t)), ("dB", f64(dB.t))):
        err = np.linalg.norm(got - exact[name]) / np.linalg.norm(exact[name])
        assert err < 0.2, (name, err)
    # the gradient state was updated (E5M2 maximum 57344), this step's amaxes reset
    for i, k in enumerate(("dY", "dHpre")):
        h = grad_hist[i].cpu().double().numpy()
        assert abs(h[-1] / ref["amax"][k] - 1) < 1e-3, k
        expect = oracle.fp8_scale(oracle.roll_amax_history(np.ones(L), ref["amax"][k]), fp8_max=57344.0)
        assert abs(float(grad_scale[i].item()) / expect - 1) < 1e-3, k
    assert float(grad_amax.abs().sum().item()) == 0.0
    assert all(t.intact() for t in dX + [dA, dB, db, dga, dbe, dHq])
