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


def _code_step_agreement(got, ref, min_equal=0.999):
    """Codes equal on all but a tiny fraction; the rest one E4M3 step apart (neighbouring values)."""
    eq = got == ref
    assert eq.mean() >= min_equal, eq.mean()
    if not eq.all():
        g, r = got[~eq], ref[~eq]
        hi = np.maximum(np.abs(g), np.abs(r))
        # one step of E4M3 is at most 2**-3 of the larger magnitude (2**-9 for subnormals)
        assert np.all(np.abs(g - r) <= np.maximum(hi * 2.0 ** -3, 2.0 ** -9) + 1e-30)
        assert np.all(np.sign(g) * np.sign(r) >= 0)


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
