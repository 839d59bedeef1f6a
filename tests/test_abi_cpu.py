"""The C-ABI library without a GPU: it builds, loads, exports every function
``include/tpmlp.h`` declares, and its host-side validation and workspace
arithmetic behave as documented.  No call here reaches the CUDA runtime: each
one is rejected by argument checks or is pure host arithmetic."""
import ctypes
import os
import re

import pytest

from tensor_transformer_mlp_tp_gb300 import binding, build, inputs

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "tpmlp.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"TPMLP_API\s+[\w\s\*]+?\b(tpmlp_\w+)\s*\(", text)


def test_header_declares_the_block_calls():
    names = declared_functions()
    for required in ("tpmlp_forward", "tpmlp_sp_forward", "tpmlp_backward", "tpmlp_sp_backward",
                     "tpmlp_workspace_size", "tpmlp_get_device_status", "tpmlp_status_string"):
        assert required in names
    assert len(names) == len(set(names))


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in binding._SIGS, f"binding lacks {name}"


def test_only_abi_symbols_exported(lib):
    # the statically linked CUDA runtime stays private to the library
    with pytest.raises(AttributeError):
        getattr(lib, "cudaLaunchKernel")


def test_status_strings(lib):
    assert binding.status_string(binding.OK) == "ok"
    assert binding.status_string(binding.ERR_TIMEOUT) == "device wait timed out"
    assert binding.status_string(99) == "unknown status"


def _ws(shape, op):
    n = ctypes.c_size_t(0)
    st = binding.lib().tpmlp_workspace_size(ctypes.byref(shape), op, ctypes.byref(n))
    return st, n.value


def _r256(x):
    return (x + 255) // 256 * 256


def test_workspace_sizes(lib):
    for w in inputs.WORKLOADS.values():
        if w.dtype != "bf16":
            continue
        s = binding.make_shape(w.T, w.d, w.F, w.N)
        st, fwd = _ws(s, binding.OP_FWD)
        assert st == binding.OK and fwd == _r256(w.T * w.F * 2)          # H, bf16
        st, spf = _ws(s, binding.OP_SP_FWD)
        assert st == binding.OK and spf == fwd + _r256(w.T * w.d * 2)    # + gathered LayerNorm output
        st, spp = _ws(s, binding.OP_SP_FWD_PARTIALS)
        assert st == binding.OK and spp == spf + _r256(w.N * w.T * w.d * 2)
        st, bwd = _ws(s, binding.OP_BWD)
        assert st == binding.OK and bwd >= 3 * w.T * w.F * 2
        st, spb = _ws(s, binding.OP_SP_BWD)
        assert st == binding.OK and spb > bwd
    s = binding.make_shape(128, 64, 256, 2, binding.FP32)
    assert _ws(s, binding.OP_FWD) == (binding.OK, 128 * 256 * 4)
    assert _ws(s, binding.OP_SP_FWD)[0] == binding.ERR_UNSUPPORTED
    assert _ws(binding.make_shape(0, 64, 256, 2), binding.OP_FWD) == (binding.OK, 0)


@pytest.mark.parametrize("bad", [
    dict(tokens=-1), dict(d=0), dict(ffn=0), dict(n_shards=0), dict(n_shards=65), dict(ffn=100, n_shards=3),
    dict(d=60), dict(ffn=100, n_shards=5), dict(dtype=7)])
def test_invalid_shapes(lib, bad):
    kw = dict(tokens=256, d=64, ffn=256, n_shards=2, dtype=binding.BF16)
    kw.update(bad)
    s = binding.make_shape(kw["tokens"], kw["d"], kw["ffn"], kw["n_shards"], kw["dtype"])
    assert _ws(s, binding.OP_FWD)[0] == binding.ERR_INVALID_ARG


def test_largest_shard_count_accepted(lib):
    """N = 64 (the most shards a call takes) with 8-column shards: every operation sizes its workspace."""
    s = binding.make_shape(1024, 128, 512, 64)
    for op in (binding.OP_FWD, binding.OP_SP_FWD, binding.OP_BWD, binding.OP_SP_BWD):
        assert _ws(s, op)[0] == binding.OK


def test_sp_requires_divisible_tokens(lib):
    s = binding.make_shape(100, 64, 256, 8)
    assert _ws(s, binding.OP_SP_FWD)[0] == binding.ERR_INVALID_ARG
    assert _ws(s, binding.OP_FWD)[0] == binding.OK


def test_null_and_misaligned_pointers_rejected(lib):
    L = binding.lib()
    s = binding.make_shape(256, 64, 256, 2)
    good = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 2)
    ws = ctypes.c_void_p(1 << 24)
    args = lambda X, A, B, Y: (X, A, B, None, ctypes.byref(s), Y, None, None, ws, 1 << 30, None)
    assert L.tpmlp_forward(*args(None, good, good, good)) == binding.ERR_INVALID_ARG
    assert L.tpmlp_forward(*args(good, good, good, None)) == binding.ERR_INVALID_ARG
    assert L.tpmlp_forward(*args(odd, good, good, good)) == binding.ERR_INVALID_ARG
    assert L.tpmlp_forward(good, good, good, None, ctypes.byref(s), good, None, None, ws, 16, None) == binding.ERR_WORKSPACE
    assert L.tpmlp_gemm2_partials(good, good, ctypes.byref(binding.make_shape(256, 64, 96, 2)), good, None) \
        == binding.ERR_UNSUPPORTED                                      # (ffn / N) % 64 != 0
    assert L.tpmlp_selftest_wait_timeout(0, None) == binding.ERR_INVALID_ARG


def test_empty_batch_needs_no_device(lib):
    L = binding.lib()
    s = binding.make_shape(0, 64, 256, 2)
    good = ctypes.c_void_p(1 << 20)
    assert L.tpmlp_forward(good, good, good, None, ctypes.byref(s), good, None, None, None, 0, None) == binding.OK


def test_sp_region_workspace_sizes(lib):
    for w in inputs.WORKLOADS.values():
        if w.dtype != "bf16" or not w.sp:
            continue
        s = binding.make_shape(w.T, w.d, w.F, w.N)
        dropcol = _r256(-(-w.T // 128) * w.d * 4)      # fp32 column partials, one row per 128 token rows
        assert _ws(s, binding.OP_DROPOUT_BWD) == (binding.OK, dropcol)
        st, spb = _ws(s, binding.OP_SP_BWD)
        assert _ws(s, binding.OP_SP_BLOCK_BWD) == (binding.OK, spb + dropcol)
    assert _ws(binding.make_shape(256, 64, 256, 2), 11)[0] == binding.ERR_INVALID_ARG


@pytest.mark.parametrize("p", [1.0, -0.25, float("nan"), float("inf")])
def test_dropout_probability_outside_zero_one_rejected(lib, p):
    L = binding.lib()
    s = binding.make_shape(256, 64, 256, 2)
    good = ctypes.c_void_p(1 << 20)
    chunks = (ctypes.c_void_p * 2)(1 << 20, 1 << 21)
    cp = ctypes.cast(chunks, binding._PP)
    drop = ctypes.byref(binding.Dropout(p, 1, 2))
    assert L.tpmlp_dropout_backward(cp, drop, ctypes.byref(s), good, None, None, 0, None) == binding.ERR_INVALID_ARG
    assert L.tpmlp_gemm2_bias_dropout_add(good, good, None, drop, None, ctypes.byref(s), cp, None) \
        == binding.ERR_INVALID_ARG
    assert L.tpmlp_reduce_scatter_bias_dropout_add(good, None, drop, None, ctypes.byref(s), cp, None) \
        == binding.ERR_INVALID_ARG


def test_sp_region_argument_checks(lib):
    L = binding.lib()
    s = binding.make_shape(256, 64, 256, 2)
    good = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 4)
    chunks = (ctypes.c_void_p * 2)(1 << 20, 1 << 21)
    cp = ctypes.cast(chunks, binding._PP)
    bad_chunks = ctypes.cast((ctypes.c_void_p * 2)(1 << 20, None), binding._PP)
    drop = ctypes.byref(binding.Dropout(0.1, 1, 2))
    # misaligned row bias, a missing residual chunk
    assert L.tpmlp_gemm2_bias_dropout_add(good, good, odd, drop, None, ctypes.byref(s), cp, None) \
        == binding.ERR_INVALID_ARG
    assert L.tpmlp_reduce_scatter_bias_dropout_add(good, None, drop, bad_chunks, ctypes.byref(s), cp, None) \
        == binding.ERR_INVALID_ARG
    # dbias2 wanted without a workspace
    assert L.tpmlp_dropout_backward(cp, drop, ctypes.byref(s), good, good, None, 0, None) == binding.ERR_WORKSPACE
    # the residual-gradient LayerNorm backward needs its residual chunks
    assert L.tpmlp_layernorm_backward_add(cp, good, 1e-5, good, None, ctypes.byref(s), cp, good, good, good, 1 << 30,
                                          None) == binding.ERR_INVALID_ARG
    # empty batch: nothing launched, NULL pointers accepted
    e = binding.make_shape(0, 64, 256, 2)
    assert L.tpmlp_sp_block_forward(None, None, None, 1e-5, None, None, None, None, drop, ctypes.byref(e), None, 0,
                                    None, None, None, None, 0, None) == binding.OK
    assert L.tpmlp_sp_block_backward(None, None, None, 1e-5, None, None, None, drop, None, None, None, None,
                                     ctypes.byref(e), None, None, None, None, None, None, None, None, 0, None) \
        == binding.OK


def test_fp8_workspace_and_argument_checks(lib):
    for w in inputs.WORKLOADS.values():
        if w.dtype != "bf16" or not w.sp:
            continue
        s = binding.make_shape(w.T, w.d, w.F, w.N)
        assert _ws(s, binding.OP_SP_FWD_FP8) == (binding.OK, 2 * _r256(w.d * w.F) + _r256(w.T * w.d) +
                                                  _r256(w.T * w.F))
    assert _ws(binding.make_shape(256, 72, 288, 2), binding.OP_SP_FWD_FP8)[0] == binding.ERR_INVALID_ARG  # d % 16
    L = binding.lib()
    good = ctypes.c_void_p(1 << 20)
    # rows or columns not multiples of 16, a missing scale or amax
    assert L.tpmlp_cast_e4m3(good, 24, 64, 0, good, good, good, None) == binding.ERR_INVALID_ARG
    assert L.tpmlp_cast_e4m3(good, 32, 64, 1, None, good, good, None) == binding.ERR_INVALID_ARG
    assert L.tpmlp_cast_e4m3(good, 32, 64, 1, good, good, None, None) == binding.ERR_INVALID_ARG
    assert L.tpmlp_cast_e4m3(None, 0, 64, 0, None, None, None, None) == binding.OK
    st = binding.Fp8State(1 << 20, 1 << 21, 1 << 22, 0, 0)          # history length 0
    assert L.tpmlp_fp8_update_scales(ctypes.byref(st), None) == binding.ERR_INVALID_ARG
    s = binding.make_shape(256, 96, 384, 2)                          # LayerNorm width without an E4M3 kernel
    chunks = ctypes.cast((ctypes.c_void_p * 2)(1 << 20, 1 << 21), binding._PP)
    assert L.tpmlp_layernorm_gather_e4m3(chunks, good, good, 1e-5, ctypes.byref(s), good, good, good, None) \
        == binding.ERR_UNSUPPORTED


def test_fp8_backward_workspace_and_argument_checks(lib):
    w = inputs.WORKLOADS["sp_block_fwd_bwd"]
    s = binding.make_shape(w.T, w.d, w.F, w.N)
    st, n = _ws(s, binding.OP_SP_BWD_FP8)
    td, td8, tf8, df8 = _r256(w.T * w.d * 2), _r256(w.T * w.d), _r256(w.T * w.F), _r256(w.d * w.F)
    assert st == binding.OK and n > 2 * td + 3 * td8 + 2 * df8 + 3 * tf8
    assert _ws(binding.make_shape(200, 64, 256, 2), binding.OP_SP_BWD_FP8)[0] == binding.ERR_INVALID_ARG  # T % 16
    L = binding.lib()
    good = ctypes.c_void_p(1 << 20)
    # formats other than E4M3 / E5M2, K not a multiple of 16, ldc < N
    assert L.tpmlp_gemm_fp8(good, 2, good, 0, 256, 256, 256, good, good, good, 256, None) == binding.ERR_INVALID_ARG
    assert L.tpmlp_gemm_fp8(good, 0, good, 1, 256, 256, 200, good, good, good, 256, None) == binding.ERR_INVALID_ARG
    assert L.tpmlp_gemm_fp8(good, 0, good, 1, 256, 256, 256, good, good, good, 128, None) == binding.ERR_INVALID_ARG
    assert L.tpmlp_gemm_fp8(None, 0, None, 1, 0, 256, 256, None, None, None, 256, None) == binding.OK
    assert L.tpmlp_transpose_bytes(good, 24, 64, good, None) == binding.ERR_INVALID_ARG


def test_attention_workspace_and_argument_checks(lib):
    L = binding.lib()
    n = ctypes.c_size_t(0)
    assert L.tpmlp_attention_workspace_size(4096, 2, 32, 128, ctypes.byref(n)) == binding.OK
    T, d = 4096 * 2, 32 * 128
    assert n.value == _r256(T * 3 * d * 2) + _r256(T * d * 2)
    assert L.tpmlp_attention_workspace_size(4096, 2, 32, 64, ctypes.byref(n)) == binding.ERR_UNSUPPORTED
    assert L.tpmlp_attention_workspace_size(-1, 2, 32, 128, ctypes.byref(n)) == binding.ERR_INVALID_ARG
    good = ctypes.c_void_p(1 << 20)
    # heads not divisible by the shards; a causal flag other than 0 / 1; misaligned pointers
    assert L.tpmlp_attention_tp_forward(good, good, None, good, None, 256, 1, 6, 4, 0, good, None, None, None, good,
                                        1 << 30, None) == binding.ERR_INVALID_ARG
    assert L.tpmlp_attention_core(good, 256, 1, 4, 128, 2, good, None, None) == binding.ERR_INVALID_ARG
    assert L.tpmlp_attention_core(ctypes.c_void_p((1 << 20) + 2), 256, 1, 4, 128, 0, good, None, None) \
        == binding.ERR_INVALID_ARG
    assert L.tpmlp_attention_core(good, 256, 1, 4, 128, 0, good, ctypes.c_void_p((1 << 20) + 4), None) \
        == binding.ERR_INVALID_ARG                                                         # misaligned LSE
    assert L.tpmlp_attention_core(None, 0, 1, 4, 128, 1, None, None, None) == binding.OK  # empty sequence


def test_attention_backward_workspace_and_argument_checks(lib):
    L = binding.lib()
    n = ctypes.c_size_t(0)
    S, B, H = 1000, 2, 4  # S_pad = 1024
    assert L.tpmlp_attention_backward_workspace_size(S, B, H, 128, ctypes.byref(n)) == binding.OK
    T, d = S * B, H * 128
    rows_per_block = 128  # 8 warps x 16 rows
    partial = (T + rows_per_block - 1) // rows_per_block * 3 * d * 4
    assert n.value == _r256(B * H * 1024 * 4) + _r256(T * d * 2) + _r256(T * 3 * d * 2) + _r256(partial)
    assert binding.attention_lse_shape(S, B, H) == (B * H, 1024)
    assert L.tpmlp_attention_backward_workspace_size(S, B, H, 96, ctypes.byref(n)) == binding.ERR_UNSUPPORTED
    good = ctypes.c_void_p(1 << 20)
    # the core backward: LSE required, a workspace of at least the D statistics
    assert L.tpmlp_attention_core_backward(good, good, good, None, S, B, H, 128, 0, good, good, 1 << 30, None) \
        == binding.ERR_INVALID_ARG
    assert L.tpmlp_attention_core_backward(good, good, good, good, S, B, H, 128, 0, good, good, 1024, None) \
        == binding.ERR_WORKSPACE
    assert L.tpmlp_attention_core_backward(good, good, good, good, S, B, H, 128, 3, good, good, 1 << 30, None) \
        == binding.ERR_INVALID_ARG
    assert L.tpmlp_attention_core_backward(None, None, None, None, 0, B, H, 128, 0, None, None, 0, None) == binding.OK
    # the block backward: shards must divide the heads; saved tensors required; workspace too small
    args = [good] * 7 + [S, B, H, 4, 0] + [good, good, None, good, None, None, good, 1 << 30, None]
    bad = list(args)
    bad[10] = 3
    assert L.tpmlp_attention_tp_backward(*bad) == binding.ERR_INVALID_ARG
    bad = list(args)
    bad[5] = None  # LSE
    assert L.tpmlp_attention_tp_backward(*bad) == binding.ERR_INVALID_ARG
    bad = list(args)
    bad[19] = 4096
    assert L.tpmlp_attention_tp_backward(*bad) == binding.ERR_WORKSPACE


def test_dropout_struct_layout():
    """tpmlp_dropout as the header lays it out: float p, then two 64-bit words and the mask pointer."""
    D = binding.Dropout
    assert ctypes.sizeof(D) == 32
    assert (D.p.offset, D.seed.offset, D.offset.offset, D.keep_mask.offset) == (0, 8, 16, 24)
    assert binding.keep_mask_bytes(3, 8) == 3 and binding.keep_mask_bytes(1, 12) == 2
