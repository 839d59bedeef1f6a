"""Python binding of ``libtpmlp.so`` (the C ABI in ``include/tpmlp.h``).

Argument marshalling only: every function here checks nothing the library
does not check itself, computes nothing, and calls exactly one ABI entry
point with the same name.  Tensors are torch tensors on the current CUDA
device; shapes are read from them.  PyTorch is used only for device memory
(the workspace) and streams.  If the library is missing the first call
raises; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

# The in-tree library; TPMLP_LIBRARY may name another build of it (the tests load the bounds-checked debug
# build, libtpmlp_debug.so beside this file, that way in a process of their own).
_LIB_PATH = os.environ.get("TPMLP_LIBRARY") or os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtpmlp.so")
_lib = None

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE = range(6)
BF16, FP32 = 0, 1
(OP_FWD, OP_SP_FWD, OP_SP_FWD_PARTIALS, OP_BWD, OP_SP_BWD, OP_DH_GELUPRIME, OP_LN_BWD, OP_SP_BLOCK_BWD,
 OP_DROPOUT_BWD, OP_SP_FWD_FP8, OP_SP_BWD_FP8) = range(11)
E4M3, E5M2 = 0, 1
RS_FUSED, RS_PARTIALS = 0, 1


class TpMlpError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


class Shape(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_int64), ("d", ctypes.c_int64), ("ffn", ctypes.c_int64),
                ("n_shards", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class Dropout(ctypes.Structure):
    _fields_ = [("p", ctypes.c_float), ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint64),
                ("keep_mask", ctypes.c_void_p)]


class Fp8State(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_void_p), ("amax", ctypes.c_void_p), ("history", ctypes.c_void_p),
                ("history_len", ctypes.c_int32), ("margin", ctypes.c_int32)]


_P = ctypes.c_void_p
_PP = ctypes.POINTER(ctypes.c_void_p)
_SP = ctypes.POINTER(Shape)
_DP = ctypes.POINTER(Dropout)
_FP = ctypes.POINTER(Fp8State)
_SIGS = {
    "tpmlp_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "tpmlp_workspace_size": ([_SP, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "tpmlp_get_device_status": ([_P, ctypes.POINTER(ctypes.c_uint32)], ctypes.c_int),
    "tpmlp_forward": ([_P, _P, _P, _P, _SP, _P, _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "tpmlp_sp_forward": ([_PP, _P, _P, ctypes.c_float, _P, _P, _P, _SP, _PP, ctypes.c_int, _P, _P, _P, _P,
                          ctypes.c_size_t, _P], ctypes.c_int),
    "tpmlp_backward": ([_P, _P, _P, _P, _P, _P, _P, _SP, _P, _P, _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "tpmlp_sp_backward": ([_PP, _P, _P, ctypes.c_float, _P, _P, _P, _P, _P, _P, _PP, _SP, _PP, _P, _P, _P, _P, _P,
                           _P, ctypes.c_size_t, _P], ctypes.c_int),
    "tpmlp_gemm1_bias_gelu": ([_P, _P, _P, _SP, _P, _P, _P], ctypes.c_int),
    "tpmlp_gemm2_shard_accum": ([_P, _P, _SP, _P, _PP, _P], ctypes.c_int),
    "tpmlp_gemm2_partials": ([_P, _P, _SP, _P, _P], ctypes.c_int),
    "tpmlp_reduce_scatter": ([_P, _SP, _PP, _P], ctypes.c_int),
    "tpmlp_layernorm_gather": ([_PP, _P, _P, ctypes.c_float, _SP, _P, _P], ctypes.c_int),
    "tpmlp_rmsnorm_gather": ([_PP, _P, ctypes.c_float, _SP, _P, _P], ctypes.c_int),
    "tpmlp_gemm_dh_geluprime": ([_P, _P, _P, _SP, _P, _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "tpmlp_gemm_wgrad_b": ([_P, _P, _SP, _P, _P], ctypes.c_int),
    "tpmlp_gemm_wgrad_a": ([_P, _P, _SP, _P, _P], ctypes.c_int),
    "tpmlp_gemm_dx_shard_accum": ([_P, _P, _SP, _P, _P], ctypes.c_int),
    "tpmlp_layernorm_backward": ([_PP, _P, ctypes.c_float, _P, _SP, _PP, _P, _P, _P, ctypes.c_size_t, _P],
                                 ctypes.c_int),
    "tpmlp_layernorm_backward_noalloc": ([_PP, _P, ctypes.c_float, _P, _SP, _PP, _P, _P, _P], ctypes.c_int),
    "tpmlp_debug_bounds_status": ([ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_uint32),
                                   ctypes.POINTER(ctypes.c_uint32)], ctypes.c_int),
    "tpmlp_layernorm_backward_blocks": ([_PP, _P, ctypes.c_float, _P, _SP, _PP, _P, _P, ctypes.c_int32, _P,
                                         ctypes.c_size_t, _P], ctypes.c_int),
    "tpmlp_selftest_wait_timeout": ([ctypes.c_uint32, _P], ctypes.c_int),
    "tpmlp_sp_block_forward": ([_PP, _P, _P, ctypes.c_float, _P, _P, _P, _P, _DP, _SP, _PP, ctypes.c_int, _P, _P, _P,
                                _P, ctypes.c_size_t, _P], ctypes.c_int),
    "tpmlp_sp_block_backward": ([_PP, _P, _P, ctypes.c_float, _P, _P, _P, _DP, _P, _P, _P, _PP, _SP, _PP, _P, _P, _P,
                                 _P, _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "tpmlp_gemm2_bias_dropout_add": ([_P, _P, _P, _DP, _PP, _SP, _PP, _P], ctypes.c_int),
    "tpmlp_reduce_scatter_bias_dropout_add": ([_P, _P, _DP, _PP, _SP, _PP, _P], ctypes.c_int),
    "tpmlp_dropout_backward": ([_PP, _DP, _SP, _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "tpmlp_layernorm_backward_add": ([_PP, _P, ctypes.c_float, _P, _PP, _SP, _PP, _P, _P, _P, ctypes.c_size_t, _P],
                                     ctypes.c_int),
    "tpmlp_cast_e4m3": ([_P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, _P, _P, _P, _P], ctypes.c_int),
    "tpmlp_layernorm_gather_e4m3": ([_PP, _P, _P, ctypes.c_float, _SP, _P, _P, _P, _P], ctypes.c_int),
    "tpmlp_gemm1_e4m3": ([_P, _P, _P, _SP, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "tpmlp_gemm2_e4m3": ([_P, _P, _SP, _P, _P, _P, _PP, _P], ctypes.c_int),
    "tpmlp_fp8_update_scales": ([_FP, _P], ctypes.c_int),
    "tpmlp_sp_forward_fp8": ([_PP, _P, _P, ctypes.c_float, _P, _P, _P, _FP, _SP, _PP, _P, _P, _P, _P,
                              ctypes.c_size_t, _P], ctypes.c_int),
    "tpmlp_cast_e5m2": ([_P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, _P, _P, _P, _P], ctypes.c_int),
    "tpmlp_transpose_bytes": ([_P, ctypes.c_int64, ctypes.c_int64, _P, _P], ctypes.c_int),
    "tpmlp_gemm_dh_geluprime_e5m2": ([_P, _P, _P, _SP, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
                                     ctypes.c_int),
    "tpmlp_gemm_fp8": ([_P, ctypes.c_int, _P, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _P, _P,
                        _P, ctypes.c_int64, _P], ctypes.c_int),
    "tpmlp_attention_workspace_size": ([ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "tpmlp_attention_core": ([_P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, _P, _P,
                              _P], ctypes.c_int),
    "tpmlp_attention_backward_workspace_size": ([ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                                 ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "tpmlp_attention_core_backward": ([_P, _P, _P, _P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_int, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "tpmlp_attention_tp_forward": ([_P, _P, _P, _P, _P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                    ctypes.c_int, _P, _P, _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "tpmlp_attention_tp_backward": ([_P, _P, _P, _P, _P, _P, _P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_int32, ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
                                    ctypes.c_int),
    "tpmlp_sp_backward_fp8": ([_PP, _P, ctypes.c_float, _P, _P, _P, _P, _P, _PP, _FP, _FP, _SP, _PP, _P, _P, _P, _P,
                               _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
}


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with tensor_transformer_mlp_tp_gb300.build "
                               "(the CUDA path has no fallback)")
        l = ctypes.CDLL(_LIB_PATH)
        for name, (args, res) in _SIGS.items():
            f = getattr(l, name)
            f.argtypes = args
            f.restype = res
        _lib = l
    return _lib


def lib_path() -> str:
    return _LIB_PATH


def status_string(status: int) -> str:
    return lib().tpmlp_status_string(status).decode()


def _check(fn: str, status: int):
    if status != OK:
        raise TpMlpError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _ptrs(ts):
    arr = (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])
    return ctypes.cast(arr, _PP), arr


def _dropout(p, seed, offset, keep_mask=None):
    if p is None:
        return None
    return ctypes.byref(Dropout(p, seed, offset, None if keep_mask is None else keep_mask.data_ptr()))


def keep_mask_bytes(T, d):
    """Bytes of a dropout keep mask for a gathered [T x d] output: one bit per element."""
    return (T * d + 7) // 8


def _opt_ptrs(ts):
    return (None, None) if ts is None else _ptrs(ts)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def make_shape(tokens: int, d: int, ffn: int, n_shards: int, dtype: int = BF16) -> Shape:
    return Shape(tokens, d, ffn, n_shards, dtype)


def _dtype_code(t) -> int:
    return FP32 if t.dtype == torch.float32 else BF16


def tpmlp_workspace_size(shape: Shape, op: int) -> int:
    n = ctypes.c_size_t(0)
    _check("tpmlp_workspace_size", lib().tpmlp_workspace_size(ctypes.byref(shape), op, ctypes.byref(n)))
    return n.value


def workspace(shape: Shape, op: int, device=None) -> torch.Tensor:
    """A device buffer large enough for `op` (torch allocation; contents undefined)."""
    return torch.empty(max(tpmlp_workspace_size(shape, op), 256), dtype=torch.uint8, device=device or "cuda")


def tpmlp_debug_bounds_status():
    """(checked, violations, first_site): whether the loaded library checks global indices, and what it found since
    the previous call (cleared)."""
    c, n, site = ctypes.c_int32(0), ctypes.c_uint32(0), ctypes.c_uint32(0)
    _check("tpmlp_debug_bounds_status", lib().tpmlp_debug_bounds_status(ctypes.byref(c), ctypes.byref(n),
                                                                        ctypes.byref(site)))
    return bool(c.value), n.value, site.value


def tpmlp_get_device_status(stream=None):
    site = ctypes.c_uint32(0)
    st = lib().tpmlp_get_device_status(_stream(stream), ctypes.byref(site))
    return st, site.value


# ----------------------------------------------------------------------------- block calls

def tpmlp_forward(X, A, B, bias, N, Y, Hpre_out=None, H_out=None, ws=None, stream=None):
    T, d = X.shape
    shape = make_shape(T, d, A.shape[1], N, _dtype_code(X))
    ws = workspace(shape, OP_FWD, X.device) if ws is None else ws
    _check("tpmlp_forward", lib().tpmlp_forward(_ptr(X), _ptr(A), _ptr(B), _ptr(bias), ctypes.byref(shape), _ptr(Y),
                                                _ptr(Hpre_out), _ptr(H_out), _ptr(ws), ws.numel(), _stream(stream)))
    return Y


def tpmlp_sp_forward(X_chunks, gamma, beta, A, B, N, Y_chunks, bias=None, eps=1e-5, rs_mode=RS_FUSED,
                     Hpre_out=None, H_out=None, Xg_out=None, ws=None, stream=None):
    rows, d = X_chunks[0].shape
    shape = make_shape(rows * N, d, A.shape[1], N)
    op = OP_SP_FWD if rs_mode == RS_FUSED else OP_SP_FWD_PARTIALS
    ws = workspace(shape, op, A.device) if ws is None else ws
    xp, _xa = _ptrs(X_chunks)
    yp, _ya = _ptrs(Y_chunks)
    _check("tpmlp_sp_forward", lib().tpmlp_sp_forward(xp, _ptr(gamma), _ptr(beta), eps, _ptr(A), _ptr(B), _ptr(bias),
                                                      ctypes.byref(shape), yp, rs_mode, _ptr(Hpre_out), _ptr(H_out),
                                                      _ptr(Xg_out), _ptr(ws), ws.numel(), _stream(stream)))
    return Y_chunks


def tpmlp_backward(X, A, B, bias, Hpre, dY, N, dX, dA, dB, dbias=None, H=None, ws=None, stream=None):
    T, d = X.shape
    shape = make_shape(T, d, A.shape[1], N)
    ws = workspace(shape, OP_BWD, X.device) if ws is None else ws
    _check("tpmlp_backward", lib().tpmlp_backward(_ptr(X), _ptr(A), _ptr(B), _ptr(bias), _ptr(Hpre), _ptr(H), _ptr(dY),
                                                  ctypes.byref(shape), _ptr(dX), _ptr(dA), _ptr(dB), _ptr(dbias),
                                                  _ptr(ws), ws.numel(), _stream(stream)))


def tpmlp_sp_backward(X_chunks, gamma, beta, A, B, Hpre, dY_chunks, N, dX_chunks, dA, dB, dgamma, dbeta,
                      bias=None, dbias=None, eps=1e-5, H=None, Xg=None, ws=None, stream=None):
    rows, d = X_chunks[0].shape
    shape = make_shape(rows * N, d, A.shape[1], N)
    ws = workspace(shape, OP_SP_BWD, A.device) if ws is None else ws
    xp, _xa = _ptrs(X_chunks)
    dyp, _dya = _ptrs(dY_chunks)
    dxp, _dxa = _ptrs(dX_chunks)
    _check("tpmlp_sp_backward", lib().tpmlp_sp_backward(
        xp, _ptr(gamma), _ptr(beta), eps, _ptr(A), _ptr(B), _ptr(bias), _ptr(Hpre), _ptr(H), _ptr(Xg), dyp,
        ctypes.byref(shape), dxp,
        _ptr(dA), _ptr(dB), _ptr(dbias), _ptr(dgamma), _ptr(dbeta), _ptr(ws), ws.numel(), _stream(stream)))


def tpmlp_sp_block_forward(X_chunks, gamma, beta, A, B, N, Y_chunks, bias=None, bias2=None, p=None, seed=0, offset=0,
                           eps=1e-5, rs_mode=RS_FUSED, Hpre_out=None, H_out=None, Xg_out=None, ws=None, keep_mask=None, stream=None):
    """Y_j = X_j + dropout(Z_j + bias2); p=None passes a NULL dropout (p = 0)."""
    rows, d = X_chunks[0].shape
    shape = make_shape(rows * N, d, A.shape[1], N)
    op = OP_SP_FWD if rs_mode == RS_FUSED else OP_SP_FWD_PARTIALS
    ws = workspace(shape, op, A.device) if ws is None else ws
    xp, _xa = _ptrs(X_chunks)
    yp, _ya = _ptrs(Y_chunks)
    _check("tpmlp_sp_block_forward", lib().tpmlp_sp_block_forward(
        xp, _ptr(gamma), _ptr(beta), eps, _ptr(A), _ptr(B), _ptr(bias), _ptr(bias2), _dropout(p, seed, offset, keep_mask),
        ctypes.byref(shape), yp, rs_mode, _ptr(Hpre_out), _ptr(H_out), _ptr(Xg_out), _ptr(ws), ws.numel(),
        _stream(stream)))
    return Y_chunks


def tpmlp_sp_block_backward(X_chunks, gamma, beta, A, B, Hpre, dY_chunks, N, dX_chunks, dA, dB, dgamma, dbeta,
                            bias=None, dbias=None, dbias2=None, p=None, seed=0, offset=0, eps=1e-5, H=None, Xg=None,
                            ws=None, keep_mask=None, stream=None):
    rows, d = X_chunks[0].shape
    shape = make_shape(rows * N, d, A.shape[1], N)
    ws = workspace(shape, OP_SP_BLOCK_BWD, A.device) if ws is None else ws
    xp, _xa = _ptrs(X_chunks)
    dyp, _dya = _ptrs(dY_chunks)
    dxp, _dxa = _ptrs(dX_chunks)
    _check("tpmlp_sp_block_backward", lib().tpmlp_sp_block_backward(
        xp, _ptr(gamma), _ptr(beta), eps, _ptr(A), _ptr(B), _ptr(bias), _dropout(p, seed, offset, keep_mask), _ptr(Hpre),
        _ptr(H), _ptr(Xg), dyp, ctypes.byref(shape), dxp, _ptr(dA), _ptr(dB), _ptr(dbias), _ptr(dbias2),
        _ptr(dgamma), _ptr(dbeta), _ptr(ws), ws.numel(), _stream(stream)))


# ----------------------------------------------------------------------------- single steps

def tpmlp_gemm1_bias_gelu(X, A, bias, N, H, Hpre=None, stream=None):
    shape = make_shape(X.shape[0], X.shape[1], A.shape[1], N)
    _check("tpmlp_gemm1_bias_gelu", lib().tpmlp_gemm1_bias_gelu(_ptr(X), _ptr(A), _ptr(bias), ctypes.byref(shape),
                                                                _ptr(H), _ptr(Hpre), _stream(stream)))


def tpmlp_gemm2_shard_accum(H, B, N, Y=None, Y_chunks=None, stream=None):
    shape = make_shape(H.shape[0], B.shape[1], H.shape[1], N)
    if Y_chunks is not None:
        yp, _ya = _ptrs(Y_chunks)
    else:
        yp = None
    _check("tpmlp_gemm2_shard_accum", lib().tpmlp_gemm2_shard_accum(_ptr(H), _ptr(B), ctypes.byref(shape), _ptr(Y),
                                                                    yp, _stream(stream)))


def tpmlp_gemm2_bias_dropout_add(H, B, N, Y_chunks, bias2=None, p=None, seed=0, offset=0, R_chunks=None,
                                 keep_mask=None, stream=None):
    shape = make_shape(H.shape[0], B.shape[1], H.shape[1], N)
    yp, _ya = _ptrs(Y_chunks)
    rp, _ra = _opt_ptrs(R_chunks)
    _check("tpmlp_gemm2_bias_dropout_add", lib().tpmlp_gemm2_bias_dropout_add(
        _ptr(H), _ptr(B), _ptr(bias2), _dropout(p, seed, offset, keep_mask), rp, ctypes.byref(shape), yp, _stream(stream)))


def tpmlp_gemm2_partials(H, B, N, P, stream=None):
    shape = make_shape(H.shape[0], B.shape[1], H.shape[1], N)
    _check("tpmlp_gemm2_partials", lib().tpmlp_gemm2_partials(_ptr(H), _ptr(B), ctypes.byref(shape), _ptr(P),
                                                              _stream(stream)))


def tpmlp_reduce_scatter(P, N, Y_chunks, stream=None):
    _, T, d = P.shape
    shape = make_shape(T, d, 8 * N, N)  # ffn unused by this step
    yp, _ya = _ptrs(Y_chunks)
    _check("tpmlp_reduce_scatter", lib().tpmlp_reduce_scatter(_ptr(P), ctypes.byref(shape), yp, _stream(stream)))


def tpmlp_reduce_scatter_bias_dropout_add(P, N, Y_chunks, bias2=None, p=None, seed=0, offset=0, R_chunks=None,
                                          keep_mask=None, stream=None):
    _, T, d = P.shape
    shape = make_shape(T, d, 8 * N, N)  # ffn unused by this step
    yp, _ya = _ptrs(Y_chunks)
    rp, _ra = _opt_ptrs(R_chunks)
    _check("tpmlp_reduce_scatter_bias_dropout_add", lib().tpmlp_reduce_scatter_bias_dropout_add(
        _ptr(P), _ptr(bias2), _dropout(p, seed, offset, keep_mask), rp, ctypes.byref(shape), yp, _stream(stream)))


def tpmlp_dropout_backward(dY_chunks, N, dZ, dbias2=None, p=None, seed=0, offset=0, ws=None, keep_mask=None, stream=None):
    rows, d = dY_chunks[0].shape
    shape = make_shape(rows * N, d, 8 * N, N)  # ffn unused by this step
    if dbias2 is not None and ws is None:
        ws = workspace(shape, OP_DROPOUT_BWD, dZ.device)
    dyp, _dya = _ptrs(dY_chunks)
    _check("tpmlp_dropout_backward", lib().tpmlp_dropout_backward(
        dyp, _dropout(p, seed, offset, keep_mask), ctypes.byref(shape), _ptr(dZ), _ptr(dbias2), _ptr(ws),
        0 if ws is None else ws.numel(), _stream(stream)))


def tpmlp_layernorm_gather(X_chunks, gamma, beta, N, Xg, eps=1e-5, stream=None):
    rows, d = X_chunks[0].shape
    shape = make_shape(rows * N, d, 8 * N, N)  # ffn unused by this step
    xp, _xa = _ptrs(X_chunks)
    _check("tpmlp_layernorm_gather", lib().tpmlp_layernorm_gather(xp, _ptr(gamma), _ptr(beta), eps,
                                                                  ctypes.byref(shape), _ptr(Xg), _stream(stream)))


def tpmlp_rmsnorm_gather(X_chunks, weight, N, Xg, eps=1e-5, stream=None):
    rows, d = X_chunks[0].shape
    shape = make_shape(rows * N, d, 8 * N, N)  # ffn unused by this step
    xp, _xa = _ptrs(X_chunks)
    _check("tpmlp_rmsnorm_gather", lib().tpmlp_rmsnorm_gather(xp, _ptr(weight), eps, ctypes.byref(shape), _ptr(Xg),
                                                              _stream(stream)))


def tpmlp_gemm_dh_geluprime(dY, B, Hpre, N, dHpre, H=None, dbias=None, ws=None, stream=None):
    shape = make_shape(dY.shape[0], dY.shape[1], B.shape[0], N)
    if dbias is not None and ws is None:
        ws = workspace(shape, OP_DH_GELUPRIME, dY.device)
    _check("tpmlp_gemm_dh_geluprime", lib().tpmlp_gemm_dh_geluprime(
        _ptr(dY), _ptr(B), _ptr(Hpre), ctypes.byref(shape), _ptr(dHpre), _ptr(H), _ptr(dbias), _ptr(ws),
        0 if ws is None else ws.numel(), _stream(stream)))


def tpmlp_gemm_wgrad_b(H, dY, N, dB, stream=None):
    shape = make_shape(H.shape[0], dY.shape[1], H.shape[1], N)
    _check("tpmlp_gemm_wgrad_b", lib().tpmlp_gemm_wgrad_b(_ptr(H), _ptr(dY), ctypes.byref(shape), _ptr(dB),
                                                          _stream(stream)))


def tpmlp_gemm_wgrad_a(X, dHpre, N, dA, stream=None):
    shape = make_shape(X.shape[0], X.shape[1], dHpre.shape[1], N)
    _check("tpmlp_gemm_wgrad_a", lib().tpmlp_gemm_wgrad_a(_ptr(X), _ptr(dHpre), ctypes.byref(shape), _ptr(dA),
                                                          _stream(stream)))


def tpmlp_gemm_dx_shard_accum(dHpre, A, N, dX, stream=None):
    shape = make_shape(dHpre.shape[0], A.shape[0], dHpre.shape[1], N)
    _check("tpmlp_gemm_dx_shard_accum", lib().tpmlp_gemm_dx_shard_accum(_ptr(dHpre), _ptr(A), ctypes.byref(shape),
                                                                        _ptr(dX), _stream(stream)))


def tpmlp_layernorm_backward(X_chunks, gamma, dXg, N, dX_chunks, dgamma, dbeta, eps=1e-5, ws=None, stream=None):
    rows, d = X_chunks[0].shape
    shape = make_shape(rows * N, d, 8 * N, N)  # ffn unused by this step
    ws = workspace(shape, OP_LN_BWD, dXg.device) if ws is None else ws
    xp, _xa = _ptrs(X_chunks)
    dxp, _dxa = _ptrs(dX_chunks)
    _check("tpmlp_layernorm_backward", lib().tpmlp_layernorm_backward(
        xp, _ptr(gamma), eps, _ptr(dXg), ctypes.byref(shape), dxp, _ptr(dgamma), _ptr(dbeta), _ptr(ws), ws.numel(),
        _stream(stream)))


def tpmlp_layernorm_backward_add(X_chunks, gamma, dXg, R_chunks, N, dX_chunks, dgamma, dbeta, eps=1e-5, ws=None,
                                 stream=None):
    rows, d = X_chunks[0].shape
    shape = make_shape(rows * N, d, 8 * N, N)  # ffn unused by this step
    ws = workspace(shape, OP_LN_BWD, dXg.device) if ws is None else ws
    xp, _xa = _ptrs(X_chunks)
    rp, _ra = _ptrs(R_chunks)
    dxp, _dxa = _ptrs(dX_chunks)
    _check("tpmlp_layernorm_backward_add", lib().tpmlp_layernorm_backward_add(
        xp, _ptr(gamma), eps, _ptr(dXg), rp, ctypes.byref(shape), dxp, _ptr(dgamma), _ptr(dbeta), _ptr(ws),
        ws.numel(), _stream(stream)))


def tpmlp_layernorm_backward_blocks(X_chunks, gamma, dXg, N, dX_chunks, dgamma, dbeta, max_blocks, eps=1e-5, ws=None,
                                    stream=None):
    """LayerNorm backward with its dgamma/dbeta partials on at most `max_blocks` CTAs (a workspace of
    max_blocks * 2 * d floats)."""
    rows, d = X_chunks[0].shape
    shape = make_shape(rows * N, d, 8 * N, N)  # ffn unused by this step
    if ws is None:
        ws = torch.empty(max(1, max_blocks) * 2 * d * 4, dtype=torch.uint8, device=dXg.device)
    xp, _xa = _ptrs(X_chunks)
    dxp, _dxa = _ptrs(dX_chunks)
    _check("tpmlp_layernorm_backward_blocks", lib().tpmlp_layernorm_backward_blocks(
        xp, _ptr(gamma), eps, _ptr(dXg), ctypes.byref(shape), dxp, _ptr(dgamma), _ptr(dbeta), max_blocks, _ptr(ws),
        ws.numel(), _stream(stream)))


def tpmlp_layernorm_backward_noalloc(X_chunks, gamma, dXg, N, dX_chunks, dgamma, dbeta, eps=1e-5, stream=None):
    """LayerNorm backward without a workspace (scratch is a fixed array inside the library)."""
    rows, d = X_chunks[0].shape
    shape = make_shape(rows * N, d, 8 * N, N)  # ffn unused by this step
    xp, _xa = _ptrs(X_chunks)
    dxp, _dxa = _ptrs(dX_chunks)
    _check("tpmlp_layernorm_backward_noalloc", lib().tpmlp_layernorm_backward_noalloc(
        xp, _ptr(gamma), eps, _ptr(dXg), ctypes.byref(shape), dxp, _ptr(dgamma), _ptr(dbeta), _stream(stream)))


# ----------------------------------------------------------------------------- FP8 (E4M3) forward

def fp8_state(scale, amax, history, margin=0):
    """A tpmlp_fp8_state over device fp32 tensors scale [n], amax [n], history [n x L] (n = 4 for the
    forward's X, A, B, H; 2 for the backward's dY, dHpre).  The returned struct holds references to the
    tensors, so their memory stays allocated while the struct is alive."""
    st = Fp8State(scale.data_ptr(), amax.data_ptr(), history.data_ptr(), history.shape[-1], margin)
    st._tensors = (scale, amax, history)
    return st


def tpmlp_cast_e4m3(src, scale, dst, amax, transpose=False, stream=None):
    rows, cols = src.shape
    _check("tpmlp_cast_e4m3", lib().tpmlp_cast_e4m3(_ptr(src), rows, cols, 1 if transpose else 0, _ptr(scale),
                                                    _ptr(dst), _ptr(amax), _stream(stream)))


def tpmlp_layernorm_gather_e4m3(X_chunks, gamma, beta, N, scale, Xq, amax, eps=1e-5, stream=None):
    rows, d = X_chunks[0].shape
    shape = make_shape(rows * N, d, 16 * N, N)  # ffn unused by this step
    xp, _xa = _ptrs(X_chunks)
    _check("tpmlp_layernorm_gather_e4m3", lib().tpmlp_layernorm_gather_e4m3(
        xp, _ptr(gamma), _ptr(beta), eps, ctypes.byref(shape), _ptr(scale), _ptr(Xq), _ptr(amax), _stream(stream)))


def tpmlp_gemm1_e4m3(Xq, AqT, bias, N, scale_x, scale_a, scale_h, Hq, amax_h, Hpre=None, stream=None):
    shape = make_shape(Xq.shape[0], Xq.shape[1], AqT.shape[0], N)
    _check("tpmlp_gemm1_e4m3", lib().tpmlp_gemm1_e4m3(
        _ptr(Xq), _ptr(AqT), _ptr(bias), ctypes.byref(shape), _ptr(scale_x), _ptr(scale_a), _ptr(scale_h), _ptr(Hq),
        _ptr(amax_h), _ptr(Hpre), _stream(stream)))


def tpmlp_gemm2_e4m3(Hq, BqT, N, scale_h, scale_b, Y=None, Y_chunks=None, stream=None):
    shape = make_shape(Hq.shape[0], BqT.shape[0], Hq.shape[1], N)
    yp, _ya = _opt_ptrs(Y_chunks)
    _check("tpmlp_gemm2_e4m3", lib().tpmlp_gemm2_e4m3(_ptr(Hq), _ptr(BqT), ctypes.byref(shape), _ptr(scale_h),
                                                      _ptr(scale_b), _ptr(Y), yp, _stream(stream)))


def tpmlp_fp8_update_scales(state, stream=None):
    _check("tpmlp_fp8_update_scales", lib().tpmlp_fp8_update_scales(ctypes.byref(state), _stream(stream)))


def tpmlp_sp_forward_fp8(X_chunks, gamma, beta, A, B, N, Y_chunks, state, bias=None, eps=1e-5, Hpre_out=None,
                         Xq_out=None, Hq_out=None, ws=None, stream=None):
    """The E4M3 block forward; the scales are updated by tpmlp_fp8_update_scales once the step is over."""
    rows, d = X_chunks[0].shape
    shape = make_shape(rows * N, d, A.shape[1], N)
    ws = workspace(shape, OP_SP_FWD_FP8, A.device) if ws is None else ws
    xp, _xa = _ptrs(X_chunks)
    yp, _ya = _ptrs(Y_chunks)
    _check("tpmlp_sp_forward_fp8", lib().tpmlp_sp_forward_fp8(
        xp, _ptr(gamma), _ptr(beta), eps, _ptr(A), _ptr(B), _ptr(bias), ctypes.byref(state), ctypes.byref(shape), yp,
        _ptr(Hpre_out), _ptr(Xq_out), _ptr(Hq_out), _ptr(ws), ws.numel(), _stream(stream)))
    return Y_chunks


def tpmlp_cast_e5m2(src, scale, dst, amax, transpose=False, stream=None):
    rows, cols = src.shape
    _check("tpmlp_cast_e5m2", lib().tpmlp_cast_e5m2(_ptr(src), rows, cols, 1 if transpose else 0, _ptr(scale),
                                                    _ptr(dst), _ptr(amax), _stream(stream)))


def tpmlp_transpose_bytes(src, dst, stream=None):
    rows, cols = src.shape
    _check("tpmlp_transpose_bytes", lib().tpmlp_transpose_bytes(_ptr(src), rows, cols, _ptr(dst), _stream(stream)))


def tpmlp_gemm_dh_geluprime_e5m2(dYq, Bq, Hpre, N, scale_dy, scale_b, scale_g, dHq, amax_g, dbias=None, ws=None,
                                 stream=None):
    shape = make_shape(dYq.shape[0], dYq.shape[1], Bq.shape[0], N)
    if dbias is not None and ws is None:
        ws = workspace(shape, OP_DH_GELUPRIME, dYq.device)
    _check("tpmlp_gemm_dh_geluprime_e5m2", lib().tpmlp_gemm_dh_geluprime_e5m2(
        _ptr(dYq), _ptr(Bq), _ptr(Hpre), ctypes.byref(shape), _ptr(scale_dy), _ptr(scale_b), _ptr(scale_g), _ptr(dHq),
        _ptr(amax_g), _ptr(dbias), _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))


def tpmlp_gemm_fp8(A8, a_fmt, B8, b_fmt, scale_a, scale_b, C, stream=None):
    """C [M x N] bf16 = (A8 [M x K] . B8 [N x K]^T) / (scale_a scale_b); formats E4M3 / E5M2."""
    M, K = A8.shape
    N = B8.shape[0]
    _check("tpmlp_gemm_fp8", lib().tpmlp_gemm_fp8(_ptr(A8), a_fmt, _ptr(B8), b_fmt, M, N, K, _ptr(scale_a),
                                                  _ptr(scale_b), _ptr(C), C.stride(0), _stream(stream)))


def tpmlp_sp_backward_fp8(X_chunks, gamma, A, B, Hpre, Xq, Hq, dY_chunks, N, fwd_state, grad_state, dX_chunks, dA, dB,
                          dgamma, dbeta, dbias=None, eps=1e-5, dHq_out=None, ws=None, stream=None):
    rows, d = X_chunks[0].shape
    shape = make_shape(rows * N, d, A.shape[1], N)
    ws = workspace(shape, OP_SP_BWD_FP8, A.device) if ws is None else ws
    xp, _xa = _ptrs(X_chunks)
    dyp, _dya = _ptrs(dY_chunks)
    dxp, _dxa = _ptrs(dX_chunks)
    _check("tpmlp_sp_backward_fp8", lib().tpmlp_sp_backward_fp8(
        xp, _ptr(gamma), eps, _ptr(A), _ptr(B), _ptr(Hpre), _ptr(Xq), _ptr(Hq), dyp, ctypes.byref(fwd_state),
        ctypes.byref(grad_state), ctypes.byref(shape), dxp, _ptr(dA), _ptr(dB), _ptr(dbias), _ptr(dgamma),
        _ptr(dbeta), _ptr(dHq_out), _ptr(ws), ws.numel(), _stream(stream)))


# ----------------------------------------------------------------------------- tensor-parallel attention

def tpmlp_attention_workspace_size(S, B, H, head_dim=128):
    n = ctypes.c_size_t(0)
    _check("tpmlp_attention_workspace_size", lib().tpmlp_attention_workspace_size(S, B, H, head_dim, ctypes.byref(n)))
    return n.value


def attention_lse_shape(S, B, H):
    """Shape of the log-sum-exp statistics the attention forward saves: ``[B·H, 128·ceil(S/128)]``."""
    return (B * H, (S + 127) // 128 * 128)


def tpmlp_attention_core(QKV, S, B, H, O, causal=False, LSE=None, head_dim=128, stream=None):
    _check("tpmlp_attention_core", lib().tpmlp_attention_core(_ptr(QKV), S, B, H, head_dim, 1 if causal else 0, _ptr(O),
                                                              _ptr(LSE), _stream(stream)))


def tpmlp_attention_backward_workspace_size(S, B, H, head_dim=128):
    n = ctypes.c_size_t(0)
    _check("tpmlp_attention_backward_workspace_size",
           lib().tpmlp_attention_backward_workspace_size(S, B, H, head_dim, ctypes.byref(n)))
    return n.value


def tpmlp_attention_core_backward(QKV, O, dO, LSE, S, B, H, dQKV, causal=False, head_dim=128, ws=None, stream=None):
    if ws is None:
        ws = torch.empty(max(tpmlp_attention_backward_workspace_size(S, B, H), 256), dtype=torch.uint8,
                         device=QKV.device)
    _check("tpmlp_attention_core_backward", lib().tpmlp_attention_core_backward(
        _ptr(QKV), _ptr(O), _ptr(dO), _ptr(LSE), S, B, H, head_dim, 1 if causal else 0, _ptr(dQKV), _ptr(ws),
        ws.numel(), _stream(stream)))
    return dQKV


def tpmlp_attention_tp_forward(X, Wqkv, Wo, S, B, H, N, Y, bqkv=None, bo=None, causal=False, QKV_out=None,
                               O_out=None, LSE_out=None, ws=None, stream=None):
    if ws is None:
        ws = torch.empty(max(tpmlp_attention_workspace_size(S, B, H), 256), dtype=torch.uint8, device=X.device)
    _check("tpmlp_attention_tp_forward", lib().tpmlp_attention_tp_forward(
        _ptr(X), _ptr(Wqkv), _ptr(bqkv), _ptr(Wo), _ptr(bo), S, B, H, N, 1 if causal else 0, _ptr(Y), _ptr(QKV_out),
        _ptr(O_out), _ptr(LSE_out), _ptr(ws), ws.numel(), _stream(stream)))
    return Y


def tpmlp_attention_tp_backward(X, Wqkv, Wo, QKV, O, LSE, dY, S, B, H, N, dX, dWqkv, dWo, dbqkv=None, dbo=None,
                                causal=False, dQKV_out=None, ws=None, stream=None):
    if ws is None:
        ws = torch.empty(max(tpmlp_attention_backward_workspace_size(S, B, H), 256), dtype=torch.uint8,
                         device=X.device)
    _check("tpmlp_attention_tp_backward", lib().tpmlp_attention_tp_backward(
        _ptr(X), _ptr(Wqkv), _ptr(Wo), _ptr(QKV), _ptr(O), _ptr(LSE), _ptr(dY), S, B, H, N, 1 if causal else 0,
        _ptr(dX), _ptr(dWqkv), _ptr(dbqkv), _ptr(dWo), _ptr(dbo), _ptr(dQKV_out), _ptr(ws), ws.numel(),
        _stream(stream)))
    return dX


def tpmlp_selftest_wait_timeout(budget_us: int, stream=None):
    _check("tpmlp_selftest_wait_timeout", lib().tpmlp_selftest_wait_timeout(budget_us, _stream(stream)))
