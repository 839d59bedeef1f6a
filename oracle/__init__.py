"""Plain CPU fp64 oracle of the tensor-parallel MLP block and its sequence-parallel variant.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import this module.  The
CUDA library never calls it, shares no code with it, and the product path
fails rather than fall back to it.

Everything is float64 numpy; the matrix product is ``numpy.matmul`` and the
error function is ``scipy.special.erf`` (library primitives); there is no
blocking, fusion or reordering beyond what the definitions state.  Inputs are
the exact bf16 (or fp32) values the GPU consumes, widened to float64; no
intermediate is rounded.

Sources (pages by title, then section):

* [6D] "Megatron 架构与 6D 并行完整指南" (walkerchi.com), §3.1 "原理": the MLP
  is ``Y = GeLU(X·A)·B`` with ``A ∈ R^{d×4d}``, ``B ∈ R^{4d×d}``; with TP=2
  ``A0 = A[:, :2d]``, ``A1 = A[:, 2d:]``, ``B0 = B[:2d, :]``, ``B1 = B[2d:, :]``;
  each shard computes ``Y_i = GeLU(X·A_i)·B_i`` and an AllReduce gives
  ``Y = Y_0 + Y_1``; GeLU is elementwise so the column split commutes with it.
* [DEEP] "Megatron-LM 심층 아키텍처: 3D 하이브리드 병렬화(TP·SP·PP)…"
  (techknowgenie.com):
  - section "열 병렬(Column Parallel)과 행 병렬(Row Parallel)의 결합":
    ``Z = GeLU(X W1)``, ``Output = Z W2 = Σ_i Z_i W2_i = Σ_i Y_i``, W1 split
    into N column blocks, W2 into N row blocks;
  - section "All-Reduce 통신의 All-Gather 및 Reduce-Scatter 분해":
    ``AllReduce(X) = AllGather(ReduceScatter(X))``; LayerNorm runs on the
    S/N sequence slice, an All-Gather restores the full sequence before the
    GEMMs and a Reduce-Scatter after them sums the partials and splits the
    result by sequence;
  - section "분산 제어 소스코드 구조 패턴" (listing of ColumnParallelLinear,
    RowParallelLinear, SequenceParallelLayerNorm): the column layer adds a
    bias of ``out_features // world`` entries, ``split = out // world`` sizes
    the shards, the norm uses fp32 statistics and ``eps = 1e-5`` on a
    ``[S/N, batch, hidden]`` slice.
* [GLOSS] "Megatron-LM" glossary (jisaku.com), tensor-parallel table and the
  sequence-parallel paragraph: FFN layer 1 column-parallel, GeLU per GPU,
  layer 2 row-parallel with an AllReduce in forward; two AllReduces per
  block in backward; SP splits LayerNorm/Dropout along the sequence and
  replaces the AllReduce by ReduceScatter + AllGather.

Readings where the pages are silent or disagree (each is listed with its
reason in the design notes):

* GeLU is the exact ``0.5·x·(1 + erf(x/√2))`` ("GeLU" is all the pages say).
* ``bias`` is the column layer's bias, one entry per FFN column, split with
  A's columns; the row layer's bias is not part of this block.
* The sequence-parallel norm is a standard LayerNorm (the text says
  LayerNorm; the listing computes an RMS norm): biased variance (divide by
  d), ``eps`` inside the square root, scale ``gamma`` and shift ``beta``.
* Chunk ``j`` of the sequence is the contiguous row range
  ``[j·T/N, (j+1)·T/N)`` (tokens are sequence-major, ``[S/N, batch, hidden]``).
* The backward pass is not written on the pages; it is the chain rule of
  the forward definitions (``GeLU'(x) = Φ(x) + x·φ(x)``), with the backward
  AllReduce of the MLP summing the shards' input gradients, and in the SP
  block the mirror collectives: AllGather of dY, ReduceScatter of the input
  gradient.  dgamma and dbeta sum over all chunks.
* Non-divisible sizes (``F % N``, ``T % N``) are rejected, not truncated.
* The rest of the sequence-parallel region (bias of the row layer, Dropout,
  residual) reads: ``Y_j = X_j + dropout(Z_j + b2)``.  ``Z_j`` is chunk j
  of the reduced MLP output and ``b2`` is the row layer's bias, added after
  the reduction as the RowParallelLinear listing does.  Dropout lives in the
  sequence-split region (SP section, [GLOSS] SP paragraph).  The residual,
  which the pages never mention, is the block input ``X_j``.  Dropout keeps
  an element with probability ``1 - p`` and scales kept elements by
  ``1/(1 - p)``.  The pages give no generator, so the keep decision is drawn
  from Philox4x64-10 (Salmon, Moraes, Dror and Shaw, "Parallel random
  numbers: as easy as 1, 2, 3", SC 2011) on the element's index in the
  gathered ``[T x d]`` output (details at :func:`dropout_keep`).
* The RMS norm variant follows the SequenceParallelLayerNorm listing as
  written: fp32 mean of squares, ``rsqrt(ms + eps)``, the normalised row
  rounded to bf16 before the weight multiply (the listing's ``.to(dtype)``).
  Here the normalised value is computed in float64 and then rounded to bf16
  (round to nearest, ties to even, 8 significant bits).

* FP8 ([DEEP] section "FP8 하이브리드 정밀도 및 지연 스케일링(Delayed Scaling)"):
  forward matmul operands in E4M3 (1 sign, 4 exponent bits, 3 mantissa
  bits), each tensor multiplied by its scale factor ``S`` before the cast,
  ``q = E4M3(x·S)``, and the product divided by both scales afterwards.
  E4M3 is read as the OCP 8-bit format without infinities (bias 7, largest
  finite value 448, subnormals down to 2**-9); the cast rounds to nearest,
  ties to even, and saturates at ±448.  ``x·S`` is formed in float32, as the
  GPU forms it.  Delayed scaling: the page predicts the next step's scale
  from the moving average of the amaxes recorded in earlier steps; here the
  average is the mean of a fixed-length amax history and ``S = 448 / mean``
  (``2**-margin`` headroom optional; ``S = 1`` while the history is zero).
  Which tensors run in FP8 in the forward: the gathered norm output, both
  weights and the GeLU output ``H`` (the operands of the two GEMMs); the
  bias and GeLU act on the dequantised fp32 product.  In the backward the
  gradients that enter GEMMs (``dY`` and ``dHpre``) are cast to E5M2 (1
  sign, 5 exponent bits with bias 15, 2 mantissa bits, largest finite 57344,
  subnormals down to 2**-16; same rounding and saturation), the forward's
  E4M3 operands are reused, and the bias gradient and GeLU' act on fp32
  values.

* Attention ([6D] §3.2 "Attention 的 TP"; [GLOSS] tensor-parallel section;
  [DEEP] column/row-parallel section, multi-head attention paragraph): the
  Q, K, V projections are split by columns along heads, each shard computes
  complete attention for its heads, the output projection is split by rows
  (the same heads) and an AllReduce sums the shards.  Readings: attention
  is ``softmax(Q Kᵀ / sqrt(hd)) V`` per head and sequence, optionally causal
  (position s attends to positions <= s); the projection weight is one
  ``[d x 3d]`` matrix whose columns are Q, K, V in that order, head h taking
  columns ``h·hd .. (h+1)·hd`` of each; tokens are sequence-major
  (``[S, batch, hidden]``, row ``s·B + b``) and attend only within their
  batch element; the output projection's bias is added once, after the sum.

Every function is pinned by tests in ``tests/test_oracle_pins.py`` (values
printed on the pages, closed forms, invariants, brute force, library
witnesses and finite differences); none is parity-unpinned.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf as _erf

SQRT_HALF = 1.0 / math.sqrt(2.0)
INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)


# --------------------------------------------------------------------------- partition

def shard_ranges(F: int, N: int) -> list[tuple[int, int]]:
    """Column shard ``i`` of A (row shard ``i`` of B): ``[i·F/N, (i+1)·F/N)``.

    [6D] §3.1 (TP=2: ``A[:, :2d]``, ``A[:, 2d:]``); [DEEP] listing
    (``split_out_features = out_features // world``).  Rejects ``F % N != 0``.
    """
    if N <= 0 or F <= 0 or F % N:
        raise ValueError(f"F={F} is not split evenly into N={N} shards")
    w = F // N
    return [(i * w, (i + 1) * w) for i in range(N)]


def chunk_ranges(T: int, N: int) -> list[tuple[int, int]]:
    """Sequence chunk ``j``: rows ``[j·T/N, (j+1)·T/N)`` ([DEEP] SP section: S/N per GPU)."""
    if N <= 0 or T <= 0 or T % N:
        raise ValueError(f"T={T} is not split evenly into N={N} chunks")
    w = T // N
    return [(j * w, (j + 1) * w) for j in range(N)]


# --------------------------------------------------------------------------- elementwise

def gelu(x):
    """Exact GeLU: ``x·Φ(x) = 0.5·x·(1 + erf(x/√2))``."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + _erf(x * SQRT_HALF))


def gelu_prime(x):
    """Derivative of the exact GeLU: ``Φ(x) + x·φ(x)``."""
    x = np.asarray(x, dtype=np.float64)
    cdf = 0.5 * (1.0 + _erf(x * SQRT_HALF))
    pdf = INV_SQRT_2PI * np.exp(-0.5 * x * x)
    return cdf + x * pdf


# --------------------------------------------------------------------------- collectives (on explicit per-shard buffers)

def all_reduce(parts):
    """Sum of the shards' partial outputs, shard 0 first ([DEEP] eq. ``Output = Σ_i Y_i``)."""
    total = np.zeros_like(np.asarray(parts[0], dtype=np.float64))
    for p in parts:
        total = total + p
    return total


def reduce_scatter(parts, N: int):
    """Sum the partials, then split the rows into N sequence chunks ([DEEP] SP section)."""
    total = all_reduce(parts)
    return [total[lo:hi] for lo, hi in chunk_ranges(total.shape[0], N)]


def all_gather(chunks):
    """Concatenate sequence chunks back into the full sequence ([DEEP] SP section)."""
    return np.concatenate([np.asarray(c, dtype=np.float64) for c in chunks], axis=0)


# --------------------------------------------------------------------------- forward

def _bias_or_zero(b, F):
    return np.zeros(F, dtype=np.float64) if b is None else np.asarray(b, dtype=np.float64)


def mlp_reference(X, A, B, b=None):
    """Unsharded block: ``Y = GeLU(X·A + b)·B`` ([6D] §3.1 ``Y = GeLU(X·A)·B``; bias of the column layer)."""
    X = np.asarray(X, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    Z = gelu(X @ A + _bias_or_zero(b, A.shape[1]))
    return Z @ B


def column_parallel(X, A_i, b_i):
    """Shard i of the first layer: ``Z_i = GeLU(X·A_i + b_i)`` (no communication)."""
    return gelu(np.asarray(X, dtype=np.float64) @ np.asarray(A_i, dtype=np.float64) + b_i)


def row_parallel_partial(Z_i, B_i):
    """Shard i of the second layer: the partial ``Y_i = Z_i·B_i``."""
    return Z_i @ np.asarray(B_i, dtype=np.float64)


def mlp_partials(X, A, B, b, N: int):
    """The N partial outputs ``Y_i = GeLU(X·A_i + b_i)·B_i``, one per shard."""
    F = np.asarray(A).shape[1]
    bias = _bias_or_zero(b, F)
    parts = []
    for lo, hi in shard_ranges(F, N):
        Z_i = column_parallel(X, np.asarray(A)[:, lo:hi], bias[lo:hi])
        parts.append(row_parallel_partial(Z_i, np.asarray(B)[lo:hi, :]))
    return parts


def mlp_tp(X, A, B, b, N: int):
    """Tensor-parallel block: AllReduce of the shard partials."""
    return all_reduce(mlp_partials(X, A, B, b, N))


def layer_norm(x, gamma, beta, eps: float = 1e-5):
    """LayerNorm of each row: ``(x - mean)/sqrt(var + eps)·gamma + beta``, biased variance."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * np.asarray(gamma, dtype=np.float64) + np.asarray(beta, dtype=np.float64)


def sp_forward(X_chunks, gamma, beta, eps, A, B, b, N: int, return_intermediates: bool = False):
    """Sequence-parallel block forward.

    LayerNorm on each S/N chunk, AllGather, the N shard partials, then
    ReduceScatter back to chunks ([DEEP] SP section).
    """
    if len(X_chunks) != N:
        raise ValueError("one input chunk per shard")
    normed = [layer_norm(c, gamma, beta, eps) for c in X_chunks]
    Xg = all_gather(normed)
    parts = mlp_partials(Xg, A, B, b, N)
    Y_chunks = reduce_scatter(parts, N)
    if return_intermediates:
        return Y_chunks, {"Xg": Xg, "partials": parts}
    return Y_chunks


def round_bf16(x):
    """Round to the nearest bfloat16 value (8 significant bits, ties to even), returned as float64.

    ``x = m·2**e`` with ``0.5 <= |m| < 1``; ``m·2**8`` rounded half-to-even and scaled back.  Values
    stay inside bf16's normal range here (no overflow or subnormal handling).
    """
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(np.rint(m * 256.0), e - 8)


def rms_norm(x, weight, eps: float = 1e-5):
    """The norm of the SequenceParallelLayerNorm listing ([DEEP] "분산 제어 소스코드 구조 패턴"):
    ``x·rsqrt(mean(x²) + eps)`` rounded to bf16, then times ``weight``."""
    x = np.asarray(x, dtype=np.float64)
    rstd = 1.0 / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)
    return round_bf16(x * rstd) * np.asarray(weight, dtype=np.float64)


# --------------------------------------------------------------------------- dropout generator

# Philox4x64 round multipliers and key increments (Salmon et al., SC 2011, table of Philox parameters).
PHILOX4X64_M = (0xD2E7470EE14C6C93, 0xCA5A826395121157)
PHILOX4X64_W = (0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B)
_MASK64 = (1 << 64) - 1
_LO32 = np.uint64(0xFFFFFFFF)
_S32 = np.uint64(32)


def _mulhilo64(m: int, x):
    """High and low 64-bit halves of the 128-bit products ``m·x`` (``x`` a uint64 array), by 32-bit limbs."""
    a_lo, a_hi = np.uint64(m & 0xFFFFFFFF), np.uint64(m >> 32)
    x_lo, x_hi = x & _LO32, x >> _S32
    with np.errstate(over="ignore"):
        ll, lh, hl, hh = a_lo * x_lo, a_lo * x_hi, a_hi * x_lo, a_hi * x_hi
        mid = (ll >> _S32) + (lh & _LO32) + (hl & _LO32)
        hi = hh + (lh >> _S32) + (hl >> _S32) + (mid >> _S32)
        lo = np.uint64(m) * x
    return hi, lo


def philox4x64(counter, key, rounds: int = 10):
    """Philox4x64-``rounds`` blocks: ``counter`` [..., 4] uint64, ``key`` = (k0, k1) -> [..., 4] uint64.

    One round takes ``(hi0, lo0) = M0·x0`` and ``(hi1, lo1) = M1·x2`` and sets
    ``x = (hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0)``; the key advances by the
    Weyl increments ``(W0, W1)`` between rounds (the first round uses the key
    as given).
    """
    c = np.asarray(counter, dtype=np.uint64)
    x = [c[..., i] for i in range(4)]
    k0, k1 = int(key[0]) & _MASK64, int(key[1]) & _MASK64
    for r in range(rounds):
        if r:
            k0 = (k0 + PHILOX4X64_W[0]) & _MASK64
            k1 = (k1 + PHILOX4X64_W[1]) & _MASK64
        hi0, lo0 = _mulhilo64(PHILOX4X64_M[0], x[0])
        hi1, lo1 = _mulhilo64(PHILOX4X64_M[1], x[2])
        x = [hi1 ^ x[1] ^ np.uint64(k0), lo1, hi0 ^ x[3] ^ np.uint64(k1), lo0]
    return np.stack(x, axis=-1)


def dropout_threshold(p) -> int:
    """Keep threshold for drop probability ``p`` (taken as float32): ``floor((1 - p)·2**32)``."""
    p = float(np.float32(p))
    if not 0.0 <= p < 1.0:
        raise ValueError("dropout probability must lie in [0, 1)")
    return math.floor((1.0 - p) * 2.0 ** 32)


def dropout_keep(rows: int, d: int, row0: int, p, seed: int, offset: int):
    """Keep mask of rows ``[row0, row0 + rows)`` of a ``[T x d]`` output.

    Element ``(r, c)`` has index ``e = r·d + c``.  Block ``e // 8`` is one
    Philox4x64-10 call with counter ``(e // 8, offset, 0, 0)`` and key
    ``(seed, 0)``; element ``e`` takes 32 bits of it: word ``(e % 8) // 2``,
    its low half for even ``e`` and its high half for odd ``e``.  The element
    is kept when those 32 bits, read as an unsigned integer, are below
    :func:`dropout_threshold`.
    """
    r = np.arange(row0, row0 + rows, dtype=np.uint64)[:, None]
    e = r * np.uint64(d) + np.arange(d, dtype=np.uint64)[None, :]
    ctr = np.zeros(e.shape + (4,), dtype=np.uint64)
    ctr[..., 0] = e >> np.uint64(3)
    ctr[..., 1] = np.uint64(offset)
    words = philox4x64(ctr, (seed, 0))
    lane = e & np.uint64(7)
    w = np.take_along_axis(words, (lane >> np.uint64(1)).astype(np.intp)[..., None], axis=-1)[..., 0]
    u = (w >> (_S32 * (lane & np.uint64(1)))) & _LO32
    return u < np.uint64(dropout_threshold(p)) if dropout_threshold(p) < 2 ** 32 else np.ones(e.shape, dtype=bool)


def sp_block_forward(X_chunks, gamma, beta, eps, A, B, b, b2, p, seed: int, offset: int, N: int):
    """The whole sequence-parallel region: ``Y_j = X_j + dropout(Z_j + b2)``, ``Z_j`` = :func:`sp_forward`."""
    Z = sp_forward(X_chunks, gamma, beta, eps, A, B, b, N)
    T = sum(np.asarray(x).shape[0] for x in X_chunks)
    d = np.asarray(X_chunks[0]).shape[1]
    bias2 = _bias_or_zero(b2, d)
    scale = 1.0 / (1.0 - float(np.float32(p)))
    out = []
    for (lo, hi), xj, zj in zip(chunk_ranges(T, N), X_chunks, Z):
        keep = dropout_keep(hi - lo, d, lo, p, seed, offset)
        out.append(np.asarray(xj, dtype=np.float64) + np.where(keep, (zj + bias2) * scale, 0.0))
    return out


# --------------------------------------------------------------------------- FP8 (E4M3) forward with delayed scaling

E4M3_MAX = 448.0


def round_e4m3(x):
    """Nearest E4M3 value, ties to even, magnitudes above 448 saturated to 448; returned as float64.

    ``|x| = m·2**e`` with ``0.5 <= m < 1``; a normal E4M3 number ``1.fff·2**E`` has
    quantum ``2**(E-3)`` with ``E = e - 1``; below ``2**-6`` the subnormals keep the
    quantum ``2**-9``.  Rounding ``|x|/quantum`` half-to-even rounds the last mantissa
    bit to even.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)
    quantum = np.ldexp(1.0, np.maximum(e - 1, -6) - 3)
    r = np.minimum(np.rint(a / quantum) * quantum, E4M3_MAX)
    return np.copysign(r, x)


E5M2_MAX = 57344.0


def round_e5m2(x):
    """Nearest E5M2 value, ties to even, magnitudes above 57344 saturated to 57344; returned as float64.

    As :func:`round_e4m3` with two mantissa bits (quantum ``2**(E-2)``) and normal exponents
    down to ``E = -14`` (subnormal quantum ``2**-16``).
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)
    quantum = np.ldexp(1.0, np.maximum(e - 1, -14) - 2)
    r = np.minimum(np.rint(a / quantum) * quantum, E5M2_MAX)
    return np.copysign(r, x)


def quantize_e5m2(x, scale):
    """``E5M2(x·S)`` with the product formed in float32."""
    return round_e5m2(np.asarray(x, dtype=np.float32) * np.float32(scale))


def quantize_e4m3(x, scale):
    """``E4M3(x·S)`` with the product formed in float32 (``x`` taken to float32 first)."""
    return round_e4m3(np.asarray(x, dtype=np.float32) * np.float32(scale))


def fp8_scale(amax_history, fp8_max: float = E4M3_MAX, margin: int = 0) -> float:
    """Delayed scaling: ``S = fp8_max / mean(history) / 2**margin``; 1 while the mean is not positive."""
    est = float(np.mean(np.asarray(amax_history, dtype=np.float64)))
    if not est > 0.0 or not math.isfinite(est):
        return 1.0
    return fp8_max / est / 2.0 ** margin


def roll_amax_history(amax_history, amax):
    """The history after a step: the oldest entry drops out, this step's amax is appended."""
    h = np.asarray(amax_history, dtype=np.float64)
    return np.concatenate([h[1:], [float(amax)]])


def mlp_fp8(X, A, B, b, N: int, scales):
    """The MLP with E4M3 GEMM operands: ``scales = (S_X, S_A, S_B, S_H)``.

    ``H = GeLU((q_X·q_A)/(S_X S_A) + b)``, ``Y = Σ_i (q_H,i·q_B,i)/(S_H S_B)`` over the
    N row shards of the second layer (one shard sum, as :func:`mlp_tp`).  Also
    returns the amaxes a step records: ``max|X|``, ``max|A|``, ``max|B|``,
    ``max|H|`` (before the casts).
    """
    sx, sa, sb, sh = scales
    X = np.asarray(X, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    qx, qa, qb = quantize_e4m3(X, sx), quantize_e4m3(A, sa), quantize_e4m3(B, sb)
    H = gelu((qx @ qa) / (float(np.float32(sx)) * float(np.float32(sa))) + _bias_or_zero(b, A.shape[1]))
    qh = quantize_e4m3(H, sh)
    F = A.shape[1]
    parts = [(qh[:, lo:hi] @ qb[lo:hi, :]) / (float(np.float32(sh)) * float(np.float32(sb)))
             for lo, hi in shard_ranges(F, N)]
    amax = {"X": float(np.max(np.abs(X), initial=0.0)), "A": float(np.max(np.abs(A), initial=0.0)),
            "B": float(np.max(np.abs(B), initial=0.0)), "H": float(np.max(np.abs(H), initial=0.0))}
    return {"Y": all_reduce(parts), "H": H, "qH": qh, "amax": amax}


def mlp_backward_fp8(X, A, B, b, dY, N: int, scales, grad_scales, saved=None):
    """Backward of :func:`mlp_fp8` with E5M2 gradients: ``grad_scales = (S_dY, S_dHpre)``.

    With the forward's ``q_X, q_A, q_B``, ``Hpre = (q_X·q_A)/(S_X S_A) + b``, ``H = GeLU(Hpre)``,
    ``q_H = E4M3(H·S_H)`` and ``q_dY = E5M2(dY·S_dY)``:
    ``dHpre = (q_dY·q_Bᵀ)/(S_dY S_B) ⊙ GeLU'(Hpre)``, ``q_g = E5M2(dHpre·S_dHpre)``,
    ``dB = (q_Hᵀ·q_dY)/(S_H S_dY)``, ``dA = (q_Xᵀ·q_g)/(S_X S_dHpre)``, ``db = Σ_rows dHpre``,
    ``dX = Σ_i (q_g,i·q_A,iᵀ)/(S_dHpre S_A)`` (the backward shard sum).  Also the amaxes of
    ``dY`` and ``dHpre``.

    ``saved``: None, or a dict whose entries replace the values this function would form itself:
    ``"qX"``, ``"qH"`` (E4M3 code values of the norm output and of H, as a forward saved them),
    ``"Hpre"`` (the saved pre-activation) and ``"qdHpre"`` (E5M2 code values of the gradient that enters
    the weight- and input-gradient GEMMs).  A backward works from the activations its forward kept; where
    a cast's input lies within rounding of a midpoint, another implementation's saved codes can differ from
    these by one step, and this lets the rest of the chain be formed from exactly those codes.
    """
    saved = {} if saved is None else saved
    sx, sa, sb, sh = (float(np.float32(v)) for v in scales)
    sdy, sg = (float(np.float32(v)) for v in grad_scales)
    X = np.asarray(X, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    qx, qa, qb = quantize_e4m3(X, sx), quantize_e4m3(A, sa), quantize_e4m3(B, sb)
    if "qX" in saved:
        qx = np.asarray(saved["qX"], dtype=np.float64)
    if "Hpre" in saved:
        Hpre = np.asarray(saved["Hpre"], dtype=np.float64)
    else:
        Hpre = (qx @ qa) / (sx * sa) + _bias_or_zero(b, A.shape[1])
    qh = np.asarray(saved["qH"], dtype=np.float64) if "qH" in saved else quantize_e4m3(gelu(Hpre), sh)
    qdy = quantize_e5m2(dY, sdy)
    dHpre = (qdy @ qb.T) / (sdy * sb) * gelu_prime(Hpre)
    qg = np.asarray(saved["qdHpre"], dtype=np.float64) if "qdHpre" in saved else quantize_e5m2(dHpre, sg)
    F = A.shape[1]
    dX_parts = [(qg[:, lo:hi] @ qa[:, lo:hi].T) / (sg * sa) for lo, hi in shard_ranges(F, N)]
    return {"dX": all_reduce(dX_parts), "dX_parts": dX_parts, "dA": (qx.T @ qg) / (sx * sg),
            "dB": (qh.T @ qdy) / (sh * sdy), "db": dHpre.sum(axis=0), "dHpre": dHpre, "qdHpre": qg,
            "amax": {"dY": float(np.max(np.abs(dY), initial=0.0)), "dHpre": float(np.max(np.abs(dHpre), initial=0.0))}}


def sp_backward_fp8(X_chunks, gamma, beta, eps, A, B, b, dY_chunks, N: int, scales, grad_scales, saved=None):
    """:func:`sp_backward` with the FP8 GEMMs of :func:`mlp_backward_fp8`: gather the norm output and
    dY, the FP8 MLP backward, reduce-scatter of the input-gradient shard partials, LayerNorm backward
    per chunk (on the unquantised gradient).  ``saved`` as in :func:`mlp_backward_fp8`."""
    Xg = all_gather([layer_norm(c, gamma, beta, eps) for c in X_chunks])
    g = mlp_backward_fp8(Xg, A, B, b, all_gather(dY_chunks), N, scales, grad_scales, saved=saved)
    dXg_chunks = reduce_scatter(g["dX_parts"], N)
    dX_chunks, dgamma, dbeta = [], 0.0, 0.0
    for xc, dyc in zip(X_chunks, dXg_chunks):
        dx, dga, dbe = layer_norm_backward(xc, gamma, eps, dyc)
        dX_chunks.append(dx)
        dgamma = dgamma + dga
        dbeta = dbeta + dbe
    g.update({"dX_chunks": dX_chunks, "dgamma": dgamma, "dbeta": dbeta, "dXg_chunks": dXg_chunks})
    return g


def sp_forward_fp8(X_chunks, gamma, beta, eps, A, B, b, N: int, scales):
    """:func:`sp_forward` with the E4M3 GEMMs of :func:`mlp_fp8`: LayerNorm per chunk,
    gather, the FP8 MLP, reduce-scatter of its row-shard partials."""
    Xg = all_gather([layer_norm(c, gamma, beta, eps) for c in X_chunks])
    out = mlp_fp8(Xg, A, B, b, N, scales)
    T = Xg.shape[0]
    out["Y_chunks"] = [out["Y"][lo:hi] for lo, hi in chunk_ranges(T, N)]
    out["Xg"] = Xg
    return out


# --------------------------------------------------------------------------- tensor-parallel attention

def attention_head(Q, K, V, causal: bool):
    """``softmax(Q·Kᵀ/sqrt(hd))·V`` for one head of one sequence: Q, K, V ``[S x hd]``; with ``causal``
    position s sees keys 0..s only."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    scores = Q @ K.T / math.sqrt(Q.shape[1])
    if causal:
        S = Q.shape[0]
        scores = np.where(np.tril(np.ones((S, S), dtype=bool)), scores, -np.inf)
    scores = scores - scores.max(axis=1, keepdims=True)
    w = np.exp(scores)
    return (w / w.sum(axis=1, keepdims=True)) @ V


def head_ranges(H: int, N: int) -> list[tuple[int, int]]:
    """Heads of shard i: ``[i·H/N, (i+1)·H/N)`` (H % N == 0)."""
    if N <= 0 or H % N != 0:
        raise ValueError("the heads must split evenly over the shards")
    return [(i * H // N, (i + 1) * H // N) for i in range(N)]


def attention_tp(X, Wqkv, bqkv, Wo, bo, H: int, N: int, B: int, causal: bool, return_parts: bool = False):
    """The tensor-parallel attention block: ``Y = Σ_i O_i·Wo[rows of shard i] + bo``.

    ``X [T x d]`` with ``T = S·B`` (row ``s·B + b``); ``Wqkv [d x 3d]``, ``bqkv [3d]`` or None;
    ``Wo [d x d]``, ``bo [d]`` or None.  Shard i projects its heads' Q, K, V columns, computes their
    attention per batch element, and multiplies by its rows of ``Wo``; the shards' partials are summed
    (the AllReduce) and ``bo`` is added once.
    """
    X = np.asarray(X, dtype=np.float64)
    Wqkv = np.asarray(Wqkv, dtype=np.float64)
    Wo = np.asarray(Wo, dtype=np.float64)
    T, d = X.shape
    if T % B != 0 or d % H != 0:
        raise ValueError("T must be a multiple of the batch and d of the head count")
    hd = d // H
    bias_qkv = np.zeros(3 * d) if bqkv is None else np.asarray(bqkv, dtype=np.float64)
    parts, Os = [], []
    for lo, hi in head_ranges(H, N):
        O_i = np.zeros((T, (hi - lo) * hd))
        for h in range(lo, hi):
            cols = [slice(part * d + h * hd, part * d + (h + 1) * hd) for part in range(3)]
            Qh, Kh, Vh = (X @ Wqkv[:, c] + bias_qkv[c] for c in cols)
            for b in range(B):
                rows = slice(b, T, B)
                O_i[rows, (h - lo) * hd:(h - lo + 1) * hd] = attention_head(Qh[rows], Kh[rows], Vh[rows], causal)
        Os.append(O_i)
        parts.append(O_i @ Wo[lo * hd:hi * hd, :])
    Y = all_reduce(parts) + (0.0 if bo is None else np.asarray(bo, dtype=np.float64))
    if return_parts:
        return Y, {"O": np.concatenate(Os, axis=1), "partials": parts}
    return Y


def attention_head_backward(Q, K, V, dO, causal: bool, O=None):
    """Gradients of :func:`attention_head` (chain rule): with ``P = softmax(Q Kᵀ/√hd)`` and ``O = P V``,
    ``dV = Pᵀ dO``, ``dP = dO Vᵀ``, ``dS = P ⊙ (dP - D)`` with ``D = rowsum(dO ⊙ O)``,
    ``dQ = dS K / √hd``, ``dK = dSᵀ Q / √hd``.  ``O``: None for the exact forward output, or the output
    as the forward saved it (e.g. rounded to bf16), from which ``D`` is then formed."""
    Q, K, V, dO = (np.asarray(a, dtype=np.float64) for a in (Q, K, V, dO))
    hd = Q.shape[1]
    scores = Q @ K.T / math.sqrt(hd)
    if causal:
        S = Q.shape[0]
        scores = np.where(np.tril(np.ones((S, S), dtype=bool)), scores, -np.inf)
    scores = scores - scores.max(axis=1, keepdims=True)
    P = np.exp(scores)
    P = P / P.sum(axis=1, keepdims=True)
    O = P @ V if O is None else np.asarray(O, dtype=np.float64)
    dV = P.T @ dO
    dP = dO @ V.T
    D = (dO * O).sum(axis=1, keepdims=True)
    dS = P * (dP - D)
    return dS @ K / math.sqrt(hd), dS.T @ Q / math.sqrt(hd), dV


def attention_tp_backward(X, Wqkv, bqkv, Wo, bo, H: int, N: int, B: int, causal: bool, dY):
    """Gradients of :func:`attention_tp` (chain rule), shard by shard as the forward splits the work:
    ``dO_i = dY Wo[rows of shard i]ᵀ``, ``dWo[rows of shard i] = O_iᵀ dY``, ``dbo = Σ_rows dY``; per
    head the attention backward; the projection ``dWqkv = Xᵀ dQKV``, ``dbqkv = Σ_rows dQKV`` and
    ``dX = Σ_i dQKV_i Wqkv_iᵀ`` (the backward AllReduce over the shards' columns)."""
    X = np.asarray(X, dtype=np.float64)
    Wqkv = np.asarray(Wqkv, dtype=np.float64)
    Wo = np.asarray(Wo, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    T, d = X.shape
    hd = d // H
    bias_qkv = np.zeros(3 * d) if bqkv is None else np.asarray(bqkv, dtype=np.float64)
    QKV = X @ Wqkv + bias_qkv
    dQKV = np.zeros_like(QKV)
    dWo = np.zeros_like(Wo)
    dX_parts = []
    for lo, hi in head_ranges(H, N):
        cols = np.concatenate([np.arange(part * d + lo * hd, part * d + hi * hd) for part in range(3)])
        O_i = np.zeros((T, (hi - lo) * hd))
        for h in range(lo, hi):
            c = [slice(part * d + h * hd, part * d + (h + 1) * hd) for part in range(3)]
            for b in range(B):
                rows = slice(b, T, B)
                O_i[rows, (h - lo) * hd:(h - lo + 1) * hd] = attention_head(QKV[rows, c[0]], QKV[rows, c[1]],
                                                                             QKV[rows, c[2]], causal)
        dO_i = dY @ Wo[lo * hd:hi * hd, :].T
        dWo[lo * hd:hi * hd, :] = O_i.T @ dY
        for h in range(lo, hi):
            c = [slice(part * d + h * hd, part * d + (h + 1) * hd) for part in range(3)]
            for b in range(B):
                rows = slice(b, T, B)
                dq, dk, dv = attention_head_backward(QKV[rows, c[0]], QKV[rows, c[1]], QKV[rows, c[2]],
                                                     dO_i[rows, (h - lo) * hd:(h - lo + 1) * hd], causal)
                dQKV[rows, c[0]], dQKV[rows, c[1]], dQKV[rows, c[2]] = dq, dk, dv
        dX_parts.append(dQKV[:, cols] @ Wqkv[:, cols].T)
    return {"dX": all_reduce(dX_parts), "dWqkv": X.T @ dQKV, "dbqkv": dQKV.sum(axis=0), "dWo": dWo,
            "dbo": dY.sum(axis=0), "dQKV": dQKV}


# --------------------------------------------------------------------------- backward (chain rule)

def mlp_backward(X, A, B, b, dY):
    """Gradients of ``Y = GeLU(X·A + b)·B`` (unsharded).

    ``Hpre = X·A + b``, ``H = GeLU(Hpre)``, ``dH = dY·Bᵀ``,
    ``dHpre = dH ⊙ GeLU'(Hpre)``, ``dB = Hᵀ·dY``, ``dA = Xᵀ·dHpre``,
    ``db = Σ_rows dHpre``, ``dX = dHpre·Aᵀ``.
    """
    X = np.asarray(X, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    Hpre = X @ A + _bias_or_zero(b, A.shape[1])
    H = gelu(Hpre)
    dH = dY @ B.T
    dHpre = dH * gelu_prime(Hpre)
    return {"dX": dHpre @ A.T, "dA": X.T @ dHpre, "dB": H.T @ dY, "db": dHpre.sum(axis=0),
            "Hpre": Hpre, "H": H, "dHpre": dHpre}


def mlp_backward_tp(X, A, B, b, dY, N: int):
    """Per-shard gradients; the input gradient is the AllReduce of the shards' ``dX_i``.

    Shard i owns ``A_i``, ``B_i``, ``b_i`` and so ``dA_i``, ``dB_i``, ``db_i``
    (concatenated here); ``dX_i = dHpre_i·A_iᵀ`` is a partial that the
    backward AllReduce sums ([GLOSS] tensor-parallel section: two AllReduces
    per block in backward).
    """
    F = np.asarray(A).shape[1]
    bias = _bias_or_zero(b, F)
    dA = np.zeros(np.asarray(A).shape)
    dB = np.zeros(np.asarray(B).shape)
    db = np.zeros(F)
    dX_parts = []
    for lo, hi in shard_ranges(F, N):
        g = mlp_backward(X, np.asarray(A)[:, lo:hi], np.asarray(B)[lo:hi, :], bias[lo:hi], dY)
        dA[:, lo:hi] = g["dA"]
        dB[lo:hi, :] = g["dB"]
        db[lo:hi] = g["db"]
        dX_parts.append(g["dX"])
    return {"dX": all_reduce(dX_parts), "dX_parts": dX_parts, "dA": dA, "dB": dB, "db": db}


def layer_norm_backward(x, gamma, eps, dy):
    """Gradients of :func:`layer_norm` for one chunk of rows.

    With ``x̂ = (x - mean)·rstd`` and ``g = dy·gamma``:
    ``dx = rstd·(g - mean(g) - x̂·mean(g·x̂))``, ``dgamma = Σ_rows dy·x̂``,
    ``dbeta = Σ_rows dy``.
    """
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (x - mu) * rstd
    g = dy * np.asarray(gamma, dtype=np.float64)
    dx = rstd * (g - g.mean(axis=-1, keepdims=True) - xhat * (g * xhat).mean(axis=-1, keepdims=True))
    return dx, (dy * xhat).sum(axis=0), dy.sum(axis=0)


def sp_backward(X_chunks, gamma, beta, eps, A, B, b, dY_chunks, N: int):
    """Sequence-parallel block backward: the mirror of :func:`sp_forward`.

    AllGather of the output-gradient chunks (mirror of the forward
    ReduceScatter), per-shard MLP gradients, ReduceScatter of the shards'
    input-gradient partials (mirror of the forward AllGather), then the
    LayerNorm backward on each chunk.
    """
    normed = [layer_norm(c, gamma, beta, eps) for c in X_chunks]
    Xg = all_gather(normed)
    dYg = all_gather(dY_chunks)
    g = mlp_backward_tp(Xg, A, B, b, dYg, N)
    dXg_chunks = reduce_scatter(g["dX_parts"], N)
    dX_chunks, dgamma, dbeta = [], 0.0, 0.0
    for xc, dyc in zip(X_chunks, dXg_chunks):
        dx, dga, dbe = layer_norm_backward(xc, gamma, eps, dyc)
        dX_chunks.append(dx)
        dgamma = dgamma + dga
        dbeta = dbeta + dbe
    return {"dX_chunks": dX_chunks, "dA": g["dA"], "dB": g["dB"], "db": g["db"],
            "dgamma": dgamma, "dbeta": dbeta, "dXg_chunks": dXg_chunks}


def sp_block_backward(X_chunks, gamma, beta, eps, A, B, b, p, seed: int, offset: int, dY_chunks, N: int):
    """Gradients of :func:`sp_block_forward`.

    ``dZ_j = dY_j ⊙ keep_j / (1 - p)``; ``db2 = Σ_j Σ_rows dZ_j``; the MLP and
    norm gradients are :func:`sp_backward` driven by ``dZ``; the residual
    adds ``dY_j`` to the input gradient of chunk j.
    """
    T = sum(np.asarray(x).shape[0] for x in X_chunks)
    d = np.asarray(X_chunks[0]).shape[1]
    scale = 1.0 / (1.0 - float(np.float32(p)))
    dZ = [np.where(dropout_keep(hi - lo, d, lo, p, seed, offset), np.asarray(dy, dtype=np.float64) * scale, 0.0)
          for (lo, hi), dy in zip(chunk_ranges(T, N), dY_chunks)]
    g = sp_backward(X_chunks, gamma, beta, eps, A, B, b, dZ, N)
    g["dX_chunks"] = [dx + np.asarray(dy, dtype=np.float64) for dx, dy in zip(g["dX_chunks"], dY_chunks)]
    g["db2"] = sum(z.sum(axis=0) for z in dZ)
    g["dZ_chunks"] = dZ
    return g
