"""Seeded synthetic inputs for the tensor-parallel MLP block.

This module is shared by the tests, the bench and the smoke check.  It holds
no arithmetic of the method itself: only a counter-based random generator,
the bf16 round-to-nearest-even quantisation that turns the draws into the
exact values both the CUDA path and the CPU oracle consume, and the recipe
(shapes and distributions) of each named workload.

Generator: splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) evaluated on the counter ``k`` of each
element, so element ``k`` of a tensor is independent of how the tensor is
generated in blocks.  Two 53-bit uniforms per pair of elements feed the
Box-Muller transform (Box & Muller 1958) to give standard normals.  Each
tensor has its own stream, keyed by FNV-1a-64 of ``"<workload>/<tensor>"``
mixed with the seed.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_BLOCK = 1 << 22


def _fnv1a64(text: str) -> int:
    h = 0xCBF29CE484222325
    for byte in text.encode("utf-8"):
        h ^= byte
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def _splitmix64(z: np.ndarray) -> np.ndarray:
    """The splitmix64 output mix applied to ``state + golden`` (uint64, wrapping)."""
    with np.errstate(over="ignore"):
        z = z + _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def stream_key(seed: int, workload: str, tensor: str) -> int:
    """64-bit key of one tensor's stream."""
    s = np.array([(_fnv1a64(f"{workload}/{tensor}") ^ (seed * 0xD1B54A32D192ED03)) & 0xFFFFFFFFFFFFFFFF],
                 dtype=np.uint64)
    return int(_splitmix64(s)[0])


def uniforms(key: int, start: int, count: int) -> np.ndarray:
    """``count`` doubles in [0, 1): 53-bit uniforms of counters ``start .. start+count-1``."""
    ctr = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = _splitmix64(np.uint64(key) + ctr * _GOLDEN)
    return (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normals(key: int, n: int) -> np.ndarray:
    """``n`` standard normal doubles from the stream ``key`` (Box-Muller, pairs of counters).

    Blocks of counters are independent, so large draws run their blocks on a thread pool (numpy's
    array operations release the interpreter lock); the values do not depend on the block order."""
    out = np.empty(n, dtype=np.float64)
    pairs = (n + 1) // 2

    def block(p0):
        p1 = min(pairs, p0 + _BLOCK)
        u = uniforms(key, 2 * p0, 2 * (p1 - p0))
        u1 = 1.0 - u[0::2]                      # (0, 1]: log is finite
        u2 = u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        th = 2.0 * math.pi * u2
        z = np.empty(2 * (p1 - p0), dtype=np.float64)
        z[0::2] = r * np.cos(th)
        z[1::2] = r * np.sin(th)
        lo = 2 * p0
        hi = min(n, 2 * p1)
        out[lo:hi] = z[: hi - lo]

    starts = range(0, pairs, _BLOCK)
    if len(starts) <= 1:
        for p0 in starts:
            block(p0)
        return out
    import concurrent.futures as cf
    import os

    with cf.ThreadPoolExecutor(max_workers=min(len(starts), os.cpu_count() or 1, 32)) as ex:
        list(ex.map(block, starts))
    return out


# --------------------------------------------------------------------------- bf16 helpers

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16, nearest-even; returns the uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    with np.errstate(over="ignore"):
        rounding = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
        return ((b + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to the float32 values they denote (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


# --------------------------------------------------------------------------- workloads

@dataclass(frozen=True)
class Workload:
    """One named workload: shapes plus the distribution of every tensor.

    ``T`` tokens (rows), hidden size ``d``, FFN width ``F`` (= 4d), ``N`` shards.
    ``sp`` marks the sequence-parallel block (LayerNorm on T/N-row chunks);
    ``backward`` adds an upstream gradient dY.  ``dtype`` is the arithmetic
    type the path computes in.  ``dists`` maps tensor name to
    ``(mean, std)`` of a normal draw, or ``None`` for a tensor that is absent
    (a NULL bias) and ``"zero"`` for an all-zero one.
    """
    name: str
    T: int
    d: int
    F: int
    N: int
    dtype: str = "bf16"
    sp: bool = False
    backward: bool = False
    batch: int = 1
    seq: int = 0
    dists: dict = field(default_factory=dict)

    @property
    def rows_per_chunk(self) -> int:
        return self.T // self.N


_W = 0.02
WORKLOADS = {
    "tiny_fp32_fwd": Workload(
        "tiny_fp32_fwd", T=128, d=64, F=256, N=2, dtype="fp32", batch=1, seq=128,
        dists={"X": (0.0, 1.0), "A": (0.0, _W), "B": (0.0, _W), "bias": "zero"}),
    "gpt2_medium_fwd": Workload(
        "gpt2_medium_fwd", T=4096, d=1024, F=4096, N=8, batch=4, seq=1024,
        dists={"X": (0.0, 1.0), "A": (0.0, _W), "B": (0.0, _W), "bias": (0.0, _W)}),
    "mlp7b_fwd": Workload(
        "mlp7b_fwd", T=8192, d=4096, F=16384, N=8, batch=2, seq=4096,
        dists={"X": (0.0, 1.0), "A": (0.0, _W), "B": (0.0, _W / math.sqrt(2 * 32)), "bias": "zero"}),
    "sp_block_fwd_bwd": Workload(
        "sp_block_fwd_bwd", T=8192, d=4096, F=16384, N=8, sp=True, backward=True, batch=1, seq=8192,
        dists={"X": (0.0, 1.0), "gamma": (1.0, _W), "beta": (0.0, _W), "A": (0.0, _W), "B": (0.0, _W),
               "bias": None, "dY": (0.0, 1.0)}),
    "sp_large_fwd": Workload(
        "sp_large_fwd", T=4096, d=8192, F=32768, N=8, sp=True, batch=1, seq=4096,
        dists={"X": (0.0, 1.0), "gamma": (1.0, _W), "beta": (0.0, _W), "A": (0.0, _W), "B": (0.0, _W),
               "bias": None}),
}


def tensor_shape(w: Workload, name: str) -> tuple:
    return {"X": (w.T, w.d), "A": (w.d, w.F), "B": (w.F, w.d), "bias": (w.F,),
            "gamma": (w.d,), "beta": (w.d,), "dY": (w.T, w.d)}[name]


def draw(w: Workload, name: str, seed: int = 0, rows: np.ndarray | None = None,
         shape: tuple | None = None, dist=None):
    """Draw one tensor of workload ``w``.

    Returns ``None`` for an absent tensor, else ``(bits, values)``: for bf16
    workloads ``bits`` are the uint16 bfloat16 patterns and ``values`` the
    float64 numbers they denote; for fp32 workloads ``bits`` is the float32
    array and ``values`` its float64 widening.  ``rows`` selects a subset of
    rows of a 2-D tensor (element counters are those of the full tensor, so a
    sample equals the matching rows of the whole).
    """
    dist = w.dists.get(name) if dist is None else dist
    shape = tensor_shape(w, name) if shape is None else shape
    if dist is None:
        return None
    key = stream_key(seed, w.name, name)
    if dist == "zero":
        raw = np.zeros(shape, dtype=np.float64)
    elif rows is None:
        n = int(np.prod(shape))
        mean, std = dist
        raw = (mean + std * normals(key, n)).reshape(shape)
    else:
        mean, std = dist
        cols = shape[1]
        out = np.empty((len(rows), cols), dtype=np.float64)
        for j, r in enumerate(rows):
            out[j] = _row_normals(key, int(r), cols)
        raw = mean + std * out
    f32 = raw.astype(np.float32)
    if w.dtype == "fp32":
        return f32, f32.astype(np.float64)
    bits = f32_to_bf16_bits(f32).reshape(f32.shape)
    return bits, bf16_bits_to_f64(bits).reshape(f32.shape)


def _row_normals(key: int, row: int, cols: int) -> np.ndarray:
    """Normals of elements ``row*cols .. row*cols+cols-1`` of a stream."""
    start = row * cols
    p0 = start // 2
    p1 = (start + cols + 1) // 2
    u = uniforms(key, 2 * p0, 2 * (p1 - p0))
    u1 = 1.0 - u[0::2]
    r = np.sqrt(-2.0 * np.log(u1))
    th = 2.0 * math.pi * u[1::2]
    z = np.empty(2 * (p1 - p0), dtype=np.float64)
    z[0::2] = r * np.cos(th)
    z[1::2] = r * np.sin(th)
    off = start - 2 * p0
    return z[off: off + cols]


def small_workload(T: int, d: int, N: int, *, F: int | None = None, sp: bool = False,
                   backward: bool = False, bias=(0.0, _W), name: str | None = None,
                   dtype: str = "bf16") -> Workload:
    """A reduced-size workload with the same distributions as the full ones."""
    F = 4 * d if F is None else F
    dists = {"X": (0.0, 1.0), "A": (0.0, _W), "B": (0.0, _W), "bias": bias}
    if sp:
        dists.update({"gamma": (1.0, _W), "beta": (0.0, _W)})
    if backward:
        dists["dY"] = (0.0, 1.0)
    return Workload(name or f"small_T{T}_d{d}_F{F}_N{N}", T=T, d=d, F=F, N=N, dtype=dtype,
                    sp=sp, backward=backward, seq=T, dists=dists)
