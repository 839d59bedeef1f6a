// HBM-bound row kernels of the sequence-parallel block:
//   LayerNorm of each S/N chunk written straight into its row slot of the
//   gathered activation (the All-Gather is a layout, not a copy);
//   LayerNorm backward per chunk with deterministic dgamma/dbeta partials;
//   the explicit Reduce-Scatter over per-shard bf16 partials;
//   a row gather and a fixed-order column sum.
// All global traffic is 16-byte vectors; reductions are warp shuffles.
#include <cuda_bf16.h>

#include <atomic>

#include "debug_bounds.cuh"
#include "fp8.cuh"
#include "launch.h"
#include "philox.cuh"
#include "ptx.cuh"

namespace tpmlp {
namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z), d = unpack_bf16x2(u.w);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y; f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

// The two bf16 values of a 32-bit word as a float pair (low half first), and word w of a 16-byte vector.
__device__ __forceinline__ float2 bf2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ uint32_t word(const uint4& u, int w) { return w == 0 ? u.x : w == 1 ? u.y : w == 2 ? u.z : u.w; }

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// Row `row` of the chunked input (a debug build that finds the row or its chunk out of range counts it and
// reads the first row instead).
__device__ __forceinline__ const __nv_bfloat16* chunk_row(const RowParams& p, int row) {
  int j = row / p.rows_per_chunk;
  if (!(TPMLP_IN_BOUNDS(row, p.rows, kBoundsInChunk) && TPMLP_IN_BOUNDS(j, p.n_chunks, kBoundsInChunk))) j = row = 0;
  return static_cast<const __nv_bfloat16*>(p.in_chunks.p[j]) +
         static_cast<long long>(row - j * p.rows_per_chunk) * p.d;
}

__device__ __forceinline__ const __nv_bfloat16* add_chunk_row(const RowParams& p, int row) {
  int j = row / p.rows_per_chunk;
  if (!(TPMLP_IN_BOUNDS(row, p.rows, kBoundsAddChunk) && TPMLP_IN_BOUNDS(j, p.n_chunks, kBoundsAddChunk))) j = row = 0;
  return static_cast<const __nv_bfloat16*>(p.add_chunks.p[j]) +
         static_cast<long long>(row - j * p.rows_per_chunk) * p.d;
}

// Debug builds: is 16-byte vector `v` of row `row` inside a [rows x d] tensor (a store is skipped if not)?
__device__ __forceinline__ bool row_vec_ok(const RowParams& p, long long row, long long v, uint32_t site) {
  return TPMLP_IN_BOUNDS(row, p.rows, site) && TPMLP_IN_BOUNDS(v, p.d / 8, site);
}

// The sequence-parallel tail on 8 elements of vector q (= element index / 8) of row `row`, column `col`.
__device__ __forceinline__ void sp_tail_8(const RowParams& p, float (&a)[8], long long q, int row, int col) {
  if (p.bias2 != nullptr) {
    float b[8];
    unpack8(__ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.bias2) + col)), b);
#pragma unroll
    for (int e = 0; e < 8; ++e) a[e] += b[e];
  }
  uint32_t m = 0xFFu;
  if (p.drop_thr < kKeepAll) {
    m = dropout_keep8(static_cast<unsigned long long>(q), p.drop_offset, p.drop_seed, p.drop_thr);
    if (p.drop_mask != nullptr) p.drop_mask[q] = static_cast<uint8_t>(m);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) a[e] = (m >> e) & 1u ? a[e] * p.drop_scale : 0.f;
  if (p.add_chunks.p[0] != nullptr) {
    float r[8];
    unpack8(__ldg(reinterpret_cast<const uint4*>(add_chunk_row(p, row) + col)), r);
#pragma unroll
    for (int e = 0; e < 8; ++e) a[e] += r[e];
  }
}

// Row `row` of the chunked output; the stores through it check the row (row_vec_ok), this checks the chunk.
__device__ __forceinline__ __nv_bfloat16* out_chunk_row(const RowParams& p, int row) {
  int j = row / p.rows_per_chunk;
  if (!TPMLP_IN_BOUNDS(j, p.n_chunks, kBoundsOutChunk)) j = row = 0;
  return static_cast<__nv_bfloat16*>(p.out_chunks.p[j]) + static_cast<long long>(row - j * p.rows_per_chunk) * p.d;
}

// ----------------------------------------------------------------------------- LayerNorm forward

// WPR warps per row, the row held in registers: V 16-byte vectors per lane
// (d = 256 V WPR).  Mean first, then the biased variance from the centred
// values (two passes over registers), rstd = rsqrt(var + eps), one bf16
// rounding at the output.
// Warp sums of two values in five shuffles (lanes 0-15 end with a's, 16-31 with b's) and two broadcasts.
__device__ __forceinline__ float2 warp_sum2(float a, float b) {
  const bool hi = (threadIdx.x & 16) != 0;
  float v = (hi ? b : a) + __shfl_xor_sync(0xffffffffu, hi ? a : b, 16);
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return make_float2(__shfl_sync(0xffffffffu, v, 0), __shfl_sync(0xffffffffu, v, 16));
}

// Row sums of two values over the WPR warps of a row (all threads of the block call it).
template <int V, int WPR>
__device__ __forceinline__ float2 row_sum2(float a, float b, float2* red2, int warp) {
  float2 v = warp_sum2(a, b);
  if constexpr (WPR == 1) {
    return v;
  } else {
    if ((threadIdx.x & 31) == 0) red2[warp] = v;
    __syncthreads();
    float2 t = make_float2(0.f, 0.f);
    const int first = warp - warp % WPR;
#pragma unroll
    for (int k = 0; k < WPR; ++k) {
      t.x += red2[first + k].x;
      t.y += red2[first + k].y;
    }
    __syncthreads();
    return t;
  }
}

template <int V, int WPR>
__device__ __forceinline__ float row_sum(float v, float* red, int warp) {
  v = warp_sum(v);
  if constexpr (WPR == 1) {
    return v;
  } else {
    if ((threadIdx.x & 31) == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
    const int first = warp - warp % WPR;
#pragma unroll
    for (int k = 0; k < WPR; ++k) t += red[first + k];
    __syncthreads();
    return t;
  }
}

// RMS = true: the norm of the SequenceParallelLayerNorm listing instead:
// rstd = rsqrt(mean(x^2) + eps), n = bf16(x rstd), y = bf16(n * gamma).
// Q8 = true: the fp32 LayerNorm value y is written as E4M3(y * (*p.qscale)) (one byte) and max |y| is
// max-combined into *p.amax.
// A warp holds its row (V 16-byte vectors per lane) in registers; at V = 16 the register count is held to
// what kLnRegMinBlocks resident blocks allow, so enough rows are in flight to cover the memory latency.
constexpr int kLnRegMinBlocks = 4;

template <int V, int WPR, bool RMS = false, bool Q8 = false>
__global__ void __launch_bounds__(128, V >= 16 ? kLnRegMinBlocks : 1) k_layernorm_fwd_reg(const RowParams p) {
  __shared__ float red[4];
  __shared__ float2 red2[4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * static_cast<int>(blockDim.x >> 5) / WPR + warp / WPR;
  const int sub = warp % WPR;
  const bool valid = row < p.rows;
  const uint4* src = valid ? reinterpret_cast<const uint4*>(chunk_row(p, row)) : nullptr;
  uint4 x[V];
#pragma unroll
  for (int v = 0; v < V; ++v) x[v] = valid ? __ldg(src + (sub * V + v) * 32 + lane) : make_uint4(0, 0, 0, 0);
  float mean = 0.f, rstd;
  if constexpr (!RMS) {
    // Shifted sums (K = the row's first element): Σc and Σc² of c = x - K in one reduction round give
    // mean = K + Σc/d and var = Σc²/d - (Σc/d)², without the cancellation of E[x²] - mean² when the mean
    // is large against the spread.
    const float K = valid ? __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(src))) << 16)
                          : 0.f;
    const float2 nk = make_float2(-K, -K);
    float2 s1 = make_float2(0.f, 0.f), s2 = s1;
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float2 c = __fadd2_rn(bf2(word(x[v], w)), nk);
        s1 = __fadd2_rn(s1, c);
        s2 = __ffma2_rn(c, c, s2);
      }
    const float2 t = row_sum2<V, WPR>(s1.x + s1.y, s2.x + s2.y, red2, warp);
    const float m = t.x / static_cast<float>(p.d);
    mean = K + m;
    rstd = rsqrtf(fmaxf(t.y / static_cast<float>(p.d) - m * m, 0.f) + p.eps);
  } else {
    float q = 0.f;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      float f[8];
      unpack8(x[v], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) q += f[e] * f[e];
    }
    rstd = rsqrtf(row_sum<V, WPR>(q, red, warp) / static_cast<float>(p.d) + p.eps);
  }
  const uint4* g4 = reinterpret_cast<const uint4*>(p.gamma);
  const uint4* b4 = reinterpret_cast<const uint4*>(p.beta);
  const long long row_off = static_cast<long long>(valid ? row : 0) * p.d;
  uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dst) + row_off);
  uint2* dst8 = reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.dst) + row_off);
  float qs = 1.f, amax = 0.f;
  if constexpr (Q8) qs = __ldg(p.qscale);
  if (valid) {
    const float2 nm = make_float2(-mean, -mean), r2 = make_float2(rstd, rstd);
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int idx = (sub * V + v) * 32 + lane;
      const uint4 gv = __ldg(g4 + idx);
      float o[8];
      if constexpr (RMS) {
        float f[8], g[8];
        unpack8(x[v], f);
        unpack8(gv, g);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = __bfloat162float(__float2bfloat16_rn(f[e] * rstd)) * g[e];
      } else {
        // (x - mean) rstd γ + β on float pairs
        const uint4 bv = __ldg(b4 + idx);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float2 y = __ffma2_rn(__fmul2_rn(__fadd2_rn(bf2(word(x[v], w)), nm), r2), bf2(word(gv, w)),
                                      bf2(word(bv, w)));
          o[2 * w] = y.x;
          o[2 * w + 1] = y.y;
        }
      }
      if constexpr (Q8) {
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(o[e]));
        if (row_vec_ok(p, row, idx, kBoundsRowStore)) dst8[idx] = e4m3x8(o, qs);
      } else {
        if (row_vec_ok(p, row, idx, kBoundsRowStore)) dst[idx] = pack8(o);
      }
    }
  }
  if constexpr (Q8) amax_combine_warp(p.amax, amax);
}

// LayerNorm forward, persistent and software-pipelined: each warp owns rows w, w + W, w + 2W, ...
// (W = warps in the grid) and holds two rows in registers, loading the next while it normalises the
// current, so the loads of the whole SM stay in flight while it computes (a launch-per-row-group kernel
// instead idles the memory system during each group's compute phase).  d = 256 V.
template <int V>
__device__ __forceinline__ void ln_row_load(const RowParams& p, int row, int lane, uint4 (&x)[V]) {
  if (row < p.rows) {
    const uint4* src = reinterpret_cast<const uint4*>(chunk_row(p, row));
#pragma unroll
    for (int v = 0; v < V; ++v) x[v] = __ldg(src + v * 32 + lane);
  }
}

template <int V>
__device__ __forceinline__ void ln_row_store(const RowParams& p, int row, int lane, const uint4 (&x)[V],
                                             const uint4* g4, const uint4* b4) {
  float s = 0.f;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    float f[8];
    unpack8(x[v], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) s += f[e];
  }
  const float mean = warp_sum(s) / static_cast<float>(p.d);
  float q = 0.f;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    float f[8];
    unpack8(x[v], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float c = f[e] - mean;
      q += c * c;
    }
  }
  const float rstd = rsqrtf(warp_sum(q) / static_cast<float>(p.d) + p.eps);
  uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dst) + static_cast<long long>(row) * p.d);
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int idx = v * 32 + lane;
    float f[8], g[8], b[8], o[8];
    unpack8(x[v], f);
    unpack8(g4[idx], g);
    unpack8(b4[idx], b);
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = (f[e] - mean) * rstd * g[e] + b[e];
    if (row_vec_ok(p, row, idx, kBoundsRowStore)) dst[idx] = pack8(o);
  }
}

template <int V>
__global__ void __launch_bounds__(128) k_layernorm_fwd_pipe(const RowParams p) {
  __shared__ uint4 gbs[2 * 32 * V];  // gamma, beta
  for (int i = threadIdx.x; i < 32 * V; i += blockDim.x) {
    gbs[i] = __ldg(reinterpret_cast<const uint4*>(p.gamma) + i);
    gbs[32 * V + i] = __ldg(reinterpret_cast<const uint4*>(p.beta) + i);
  }
  __syncthreads();
  const uint4* g4 = gbs;
  const uint4* b4 = gbs + 32 * V;
  const int lane = threadIdx.x & 31;
  const int W = gridDim.x * (blockDim.x >> 5);
  int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  uint4 a[V], b[V];
  ln_row_load<V>(p, row, lane, a);
  // two rows per trip so that the two register sets keep fixed roles
  while (row < p.rows) {
    ln_row_load<V>(p, row + W, lane, b);
    ln_row_store<V>(p, row, lane, a, g4, b4);
    row += W;
    if (row >= p.rows) break;
    ln_row_load<V>(p, row + W, lane, a);
    ln_row_store<V>(p, row, lane, b, g4, b4);
    row += W;
  }
}

// The same with two warps per row (warps 2k and 2k + 1 of a block, each 128 V columns of the 256 V):
// the row statistics combine through shared memory and a named barrier per warp pair, double-buffered by
// row parity.  d = 512 V.
template <int V>
__device__ __forceinline__ void ln_half_load(const RowParams& p, int row, int half, int lane, uint4 (&x)[V]) {
  if (row < p.rows) {
    const uint4* src = reinterpret_cast<const uint4*>(chunk_row(p, row)) + half * 32 * V;
#pragma unroll
    for (int v = 0; v < V; ++v) x[v] = __ldg(src + v * 32 + lane);
  }
}

template <int V>
__device__ __forceinline__ void ln_half_store(const RowParams& p, int row, int half, int pair, int lane, int par,
                                              const uint4 (&x)[V], const uint4* g4, const uint4* b4,
                                              float (*red)[4][2]) {
  const int bar = 1 + pair;
  float s = 0.f;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    float f[8];
    unpack8(x[v], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) s += f[e];
  }
  s = warp_sum(s);
  if (lane == 0) red[par][pair * 2 + half][0] = s;
  asm volatile("bar.sync %0, 64;" ::"r"(bar) : "memory");
  const float mean = (red[par][pair * 2][0] + red[par][pair * 2 + 1][0]) / static_cast<float>(p.d);
  float q = 0.f;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    float f[8];
    unpack8(x[v], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float c = f[e] - mean;
      q += c * c;
    }
  }
  q = warp_sum(q);
  if (lane == 0) red[par][pair * 2 + half][1] = q;
  asm volatile("bar.sync %0, 64;" ::"r"(bar) : "memory");
  const float rstd = rsqrtf((red[par][pair * 2][1] + red[par][pair * 2 + 1][1]) / static_cast<float>(p.d) + p.eps);
  uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dst) + static_cast<long long>(row) * p.d) +
               half * 32 * V;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int idx = half * 32 * V + v * 32 + lane;
    float f[8], g[8], b[8], o[8];
    unpack8(x[v], f);
    unpack8(g4[idx], g);
    unpack8(b4[idx], b);
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = (f[e] - mean) * rstd * g[e] + b[e];
    if (row_vec_ok(p, row, idx, kBoundsRowStore)) dst[v * 32 + lane] = pack8(o);
  }
}

template <int V>
__global__ void __launch_bounds__(128) k_layernorm_fwd_pipe2(const RowParams p) {
  __shared__ uint4 gbs[2 * 64 * V];   // gamma, beta
  __shared__ float red[2][4][2];      // [row parity][warp][sum, centred sum of squares]
  for (int i = threadIdx.x; i < 64 * V; i += blockDim.x) {
    gbs[i] = __ldg(reinterpret_cast<const uint4*>(p.gamma) + i);
    gbs[64 * V + i] = __ldg(reinterpret_cast<const uint4*>(p.beta) + i);
  }
  __syncthreads();
  const uint4* g4 = gbs;
  const uint4* b4 = gbs + 64 * V;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = warp >> 1, half = warp & 1;
  const int W = gridDim.x * (blockDim.x >> 6);  // warp pairs in the grid
  int row = blockIdx.x * (blockDim.x >> 6) + pair;
  uint4 a[V], b[V];
  ln_half_load<V>(p, row, half, lane, a);
  int par = 0;
  // both warps of a pair see the same rows, so they leave the loop together (the barriers stay matched)
  while (row < p.rows) {
    ln_half_load<V>(p, row + W, half, lane, b);
    ln_half_store<V>(p, row, half, pair, lane, par, a, g4, b4, red);
    row += W;
    par ^= 1;
    if (row >= p.rows) break;
    ln_half_load<V>(p, row + W, half, lane, a);
    ln_half_store<V>(p, row, half, pair, lane, par, b, g4, b4, red);
    row += W;
    par ^= 1;
  }
}

// Any d that is a multiple of 8: one warp per row, three sweeps over the row
// (the second and third hit L1/L2).
template <bool RMS = false>
__global__ void __launch_bounds__(128) k_layernorm_fwd_any(const RowParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + warp;
  if (row >= p.rows) return;
  const int nv = p.d / 8;
  const uint4* src = reinterpret_cast<const uint4*>(chunk_row(p, row));
  float mean = 0.f;
  if constexpr (!RMS) {
    float s = 0.f;
    for (int v = lane; v < nv; v += 32) {
      float f[8];
      unpack8(__ldg(src + v), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) s += f[e];
    }
    mean = warp_sum(s) / static_cast<float>(p.d);
  }
  float q = 0.f;
  for (int v = lane; v < nv; v += 32) {
    float f[8];
    unpack8(__ldg(src + v), f);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float c = f[e] - mean;
      q += c * c;
    }
  }
  const float rstd = rsqrtf(warp_sum(q) / static_cast<float>(p.d) + p.eps);
  const uint4* g4 = reinterpret_cast<const uint4*>(p.gamma);
  const uint4* b4 = reinterpret_cast<const uint4*>(p.beta);
  uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dst) + static_cast<long long>(row) * p.d);
  for (int v = lane; v < nv; v += 32) {
    float f[8], g[8], o[8];
    unpack8(__ldg(src + v), f);
    unpack8(__ldg(g4 + v), g);
    if constexpr (RMS) {
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = __bfloat162float(__float2bfloat16_rn(f[e] * rstd)) * g[e];
    } else {
      float b[8];
      unpack8(__ldg(b4 + v), b);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = (f[e] - mean) * rstd * g[e] + b[e];
    }
    if (row_vec_ok(p, row, v, kBoundsRowStore)) dst[v] = pack8(o);
  }
}

// ----------------------------------------------------------------------------- LayerNorm backward

// Rows in groups of 8 (one warp each), grid-stride.  Phase 1 (per warp):
// mean, rstd, mean(g) and mean(g * xhat) with g = dy * gamma, then
// dx = rstd * (g - mean(g) - xhat * mean(g * xhat)) to the row's chunk.
// Phase 2 (per thread, its own columns): dgamma += dy * xhat, dbeta += dy,
// accumulated in shared memory without atomics; each block finally writes
// its [2 d] partial row, which a fixed-order column sum reduces.
constexpr int kLnBwdRowsPerGroup = 8;

__global__ void __launch_bounds__(256) k_layernorm_bwd(const RowParams p) {
  extern __shared__ float acc[];  // [2 d]: dgamma, dbeta
  __shared__ float s_mean[kLnBwdRowsPerGroup], s_rstd[kLnBwdRowsPerGroup];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nv = p.d / 8;
  for (int c = threadIdx.x; c < 2 * p.d; c += blockDim.x) acc[c] = 0.f;
  const uint4* g4 = reinterpret_cast<const uint4*>(p.gamma);
  const int groups = (p.rows + kLnBwdRowsPerGroup - 1) / kLnBwdRowsPerGroup;
  for (int grp = blockIdx.x; grp < groups; grp += gridDim.x) {
    const int row = grp * kLnBwdRowsPerGroup + warp;
    if (row < p.rows) {
      const uint4* x4 = reinterpret_cast<const uint4*>(chunk_row(p, row));
      const uint4* dy4 = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.src) +
                                                        static_cast<long long>(row) * p.d);
      float s = 0.f;
      for (int v = lane; v < nv; v += 32) {
        float f[8];
        unpack8(__ldg(x4 + v), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) s += f[e];
      }
      const float mean = warp_sum(s) / static_cast<float>(p.d);
      float q = 0.f, sg = 0.f, sgc = 0.f;
      for (int v = lane; v < nv; v += 32) {
        float f[8], dy[8], g[8];
        unpack8(__ldg(x4 + v), f);
        unpack8(__ldg(dy4 + v), dy);
        unpack8(__ldg(g4 + v), g);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float c = f[e] - mean;
          const float gg = dy[e] * g[e];
          q += c * c;
          sg += gg;
          sgc += gg * c;
        }
      }
      q = warp_sum(q);
      sg = warp_sum(sg);
      sgc = warp_sum(sgc);
      const float rstd = rsqrtf(q / static_cast<float>(p.d) + p.eps);
      const float m1 = sg / static_cast<float>(p.d);
      const float m2 = rstd * sgc / static_cast<float>(p.d);
      uint4* dx4 = reinterpret_cast<uint4*>(out_chunk_row(p, row));
      for (int v = lane; v < nv; v += 32) {
        float f[8], dy[8], g[8], o[8];
        unpack8(__ldg(x4 + v), f);
        unpack8(__ldg(dy4 + v), dy);
        unpack8(__ldg(g4 + v), g);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = rstd * (dy[e] * g[e] - m1 - (f[e] - mean) * rstd * m2);
        if (p.add_chunks.p[0] != nullptr) {
          float a[8];
          unpack8(__ldg(reinterpret_cast<const uint4*>(add_chunk_row(p, row)) + v), a);
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] += a[e];
        }
        if (row_vec_ok(p, row, v, kBoundsOutChunk)) dx4[v] = pack8(o);
      }
      if (lane == 0) {
        s_mean[warp] = mean;
        s_rstd[warp] = rstd;
      }
    }
    __syncthreads();
    const int rows_here = min(kLnBwdRowsPerGroup, p.rows - grp * kLnBwdRowsPerGroup);
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
      float dg[8], db[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) dg[e] = db[e] = 0.f;
      for (int r = 0; r < rows_here; ++r) {
        const int row = grp * kLnBwdRowsPerGroup + r;
        float f[8], dy[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(chunk_row(p, row)) + v), f);
        unpack8(__ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.src) +
                                                     static_cast<long long>(row) * p.d) + v), dy);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          dg[e] += dy[e] * (f[e] - s_mean[r]) * s_rstd[r];
          db[e] += dy[e];
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        acc[v * 8 + e] += dg[e];
        acc[p.d + v * 8 + e] += db[e];
      }
    }
    __syncthreads();
  }
  for (int c = threadIdx.x; c < 2 * p.d; c += blockDim.x)
    p.partial[static_cast<long long>(blockIdx.x) * 2 * p.d + c] = acc[c];
}

// ----------------------------------------------------------------------------- streamed row kernels
//
// Persistent CTAs (one per SM).  Warp 0 is the producer: one lane streams the
// CTA's rows (row blockIdx.x + i * gridDim.x for i = 0, 1, ...) into a ring of
// shared-memory slots with 1-D bulk copies, completion counted on `full[slot]`.
// Warps 1..8 are consumers: consumer c takes rows i = c, c + 8, ..., copies
// the row from its slot into registers (V 16-byte vectors per lane), frees the
// slot (`empty[slot]`) and computes.  Every wait is bounded.

constexpr int kStreamConsumers = 8;
constexpr int kStreamThreads = 32 * (kStreamConsumers + 1);

__device__ __forceinline__ uint8_t* align128(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 127) & ~uintptr_t(127));
}

// Producer loop shared by the streamed kernels: `copies` rows of `row_bytes`
// per slot (the second, if any, from `src2` rows of the same index).
__device__ __forceinline__ void stream_producer(const RowParams& p, uint8_t* ring, uint32_t slot_bytes,
                                                uint32_t row_bytes, uint64_t* full, uint64_t* empty, int n_rows,
                                                const WaitCtx& wc, bool second) {
  uint32_t issued_mask = 0, issued_parity = 0;
  for (int i = 0; i < n_rows; ++i) {
    const int slot = i % p.slots;
    const uint32_t ph = static_cast<uint32_t>(i / p.slots) & 1u;
    if (!wait_bounded(empty + slot, ph ^ 1u, wc, kSiteRowProducer)) break;
    const int row = blockIdx.x + i * gridDim.x;
    mbar_arrive_expect_tx(full + slot, second ? 2 * row_bytes : row_bytes);
    bulk_load(ring + slot * slot_bytes, chunk_row(p, row), row_bytes, full + slot);
    if (second)
      bulk_load(ring + slot * slot_bytes + row_bytes,
                static_cast<const __nv_bfloat16*>(p.src) +
                    static_cast<long long>(TPMLP_IN_BOUNDS(row, p.rows, kBoundsRowLoad) ? row : 0) * p.d,
                row_bytes, full + slot);
    if (slot < 32) {
      issued_mask |= 1u << slot;
      issued_parity = (issued_parity & ~(1u << slot)) | (ph << slot);
    }
  }
  // copies in flight must land before the CTA exits
  for (int s = 0; s < p.slots && s < 32; ++s)
    if (issued_mask & (1u << s)) wait_drain(full + s, (issued_parity >> s) & 1u, p.timeout_ns);
}

// The ring's phase parity is one bit, so a consumer must never wait on a slot while that slot's previous
// row is still unconsumed by someone else: each slot has to belong to one team, which takes its rows in
// order.  Rows go to slot i % slots and to team i % teams, so that holds exactly when slots is a multiple
// of teams.  A CTA given any other count records kErrConfig and returns before it touches memory.
__device__ __forceinline__ bool ring_config_ok(const RowParams& p, int teams) {
  if (p.slots >= teams && p.slots % teams == 0 && p.slots <= 32) return true;
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    atomicOr(p.err, kErrConfig);
    atomicCAS(p.err + 1, 0u, kSiteRowConfig);
  }
  return false;
}

__device__ __forceinline__ bool stream_wait(uint64_t* bar, uint32_t parity, const WaitCtx& wc) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = wait_bounded(bar, parity, wc, kSiteRowConsumer) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// LayerNorm backward in one pass over x and dy.  Teams of TW warps (CONS / TW
// teams per CTA) each take one row of the ring at a time; thread j of a team
// owns the 16-byte column vectors j + k·32·TW, k < VT (d = 256 TW VT).
// Row statistics in one reduction round from shifted sums: with K the row's
// first element and c = x - K, S1 = Σc, S2 = Σc², Sg = Σg, Sgc = Σg·c
// (g = dy·γ) give mean = K + S1/d, var = S2/d - (S1/d)² and
// Σ g·(x - mean) = Sgc - (S1/d)·Sg; the shift by a sample of the row keeps the
// variance free of the cancellation that E[x²] - mean² suffers when the mean
// is large against the spread.  Arithmetic on float pairs (the packed fp32
// instructions); c stays in registers for the output pass, or (RR) is formed
// again from the slot's x, which the team then reads twice.  dx goes to the
// row's chunk; dγ and dβ for the thread's columns accumulate in registers over
// all rows the team processes, and at the end the teams' sums are added in
// team order into the CTA's partial row [2 d], which a fixed-order column sum
// reduces.
__device__ __forceinline__ void team_sync(int team, int tw) {
  if (tw == 1) {
    __syncwarp();
  } else {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(32 * tw) : "memory");
  }
}

// Warp sums of four values in six shuffles: afterwards lane l holds the sum of value (l >> 3) & 3 (a for
// lanes 0-7, b for 8-15, c for 16-23, d for 24-31).
__device__ __forceinline__ float warp_sum4(float a, float b, float c, float d) {
  const int lane = threadIdx.x & 31;
  const bool hi16 = (lane & 16) != 0;
  const float k0 = (hi16 ? c : a) + __shfl_xor_sync(0xffffffffu, hi16 ? a : c, 16);
  const float k1 = (hi16 ? d : b) + __shfl_xor_sync(0xffffffffu, hi16 ? b : d, 16);
  const bool hi8 = (lane & 8) != 0;
  float v = (hi8 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, hi8 ? k0 : k1, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v;
}

// ADD: dx += the rows of p.add_chunks (the residual's gradient), loaded while the row statistics reduce.
// CONS consumer warps (one more warp produces).  RR: the output pass reads x and dy from the row's slot a
// second time instead of keeping them (and x - K) in registers, and the slot is freed after that pass; the
// registers saved let more consumer warps share an SM.
template <int VT, int TW, bool ADD = false, int CONS = kStreamConsumers, bool RR = false>
__global__ void __launch_bounds__(32 * (CONS + 1), 1) k_layernorm_bwd_fused(const RowParams p) {
  constexpr int kTeams = CONS / TW;
  if (!ring_config_ok(p, kTeams)) return;  // uniform over the CTA: no barrier is left waiting
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = align128(smem_raw);
  const uint32_t row_bytes = static_cast<uint32_t>(p.d) * 2u;
  uint4* gam = reinterpret_cast<uint4*>(ring + p.slots * 2 * row_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(gam + p.d / 8);
  uint64_t* empty = full + p.slots;
  int* abort_flag = reinterpret_cast<int*>(empty + p.slots);
  __shared__ float4 red4[2][CONS];
  __shared__ int vote[2][CONS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.slots; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, TW);
    }
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};
  const int n_rows = p.rows > static_cast<int>(blockIdx.x)
                         ? (p.rows - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) / gridDim.x
                         : 0;
  const int cw = warp - 1;        // consumer warp index
  const int team = cw / TW;
  const int tw = cw % TW;         // warp within the team
  const int j = tw * 32 + lane;   // thread within the team
  float2 dg[VT][4], db[VT][4];
#pragma unroll
  for (int k = 0; k < VT; ++k)
#pragma unroll
    for (int w = 0; w < 4; ++w) dg[k][w] = db[k][w] = make_float2(0.f, 0.f);
  if (warp == 0) {
    if (lane == 0) stream_producer(p, ring, 2 * row_bytes, row_bytes, full, empty, n_rows, wc, true);
  } else {
    // γ is staged by the consumer warps while the producer's first copies are in flight (measured on GB300 at
    // T = 8192, d = 4096: 0.0472 -> 0.0459 ms); named barrier 1 + kTeams (the teams use 1 .. kTeams)
    for (int i = threadIdx.x - 32; i < p.d / 8; i += 32 * CONS)
      gam[i] = __ldg(reinterpret_cast<const uint4*>(p.gamma) + i);
    asm volatile("bar.sync %0, %1;" ::"r"(1 + kTeams), "r"(32 * CONS) : "memory");
    const float inv_d = 1.f / static_cast<float>(p.d);
    int parity_buf = 0;
    for (int i = team; i < n_rows; i += kTeams, parity_buf ^= 1) {
      const int slot = i % p.slots;
      // Every warp of the team waits (bounded) on its own; the outcomes are voted at the team barrier, so
      // the team leaves the loop together and no warp is left waiting at a barrier.
      const bool ok = stream_wait(full + slot, static_cast<uint32_t>(i / p.slots) & 1u, wc);
      const uint4* xs = reinterpret_cast<const uint4*>(ring + slot * 2 * row_bytes);
      const uint4* ds = reinterpret_cast<const uint4*>(ring + slot * 2 * row_bytes + row_bytes);
      uint4 xv[RR ? 1 : VT], dv[RR ? 1 : VT];
      if constexpr (!RR) {
#pragma unroll
        for (int k = 0; k < VT; ++k) {
          xv[k] = ok ? xs[j + k * 32 * TW] : make_uint4(0, 0, 0, 0);
          dv[k] = ok ? ds[j + k * 32 * TW] : make_uint4(0, 0, 0, 0);
        }
      }
      const float shift = ok ? __uint_as_float(xs[0].x << 16) : 0.f;  // the row's first element
      if constexpr (!RR) {
        __syncwarp();
        if (lane == 0 && ok) mbar_arrive(empty + slot);
      }
      uint4 av[VT];
      if constexpr (ADD) {
        const uint4* a4 = reinterpret_cast<const uint4*>(add_chunk_row(p, blockIdx.x + i * gridDim.x));
#pragma unroll
        for (int k = 0; k < VT; ++k) av[k] = ok ? __ldg(a4 + j + k * 32 * TW) : make_uint4(0, 0, 0, 0);
      }
      const float2 nk = make_float2(-shift, -shift);
      float2 s1 = make_float2(0.f, 0.f), s2 = s1, sg = s1, sgc = s1;
      float2 c[RR ? 1 : VT][4];
#pragma unroll
      for (int k = 0; k < VT; ++k) {
        const uint4 gk = gam[j + k * 32 * TW];
        const uint4 xk = RR ? (ok ? xs[j + k * 32 * TW] : make_uint4(0, 0, 0, 0)) : xv[RR ? 0 : k];
        const uint4 dk = RR ? (ok ? ds[j + k * 32 * TW] : make_uint4(0, 0, 0, 0)) : dv[RR ? 0 : k];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float2 ck = __fadd2_rn(bf2(word(xk, w)), nk);
          if constexpr (!RR) c[k][w] = ck;
          const float2 g = __fmul2_rn(bf2(word(dk, w)), bf2(word(gk, w)));
          s1 = __fadd2_rn(s1, ck);
          s2 = __ffma2_rn(ck, ck, s2);
          sg = __fadd2_rn(sg, g);
          sgc = __ffma2_rn(g, ck, sgc);
        }
      }
      const float v = warp_sum4(s1.x + s1.y, s2.x + s2.y, sg.x + sg.y, sgc.x + sgc.y);
      float4 t;
      bool team_ok = ok;
      if (TW > 1) {
        if ((lane & 7) == 0) reinterpret_cast<float*>(&red4[parity_buf][cw])[lane >> 3] = v;
        if (lane == 0) vote[parity_buf][cw] = ok ? 1 : 0;
        team_sync(team, TW);
        t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < TW; ++w) {
          const float4 r = red4[parity_buf][team * TW + w];
          t.x += r.x;
          t.y += r.y;
          t.z += r.z;
          t.w += r.w;
          team_ok = team_ok && vote[parity_buf][team * TW + w] != 0;
        }
      } else {
        t = make_float4(__shfl_sync(0xffffffffu, v, 0), __shfl_sync(0xffffffffu, v, 8),
                        __shfl_sync(0xffffffffu, v, 16), __shfl_sync(0xffffffffu, v, 24));
      }
      if (!team_ok) break;
      const float m = t.x * inv_d;                               // mean - K
      const float rstd = rsqrtf(fmaxf(t.y * inv_d - m * m, 0.f) + p.eps);
      const float m1 = t.z * inv_d;                              // mean(g)
      const float m2 = rstd * (t.w - m * t.z) * inv_d;           // rstd mean(g (x - mean))
      const float2 r2 = make_float2(rstd, rstd);
      const float2 nmr = make_float2(-m * rstd, -m * rstd);      // xhat = c rstd - m rstd
      const float2 nm1r = make_float2(-m1 * rstd, -m1 * rstd);   // dx = g rstd - m1 rstd - xhat m2 rstd
      const float2 nm2r = make_float2(-m2 * rstd, -m2 * rstd);
      const int row = blockIdx.x + i * gridDim.x;
      uint4* dx4 = reinterpret_cast<uint4*>(out_chunk_row(p, row));
#pragma unroll
      for (int k = 0; k < VT; ++k) {
        const uint4 gk = gam[j + k * 32 * TW];
        const uint4 xk = RR ? (ok ? xs[j + k * 32 * TW] : make_uint4(0, 0, 0, 0)) : xv[RR ? 0 : k];
        const uint4 dk = RR ? (ok ? ds[j + k * 32 * TW] : make_uint4(0, 0, 0, 0)) : dv[RR ? 0 : k];
        uint32_t o[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float2 ck = RR ? __fadd2_rn(bf2(word(xk, w)), nk) : c[RR ? 0 : k][w];
          const float2 xhat = __ffma2_rn(ck, r2, nmr);
          const float2 dy = bf2(word(dk, w));
          float2 dx = __ffma2_rn(xhat, nm2r, __ffma2_rn(__fmul2_rn(dy, bf2(word(gk, w))), r2, nm1r));
          dg[k][w] = __ffma2_rn(dy, xhat, dg[k][w]);
          db[k][w] = __fadd2_rn(db[k][w], dy);
          if constexpr (ADD) dx = __fadd2_rn(dx, bf2(word(av[k], w)));
          o[w] = pack_bf16x2(dx.x, dx.y);
        }
        if (row_vec_ok(p, row, j + k * 32 * TW, kBoundsOutChunk)) dx4[j + k * 32 * TW] = make_uint4(o[0], o[1], o[2], o[3]);
      }
      if constexpr (RR) {  // this warp's reads of the slot are done
        __syncwarp();
        if (lane == 0 && ok) mbar_arrive(empty + slot);
      }
    }
  }
  __syncthreads();  // the producer has drained its copies: the ring is free for the team sums
  float* acc = reinterpret_cast<float*>(ring);  // [kTeams][2 d]
  if (warp > 0) {
#pragma unroll
    for (int k = 0; k < VT; ++k) {
      const int col = (j + k * 32 * TW) * 8;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        acc[team * 2 * p.d + col + 2 * w] = dg[k][w].x;
        acc[team * 2 * p.d + col + 2 * w + 1] = dg[k][w].y;
        acc[team * 2 * p.d + p.d + col + 2 * w] = db[k][w].x;
        acc[team * 2 * p.d + p.d + col + 2 * w + 1] = db[k][w].y;
      }
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < 2 * p.d; c += blockDim.x) {
    float t = 0.f;
#pragma unroll
    for (int tm = 0; tm < kTeams; ++tm) t += acc[tm * 2 * p.d + c];
    p.partial[static_cast<long long>(blockIdx.x) * 2 * p.d + c] = t;
  }
}

// LayerNorm forward streamed through the ring: the producer lane keeps the CTA's next rows in flight while
// teams of TW consumer warps normalise.  A team copies its row from the slot into registers (thread j of
// the team owns the 16-byte vectors j + k·32·TW, k < VT; d = 256 TW VT), frees the slot and only then
// reduces and stores, so the CTA's loads never wait on its arithmetic.  The kernel is bound by its
// instruction latencies rather than by DRAM (its time follows the SM clock), so it keeps the work per
// element small and many rows in flight: γ and β are converted to fp32 once per CTA into shared memory
// (each vector's first four values in one array, its last four in another, so that a warp's 16-byte reads
// are consecutive), statistics come from shifted sums in one reduction round (K = the row's first
// element), and the output is (x·rstd − mean·rstd)·γ + β, two fused multiply-adds per float pair, rounded
// once to bf16 and stored from registers into the row's slot of the gathered tensor.
template <int VT, int TW, int CONS = kStreamConsumers>
__global__ void __launch_bounds__(32 * (CONS + 1), 1) k_layernorm_fwd_stream(const RowParams p) {
  constexpr int kTeams = CONS / TW;
  if (!ring_config_ok(p, kTeams)) return;  // uniform over the CTA: no barrier is left waiting
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = align128(smem_raw);
  const uint32_t row_bytes = static_cast<uint32_t>(p.d) * 2u;
  const int nv = p.d / 8;                  // 16-byte vectors per row
  float4* gb = reinterpret_cast<float4*>(ring + p.slots * row_bytes);  // [4][nv]: γ lo, γ hi, β lo, β hi
  uint64_t* full = reinterpret_cast<uint64_t*>(gb + 4 * nv);
  uint64_t* empty = full + p.slots;
  int* abort_flag = reinterpret_cast<int*>(empty + p.slots);
  __shared__ float2 red2[2][CONS];
  __shared__ int vote[2][CONS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.slots; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, TW);
    }
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};
  const int n_rows = p.rows > static_cast<int>(blockIdx.x)
                         ? (p.rows - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) / gridDim.x
                         : 0;
  if (warp == 0) {
    // the producer drains its copies in flight before it leaves; no CTA-wide barrier follows
    if (lane == 0) stream_producer(p, ring, row_bytes, row_bytes, full, empty, n_rows, wc, false);
    return;
  }
  // γ and β are staged by the consumer warps while the producer's first copies are in flight (measured on
  // GB300 at T = 8192, d = 4096: 0.0252 -> 0.0245 ms); named barrier 1 + kTeams (the teams use 1 .. kTeams)
  for (int v = threadIdx.x - 32; v < nv; v += 32 * CONS) {
    float f[8];
    unpack8(__ldg(reinterpret_cast<const uint4*>(p.gamma) + v), f);
    gb[v] = make_float4(f[0], f[1], f[2], f[3]);
    gb[nv + v] = make_float4(f[4], f[5], f[6], f[7]);
    unpack8(__ldg(reinterpret_cast<const uint4*>(p.beta) + v), f);
    gb[2 * nv + v] = make_float4(f[0], f[1], f[2], f[3]);
    gb[3 * nv + v] = make_float4(f[4], f[5], f[6], f[7]);
  }
  asm volatile("bar.sync %0, %1;" ::"r"(1 + kTeams), "r"(32 * CONS) : "memory");
  const int cw = warp - 1;        // consumer warp index
  const int team = cw / TW;
  const int tw = cw % TW;         // warp within the team
  const int j = tw * 32 + lane;   // thread within the team
  const float inv_d = 1.f / static_cast<float>(p.d);
  int par = 0;
  for (int i = team; i < n_rows; i += kTeams, par ^= 1) {
    const int slot = i % p.slots;
    // every warp of the team waits (bounded) on its own; the outcomes are voted at the team barrier
    const bool ok = stream_wait(full + slot, static_cast<uint32_t>(i / p.slots) & 1u, wc);
    const uint4* xs = reinterpret_cast<const uint4*>(ring + slot * row_bytes);
    uint4 xv[VT];
#pragma unroll
    for (int k = 0; k < VT; ++k) xv[k] = ok ? xs[j + k * 32 * TW] : make_uint4(0, 0, 0, 0);
    const float shift = ok ? __uint_as_float(xs[0].x << 16) : 0.f;  // the row's first element
    __syncwarp();
    if (lane == 0 && ok) mbar_arrive(empty + slot);
    const float2 nk = make_float2(-shift, -shift);
    float2 s1 = make_float2(0.f, 0.f), s2 = s1;
#pragma unroll
    for (int k = 0; k < VT; ++k)
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float2 c = __fadd2_rn(bf2(word(xv[k], w)), nk);
        s1 = __fadd2_rn(s1, c);
        s2 = __ffma2_rn(c, c, s2);
      }
    float2 t = warp_sum2(s1.x + s1.y, s2.x + s2.y);
    bool team_ok = ok;
    if constexpr (TW > 1) {
      if (lane == 0) {
        red2[par][cw] = t;
        vote[par][cw] = ok ? 1 : 0;
      }
      team_sync(team, TW);
      t = make_float2(0.f, 0.f);
#pragma unroll
      for (int w = 0; w < TW; ++w) {
        const float2 r = red2[par][team * TW + w];
        t.x += r.x;
        t.y += r.y;
        team_ok = team_ok && vote[par][team * TW + w] != 0;
      }
    }
    if (!team_ok) break;
    const float m = t.x * inv_d;  // mean - K
    const float rstd = rsqrtf(fmaxf(t.y * inv_d - m * m, 0.f) + p.eps);
    const float nmr = -(shift + m) * rstd;  // -mean rstd
    const float2 a2 = make_float2(rstd, rstd), b2 = make_float2(nmr, nmr);
    const int row = blockIdx.x + i * gridDim.x;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dst) + static_cast<long long>(row) * p.d);
#pragma unroll
    for (int k = 0; k < VT; ++k) {
      const int idx = j + k * 32 * TW;
      const float4 gl = gb[idx], gh = gb[nv + idx], bl = gb[2 * nv + idx], bh = gb[3 * nv + idx];
      const float2 g2[4] = {make_float2(gl.x, gl.y), make_float2(gl.z, gl.w), make_float2(gh.x, gh.y),
                            make_float2(gh.z, gh.w)};
      const float2 be2[4] = {make_float2(bl.x, bl.y), make_float2(bl.z, bl.w), make_float2(bh.x, bh.y),
                             make_float2(bh.z, bh.w)};
      uint32_t o[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float2 y = __ffma2_rn(__ffma2_rn(bf2(word(xv[k], w)), a2, b2), g2[w], be2[w]);
        o[w] = pack_bf16x2(y.x, y.y);
      }
      if (row_vec_ok(p, row, idx, kBoundsRowStore)) dst[idx] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// ----------------------------------------------------------------------------- reduce-scatter, gather, column sum

// Y_chunk_j[r] = bf16(sum_{i<N} P_i[j T/N + r]) in fp32, shard 0 first.
__global__ void __launch_bounds__(256) k_reduce_scatter(const RowParams p) {
  const long long nvec = static_cast<long long>(p.rows) * p.d / 8;
  const uint4* src = static_cast<const uint4*>(p.src);
  const long long sstride = p.shard_stride / 8;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < nvec;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    float a[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) a[e] = 0.f;
    for (int s = 0; s < p.n_chunks; ++s) {
      float f[8];
      // debug builds: shard s's slice of the partials holds exactly rows x d / 8 vectors
      const long long k = TPMLP_IN_BOUNDS(i, sstride, kBoundsShard) ? s * sstride + i : 0;
      unpack8(__ldg(src + k), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) a[e] += f[e];
    }
    const long long el = i * 8;
    const int row = static_cast<int>(el / p.d);
    const int col = static_cast<int>(el - static_cast<long long>(row) * p.d);
    if (p.tail) sp_tail_8(p, a, i, row, col);
    if (row_vec_ok(p, row, col / 8, kBoundsOutChunk)) reinterpret_cast<uint4*>(out_chunk_row(p, row) + col)[0] = pack8(a);
  }
}

// Column-sum tiling of the dropout backward and the bf16 column partials: a block of kColWarps warps
// covers 256 columns (one 16-byte vector per lane) and kColWarps runs of `rows_per_warp` rows (one run per
// warp, 4 loads in flight per lane); the warps' sums are added in warp order in shared memory, so each
// block writes one fp32 partial row of its 256 columns (a fixed summation order).
constexpr int kColWarps = 8;
constexpr int kColWarpRows = 16;  // rows per warp unless the grid's y extent (65535) needs more

__device__ __forceinline__ void block_column_partial(const float (&acc)[8], bool active, int lane, int warp, int v,
                                                     int cols, float* partial) {
  __shared__ float4 red[kColWarps][32][2];
  red[warp][lane][0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  red[warp][lane][1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  __syncthreads();
  if (warp == 0 && active) {
    float4 a = red[0][lane][0], b = red[0][lane][1];
#pragma unroll
    for (int w = 1; w < kColWarps; ++w) {
      const float4 c = red[w][lane][0], d = red[w][lane][1];
      a.x += c.x; a.y += c.y; a.z += c.z; a.w += c.w;
      b.x += d.x; b.y += d.y; b.z += d.z; b.w += d.w;
    }
    float4* out = reinterpret_cast<float4*>(partial + static_cast<long long>(blockIdx.y) * cols + 8 * v);
    out[0] = a;
    out[1] = b;
  }
}

// Dropout backward: dst[r] = keep * dY[r] * scale (gathered rows); with p.partial, each block's column sums
// of those values (the row bias gradient).  KEEP: 0 = every element kept (p = 0), 1 = the forward's saved
// keep bits, 2 = the generator's bits.  The load-only variants are held to 48 registers (5 blocks per SM)
// so enough rows are in flight; the generator's 64-bit arithmetic needs more.
template <int KEEP>
__global__ void __launch_bounds__(32 * kColWarps, KEEP == 2 ? 1 : 5) k_dropout_bwd(const RowParams p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nv = p.d / 8;
  const int v = blockIdx.x * 32 + lane;
  const bool active = v < nv;
  const int r0 = (blockIdx.y * kColWarps + warp) * p.rows_per_block;
  const int r1 = min(p.rows, r0 + p.rows_per_block);
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  uint4* dst = static_cast<uint4*>(p.dst);
  if (active) {
    for (int rb = r0; rb < r1; rb += 4) {
      uint4 raw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        raw[u] = rb + u < r1 ? __ldg(reinterpret_cast<const uint4*>(chunk_row(p, rb + u)) + v) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (rb + u >= r1) break;
        const long long q = static_cast<long long>(rb + u) * nv + v;
        uint32_t m = 0xFFu;
        if constexpr (KEEP == 1) m = p.drop_mask[q];
        if constexpr (KEEP == 2)
          m = dropout_keep8(static_cast<unsigned long long>(q), p.drop_offset, p.drop_seed, p.drop_thr);
        float f[8];
        unpack8(raw[u], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          f[e] = (m >> e) & 1u ? f[e] * p.drop_scale : 0.f;
          acc[e] += f[e];
        }
        if (row_vec_ok(p, rb + u, v, kBoundsRowStore)) dst[q] = pack8(f);
      }
    }
  }
  if (p.partial != nullptr) block_column_partial(acc, active, lane, warp, v, p.d, p.partial);
}

// Contiguous dst[T x d] <- the N chunk pointers.
__global__ void __launch_bounds__(256) k_gather_rows(const RowParams p) {
  const long long nvec = static_cast<long long>(p.rows) * p.d / 8;
  uint4* dst = static_cast<uint4*>(p.dst);
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < nvec;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long el = i * 8;
    const int row = static_cast<int>(el / p.d);
    const int col = static_cast<int>(el - static_cast<long long>(row) * p.d);
    dst[i] = __ldg(reinterpret_cast<const uint4*>(chunk_row(p, row) + col));
  }
}

// out[c] = sum over r < rows of partial[r * stride + c], for c < cols; columns c < split go to
// out0[c], the rest to out1[c - split].  32 columns per block, rows split over the 8 warps and
// combined in warp order: a fixed summation order, so the result is deterministic.
__global__ void __launch_bounds__(256) k_column_sum(const float* __restrict__ partial, int rows, int cols,
                                                     long long stride, void* out0, void* out1, int split,
                                                     int out_bf16) {
  __shared__ float red[8][33];
  const int lane = threadIdx.x & 31, slice = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + lane;
  float s = 0.f;
  if (c < cols) {
    // four independent chains (rows slice + 8 (4 k + u)), combined in a fixed order: loads stay in flight
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    int r = slice;
    for (; r + 24 < rows; r += 32) {
#pragma unroll
      for (int u = 0; u < 4; ++u) a[u] += partial[static_cast<long long>(r + 8 * u) * stride + c];
    }
    for (int u = 0; r < rows; r += 8, ++u) a[u & 3] += partial[static_cast<long long>(r) * stride + c];
    s = (a[0] + a[1]) + (a[2] + a[3]);
  }
  red[slice][lane] = s;
  __syncthreads();
  if (slice == 0 && c < cols) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) t += red[k][lane];
    void* out = c < split ? out0 : out1;
    const int oc = c < split ? c : c - split;
    if (out_bf16)
      static_cast<__nv_bfloat16*>(out)[oc] = __float2bfloat16_rn(t);
    else
      static_cast<float*>(out)[oc] = t;
  }
}

// partial[y, c] = the column sums of src over block row y's rows (a bf16 matrix with row stride ld), in the
// tiling of k_dropout_bwd.
__global__ void __launch_bounds__(32 * kColWarps, 6) k_column_partial_bf16(const __nv_bfloat16* __restrict__ src, int rows,
                                                                        int cols, long long ld, int rows_per_warp,
                                                                        float* __restrict__ partial) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int v = blockIdx.x * 32 + lane;
  const bool active = v < cols / 8;
  const int r0 = (blockIdx.y * kColWarps + warp) * rows_per_warp;
  const int r1 = min(rows, r0 + rows_per_warp);
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  if (active) {
    for (int rb = r0; rb < r1; rb += 4) {
      uint4 raw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        raw[u] = rb + u < r1 ? __ldg(reinterpret_cast<const uint4*>(src + static_cast<long long>(rb + u) * ld) + v)
                             : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float f[8];
        unpack8(raw[u], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += f[e];
      }
    }
  }
  block_column_partial(acc, active, lane, warp, v, cols, partial);
}

// ----------------------------------------------------------------------------- E4M3 casts and delayed scaling

// dst[i] = FP8(src[i] * s), 16 elements (two 16-byte loads, one 16-byte store) per step, grid-stride.
// FMT 0 = E4M3, 1 = E5M2.
template <int FMT>
__global__ void __launch_bounds__(256) k_cast_fp8(const __nv_bfloat16* __restrict__ src, long long n16,
                                                  const float* scale, uint8_t* __restrict__ dst, float* amax) {
  const float s = __ldg(scale);
  float m = 0.f;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    float a[8], b[8];
    unpack8(__ldg(reinterpret_cast<const uint4*>(src) + 2 * i), a);
    unpack8(__ldg(reinterpret_cast<const uint4*>(src) + 2 * i + 1), b);
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, fmaxf(fabsf(a[e]), fabsf(b[e])));
    const uint2 lo = fp8x8<FMT>(a, s), hi = fp8x8<FMT>(b, s);
    reinterpret_cast<uint4*>(dst)[i] = make_uint4(lo.x, lo.y, hi.x, hi.y);
  }
  amax_combine_warp(amax, m);
}

// Transposing cast: src [rows x cols] -> dst [cols x rows], tiles of 128 source rows x 64 columns through
// shared memory (rows, cols multiples of 16).  Loads: 16-byte vectors along the source row, all four of a
// thread issued before any is used; stores: 16 bytes of one destination row (16 consecutive source rows of
// one column), so each destination row of the tile is one 128-byte line.  Measured on GB300 against 64 x 64
// tiles: the weight casts at d = 4096, F = 16384 54 -> 52 µs.
constexpr int kCastTile = 64;   // columns per tile
constexpr int kCastRows = 128;  // rows per tile
template <int FMT>
__global__ void __launch_bounds__(256) k_cast_fp8_t(const __nv_bfloat16* __restrict__ src, int rows, int cols,
                                                    const float* scale, uint8_t* __restrict__ dst, float* amax) {
  __shared__ float tile[kCastRows][kCastTile + 1];
  const float s = __ldg(scale);
  const int r0 = blockIdx.y * kCastRows, c0 = blockIdx.x * kCastTile;
  const int t = threadIdx.x;
  float m = 0.f;
  uint4 raw[kCastRows / 32];
#pragma unroll
  for (int h = 0; h < kCastRows / 32; ++h) {
    const int r = t / 8 + 32 * h, cv = (t % 8) * 8;
    raw[h] = (r0 + r < rows && c0 + cv < cols)
                 ? __ldg(reinterpret_cast<const uint4*>(src + static_cast<long long>(r0 + r) * cols + c0 + cv))
                 : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int h = 0; h < kCastRows / 32; ++h) {
    const int r = t / 8 + 32 * h, cv = (t % 8) * 8;
    float f[8];
    unpack8(raw[h], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      m = fmaxf(m, fabsf(f[e]));
      tile[r][cv + e] = f[e];
    }
  }
  __syncthreads();
  const int oc = t / 4;  // destination row c0 + oc, bytes [r0 + rb, r0 + rb + 16)
#pragma unroll
  for (int q = 0; q < kCastRows / 64; ++q) {
    const int rb = (t % 4) * 16 + 64 * q;
    if (c0 + oc < cols && r0 + rb < rows) {
      float f[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) f[i] = tile[rb + i][oc];
      uint4 o;
      o.x = fp8x4<FMT>(f[0], f[1], f[2], f[3], s);
      o.y = fp8x4<FMT>(f[4], f[5], f[6], f[7], s);
      o.z = fp8x4<FMT>(f[8], f[9], f[10], f[11], s);
      o.w = fp8x4<FMT>(f[12], f[13], f[14], f[15], s);
      *reinterpret_cast<uint4*>(dst + static_cast<long long>(c0 + oc) * rows + r0 + rb) = o;
    }
  }
  amax_combine_warp(amax, m);
}

// dst [cols x rows] = transpose of src [rows x cols], bytes, in registers.  A thread loads 16 bytes from
// each of 4 consecutive rows, transposes the four 4 x 4 byte blocks with byte permutes and stores 16
// words of 4 bytes (4 consecutive source rows of one column each).  A block covers 256 rows x 64 columns:
// thread t takes rows 4 (t / 4) .. + 3 and columns 16 (t % 4) .. + 15; the stores of one destination row
// by the 64 threads with the same t % 4 are 256 consecutive bytes.
constexpr int kTrRows = 256, kTrCols = 64;
__global__ void __launch_bounds__(256) k_transpose_bytes(const uint8_t* __restrict__ src, int rows, int cols,
                                                         uint8_t* __restrict__ dst) {
  const int t = threadIdx.x;
  const int r = blockIdx.y * kTrRows + 4 * (t / 4);
  const int c = blockIdx.x * kTrCols + 16 * (t % 4);
  if (r >= rows || c >= cols) return;  // rows % 4 == 0 and cols % 16 == 0: a strip is wholly in or out
  uint4 v[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) v[k] = __ldg(reinterpret_cast<const uint4*>(src + static_cast<long long>(r + k) * cols + c));
  const uint32_t w[4][4] = {{v[0].x, v[0].y, v[0].z, v[0].w}, {v[1].x, v[1].y, v[1].z, v[1].w},
                            {v[2].x, v[2].y, v[2].z, v[2].w}, {v[3].x, v[3].y, v[3].z, v[3].w}};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    // block q: bytes 4q .. 4q+3 of the four rows; word k of row k holds (row k, columns 4q .. 4q+3)
    const uint32_t lo01 = __byte_perm(w[0][q], w[1][q], 0x5140), hi01 = __byte_perm(w[0][q], w[1][q], 0x7362);
    const uint32_t lo23 = __byte_perm(w[2][q], w[3][q], 0x5140), hi23 = __byte_perm(w[2][q], w[3][q], 0x7362);
    const uint32_t o[4] = {__byte_perm(lo01, lo23, 0x5410), __byte_perm(lo01, lo23, 0x7632),
                           __byte_perm(hi01, hi23, 0x5410), __byte_perm(hi01, hi23, 0x7632)};
#pragma unroll
    for (int m = 0; m < 4; ++m)
      *reinterpret_cast<uint32_t*>(dst + static_cast<long long>(c + 4 * q + m) * rows + r) = o[m];
  }
}

// One warp per tensor: shift the history by one (oldest out, this step's amax in), mean in a fixed order,
// next scale = fp8_max / mean / 2^margin (1 while the mean is not positive), reset this step's amax.
__global__ void __launch_bounds__(128) k_fp8_update(float* scale, float* amax, float* history, int n, int len,
                                                    float fp8_max, int margin) {
  const int lane = threadIdx.x & 31;
  for (int i = threadIdx.x >> 5; i < n; i += blockDim.x >> 5) {
    float* h = history + static_cast<long long>(i) * len;
    const float cur = amax[i];
    for (int base = 0; base < len; base += 32) {
      const int j = base + lane;
      float v = 0.f;
      if (j < len) v = j + 1 < len ? h[j + 1] : cur;
      __syncwarp();
      if (j < len) h[j] = v;
      __syncwarp();
    }
    float sum = 0.f;
    for (int j = lane; j < len; j += 32) sum += h[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) {
      const float mean = sum / static_cast<float>(len);
      scale[i] = mean > 0.f && isfinite(mean) ? fp8_max / mean / exp2f(static_cast<float>(margin)) : 1.f;
      amax[i] = 0.f;
    }
  }
}

}  // namespace

cudaError_t rowwise_bounds_status(unsigned int* count, unsigned int* site) {
#ifdef TPMLP_DEBUG_BOUNDS
  return bounds_read_and_clear(count, site);
#else
  *count = *site = 0;
  return cudaSuccess;
#endif
}

namespace {

int stream_grid(long long work_items, int sm_count) {
  const long long per = 256;
  long long g = (work_items + per - 1) / per;
  const long long cap = static_cast<long long>(sm_count) * 8;
  if (g > cap) g = cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

template <typename K>
static cudaError_t launch_stream(K kern, const RowParams& r, size_t smem, int grid, cudaStream_t s,
                                 int threads = kStreamThreads) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  // programmatic dependent launch: the kernel's set-up overlaps the previous kernel's tail; it waits for that
  // kernel (griddepcontrol.wait) before its first global access (measured on GB300, T = 8192, d = 4096: the
  // forward 0.0243 -> 0.0235 ms graph-timed, 0.0271 -> 0.0244 ms eager)
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, r);
}

// Shared-memory row slots for rows of `slot_bytes`: about 128 KB of rows in flight per SM.
static int stream_slots(size_t slot_bytes) {
  const size_t n = (128u * 1024u) / slot_bytes;
  return static_cast<int>(n < 2 ? 2 : (n > 32 ? 32 : n));
}

// Persistent launch of a pipelined LayerNorm kernel, or cudaErrorNotReady when the grid would give each
// warp (pair) fewer than kLnPipeMinRows rows: below that the exposed first load and the tail outweigh the
// overlap (measured on GB300: at T = 8192, d = 4096 the launch-per-group kernel is 7% faster; at T = 65536
// the pipelined one reaches 0.94 of HBM against 0.80).
constexpr int kLnPipeMinRows = 24;

template <typename K>
static cudaError_t launch_ln_persistent(K kern, int rows_per_block, const RowParams& r, const DeviceCtx& ctx,
                                        cudaStream_t s, std::atomic<int>* per_sm_cache) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int per_sm = per_sm_cache[dev & 63].load(std::memory_order_relaxed);
  if (per_sm == 0) {
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 128, 0);
    if (e != cudaSuccess) return e;
    per_sm = n < 1 ? 1 : n;
    per_sm_cache[dev & 63].store(per_sm, std::memory_order_relaxed);  // concurrent callers store the same value
  }
  const long long grid = static_cast<long long>(per_sm) * ctx.sm_count;
  if (static_cast<long long>(r.rows) < grid * rows_per_block * kLnPipeMinRows) return cudaErrorNotReady;
  kern<<<static_cast<int>(grid), 128, 0, s>>>(r);
  return cudaGetLastError();
}

template <int V>
static cudaError_t launch_ln_pipe(const RowParams& r, const DeviceCtx& ctx, cudaStream_t s) {
  static std::atomic<int> per_sm[64] = {};
  return launch_ln_persistent(k_layernorm_fwd_pipe<V>, 4, r, ctx, s, per_sm);
}

template <int V>
static cudaError_t launch_ln_pipe2(const RowParams& r, const DeviceCtx& ctx, cudaStream_t s) {
  static std::atomic<int> per_sm[64] = {};
  return launch_ln_persistent(k_layernorm_fwd_pipe2<V>, 2, r, ctx, s, per_sm);
}

// The streamed LayerNorm forward, VT vectors per thread and TW warps per row (d = 256 TW VT), CONS consumer
// warps: `per_sm` CTAs per SM (fewer for short inputs), each with a ring of about `ring_bytes` of row
// slots, the slot count a multiple of the teams (see ring_config_ok).
template <int VT, int TW, int CONS>
static cudaError_t launch_ln_stream_cfg(const RowParams& r0, const DeviceCtx& ctx, cudaStream_t s,
                                        size_t ring_bytes, int per_sm) {
  constexpr int kTeams = CONS / TW;
  constexpr size_t kMaxSmem = 227u * 1024u;
  RowParams r = r0;
  r.err = ctx.err;
  r.timeout_ns = ctx.timeout_ns;
  const size_t row_bytes = static_cast<size_t>(r.d) * 2;
  const size_t fixed = 128 + 4 * row_bytes + 16;  // alignment, fp32 γ/β (8 d bytes), abort flag
  size_t slots = ring_bytes / row_bytes / kTeams * kTeams;
  if (slots < static_cast<size_t>(kTeams)) slots = kTeams;
  while (slots > 32 || (slots > static_cast<size_t>(kTeams) && fixed + slots * (row_bytes + 16) > kMaxSmem))
    slots -= kTeams;
  if (fixed + slots * (row_bytes + 16) > kMaxSmem) return cudaErrorNotSupported;
  r.slots = static_cast<int>(slots);
  const size_t smem = fixed + slots * (row_bytes + 16);  // + the ring and its two barriers per slot
  const long long cap = static_cast<long long>(per_sm) * ctx.sm_count;
  const int grid = static_cast<int>(r.rows < cap ? r.rows : cap);
  return launch_stream(k_layernorm_fwd_stream<VT, TW, CONS>, r, smem, grid, s, 32 * (CONS + 1));
}

// Ring bytes per CTA of the streamed forward.  Measured on GB300 (CUDA graphs of back-to-back launches,
// fraction of the measured HBM bandwidth at T = 8192, d = 4096 / T = 4096, d = 8192): teams of two warps
// on a 64 KB ring 0.80 / 0.79; one-warp teams 0.74 / 0.78; a 190 KB ring 0.74 / 0.66 (every SM's first
// rows wait behind the whole start-up burst); two CTAs per SM with 48 KB rings 0.65 / 0.60; the
// register kernels 0.69 / 0.65.
constexpr size_t kLnFwdRingBytes = 64u * 1024u;
constexpr int kLnFwdCtasPerSm = 1;

// cudaErrorNotSupported for widths it does not cover.
static cudaError_t launch_ln_stream(const RowParams& r, const DeviceCtx& ctx, cudaStream_t s) {
  constexpr size_t kRing = kLnFwdRingBytes;
  constexpr int kPer = kLnFwdCtasPerSm;
  // four teams of VT = 8 vectors per thread where the width allows (measured best at d = 4096 and 8192:
  // fewer teams leave the SM idle between rows, more run out of registers or issue slots)
  switch (r.d) {
    case 256: return launch_ln_stream_cfg<1, 1, 8>(r, ctx, s, kRing, kPer);
    case 512: return launch_ln_stream_cfg<2, 1, 8>(r, ctx, s, kRing, kPer);
    case 1024: return launch_ln_stream_cfg<4, 1, 8>(r, ctx, s, kRing, kPer);
    case 2048: return launch_ln_stream_cfg<8, 1, 8>(r, ctx, s, kRing, kPer);
    case 4096: return launch_ln_stream_cfg<8, 2, 8>(r, ctx, s, kRing, kPer);
    case 8192: return launch_ln_stream_cfg<8, 4, 16>(r, ctx, s, kRing, kPer);
    default: return cudaErrorNotSupported;
  }
}

cudaError_t launch_layernorm_fwd(const RowParams& r, const DeviceCtx& ctx, cudaStream_t s) {
  if (r.rows <= 0) return cudaSuccess;
  {
    // long inputs: the persistent register-pipelined kernels (T = 65536, d = 4096: 0.95 of HBM, the
    // streamed kernel 0.92)
    cudaError_t e = cudaErrorNotReady;
    switch (r.d) {
      case 1024: e = launch_ln_pipe<4>(r, ctx, s); break;
      case 2048: e = launch_ln_pipe<8>(r, ctx, s); break;
      case 4096: e = launch_ln_pipe2<8>(r, ctx, s); break;
      default: break;
    }
    if (e != cudaErrorNotReady) return e;  // launched (or failed); otherwise too few rows per warp
  }
  {
    const cudaError_t e = launch_ln_stream(r, ctx, s);
    if (e != cudaErrorNotSupported) return e;  // launched (or failed); otherwise a width it does not cover
  }
  // any other multiple of 8
  k_layernorm_fwd_any<false><<<(r.rows + 3) / 4, 128, 0, s>>>(r);
  return cudaGetLastError();
}

cudaError_t launch_layernorm_fwd_e4m3(const RowParams& r0, const float* scale, float* amax, cudaStream_t s) {
  if (r0.rows <= 0) return cudaSuccess;
  RowParams r = r0;
  r.qscale = scale;
  r.amax = amax;
  const int grid4 = (r.rows + 3) / 4;
  const int grid2 = (r.rows + 1) / 2;
  switch (r.d) {
    case 256: k_layernorm_fwd_reg<1, 1, false, true><<<grid4, 128, 0, s>>>(r); break;
    case 512: k_layernorm_fwd_reg<2, 1, false, true><<<grid4, 128, 0, s>>>(r); break;
    case 1024: k_layernorm_fwd_reg<4, 1, false, true><<<grid4, 128, 0, s>>>(r); break;
    case 2048: k_layernorm_fwd_reg<8, 1, false, true><<<grid4, 128, 0, s>>>(r); break;
    case 4096: k_layernorm_fwd_reg<16, 1, false, true><<<grid4, 128, 0, s>>>(r); break;
    case 8192: k_layernorm_fwd_reg<16, 2, false, true><<<grid2, 128, 0, s>>>(r); break;
    default: return cudaErrorNotSupported;
  }
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_fwd(const RowParams& r, cudaStream_t s) {
  if (r.rows <= 0) return cudaSuccess;
  const int grid4 = (r.rows + 3) / 4;
  const int grid2 = (r.rows + 1) / 2;
  switch (r.d) {
    case 1024: k_layernorm_fwd_reg<4, 1, true><<<grid4, 128, 0, s>>>(r); break;
    case 2048: k_layernorm_fwd_reg<8, 1, true><<<grid4, 128, 0, s>>>(r); break;
    case 4096: k_layernorm_fwd_reg<16, 1, true><<<grid4, 128, 0, s>>>(r); break;
    case 8192: k_layernorm_fwd_reg<16, 2, true><<<grid2, 128, 0, s>>>(r); break;
    default: k_layernorm_fwd_any<true><<<grid4, 128, 0, s>>>(r); break;
  }
  return cudaGetLastError();
}

int layernorm_bwd_blocks(int rows, int max_blocks) {
  const int groups = (rows + kLnBwdRowsPerGroup - 1) / kLnBwdRowsPerGroup;
  return groups < max_blocks ? (groups < 1 ? 1 : groups) : max_blocks;
}

namespace {

constexpr int kLnBwdMaxBlocksOld = 304;   // CTAs of the generic backward
constexpr int kLnBwdMaxBlocksFused = 256; // upper bound on the fused backward's CTAs (one per SM)

// (team warps, vectors per thread) of the fused backward for row width d, or {0, 0}.
struct TeamShape {
  int tw, vt;
};
// The fused backward with CONS consumer warps in teams of TW: a ring of x/dy row-pair slots (a multiple of
// the teams, at most ring_max bytes; 192 KB when the slots are held through the output pass), the γ row
// and the barriers, or the teams' dγ/dβ sums if those need more.
template <int VT, int TW, int CONS, bool RR>
static cudaError_t launch_ln_bwd_cfg(RowParams r, int grid, bool add, cudaStream_t s) {
  constexpr int kTeams = CONS / TW;
  const size_t row_bytes = static_cast<size_t>(r.d) * 2;
  const size_t ring_max = RR ? 192u * 1024u : 128u * 1024u;
  int slots = static_cast<int>(ring_max / (2 * row_bytes)) / kTeams * kTeams;
  if (slots > 32) slots = 32 / kTeams * kTeams;
  if (slots < kTeams) slots = kTeams;
  size_t smem = 128 + static_cast<size_t>(slots) * (2 * row_bytes + 16) + row_bytes + 16;
  const size_t team_sums = static_cast<size_t>(kTeams) * 2 * r.d * 4 + 128;
  if (smem < team_sums) smem = team_sums;
  if (smem > 227u * 1024u) return cudaErrorInvalidValue;
  r.slots = slots;
  return add ? launch_stream(k_layernorm_bwd_fused<VT, TW, true, CONS, RR>, r, smem, grid, s, 32 * (CONS + 1))
             : launch_stream(k_layernorm_bwd_fused<VT, TW, false, CONS, RR>, r, smem, grid, s, 32 * (CONS + 1));
}


TeamShape fused_shape(int d) {
  switch (d) {
    case 256: return {1, 1};
    case 512: return {2, 1};
    case 1024: return {4, 1};
    case 2048: return {4, 2};
    case 4096: return {4, 4};
    case 8192: return {8, 4};
    default: return {0, 0};
  }
}

}  // namespace

size_t layernorm_bwd_scratch_floats(int rows, int d) {
  if (fused_shape(d).tw > 0) {
    const int blocks = rows < kLnBwdMaxBlocksFused ? (rows < 1 ? 1 : rows) : kLnBwdMaxBlocksFused;
    return static_cast<size_t>(blocks) * 2 * d;
  }
  return static_cast<size_t>(layernorm_bwd_blocks(rows, kLnBwdMaxBlocksOld)) * 2 * d;
}

cudaError_t launch_layernorm_bwd(const RowParams& r0, float* scratch, size_t cap_floats, const DeviceCtx& ctx,
                                 float* dgamma, float* dbeta, cudaStream_t s) {
  if (r0.rows <= 0) return cudaSuccess;
  RowParams r = r0;
  r.err = ctx.err;
  r.timeout_ns = ctx.timeout_ns;
  r.partial = scratch;
  const size_t per_block = 2 * static_cast<size_t>(r.d);
  const TeamShape ts = fused_shape(r.d);
  if (ts.tw > 0) {
    int grid = r.rows < ctx.sm_count ? r.rows : ctx.sm_count;
    if (grid > kLnBwdMaxBlocksFused) grid = kLnBwdMaxBlocksFused;
    if (static_cast<size_t>(grid) * per_block > cap_floats) grid = static_cast<int>(cap_floats / per_block);
    if (grid >= 1) {
      cudaError_t e;
      if (r.d == 4096) {
        // three teams of four warps that read x and dy from the slot twice fit 13 warps' 128 registers a
        // thread (measured on GB300 at T = 8192: 0.638 of HBM against 0.632 for two teams holding them in
        // registers; at T = 32768 0.82 against 0.78); at d = 8192 neither one team (0.535) nor two
        // (spilling at 96 registers, 0.433) beat the register kernel (0.565)
        e = launch_ln_bwd_cfg<4, 4, 12, true>(r, grid, r.add_chunks.p[0] != nullptr, s);
        if (e != cudaSuccess) return e;
        k_column_sum<<<(2 * r.d + 31) / 32, 256, 0, s>>>(r.partial, grid, 2 * r.d, 2LL * r.d, dgamma, dbeta, r.d, 0);
        return cudaGetLastError();
      }
      const size_t row_bytes = static_cast<size_t>(r.d) * 2;
      // a multiple of the consumer teams (see ring_config_ok)
      const int teams = kStreamConsumers / ts.tw;
      r.slots = stream_slots(2 * row_bytes) / teams * teams;
      if (r.slots < teams) r.slots = teams;
      size_t smem = 128 + r.slots * 2 * row_bytes + row_bytes + 16 * static_cast<size_t>(r.slots) + 16;
      const size_t team_sums = static_cast<size_t>(kStreamConsumers / ts.tw) * per_block * 4 + 128;
      if (smem < team_sums) smem = team_sums;
      if (r.add_chunks.p[0] == nullptr) {
        switch (r.d) {
          case 256: e = launch_stream(k_layernorm_bwd_fused<1, 1>, r, smem, grid, s); break;
          case 512: e = launch_stream(k_layernorm_bwd_fused<1, 2>, r, smem, grid, s); break;
          case 1024: e = launch_stream(k_layernorm_bwd_fused<1, 4>, r, smem, grid, s); break;
          case 2048: e = launch_stream(k_layernorm_bwd_fused<2, 4>, r, smem, grid, s); break;
          default: e = launch_stream(k_layernorm_bwd_fused<4, 8>, r, smem, grid, s); break;
        }
      } else {
        switch (r.d) {
          case 256: e = launch_stream(k_layernorm_bwd_fused<1, 1, true>, r, smem, grid, s); break;
          case 512: e = launch_stream(k_layernorm_bwd_fused<1, 2, true>, r, smem, grid, s); break;
          case 1024: e = launch_stream(k_layernorm_bwd_fused<1, 4, true>, r, smem, grid, s); break;
          case 2048: e = launch_stream(k_layernorm_bwd_fused<2, 4, true>, r, smem, grid, s); break;
          default: e = launch_stream(k_layernorm_bwd_fused<4, 8, true>, r, smem, grid, s); break;
        }
      }
      if (e != cudaSuccess) return e;
      k_column_sum<<<(2 * r.d + 31) / 32, 256, 0, s>>>(r.partial, grid, 2 * r.d, 2LL * r.d, dgamma, dbeta, r.d, 0);
      return cudaGetLastError();
    }
  }
  // any other width: per-block shared-memory accumulation of dgamma/dbeta
  int max_blocks = static_cast<int>(cap_floats / per_block);
  if (max_blocks > kLnBwdMaxBlocksOld) max_blocks = kLnBwdMaxBlocksOld;
  if (max_blocks < 1) return cudaErrorInvalidValue;
  const int grid = layernorm_bwd_blocks(r.rows, max_blocks);
  const size_t smem = static_cast<size_t>(2) * r.d * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(k_layernorm_bwd, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k_layernorm_bwd<<<grid, 256, smem, s>>>(r);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // dgamma = column sums of partial[:, 0:d], dbeta = column sums of partial[:, d:2d]
  k_column_sum<<<(2 * r.d + 31) / 32, 256, 0, s>>>(r.partial, grid, 2 * r.d, 2LL * r.d, dgamma, dbeta, r.d, 0);
  return cudaGetLastError();
}

cudaError_t launch_reduce_scatter(const RowParams& r, const DeviceCtx& ctx, cudaStream_t s) {
  if (r.rows <= 0) return cudaSuccess;
  k_reduce_scatter<<<stream_grid(static_cast<long long>(r.rows) * r.d / 8, ctx.sm_count), 256, 0, s>>>(r);
  return cudaGetLastError();
}

// Rows per warp of the column-sum tiling: kColWarpRows, or more when the grid's y extent would pass 65535.
int dropout_rows_per_block(int rows) {
  const long long per_block_row = 65535LL * kColWarps;
  const int need = static_cast<int>((rows + per_block_row - 1) / per_block_row);
  return need <= kColWarpRows ? kColWarpRows : need;
}

int column_block_rows(int rows, int rows_per_warp) {
  const int per = rows_per_warp * kColWarps;
  return (rows + per - 1) / per;
}

// Rows per warp for one wave of `resident` blocks per SM (never fewer than dropout_rows_per_block, so the
// partial rows stay within what dropout_bwd_scratch_floats sized).
int rows_per_warp_one_wave(int rows, int cols, int resident) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms < 1)
    sms = 1;
  const int col_blocks = (cols / 8 + 31) / 32;
  int row_blocks = resident * sms / col_blocks;
  if (row_blocks < 1) row_blocks = 1;
  const int want = (rows + kColWarps * row_blocks - 1) / (kColWarps * row_blocks);
  const int least = dropout_rows_per_block(rows);
  return want > least ? want : least;
}

size_t dropout_bwd_scratch_floats(int rows, int d) {
  return static_cast<size_t>(column_block_rows(rows, dropout_rows_per_block(rows))) * static_cast<size_t>(d);
}

cudaError_t launch_dropout_bwd(const RowParams& r, float* partial, void* dbias2, cudaStream_t s) {
  if (r.rows <= 0) return cudaSuccess;
  RowParams q = r;
  q.partial = dbias2 != nullptr ? partial : nullptr;
  q.rows_per_block = rows_per_warp_one_wave(r.rows, r.d, r.drop_thr < kKeepAll && r.drop_mask == nullptr ? 2 : 5);
  const dim3 grid((r.d / 8 + 31) / 32, column_block_rows(r.rows, q.rows_per_block));
  // the forward's keep bits when it saved them, else the generator's
  if (q.drop_thr >= kKeepAll) {
    k_dropout_bwd<0><<<grid, 32 * kColWarps, 0, s>>>(q);
  } else if (q.drop_mask != nullptr) {
    k_dropout_bwd<1><<<grid, 32 * kColWarps, 0, s>>>(q);
  } else {
    k_dropout_bwd<2><<<grid, 32 * kColWarps, 0, s>>>(q);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || dbias2 == nullptr) return e;
  return launch_column_sum(partial, static_cast<int>(grid.y), r.d, dbias2, true, s);
}

cudaError_t launch_gather_rows(const RowParams& r, const DeviceCtx& ctx, cudaStream_t s) {
  if (r.rows <= 0) return cudaSuccess;
  k_gather_rows<<<stream_grid(static_cast<long long>(r.rows) * r.d / 8, ctx.sm_count), 256, 0, s>>>(r);
  return cudaGetLastError();
}

size_t column_sum_bf16_scratch_floats(int rows, int cols) { return dropout_bwd_scratch_floats(rows, cols); }

cudaError_t launch_column_sum_bf16(const void* src, int rows, int cols, long long ld, float* partial, void* out,
                                   cudaStream_t s) {
  if (rows <= 0 || cols <= 0 || out == nullptr) return cudaSuccess;
  if (cols % 8 != 0 || ld % 8 != 0) return cudaErrorInvalidValue;
  const int rpw = rows_per_warp_one_wave(rows, cols, 6);
  const dim3 grid((cols / 8 + 31) / 32, column_block_rows(rows, rpw));
  k_column_partial_bf16<<<grid, 32 * kColWarps, 0, s>>>(static_cast<const __nv_bfloat16*>(src), rows, cols, ld, rpw,
                                                   partial);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_column_sum(partial, static_cast<int>(grid.y), cols, out, true, s);
}

cudaError_t launch_column_sum(const float* partial, int rows, int cols, void* out, bool out_bf16, cudaStream_t s) {
  if (cols <= 0 || out == nullptr) return cudaSuccess;
  k_column_sum<<<(cols + 31) / 32, 256, 0, s>>>(partial, rows, cols, cols, out, out, cols, out_bf16 ? 1 : 0);
  return cudaGetLastError();
}


cudaError_t launch_cast_fp8(const void* src, int rows, int cols, bool transpose, int fmt, const float* scale,
                            void* dst, float* amax, cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  if (fmt != 0 && fmt != 1) return cudaErrorInvalidValue;
  const auto* in = static_cast<const __nv_bfloat16*>(src);
  auto* out = static_cast<uint8_t*>(dst);
  if (transpose) {
    const dim3 grid((cols + kCastTile - 1) / kCastTile, (rows + kCastRows - 1) / kCastRows);
    if (grid.y > 65535) return cudaErrorInvalidValue;
    if (fmt == 0) {
      k_cast_fp8_t<0><<<grid, 256, 0, s>>>(in, rows, cols, scale, out, amax);
    } else {
      k_cast_fp8_t<1><<<grid, 256, 0, s>>>(in, rows, cols, scale, out, amax);
    }
  } else {
    const long long n16 = static_cast<long long>(rows) * cols / 16;
    long long g = (n16 + 255) / 256;
    if (g > 152 * 8) g = 152 * 8;
    if (fmt == 0) {
      k_cast_fp8<0><<<static_cast<int>(g), 256, 0, s>>>(in, n16, scale, out, amax);
    } else {
      k_cast_fp8<1><<<static_cast<int>(g), 256, 0, s>>>(in, n16, scale, out, amax);
    }
  }
  return cudaGetLastError();
}

cudaError_t launch_cast_e4m3(const void* src, int rows, int cols, bool transpose, const float* scale, void* dst,
                             float* amax, cudaStream_t s) {
  return launch_cast_fp8(src, rows, cols, transpose, 0, scale, dst, amax, s);
}

cudaError_t launch_transpose_bytes(const void* src, int rows, int cols, void* dst, cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const dim3 grid((cols + kTrCols - 1) / kTrCols, (rows + kTrRows - 1) / kTrRows);
  if (grid.y > 65535) return cudaErrorInvalidValue;
  k_transpose_bytes<<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(src), rows, cols, static_cast<uint8_t*>(dst));
  return cudaGetLastError();
}

cudaError_t launch_fp8_update(float* scale, float* amax, float* history, int n, int len, float fp8_max, int margin,
                              cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  k_fp8_update<<<1, 128, 0, s>>>(scale, amax, history, n, len, fp8_max, margin);
  return cudaGetLastError();
}

}  // namespace tpmlp
