// Persistent tcgen05 GEMM for sm_103a with fused epilogues.
//
//   C[M x N] = sum_k A[m, k] * B[k, n]     (bf16 in, fp32 accumulate in TMEM)
//
// One CTA per SM walks output tiles of kBM x BN.  Warp roles:
//   warp 0      TMA producer (one lane): k-blocks of A and B into a STAGES-deep
//               shared-memory ring, completion counted on `full[stage]`;
//   warp 1      TMEM allocator, then UMMA issuer (one lane): four
//               128 x BN x 16 MMAs per k-block, `tcgen05.commit` frees the
//               ring slot; after the last k-block of a tile, commits the
//               accumulator to the epilogue;
//   warps 2..   epilogue: tcgen05.ld of the accumulator (double-buffered in
//               TMEM, 2 x BN fp32 columns), the fused epilogue math and
//               16-byte global stores.
//
// The K loop of one tile is where the tensor-parallel reduction happens:
// for the row-parallel GEMMs the k-blocks of shard 0, 1, ... N-1 follow each
// other into the same fp32 accumulator, so the sum over shards costs no
// extra pass over memory.  In the per-shard-partials mode the tile space is
// multiplied by the shard count and each tile sums only its shard's K range.
//
// Every wait is bounded (see wait_bounded): on timeout the CTA records an
// error word, stops issuing work, drains copies and MMAs still in flight and
// releases its TMEM before exiting.
#pragma once

#include "debug_bounds.cuh"
#include "fp8.cuh"
#include "philox.cuh"
#include "ptx.cuh"

namespace tpmlp {

template <int BN, int STAGES, int EPI_WARPS>
struct GemmShape {
  static_assert(BN == 64 || BN == 128 || BN == 256, "BN");
  static constexpr int kATile = kBM * kBK * 2;  // bytes of one A k-block
  static constexpr int kBTile = BN * kBK * 2;   // bytes of one B k-block
  static constexpr int kStage = kATile + kBTile;
  static constexpr int kTmemCols = 2 * BN;      // two fp32 accumulators of BN columns
  static constexpr int kThreads = 64 + 32 * EPI_WARPS;
  static constexpr int kBarrierBytes = 256;
  static constexpr int kSmem = 1024 + STAGES * kStage + kBarrierBytes;
};

__device__ __forceinline__ void tile_coords(const GemmParams& p, int tile, int& shard, int& mb, int& nb) {
  const int per_shard = p.m_blocks * p.n_blocks;
  shard = tile / per_shard;
  const int t = tile - shard * per_shard;
  const int group = p.group_m * p.n_blocks;
  const int g = t / group;
  const int first_m = g * p.group_m;
  const int gm = min(p.m_blocks - first_m, p.group_m);
  const int in = t - g * group;
  mb = first_m + in % gm;
  nb = in / gm;
}

// 32 consecutive bf16 of one row; columns at or beyond N (a multiple of 8) are skipped.
__device__ __forceinline__ void store_row32(__nv_bfloat16* row_ptr, int col0, int N, const float (&x)[32]) {
  uint4* d = reinterpret_cast<uint4*>(row_ptr + col0);
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    if (col0 + 8 * g < N) {
      uint4 u;
      u.x = pack_bf16x2(x[8 * g + 0], x[8 * g + 1]);
      u.y = pack_bf16x2(x[8 * g + 2], x[8 * g + 3]);
      u.z = pack_bf16x2(x[8 * g + 4], x[8 * g + 5]);
      u.w = pack_bf16x2(x[8 * g + 6], x[8 * g + 7]);
      d[g] = u;
    }
  }
}

__device__ __forceinline__ void load_row32(const __nv_bfloat16* row_ptr, int col0, int N, float (&x)[32]) {
  const uint4* s = reinterpret_cast<const uint4*>(row_ptr + col0);
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint4 u = make_uint4(0, 0, 0, 0);
    if (col0 + 8 * g < N) u = __ldg(s + g);
    float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z), e = unpack_bf16x2(u.w);
    x[8 * g + 0] = a.x; x[8 * g + 1] = a.y; x[8 * g + 2] = b.x; x[8 * g + 3] = b.y;
    x[8 * g + 4] = c.x; x[8 * g + 5] = c.y; x[8 * g + 6] = e.x; x[8 * g + 7] = e.y;
  }
}

// Raw 64-byte load of 32 bf16 (zeros past N or for rows past M), unpacked later.
__device__ __forceinline__ void load_raw32(const __nv_bfloat16* row_ptr, int col0, int N, bool ok, uint4 (&u)[4]) {
  const uint4* s = reinterpret_cast<const uint4*>(row_ptr + col0);
#pragma unroll
  for (int g = 0; g < 4; ++g) u[g] = (ok && col0 + 8 * g < N) ? __ldg(s + g) : make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ void unpack_row32(const uint4 (&u)[4], float (&x)[32]) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    float2 a = unpack_bf16x2(u[g].x), b = unpack_bf16x2(u[g].y), c = unpack_bf16x2(u[g].z), e = unpack_bf16x2(u[g].w);
    x[8 * g + 0] = a.x; x[8 * g + 1] = a.y; x[8 * g + 2] = b.x; x[8 * g + 3] = b.y;
    x[8 * g + 4] = c.x; x[8 * g + 5] = c.y; x[8 * g + 6] = e.x; x[8 * g + 7] = e.y;
  }
}

// Sum of each of the 32 columns over the warp's 32 rows, by recursive halving
// (31 shuffles).  Lane l ends with the sum of column l; the order of the
// additions is fixed, so the result is deterministic.
__device__ __forceinline__ float warp_column_sums(float (&v)[32], uint32_t lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

// Per-thread epilogue state: the FP8 dequantisation factor, the output scale and the running amax.
struct EpiState {
  float descale;
  float scale_out;
  float amax;
};

// FP8(x * s) for 32 values -> 32 bytes of one row (columns at or beyond N, a multiple of 16, skipped);
// FMT 0 = E4M3, 1 = E5M2.
template <int FMT>
__device__ __forceinline__ void store_row32_fp8(uint8_t* row_ptr, int col0, int N, const float (&x)[32], float s) {
  uint4* d = reinterpret_cast<uint4*>(row_ptr + col0);
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    if (col0 + 16 * g < N) {
      const float* y = x + 16 * g;
      d[g] = make_uint4(fp8x4<FMT>(y[0], y[1], y[2], y[3], s), fp8x4<FMT>(y[4], y[5], y[6], y[7], s),
                        fp8x4<FMT>(y[8], y[9], y[10], y[11], s), fp8x4<FMT>(y[12], y[13], y[14], y[15], s));
    }
  }
}

// The sequence-parallel tail on 32 columns of one output row:
// v = res + keep * (v + bias2) * scale, res from the residual chunk of the row.
__device__ __forceinline__ void sp_tail_32(const GemmParams& p, float (&v)[32], int row, int col0) {
  if (p.bias != nullptr) {
    float b[32];
    load_row32(static_cast<const __nv_bfloat16*>(p.bias), col0, p.N, b);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] += b[i];
  }
  if (p.drop_thr < kKeepAll) {
    // element index row * N + col0 is a multiple of 8 (N % 8 == 0, col0 % 32 == 0): four whole blocks
    const unsigned long long q0 = (static_cast<unsigned long long>(row) * p.N + col0) >> 3;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint32_t m = dropout_keep8(q0 + g, p.drop_offset, p.drop_seed, p.drop_thr);
      if (p.drop_mask != nullptr && col0 + 8 * g < p.N) p.drop_mask[q0 + g] = static_cast<uint8_t>(m);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[8 * g + j] = (m >> j) & 1u ? v[8 * g + j] * p.drop_scale : 0.f;
    }
  } else if (p.drop_scale != 1.f) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] *= p.drop_scale;
  }
  if (p.res_chunks.p[0] != nullptr) {
    const int j = row / p.rows_per_chunk;
    float r[32];
    load_row32(static_cast<const __nv_bfloat16*>(p.res_chunks.p[j]) + static_cast<long long>(row - j * p.rows_per_chunk) * p.N,
               col0, p.N, r);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] += r[i];
  }
}

// The warp's 32 rows x 32 columns (row `lane` in lane `lane`) leave through one TMA box store from `buf`
// (2 KB, 1024-byte aligned): bf16 row `lane` at buf + 64 lane, its 16-byte piece j at piece
// j ^ ((lane >> 1) & 3) -- the tensor map's 64-byte swizzle, which also keeps each quarter warp's
// shared-memory writes on distinct banks.  Rows at or beyond M and columns at or beyond N are clipped by
// the copy.  The previous box store from `buf` must have finished reading it first.
__device__ __forceinline__ void box_store_bf16_32(const CUtensorMap* map, uint8_t* buf, const float (&x)[32],
                                                  uint32_t lane, int col0, int row0, int M, int N) {
  if (lane == 0) bulk_wait_read_all();
  __syncwarp();
  uint8_t* r = buf + lane * 64;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint4 u;
    u.x = pack_bf16x2(x[8 * j + 0], x[8 * j + 1]);
    u.y = pack_bf16x2(x[8 * j + 2], x[8 * j + 3]);
    u.z = pack_bf16x2(x[8 * j + 4], x[8 * j + 5]);
    u.w = pack_bf16x2(x[8 * j + 6], x[8 * j + 7]);
    *reinterpret_cast<uint4*>(r + ((j ^ ((lane >> 1) & 3)) << 4)) = u;
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0 && row0 < M && col0 < N) {
    tma_store_2d(map, buf, col0, row0);
    bulk_commit_group();
  }
}

// `sbuf` != nullptr: the bf16 outputs that p.tma_out marks leave through box_store_bf16_32.
template <int EPI>
__device__ __forceinline__ void epilogue_32(const GemmParams& p, float (&v)[32], const uint4 (&aux_raw)[4], int row,
                                            int col0, int shard, int mb, int quad, uint32_t lane, EpiState& st,
                                            uint8_t* sbuf = nullptr) {
  const bool row_ok = row < p.M;
  if (st.descale != 1.f) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] *= st.descale;
  }
  if constexpr (EPI == kEpiBiasGeluQ) {
    if (p.bias != nullptr) {
      float b[32];
      load_row32(static_cast<const __nv_bfloat16*>(p.bias), col0, p.N, b);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] += b[i];
    }
    if (row_ok) {
      if (p.out1 != nullptr)
        store_row32(static_cast<__nv_bfloat16*>(p.out1) + static_cast<long long>(row) * p.ld1, col0, p.N, v);
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float2 y = gelu2(make_float2(v[i], v[i + 1]));
        v[i] = y.x;
        v[i + 1] = y.y;
      }
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (col0 + i < p.N) st.amax = fmaxf(st.amax, fabsf(v[i]));
      store_row32_fp8<0>(static_cast<uint8_t*>(p.out0) + static_cast<long long>(row) * p.ld0, col0, p.N, v,
                         st.scale_out);
    }
  } else if constexpr (EPI == kEpiBiasGelu || EPI == kEpiBias) {
    if (p.bias != nullptr) {
      float b[32];
      load_row32(static_cast<const __nv_bfloat16*>(p.bias), col0, p.N, b);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] += b[i];
    }
    if (sbuf != nullptr && (p.tma_out & 1)) {
      const int row0 = row - static_cast<int>(lane);
      if constexpr (EPI == kEpiBiasGelu) {
        if (p.tma_out & 2) box_store_bf16_32(&p.tmC1, sbuf, v, lane, col0, row0, p.M, p.N);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 y = gelu2(make_float2(v[i], v[i + 1]));
          v[i] = y.x;
          v[i + 1] = y.y;
        }
      }
      box_store_bf16_32(&p.tmC0, sbuf, v, lane, col0, row0, p.M, p.N);
    } else if (row_ok) {
      if constexpr (EPI == kEpiBiasGelu) {
        if (p.out1 != nullptr) store_row32(static_cast<__nv_bfloat16*>(p.out1) + row * p.ld1, col0, p.N, v);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 y = gelu2(make_float2(v[i], v[i + 1]));
          v[i] = y.x;
          v[i + 1] = y.y;
        }
      }
      store_row32(static_cast<__nv_bfloat16*>(p.out0) + row * p.ld0, col0, p.N, v);
    }
  } else if constexpr (EPI == kEpiStore) {
    if (sbuf != nullptr && (p.tma_out & 1)) {
      box_store_bf16_32(&p.tmC0, sbuf, v, lane, col0, row - static_cast<int>(lane), p.M, p.N);
    } else if (row_ok) {
      __nv_bfloat16* dst;
      bool ok = true;
      if (p.rows_per_chunk > 0) {
        if (p.tail) sp_tail_32(p, v, row, col0);
        const int j = row / p.rows_per_chunk;
        ok = TPMLP_IN_BOUNDS(j, (p.M + p.rows_per_chunk - 1) / p.rows_per_chunk, kBoundsGemmChunk);
        dst = static_cast<__nv_bfloat16*>(p.chunks.p[ok ? j : 0]) +
              static_cast<long long>(row - j * p.rows_per_chunk) * p.ld0;
      } else {
        ok = TPMLP_IN_BOUNDS(shard, p.shards, kBoundsGemmShard);
        dst = static_cast<__nv_bfloat16*>(p.out0) + shard * p.shard_stride0 + static_cast<long long>(row) * p.ld0;
      }
      if (ok) store_row32(dst, col0, p.N, v);
    }
  } else if constexpr (EPI == kEpiDGeluQ) {
    // v = dH (dequantised); aux = Hpre.  g = dH * GeLU'(Hpre) -> E5M2 with the output scale, amax, column sums.
    float h[32];
    unpack_row32(aux_raw, h);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float2 x = make_float2(h[i], h[i + 1]);
      const NormalCdfPdf2 n = normal_cdf_pdf2(x);
      const float2 d = __fmul2_rn(make_float2(v[i], v[i + 1]), __ffma2_rn(x, n.pdf, n.cdf));  // dH GeLU'(h)
      v[i] = row_ok && col0 + i < p.N ? d.x : 0.f;
      v[i + 1] = row_ok && col0 + i + 1 < p.N ? d.y : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) st.amax = fmaxf(st.amax, fabsf(v[i]));
    if (row_ok)
      store_row32_fp8<1>(static_cast<uint8_t*>(p.out0) + static_cast<long long>(row) * p.ld0, col0, p.N, v,
                         st.scale_out);
    if (p.colsum != nullptr) {
      const float s = warp_column_sums(v, lane);
      const int col = col0 + static_cast<int>(lane);
      // a 128-row block that starts at or past row M (the odd CTA of a last, half-empty pair tile) writes
      // nothing: the partial rows stay 4 per 128-row block of M
      if (col < p.N && mb * kBM < p.M &&
          TPMLP_IN_BOUNDS(mb * 4 + quad, 4 * ((p.M + kBM - 1) / kBM), kBoundsGemmColsum))
        p.colsum[static_cast<long long>(mb * 4 + quad) * p.N + col] = s;
    }
  } else if constexpr (EPI == kEpiDGelu) {
    // v = dH = dY B^T; aux = Hpre.  dHpre = dH * (Phi(h) + h phi(h)); with out1 also H = h Phi(h),
    // Phi and phi sharing one exponential.
    float h[32];
    unpack_row32(aux_raw, h);
    const bool want_h = p.out1 != nullptr;
    float g[32];
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float2 x = make_float2(h[i], h[i + 1]);
      const NormalCdfPdf2 n = normal_cdf_pdf2(x);
      const float2 gg = __fmul2_rn(x, n.cdf);                                                  // H = h Phi(h)
      const float2 d = __fmul2_rn(make_float2(v[i], v[i + 1]), __ffma2_rn(x, n.pdf, n.cdf));  // dH GeLU'(h)
      g[i] = gg.x;
      g[i + 1] = gg.y;
      v[i] = row_ok ? d.x : 0.f;
      v[i + 1] = row_ok ? d.y : 0.f;
    }
    if (row_ok) {
      store_row32(static_cast<__nv_bfloat16*>(p.out0) + static_cast<long long>(row) * p.ld0, col0, p.N, v);
      if (want_h)
        store_row32(static_cast<__nv_bfloat16*>(p.out1) + static_cast<long long>(row) * p.ld1, col0, p.N, g);
    }
    if (p.colsum != nullptr) {
      const float s = warp_column_sums(v, lane);
      const int col = col0 + static_cast<int>(lane);
      // a 128-row block that starts at or past row M (the odd CTA of a last, half-empty pair tile) writes
      // nothing: the partial rows stay 4 per 128-row block of M
      if (col < p.N && mb * kBM < p.M &&
          TPMLP_IN_BOUNDS(mb * 4 + quad, 4 * ((p.M + kBM - 1) / kBM), kBoundsGemmColsum))
        p.colsum[static_cast<long long>(mb * 4 + quad) * p.N + col] = s;
    }
  }
}

template <int BN, bool A_MN, bool B_MN, int EPI, int STAGES, int EPI_WARPS>
__global__ void __launch_bounds__(64 + 32 * EPI_WARPS, 1) k_gemm_tc(const __grid_constant__ GemmParams p) {
  using S = GemmShape<BN, STAGES, EPI_WARPS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * S::kATile;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * S::kBTile);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull + a, 1);
      mbar_init(tempty + a, EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA);
    tma_prefetch_desc(&p.tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, S::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};
  const int num_tiles = p.m_blocks * p.n_blocks * p.shards;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------------ producer
      const uint64_t pol_a = policy_evict_normal();
      const uint64_t pol_b = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        int shard, mb, nb;
        tile_coords(p, tile, shard, mb, nb);
        const int kb0 = shard * p.k_blocks_per_shard;
        for (int kb = 0; kb < p.k_blocks_per_shard; ++kb) {
          if (!wait_bounded(empty + stage, phase ^ 1u, wc, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full + stage, S::kStage);
          const int k0 = (kb0 + kb) * kBK;
          uint8_t* a_dst = sA + stage * S::kATile;
          uint8_t* b_dst = sB + stage * S::kBTile;
          if constexpr (!A_MN) {
            tma_load_2d(a_dst, &p.tmA, full + stage, k0, mb * kBM, pol_a);
          } else {
#pragma unroll
            for (int j = 0; j < kBM / 64; ++j)
              tma_load_2d(a_dst + j * 64 * kBK * 2, &p.tmA, full + stage, mb * kBM + 64 * j, k0, pol_a);
          }
          if constexpr (!B_MN) {
            tma_load_2d(b_dst, &p.tmB, full + stage, k0, nb * BN, pol_b);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(b_dst + j * 64 * kBK * 2, &p.tmB, full + stage, nb * BN + 64 * j, k0, pol_b);
          }
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Copies still in flight must land before the CTA's shared memory goes away.
      for (int s = 0; s < STAGES; ++s)
        if (issued & (1u << s)) wait_drain(full + s, (issued_parity >> s) & 1u, p.timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!wait_bounded(tempty + acc, acc_phase ^ 1u, wc, kSiteMmaTmemEmpty)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < p.k_blocks_per_shard; ++kb) {
          if (!wait_bounded(full + stage, phase, wc, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_base = smem_u32(sA + stage * S::kATile);
          const uint32_t b_base = smem_u32(sB + stage * S::kBTile);
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            // K-major: the 16-element k step is 32 bytes inside the 128-byte swizzled row.
            // MN-major: 16 k rows of 128 bytes; 64-wide MN blocks are one TMA box (LBO) apart.
            const uint64_t ad = A_MN ? sdesc_sw128(a_base + k * 2048, 64 * kBK * 2, 1024)
                                     : sdesc_sw128(a_base + k * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(b_base + k * 2048, 64 * kBK * 2, 1024)
                                     : sdesc_sw128(b_base + k * 32, 16, 1024);
            umma_bf16(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          umma_commit(empty + stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(tfull + acc);
      }
      // Every MMA issued above must finish before TMEM is released.
      umma_commit(drain);
      wait_drain(drain, 0, p.timeout_ns);
    }
  } else {
    // -------------------------------------------------------------------- epilogue
    const int ew = warp - 2;
    const int quad = warp & 3;                      // TMEM lanes this warp may read
    constexpr int kSplit = EPI_WARPS / 4;           // warps sharing a quadrant split the columns
    constexpr int kColsPerPart = BN / kSplit;
    const int part = ew / 4;
    EpiState est{1.f, 1.f, 0.f};  // the single-CTA kernel runs bf16 operands only
    int local = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
      int shard, mb, nb;
      tile_coords(p, tile, shard, mb, nb);
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if constexpr (EPI == kEpiDGelu) {
        // While this tile's MMAs run, pull the warp's 32 rows of the pre-activation tile into L2.
        const int prow = mb * kBM + quad * 32 + static_cast<int>(lane);
        const int pcol = nb * BN + part * kColsPerPart;
        if (prow < p.M && pcol < p.N) {
          const int ncols = min(kColsPerPart, p.N - pcol);
          prefetch_l2_bulk(static_cast<const __nv_bfloat16*>(p.aux) + static_cast<long long>(prow) * p.ld_aux + pcol,
                           static_cast<uint32_t>(ncols) * 2u);
        }
      }
      int ok = 1;
      if (lane == 0) ok = wait_bounded(tfull + acc, acc_phase, wc, kSiteEpiTmemFull) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      const int row = mb * kBM + quad * 32 + static_cast<int>(lane);
      const int c_begin = part * kColsPerPart, c_end = (part + 1) * kColsPerPart;
      // The pre-activation operand of the GeLU' epilogue is fetched one chunk ahead.
      const __nv_bfloat16* aux_row = nullptr;
      uint4 aux_next[4] = {};
      if constexpr (EPI == kEpiDGelu) {
        aux_row = static_cast<const __nv_bfloat16*>(p.aux) + static_cast<long long>(row < p.M ? row : 0) * p.ld_aux;
        load_raw32(aux_row, nb * BN + c_begin, p.N, row < p.M, aux_next);
      }
#pragma unroll 1
      for (int c = c_begin; c < c_end; c += 32) {
        uint4 aux_cur[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) aux_cur[g] = aux_next[g];
        if constexpr (EPI == kEpiDGelu) {
          if (c + 32 < c_end) load_raw32(aux_row, nb * BN + c + 32, p.N, row < p.M, aux_next);
        }
        float v[32];
        tmem_load_32cols(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN + c), v);
        epilogue_32<EPI>(p, v, aux_cur, row, nb * BN + c, shard, mb, quad, lane, est);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty + acc);
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, S::kTmemCols);
  }
}

}  // namespace tpmlp
