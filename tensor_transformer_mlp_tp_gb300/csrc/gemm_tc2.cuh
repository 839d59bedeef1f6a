// The tcgen05 GEMM on CTA pairs (cta_group::2): a cluster of two CTAs on two
// SMs computes a 256 x BN output tile with one 256 x BN x 16 UMMA per k-step.
//
// CTA r of the pair (r = %cluster_ctarank) loads rows [128 r, 128 r + 128) of
// the A tile and columns [r BN/2, (r+1) BN/2) of the B tile, 32 KB per k-block
// for BN = 256 instead of the 48 KB a single CTA needs for a 128 x 256 tile:
// a third less L2 -> SM traffic per flop and room for a deeper ring.  Each
// CTA's TMEM holds its 128 rows of the accumulator (double-buffered), and each
// CTA runs its own epilogue on them.
//
// Synchronisation:
//   full[s]    lives in the even CTA; both CTAs' TMA copies count their bytes
//              on it (cta_group::2 copies may signal the peer's barrier), the
//              even CTA arms it with the pair's total.
//   empty[s]   one per CTA; the MMA commit multicasts to both.
//   tfull[a]   one per CTA; the MMA commit multicasts to both.
//   tempty[a]  lives in the even CTA; every epilogue warp of both CTAs arrives.
// Epilogue warps: warps 2..5 own the four TMEM lane quadrants (quadrant =
// warp % 4).  The quadrant-0 and quadrant-1 warps share SM sub-partitions with
// the TMA producer (warp 0) and the MMA issuer (warp 1); measured on GB300, the
// ALU stream of a GeLU epilogue next to the MMA issuer slows the MMAs by ~8%.
// So those two warps only copy their accumulator rows TMEM -> shared memory
// (a swizzled double buffer per quadrant, `filled`/`drained` barriers), and
// helper warps 6 and 7 (sub-partitions 2 and 3) run the epilogue math and the
// stores for them.
// Only the even CTA's warp 1 issues MMAs.  Waits are bounded as in the
// single-CTA kernel; the pair meets at a cluster barrier before TMEM is
// released and before either CTA exits (the even CTA's MMAs read the odd
// CTA's shared memory).
// bf16 outputs that a tensor map describes leave as 32 x 32 TMA box stores
// from a 2 KB shared-memory buffer per storing warp.  A last wave of at most
// half the pairs' tiles runs as one round of half-width tiles (unit_of).  The
// kernel is launched with programmatic stream serialisation: its set-up
// overlaps the previous kernel's tail, and griddepcontrol.wait precedes its
// first global access.
#pragma once

#include "gemm_tc.cuh"

namespace tpmlp {

template <int BN, int STAGES, int EPI_WARPS, int BAL = 0>
struct PairShape {
  static_assert(BN == 128 || BN == 256, "BN");
  static constexpr int kHalfN = BN / 2;
  static constexpr int kATile = 128 * kBK * 2;     // this CTA's 128 rows of A
  static constexpr int kBTile = kHalfN * kBK * 2;  // this CTA's half of the B columns
  static constexpr int kStage = kATile + kBTile;
  static constexpr int kTmemCols = 2 * BN;
  static constexpr int kThreads = BAL > 0 ? 64 + 32 * BAL : 64 + 32 * EPI_WARPS + 64;  // + two helper warps
  // reader -> helper staging [quadrant 0/1][buffer][32 rows][32 fp32] (BAL = 0 only)
  static constexpr int kStaging = BAL > 0 ? 0 : 2 * 2 * 32 * 32 * 4;
  // one 2 KB TMA box-store buffer per warp that stores: the BAL epilogue warps, or warps 2, 3, 6, 7
  static constexpr int kStoreWarps = BAL > 0 ? BAL : 4;
  static constexpr int kStoreBuf = 32 * 32 * 2;
  static constexpr int kSmem = 1024 + STAGES * kStage + kStaging + kStoreWarps * kStoreBuf + 256;
  static_assert(EPI_WARPS == 4, "one epilogue warp per TMEM lane quadrant");
  static_assert(kSmem <= 232448, "shared memory per block");
};

// Work unit u of the pair kernel (see GemmParams::full_units): its tile, the tile's first output column
// relative to the tile (0, or BN / 2 for the upper half) and its width (BN, or BN / 2 for a half).
template <int BN>
__device__ __forceinline__ void unit_of(const GemmParams& p, int u, int& tile, int& col_off, int& width) {
  if (u < p.full_units) {
    tile = u;
    col_off = 0;
    width = BN;
  } else {
    const int j = u - p.full_units;
    tile = p.full_units + (j >> 1);
    col_off = (j & 1) * (BN / 2);
    width = BN / 2;
  }
}

// FP8: E4M3 A and B (both K-major), .kind::f8f6f4; a 128-byte k-block row then holds 128 elements and
// one UMMA covers 32 of them, so shared-memory layouts, descriptors and byte counts are those of bf16.
// BAL > 0: BAL epilogue warps (warps 2 .. BAL + 1), each reading TMEM itself, with the epilogue math
// spread evenly over all four SM sub-partitions (for epilogue-bound launches: short K or the FP8 rate);
// BAL = 0: the two warps on the TMA and MMA sub-partitions only copy TMEM to shared memory for the
// two helper warps.
template <int BN, bool A_MN, bool B_MN, int EPI, int STAGES, int EPI_WARPS, bool FP8 = false, int BAL = 0>
__global__ void __launch_bounds__(BAL > 0 ? 64 + 32 * BAL : 128 + 32 * EPI_WARPS, 1)
    k_gemm_tc2(const __grid_constant__ GemmParams p) {
  static_assert(!FP8 || (!A_MN && !B_MN), "FP8 operands are K-major");
  static_assert(FP8 || (EPI != kEpiBiasGeluQ && EPI != kEpiDGeluQ), "the quantising epilogues follow FP8 operands");
  constexpr bool kAux = EPI == kEpiDGelu || EPI == kEpiDGeluQ;  // reads the pre-activation tile
  // FP8 GEMMs with a GeLU / GeLU' epilogue are epilogue-bound at the doubled MMA rate: there every epilogue
  // warp reads TMEM itself and the math is spread over all four SM sub-partitions (see the epilogue).
  static_assert(BAL == 0 || (BAL >= 4 && BAL <= 14), "balanced epilogue: 4 to 14 warps");
  constexpr bool kBalanced = BAL > 0;
  constexpr int kTemptyArrivals = 2 * (kBalanced ? BAL : EPI_WARPS);
  constexpr int kKElems = FP8 ? 128 : kBK;  // elements of one 128-byte k-block row
  using S = PairShape<BN, STAGES, EPI_WARPS, BAL>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * S::kATile;
  float* staging = reinterpret_cast<float*>(sB + STAGES * S::kBTile);
  uint8_t* store_bufs = reinterpret_cast<uint8_t*>(staging) + S::kStaging;  // 1024-byte aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(store_bufs + S::kStoreWarps * S::kStoreBuf);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* filled = drain + 1;    // [quadrant 0/1][buffer]
  uint64_t* drained = filled + 4;  // [quadrant 0/1][buffer]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drained + 4);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull + a, 1);
      mbar_init(tempty + a, kTemptyArrivals);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(filled + i, 1);
      mbar_init(drained + i, 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA);
    tma_prefetch_desc(&p.tmB);
    if (!B_MN && p.full_units < p.m_blocks * p.n_blocks * p.shards) tma_prefetch_desc(&p.tmB_half);
    if (p.tma_out & 1) tma_prefetch_desc(&p.tmC0);
    if (p.tma_out & 2) tma_prefetch_desc(&p.tmC1);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, S::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers are initialised before any remote arrive or copy
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // The set-up above touches no global memory; with a programmatic launch it overlaps the previous
  // kernel's tail.  Every global read and write below comes after that kernel has completed.  The next
  // kernel may launch now: its blocks take an SM as this kernel's blocks leave.
  griddep_wait();
  griddep_launch_dependents();

  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};
  const int num_tiles = p.m_blocks * p.n_blocks * p.shards;  // m_blocks counts 256-row pair tiles
  const int num_units = p.full_units + 2 * (num_tiles - p.full_units);
  const int cluster_id = blockIdx.x >> 1;
  const int num_clusters = gridDim.x >> 1;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------------ producer (both CTAs)
      const uint64_t pol_a = policy_evict_normal();
      const uint64_t pol_b = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;
      bool ok = true;
      for (int u = cluster_id; ok && u < num_units; u += num_clusters) {
        int tile, col_off, width;
        unit_of<BN>(p, u, tile, col_off, width);
        int shard, mb, nb;
        tile_coords(p, tile, shard, mb, nb);
        const int kb0 = shard * p.k_blocks_per_shard;
        const int m0 = mb * 256 + static_cast<int>(rank) * 128;
        const int n0 = nb * BN + col_off + static_cast<int>(rank) * (width / 2);  // this CTA's half of the columns
        const uint32_t stage_bytes = static_cast<uint32_t>(S::kATile + (width / 2) * kBK * 2);
        for (int kb = 0; kb < p.k_blocks_per_shard; ++kb) {
          if (!wait_bounded(empty + stage, phase ^ 1u, wc, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(full + stage, 2 * stage_bytes);
          const uint32_t bar = mapa_shared(smem_u32(full + stage), 0);
          const int k0 = (kb0 + kb) * kKElems;
          uint8_t* a_dst = sA + stage * S::kATile;
          uint8_t* b_dst = sB + stage * S::kBTile;
          if constexpr (!A_MN) {
            tma_load_2d_pair(a_dst, &p.tmA, bar, k0, m0, pol_a);
          } else {
#pragma unroll
            for (int j = 0; j < 2; ++j) tma_load_2d_pair(a_dst + j * 64 * kBK * 2, &p.tmA, bar, m0 + 64 * j, k0, pol_a);
          }
          if constexpr (!B_MN) {
            tma_load_2d_pair(b_dst, width == BN ? &p.tmB : &p.tmB_half, bar, k0, n0, pol_b);
          } else {
            for (int j = 0; j < width / 128; ++j)  // 64-column boxes
              tma_load_2d_pair(b_dst + j * 64 * kBK * 2, &p.tmB, bar, n0 + 64 * j, k0, pol_b);
          }
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Copies in flight must land before shared memory is released.  The even
      // CTA's full barriers count both CTAs' bytes; the odd CTA is held at the
      // closing cluster barrier until the even CTA has drained.
      if (leader)
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s)) wait_drain(full + s, (issued_parity >> s) & 1u, p.timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------------ MMA issuer (even CTA)
      const uint32_t idesc_full = FP8 ? idesc_f8_f32(256, BN, static_cast<uint32_t>(p.a_fmt),
                                                     static_cast<uint32_t>(p.b_fmt), false, false)
                                      : idesc_bf16_f32(256, BN, A_MN, B_MN);
      const uint32_t idesc_half = FP8 ? idesc_f8_f32(256, BN / 2, static_cast<uint32_t>(p.a_fmt),
                                                     static_cast<uint32_t>(p.b_fmt), false, false)
                                      : idesc_bf16_f32(256, BN / 2, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int u = cluster_id; ok && u < num_units; u += num_clusters, ++local) {
        const uint32_t idesc = u < p.full_units ? idesc_full : idesc_half;
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
            const uint64_t ad = A_MN ? sdesc_sw128(a_base + k * 2048, 64 * kBK * 2, 1024)
                                     : sdesc_sw128(a_base + k * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(b_base + k * 2048, 64 * kBK * 2, 1024)
                                     : sdesc_sw128(b_base + k * 32, 16, 1024);
            if constexpr (FP8) {
              umma_f8_pair(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
            } else {
              umma_bf16_pair(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
            }
          }
          umma_commit_pair_multicast(empty + stage, 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_multicast(tfull + acc, 0x3);
      }
      umma_commit_pair(drain);
      wait_drain(drain, 0, p.timeout_ns);
    }
  } else if constexpr (kBalanced) {
    // -------------------------------------------------------------------- epilogue, balanced (both CTAs)
    // Warp w may read only TMEM lane quadrant w % 4, so the warps of one quadrant (w, w + 4, ...) split
    // its BN / 32 column chunks between them; sub-partition w % 4 then runs exactly one quadrant's worth
    // of math whatever BAL is.  With BAL = 6: warp 4 (next to the TMA producer) and warp 5 (next to the
    // MMA issuer) take all columns of theirs, warps 2 + 6 and 3 + 7 half each.
    const int quad = warp & 3;
    const int first = quad >= 2 ? quad : quad + 4;  // lowest epilogue warp of this quadrant
    const int n_quad = (BAL + 2 - first + 3) / 4;    // epilogue warps of this quadrant
    const int i_quad = (warp - first) / 4;
    const int c_begin = 32 * (i_quad * (BN / 32) / n_quad);
    const int c_end = 32 * ((i_quad + 1) * (BN / 32) / n_quad);
    uint8_t* sbuf = store_bufs + (warp - 2) * S::kStoreBuf;
    EpiState est{1.f, 1.f, 0.f};
    if constexpr (FP8) est.descale = 1.f / (__ldg(p.scale_a) * __ldg(p.scale_b));
    if constexpr (EPI == kEpiBiasGeluQ || EPI == kEpiDGeluQ) est.scale_out = __ldg(p.scale_out);
    int local = 0;
    for (int u = cluster_id; u < num_units; u += num_clusters, ++local) {
      int tile, col_off, width;
      unit_of<BN>(p, u, tile, col_off, width);
      int shard, mb, nb;
      tile_coords(p, tile, shard, mb, nb);
      const int n_base = nb * BN + col_off;     // the unit's first output column
      const int c_stop = min(c_end, width);     // this warp's chunks within the unit
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      const int mb128 = mb * 2 + static_cast<int>(rank);
      const int row = mb128 * 128 + quad * 32 + static_cast<int>(lane);
      const __nv_bfloat16* aux_row = nullptr;
      uint4 aux_next[4] = {};
      if constexpr (kAux) {
        // pull this warp's rows and columns of the pre-activation tile into L2 while the tile's MMAs run
        const int pcol = n_base + c_begin;
        const int ncols = min(c_stop - c_begin, p.N - pcol);
        if (row < p.M && ncols > 0)
          prefetch_l2_bulk(static_cast<const __nv_bfloat16*>(p.aux) + static_cast<long long>(row) * p.ld_aux + pcol,
                           static_cast<uint32_t>(ncols) * 2u);
      }
      int ok = 1;
      if (lane == 0) ok = wait_bounded(tfull + acc, acc_phase, wc, kSiteEpiTmemFull) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t trow = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN);
      if constexpr (kAux) {
        aux_row = static_cast<const __nv_bfloat16*>(p.aux) + static_cast<long long>(row < p.M ? row : 0) * p.ld_aux;
        if (c_begin < c_stop) load_raw32(aux_row, n_base + c_begin, p.N, row < p.M, aux_next);
      }
#pragma unroll 1
      for (int c = c_begin; c < c_stop; c += 32) {
        uint4 aux_cur[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) aux_cur[g] = aux_next[g];
        if constexpr (kAux) {
          if (c + 32 < c_stop) load_raw32(aux_row, n_base + c + 32, p.N, row < p.M, aux_next);
        }
        float v[32];
        tmem_load_32cols(trow + static_cast<uint32_t>(c), v);
        epilogue_32<EPI>(p, v, aux_cur, row, n_base + c, shard, mb128, quad, lane, est, sbuf);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(tempty + acc), 0));
    }
    if (lane == 0) bulk_wait_all();  // box stores complete before the block's shared memory is released
    if constexpr (EPI == kEpiBiasGeluQ || EPI == kEpiDGeluQ) {
      if (p.amax_out != nullptr) amax_combine_warp(p.amax_out, est.amax);
    }
  } else {
    // -------------------------------------------------------------------- epilogue (both CTAs)
    const bool quad_warp = warp < 6;
    const int quad = quad_warp ? (warp & 3) : (warp - 6);  // helper 6 serves quadrant 0, helper 7 quadrant 1
    const bool reader = quad_warp && quad < 2;             // copies TMEM -> staging only
    const bool helper = !quad_warp;                        // epilogue math on staged rows
    float* stage_base = staging + quad * (2 * 32 * 32);    // valid for quadrants 0 and 1
    uint8_t* obuf = reader ? nullptr : store_bufs + (warp >= 6 ? warp - 4 : warp - 2) * S::kStoreBuf;
    EpiState est{1.f, 1.f, 0.f};
    if constexpr (FP8) est.descale = 1.f / (__ldg(p.scale_a) * __ldg(p.scale_b));
    if constexpr (EPI == kEpiBiasGeluQ || EPI == kEpiDGeluQ) est.scale_out = __ldg(p.scale_out);
    uint32_t chunk_ctr = 0;
    int local = 0;
    bool ok_all = true;
    for (int u = cluster_id; ok_all && u < num_units; u += num_clusters, ++local) {
      int tile, col_off, width;
      unit_of<BN>(p, u, tile, col_off, width);
      int shard, mb, nb;
      tile_coords(p, tile, shard, mb, nb);
      const int n_base = nb * BN + col_off;     // the unit's first output column
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      const int mb128 = mb * 2 + static_cast<int>(rank);
      const int row = mb128 * 128 + quad * 32 + static_cast<int>(lane);
      if constexpr (kAux) {
        // While this tile's MMAs run, pull the warp's 32 rows of the pre-activation tile into L2.
        if (!reader && row < p.M) {
          const int pcol = n_base;
          const int ncols = min(width, p.N - pcol);
          prefetch_l2_bulk(static_cast<const __nv_bfloat16*>(p.aux) + static_cast<long long>(row) * p.ld_aux + pcol,
                           static_cast<uint32_t>(ncols) * 2u);
        }
      }
      if (!helper) {
        int ok = 1;
        if (lane == 0) ok = wait_bounded(tfull + acc, acc_phase, wc, kSiteEpiTmemFull) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after_sync();
      }
      const uint32_t trow = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN);
      const __nv_bfloat16* aux_row = nullptr;
      uint4 aux_next[4] = {};
      if constexpr (kAux) {
        if (!reader) {
          aux_row = static_cast<const __nv_bfloat16*>(p.aux) + static_cast<long long>(row < p.M ? row : 0) * p.ld_aux;
          load_raw32(aux_row, n_base, p.N, row < p.M, aux_next);
        }
      }
#pragma unroll 1
      for (int c = 0; c < width; c += 32, ++chunk_ctr) {
        const uint32_t buf = chunk_ctr & 1u, par = (chunk_ctr >> 1) & 1u;
        float* sbuf = stage_base + buf * (32 * 32) + lane * 32;
        float v[32];
        if (reader) {
          int ok = 1;
          if (lane == 0) ok = wait_bounded(drained + quad * 2 + buf, par ^ 1u, wc, kSiteEpiStageDrained) ? 1 : 0;
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) {
            ok_all = false;
            break;
          }
          tmem_load_32cols(trow + static_cast<uint32_t>(c), v);
          // row `lane` of the staged chunk, 16-byte pieces swizzled by (lane & 7): conflict-free per quarter warp
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(sbuf + ((j ^ (lane & 7)) * 4)) = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          __syncwarp();
          if (lane == 0) mbar_arrive(filled + quad * 2 + buf);
          continue;
        }
        uint4 aux_cur[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) aux_cur[g] = aux_next[g];
        if constexpr (kAux) {
          if (c + 32 < width) load_raw32(aux_row, n_base + c + 32, p.N, row < p.M, aux_next);
        }
        if (helper) {
          int ok = 1;
          if (lane == 0) ok = wait_bounded(filled + quad * 2 + buf, par, wc, kSiteEpiStageFilled) ? 1 : 0;
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) {
            ok_all = false;
            break;
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 f = *reinterpret_cast<const float4*>(sbuf + ((j ^ (lane & 7)) * 4));
            v[4 * j] = f.x;
            v[4 * j + 1] = f.y;
            v[4 * j + 2] = f.z;
            v[4 * j + 3] = f.w;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(drained + quad * 2 + buf);
        } else {
          tmem_load_32cols(trow + static_cast<uint32_t>(c), v);
        }
        epilogue_32<EPI>(p, v, aux_cur, row, n_base + c, shard, mb128, quad, lane, est, obuf);
      }
      if (!helper && ok_all) {
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(tempty + acc), 0));
      }
    }
    if (lane == 0 && !reader) bulk_wait_all();  // box stores complete before shared memory is released
    if constexpr (EPI == kEpiBiasGeluQ || EPI == kEpiDGeluQ) {
      if (p.amax_out != nullptr) amax_combine_warp(p.amax_out, est.amax);
    }
  }

  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, S::kTmemCols);
  }
}

}  // namespace tpmlp
