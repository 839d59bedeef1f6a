// Tensor-parallel attention: the per-head attention core on tcgen05, forward and
// backward, and the block (QKV projection, attention, output projection with the
// shard sum, and its backward).
//
// Forward core (persistent CTAs walking 128-query tiles of one batch element and
// head each, head dim 128): softmax(Q K^T / sqrt(hd)) V with an online softmax over
// 128-key tiles.
//   warp 0   TMA producer: Q once, then K and V tiles into 3-stage rings; Q, K,
//            V come straight out of the QKV projection's [S, B, 3, H, hd] layout
//            through 4-D tensor maps (two 64-element boxes per row).
//   warp 1   MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//            buffers, then O += P_{j-1} V_{j-1} once the softmax warps have
//            written P_{j-1}: P from TMEM as the A operand, V the MN-major B
//            operand, O accumulating in TMEM.
//   warps 2..9  softmax: two warps per TMEM lane quadrant (query rows) split
//            each tile's keys; the row maximum is exchanged through shared
//            memory, a reference maximum moves (rescaling O in TMEM) only when a
//            tile's maximum exceeds it by 2^8, and P = exp2(S - m) goes to TMEM
//            in bf16 pairs; the row's denominator and log-sum-exp come at the end.
// Backward core: D = rowsum(dO O); a dQ kernel over query tiles and a dK/dV kernel
// over key tiles (persistent, like the forward) recompute S and dP in TMEM and write
// P, dS in bf16 to TMEM for the gradient MMAs (described at each kernel).  Causal attention masks inside the
// tiles that reach past a row's last key; positions at or past S are masked.
// Every wait is bounded (error word + abort flag), and each CTA drains its copies
// and MMAs before it releases TMEM.
#include <cuda_bf16.h>

#include <climits>
#include <cmath>
#include <cstring>
#include <cudaTypedefs.h>
#include <mutex>

#include "../../include/tpmlp.h"
#include "launch.h"
#include "ptx.cuh"

namespace tpmlp {
namespace {

constexpr int kHd = 128;            // head dimension this kernel is laid out for
constexpr int kQTile = 128;         // queries per CTA (one per TMEM lane)
constexpr int kKTile = 128;         // keys per step
constexpr int kKvStages = 2;
constexpr int kFwdKvStages = 3;     // K and V rings of the forward (P lives in TMEM, not shared memory)
constexpr int kAtom = 128 * 128;    // one 64-element-wide swizzled column of a 128-row tile: 16 KB
constexpr int kTileBytes = 2 * kAtom;  // a 128 x 128 bf16 tile: two atom columns
constexpr int kThreads = 320;  // producer, MMA issuer, 8 softmax warps
constexpr uint32_t kSiteAttnQ = 32, kSiteAttnKv = 33, kSiteAttnS = 34, kSiteAttnP = 35, kSiteAttnSEmpty = 36,
                   kSiteAttnKvEmpty = 37, kSiteAttnPv = 38, kSiteAttnQEmpty = 39, kSiteAttnOEmpty = 40;

struct AttnParams {
  CUtensorMap tmQ, tmK, tmV;
  void* out;          // [T x d] bf16, row s B + b, columns h hd .. (h+1) hd
  float* lse;         // nullptr, or [B H x s_pad] fp32: each row's log2 of sum exp2 (scores in log2 units)
  int s_pad;          // S rounded up to whole 128-query tiles
  int S, B, H;
  int n_qtiles;
  int causal;
  float scale_log2;   // log2(e) / sqrt(hd)
  unsigned int* err;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                            int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// 32 lanes x 32 fp32 columns from TMEM without waiting (tcgen05.wait::ld before the registers are used).
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// The same into float registers.
__device__ __forceinline__ void tmem_ld32f_nowait(uint32_t taddr, float (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7]), "=f"(r[8]),
        "=f"(r[9]), "=f"(r[10]), "=f"(r[11]), "=f"(r[12]), "=f"(r[13]), "=f"(r[14]), "=f"(r[15]), "=f"(r[16]),
        "=f"(r[17]), "=f"(r[18]), "=f"(r[19]), "=f"(r[20]), "=f"(r[21]), "=f"(r[22]), "=f"(r[23]), "=f"(r[24]),
        "=f"(r[25]), "=f"(r[26]), "=f"(r[27]), "=f"(r[28]), "=f"(r[29]), "=f"(r[30]), "=f"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 16 columns into TMEM (thread t writes its lane's 16 words).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Bounded wait without a suspend-time hint: the per-tile handoffs between producer, MMA issuer and softmax
// warps are short and on the critical path, where a sleeping wait's wake-up would add to every tile.
__device__ __forceinline__ bool spin_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool wait_spin(uint64_t* bar, uint32_t parity, const WaitCtx& w, uint32_t site) {
  if (spin_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (spin_try_wait(bar, parity)) return true;
    if (*w.abort) return false;
    if (global_timer_ns() - t0 > w.budget_ns) {
      record_error(w, kErrTimeout, site);
      return false;
    }
  }
}

// The persistent CTAs' items, sorted longest first, dealt in rounds of gridDim.x.  Causal items shrink
// along the order, so the direction is reversed every other round (CTA c takes item r G + c in even rounds r
// and r G + G - 1 - c in odd ones) and no CTA takes the longest item of every round (measured at S = 4096 x
// 2, 32 heads: forward 0.309 -> 0.298 ms, backward 1.185 -> 1.113 ms); items of equal length keep the
// plain order (the reversal measured 1.7% slower on the non-causal forward).  A CTA's first index at or
// past the item count ends its walk (every later round starts beyond it).
__device__ __forceinline__ int item_of_round(int round, bool snake) {
  const int g = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return round * g + ((snake && (round & 1)) ? g - 1 - c : c);
}

// Rows s0 .. s0 + 127 of one part (Q, K or V) of head h, batch b: two boxes of 64 elements.
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int h, int b, int s0) {
  tma_load_4d(dst, map, bar, 0, h, b, s0);
  tma_load_4d(dst + kAtom, map, bar, 64, h, b, s0);
}

// Persistent: one CTA per SM walks the work items (query tile, batch element, head), longest query tiles
// first, items blockIdx.x, blockIdx.x + gridDim.x, ...  The K/V rings, the S and P buffers and their
// barriers run on over the items (phases from a running key-tile count), so the next item's Q load, K/V
// loads and first score MMA overlap the previous item's epilogue: Q is reloaded once the previous
// item's score MMAs have read it (q_empty), and the next item's first P V overwrites O only once the
// softmax warps have read it (o_empty).
__global__ void __launch_bounds__(kThreads, 1) k_attention_fwd(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + kTileBytes;
  uint8_t* sV = sK + kFwdKvStages * kTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + kFwdKvStages * kTileBytes);
  uint64_t* q_full = bars;
  uint64_t* q_empty = q_full + 1;   // every score MMA of the item has read Q
  // K and V have their own barriers: K_j is released as soon as S_j is done, V_j after P_j V_j
  uint64_t* k_full = q_empty + 1;
  uint64_t* k_empty = k_full + kFwdKvStages;
  uint64_t* v_full = k_empty + kFwdKvStages;
  uint64_t* v_empty = v_full + kFwdKvStages;
  uint64_t* s_full = v_empty + kFwdKvStages;
  uint64_t* s_empty = s_full + 2;
  uint64_t* p_full = s_empty + 2;   // [P buffer]
  uint64_t* pv_done = p_full + 2;   // [P buffer]: P V of the tiles that used that buffer
  uint64_t* o_empty = pv_done + 2;  // the softmax warps have read the item's O
  uint64_t* drain = o_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const int bh_count = p.B * p.H;
  const int n_items = p.n_qtiles * bh_count;
  const bool snake = p.causal != 0;  // item order: see item_of_round
  const int n_kt_all = (p.S + kKTile - 1) / kKTile;
  // item w: query tile n_qtiles - 1 - w / (B H) (the longest causal tiles first), batch-head w % (B H)
  auto item_of = [&](int w, int& qt, int& b, int& h, int& nk) {
    qt = p.n_qtiles - 1 - w / bh_count;
    const int bh = w % bh_count;
    b = bh % p.B;
    h = bh / p.B;
    nk = p.causal ? min(n_kt_all, qt + 1) : n_kt_all;
  };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kFwdKvStages; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 1);
      mbar_init(v_full + s, 1);
      mbar_init(v_empty + s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(s_full + s, 1);
      mbar_init(s_empty + s, 8);
      mbar_init(p_full + s, 8);
      mbar_init(pv_done + s, 1);
    }
    mbar_init(o_empty, 8);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;  // S [0, 128) and [128, 256), O [256, 384), P [384, 448) and [448, 512)
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------------ producer
      uint32_t k_issued = 0, k_par = 0, v_issued = 0, v_par = 0, q_par = 0;
      bool q_issued = false, ok = true;
      int g = 0;  // key tiles issued so far, over all items
      for (int it = 0, w = item_of_round(0, snake); ok && w < n_items; ++it, w = item_of_round(it, snake)) {
        int qt, b, h, nk;
        item_of(w, qt, b, h, nk);
        if (it >= 1 && !wait_spin(q_empty, static_cast<uint32_t>(it - 1) & 1u, wc, kSiteAttnQEmpty)) break;
        mbar_arrive_expect_tx(q_full, kTileBytes);
        load_tile(sQ, &p.tmQ, q_full, h, b, qt * kQTile);
        q_issued = true;
        q_par = static_cast<uint32_t>(it) & 1u;
        for (int j = 0; j < nk; ++j, ++g) {
          const int st = g % kFwdKvStages;
          const uint32_t ph = static_cast<uint32_t>(g / kFwdKvStages) & 1u;
          if (!wait_spin(k_empty + st, ph ^ 1u, wc, kSiteAttnKvEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(k_full + st, kTileBytes);
          load_tile(sK + st * kTileBytes, &p.tmK, k_full + st, h, b, j * kKTile);
          k_issued |= 1u << st;
          k_par = (k_par & ~(1u << st)) | (ph << st);
          if (!wait_spin(v_empty + st, ph ^ 1u, wc, kSiteAttnKvEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(v_full + st, kTileBytes);
          load_tile(sV + st * kTileBytes, &p.tmV, v_full + st, h, b, j * kKTile);
          v_issued |= 1u << st;
          v_par = (v_par & ~(1u << st)) | (ph << st);
        }
      }
      // copies in flight land before shared memory is released
      if (q_issued) wait_drain(q_full, q_par, p.timeout_ns);
      for (int s = 0; s < kFwdKvStages; ++s) {
        if (k_issued & (1u << s)) wait_drain(k_full + s, (k_par >> s) & 1u, p.timeout_ns);
        if (v_issued & (1u << s)) wait_drain(v_full + s, (v_par >> s) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------------ MMA issuer
      // step j of an item: S_j = Q K_j^T (j < nk) into S buffer g % 2, then O += P_{j-1} V_{j-1} (j >= 1):
      // O stays in TMEM across the item's key tiles (g = the running key-tile count)
      constexpr uint32_t idesc_s = idesc_bf16_f32(kQTile, kKTile, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kQTile, kHd, false, true);
      const uint32_t q_base = smem_u32(sQ);
      const uint32_t o_tmem = tmem_base + 256;
      bool ok = true;
      int g0 = 0;
      for (int it = 0, w = item_of_round(0, snake); ok && w < n_items; ++it, w = item_of_round(it, snake)) {
        int qt, b, h, nk;
        item_of(w, qt, b, h, nk);
        if (!wait_spin(q_full, static_cast<uint32_t>(it) & 1u, wc, kSiteAttnQ)) break;
        tc_fence_after_sync();
        for (int j = 0; ok && j <= nk; ++j) {
          if (j < nk) {
            const int gj = g0 + j;
            const int sb = gj & 1;
            const int st = gj % kFwdKvStages;
            if (!wait_spin(s_empty + sb, (static_cast<uint32_t>(gj >> 1) & 1u) ^ 1u, wc, kSiteAttnSEmpty) ||
                !wait_spin(k_full + st, static_cast<uint32_t>(gj / kFwdKvStages) & 1u, wc, kSiteAttnKv)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t k_base = smem_u32(sK + st * kTileBytes);
#pragma unroll
            for (int kk = 0; kk < kHd / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
              umma_bf16(tmem_base + sb * 128, sdesc_sw128(q_base + off, 16, 1024),
                        sdesc_sw128(k_base + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
            }
            umma_commit(s_full + sb);
            umma_commit(k_empty + st);
            if (j == nk - 1) umma_commit(q_empty);  // the item's last score MMA: Q may be reloaded
          }
          if (j >= 1) {
            const int gj = g0 + j - 1;
            const int pb = gj & 1;
            const int st = gj % kFwdKvStages;
            // the item's first P V overwrites O: the previous item's epilogue must have read it
            if (j == 1 && it >= 1 && !wait_spin(o_empty, static_cast<uint32_t>(it - 1) & 1u, wc, kSiteAttnOEmpty)) {
              ok = false;
              break;
            }
            if (!wait_spin(p_full + pb, static_cast<uint32_t>(gj >> 1) & 1u, wc, kSiteAttnP) ||
                !wait_spin(v_full + st, static_cast<uint32_t>(gj / kFwdKvStages) & 1u, wc, kSiteAttnKv)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t v_base = smem_u32(sV + st * kTileBytes);
#pragma unroll
            for (int kk = 0; kk < kKTile / 16; ++kk)
              umma_bf16_tmem_a(o_tmem, tmem_base + 384 + 64 * pb + 8 * kk,
                               sdesc_sw128(v_base + kk * 2048, kAtom, 1024), idesc_pv, (j > 1 || kk > 0) ? 1u : 0u);
            umma_commit(pv_done + pb);
            umma_commit(v_empty + st);
          }
        }
        g0 += nk;
      }
      umma_commit(drain);
      wait_drain(drain, 0, p.timeout_ns);
    }
  } else {
    // -------------------------------------------------------------------- softmax (warps 2..9)
    // Warps w and w + 4 share TMEM lane quadrant w % 4 (query rows) and split every tile's keys: half 0
    // takes keys 0..63 (P atom column 0, O columns 0..63), half 1 keys 64..127 (atom column 1, O columns
    // 64..127).  The halves exchange the row maximum once per tile through shared memory (a named
    // barrier per pair); their row sums combine at the end.  m is the row's reference maximum (log2
    // units): exponents are taken against it and O, l are kept relative to it; it moves (and O, l are
    // rescaled) only when a tile's maximum exceeds it by more than kRescaleLog2, so exp2(s - m) <= 2^8.
    constexpr float kRescaleLog2 = 8.f;
    __shared__ float xchg[2][kQTile];  // [half][row]: the tile's row maximum, at the end the row sum
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int pair_bar = 1 + quad;        // named barrier of the two warps of this quadrant
    const int r = quad * 32 + static_cast<int>(lane);  // row within the tile = TMEM lane
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    bool ok = true;
    int g0 = 0;
    for (int it = 0, w = item_of_round(0, snake); ok && w < n_items; ++it, w = item_of_round(it, snake)) {
      int qt, b, h, nk;
      item_of(w, qt, b, h, nk);
      const int q = qt * kQTile + r;  // query position
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nk; ++j) {
        const int gj = g0 + j;
        const int sb = gj & 1, pb = gj & 1;
        int w_ok = 1;
        if (lane == 0) w_ok = wait_spin(s_full + sb, static_cast<uint32_t>(gj >> 1) & 1u, wc, kSiteAttnS) ? 1 : 0;
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        // both warps of the pair learn each other's outcome at the barrier below, so they leave together
        tc_fence_after_sync();
        float sc[2][32];  // this half's 64 raw scores
        if (w_ok) {
#pragma unroll
          for (int c = 0; c < 2; ++c)
            tmem_ld32f_nowait(lane_base + static_cast<uint32_t>(sb * 128 + 64 * half + 32 * c), sc[c]);
          tmem_wait_ld();
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0 && w_ok) mbar_arrive(s_empty + sb);
        const int key0 = j * kKTile + 64 * half;
        const int key_end = p.causal ? min(p.S, q + 1) : p.S;  // visible keys: [0, key_end)
        // raw scores; invisible keys become -inf (only tiles that reach past some row's last key need it)
        if (!__all_sync(0xffffffffu, key0 + 64 <= key_end)) {
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (key0 + 32 * c + i >= key_end) sc[c][i] = -INFINITY;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) mx = fmaxf(mx, sc[c][i]);
        mx *= p.scale_log2;  // the scale is positive: the maximum of the scaled scores
        // Both warps of the pair pass the same named barriers: a failed wait anywhere in a tile travels to
        // the partner as NaN through the next exchange, and the pair leaves the loop there together.
        xchg[half][r] = ok && w_ok ? mx : NAN;
        asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
        const float other = xchg[half ^ 1][r];
        asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");  // both read before the next write
        if (!(ok && w_ok) || __any_sync(0xffffffffu, isnan(other))) {
          ok = false;
          break;
        }
        mx = fmaxf(mx, other);
        const bool move = mx > m + kRescaleLog2;
        const float m_new = move ? mx : m;
        const float alpha = move ? (m == -INFINITY ? 0.f : ex2_approx(m - m_new)) : 1.f;
        l *= alpha;
        // O (the item's tiles before j, once their P V is done) rescaled in TMEM where a row of the warp
        // moved; each half rescales its 64 columns
        if (j >= 1 && __any_sync(0xffffffffu, move)) {
          const int pj = gj - 1;
          if (lane == 0)
            w_ok = wait_spin(pv_done + (pj & 1), static_cast<uint32_t>(pj >> 1) & 1u, wc, kSiteAttnPv) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
            ok = false;  // finish the tile without touching TMEM or P; the next exchange ends the pair
            continue;
          }
          tc_fence_after_sync();
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint32_t addr = lane_base + 256u + static_cast<uint32_t>(64 * half + 32 * c);
            uint32_t o[32];
            tmem_ld32_nowait(addr, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(addr, o);
          }
          tmem_wait_st();
        }
        m = m_new;
        const float m_use = m == -INFINITY ? 0.f : m;  // a row with nothing visible yet keeps p = 0
        // P into buffer g % 2, once the P V that last read that buffer (two key tiles earlier, possibly
        // in the previous item) is done
        if (gj >= 2) {
          const int pj = gj - 2;
          if (lane == 0)
            w_ok = wait_spin(pv_done + (pj & 1), static_cast<uint32_t>(pj >> 1) & 1u, wc, kSiteAttnPv) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
            ok = false;  // as above
            continue;
          }
        }
        // P in bf16 pairs into TMEM buffer g % 2 (this half's 64 keys: 32 columns), the A operand of P V
        float psum = 0.f;
        uint32_t pw[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float e0 = ex2_approx(fmaf(sc[i >> 4][2 * (i & 15)], p.scale_log2, -m_use));
          const float e1 = ex2_approx(fmaf(sc[i >> 4][2 * (i & 15) + 1], p.scale_log2, -m_use));
          psum += e0 + e1;
          pw[i] = pack_bf16x2(e0, e1);
        }
        l += psum;
        tmem_st32(lane_base + 384u + static_cast<uint32_t>(64 * pb + 32 * half), pw);
        // P (and any rescaled O) handed to the MMA
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full + pb);
      }
      // the row sum of both halves (the pair left the loop at the same tile: the exchange buffer is free);
      // the second barrier keeps the next item's first exchange from overwriting it before both have read
      xchg[half][r] = ok ? l : NAN;
      asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
      const float l_all = xchg[0][r] + xchg[1][r];
      asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
      if (ok && isnan(l_all)) ok = false;
      if (ok && nk > 0) {
        const int pj = g0 + nk - 1;
        int w_ok = 1;
        if (lane == 0)
          w_ok = wait_spin(pv_done + (pj & 1), static_cast<uint32_t>(pj >> 1) & 1u, wc, kSiteAttnPv) ? 1 : 0;
        if (__shfl_sync(0xffffffffu, w_ok, 0)) {
          tc_fence_after_sync();
          uint32_t o[2][32];
#pragma unroll
          for (int c = 0; c < 2; ++c)
            tmem_ld32_nowait(lane_base + 256u + static_cast<uint32_t>(64 * half + 32 * c), o[c]);
          tmem_wait_ld();
          if (p.lse != nullptr && half == 0 && q < p.S)
            p.lse[(static_cast<long long>(b) * p.H + h) * p.s_pad + q] = m + log2f(l_all);
          if (q < p.S) {
            const float inv_l = l_all > 0.f ? 1.f / l_all : 0.f;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                                  (static_cast<long long>(q) * p.B + b) *
                                                      (static_cast<long long>(p.H) * kHd) +
                                                  static_cast<long long>(h) * kHd + 64 * half);
#pragma unroll
            for (int gg = 0; gg < 8; ++gg) {
              const uint32_t* y = o[gg / 4] + 8 * (gg % 4);
              dst[gg] = make_uint4(pack_bf16x2(__uint_as_float(y[0]) * inv_l, __uint_as_float(y[1]) * inv_l),
                                   pack_bf16x2(__uint_as_float(y[2]) * inv_l, __uint_as_float(y[3]) * inv_l),
                                   pack_bf16x2(__uint_as_float(y[4]) * inv_l, __uint_as_float(y[5]) * inv_l),
                                   pack_bf16x2(__uint_as_float(y[6]) * inv_l, __uint_as_float(y[7]) * inv_l));
            }
          }
        }
        // a failed wait here leaves `ok` as it is: `ok` changes only where both warps of the pair see the
        // same values (the exchanges), so they leave the item loop together; the wait raised the CTA's
        // abort flag, so the next item's first wait fails in both and the exchange ends them
      }
      // this warp has read the item's O: the next item's first P V may overwrite it
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty);
      g0 += nk;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 512);
  }
}

// ----------------------------------------------------------------------------- attention backward

constexpr int kBwdComputeWarps = 16;
constexpr int kDqKStages = 3;                             // K ring of the dQ kernel
constexpr int kBwdThreads = 32 * (2 + kBwdComputeWarps);  // producer, MMA issuer, compute warps

__device__ __forceinline__ float dot8(const uint4& a, const uint4& c) {
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, cw[4] = {c.x, c.y, c.z, c.w};
  float v = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = unpack_bf16x2(aw[i]), y = unpack_bf16x2(cw[i]);
    v = fmaf(x.x, y.x, v);
    v = fmaf(x.y, y.y, v);
  }
  return v;
}

// D[b, h, s] = sum_e dO[s B + b, h hd + e] O[s B + b, h hd + e] in fp32 ([B H x s_pad]).  One warp per
// token row; each half-warp takes one head per step (16 lanes x 8 elements: 256-byte coalesced loads).
__global__ void __launch_bounds__(256) k_attention_bwd_delta(const __nv_bfloat16* __restrict__ dO,
                                                             const __nv_bfloat16* __restrict__ O, int S, int B, int H,
                                                             int s_pad, float* __restrict__ D) {
  const long long t = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;  // token row
  const int lane = threadIdx.x & 31;
  if (t >= static_cast<long long>(S) * B) return;
  const int sq = static_cast<int>(t / B), b = static_cast<int>(t % B);
  const long long row = t * (static_cast<long long>(H) * kHd);
  const int sub = lane >> 4;      // which head of the pair
  const int e = 8 * (lane & 15);  // first element within the head
#pragma unroll 2
  for (int h0 = 0; h0 < H; h0 += 2) {
    const int h = h0 + sub;
    float v = 0.f;
    if (h < H)
      v = dot8(__ldg(reinterpret_cast<const uint4*>(dO + row + h * kHd + e)),
               __ldg(reinterpret_cast<const uint4*>(O + row + h * kHd + e)));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((lane & 15) == 0 && h < H) D[(static_cast<long long>(b) * H + h) * s_pad + sq] = v;
  }
}

struct AttnBwdParams {
  CUtensorMap tmQ, tmK, tmV, tmdO;  // 4-D maps: Q, K, V parts of QKV; dO ([S, B, H, hd], O's layout)
  const float* lse;                 // [B H x s_pad], log2 units
  const float* delta;               // [B H x s_pad]
  void* dqkv;                       // [T x 3 d] bf16: dQ, dK, dV in the QKV layout
  int S, B, H, s_pad, n_tiles, causal;
  float scale_log2;                 // log2(e) / sqrt(hd)
  float scale;                      // 1 / sqrt(hd)
  unsigned int* err;
  unsigned long long timeout_ns;
};

// 32 columns of one TMEM row (this thread's lane) scaled by f, as bf16 into dst (64 bytes, 16-byte aligned).
__device__ __forceinline__ void store_row32_scaled(__nv_bfloat16* dst, const float (&o)[32], float f) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const float* y = o + 8 * g;
    d4[g] = make_uint4(pack_bf16x2(y[0] * f, y[1] * f), pack_bf16x2(y[2] * f, y[3] * f),
                       pack_bf16x2(y[4] * f, y[5] * f), pack_bf16x2(y[6] * f, y[7] * f));
  }
}

// P, dS as bf16 pairs for a TMEM A operand: word i holds elements 2i (low half) and 2i + 1.
__device__ __forceinline__ void pack_pairs(const float (&v)[32], uint32_t (&w)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
}

// TMEM column of K-step kk (16 elements) of a bf16 operand written over fp32 scores by quarter: quarter q's
// 32 elements sit as 16 packed columns at 32 q.
__device__ __forceinline__ uint32_t packed_col(int kk) { return static_cast<uint32_t>(32 * (kk >> 1) + 8 * (kk & 1)); }

// dQ, per work item (one 128-query tile of one (batch, head); persistent CTAs walk the items as the
// forward does): per key tile j, S_j = Q K_j^T into TMEM columns 0..127 and
// dP_j = dO V_j^T into 128..255; the 16 compute warps (four per lane quadrant = query rows, 32 keys each)
// release S and dP as soon as they hold them in registers (so S_{j+1}, dP_{j+1} run during their math),
// form P = exp2(S scale - lse) and dS = P (dP - D), and write dS in bf16 into one of two TMEM buffers
// (columns 384.. and 448..); dQ += dS_j K_j takes it from there as the A operand (K as the MN-major B),
// accumulating in columns 256..383.  dQ / sqrt(hd) goes to dQKV.
__global__ void __launch_bounds__(kBwdThreads, 1) k_attention_bwd_dq(const __grid_constant__ AttnBwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sdO = sQ + kTileBytes;
  uint8_t* sK = sdO + kTileBytes;                  // kDqKStages stages: K_j is held until dQ_j is done
  uint8_t* sV = sK + kDqKStages * kTileBytes;      // 2 stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + kKvStages * kTileBytes);
  uint64_t* q_full = bars;                          // Q and dO
  uint64_t* q_empty = q_full + 1;                   // the item's last S and dP MMAs have read Q and dO
  uint64_t* k_full = q_empty + 1;
  uint64_t* k_empty = k_full + kDqKStages;
  uint64_t* v_full = k_empty + kDqKStages;
  uint64_t* v_empty = v_full + kKvStages;
  uint64_t* s_full = v_empty + kKvStages;           // S_j and dP_j in TMEM
  uint64_t* s_empty = s_full + 1;                   // both read by every compute warp
  uint64_t* ds_full = s_empty + 1;                  // [buffer]: dS_j written
  uint64_t* dq_done = ds_full + 2;                  // [buffer]: dQ += dS_j K_j done (buffer free)
  uint64_t* dq_read = dq_done + 2;                  // the compute warps have read the item's dQ
  uint64_t* drain = dq_read + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const int bh_count = p.B * p.H;
  const int n_items = p.n_tiles * bh_count;
  const bool snake = p.causal != 0;  // item order: see item_of_round
  // item w: query tile n_tiles - 1 - w / (B H) (the longest causal tiles first), batch-head w % (B H)
  auto item_of = [&](int w, int& qt, int& b, int& h, int& nk) {
    qt = p.n_tiles - 1 - w / bh_count;
    const int bh = w % bh_count;
    b = bh % p.B;
    h = bh / p.B;
    nk = p.causal ? min(p.n_tiles, qt + 1) : p.n_tiles;
  };
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kDqKStages; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 1);
    }
    for (int s = 0; s < kKvStages; ++s) {
      mbar_init(v_full + s, 1);
      mbar_init(v_empty + s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_empty, kBwdComputeWarps);
    for (int x = 0; x < 2; ++x) {
      mbar_init(ds_full + x, kBwdComputeWarps);
      mbar_init(dq_done + x, 1);
    }
    mbar_init(dq_read, kBwdComputeWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;  // S [0, 128), dP [128, 256), dQ [256, 384), dS [384, 448), [448, 512)
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};

  if (warp == 0) {
    if (lane == 0) {
      uint32_t k_issued = 0, k_par = 0, v_issued = 0, v_par = 0, q_par = 0;
      bool q_issued = false, ok = true;
      int g = 0;  // key tiles issued so far, over all items
      for (int it = 0, w = item_of_round(0, snake); ok && w < n_items; ++it, w = item_of_round(it, snake)) {
        int qt, b, h, nk;
        item_of(w, qt, b, h, nk);
        if (it >= 1 && !wait_spin(q_empty, static_cast<uint32_t>(it - 1) & 1u, wc, kSiteAttnQEmpty)) break;
        mbar_arrive_expect_tx(q_full, 2 * kTileBytes);
        load_tile(sQ, &p.tmQ, q_full, h, b, qt * kQTile);
        load_tile(sdO, &p.tmdO, q_full, h, b, qt * kQTile);
        q_issued = true;
        q_par = static_cast<uint32_t>(it) & 1u;
        for (int j = 0; j < nk; ++j, ++g) {
          const int sk = g % kDqKStages, sv = g % kKvStages;
          const uint32_t pk = static_cast<uint32_t>(g / kDqKStages) & 1u;
          const uint32_t pv = static_cast<uint32_t>(g / kKvStages) & 1u;
          if (!wait_spin(k_empty + sk, pk ^ 1u, wc, kSiteAttnKvEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(k_full + sk, kTileBytes);
          load_tile(sK + sk * kTileBytes, &p.tmK, k_full + sk, h, b, j * kKTile);
          k_issued |= 1u << sk;
          k_par = (k_par & ~(1u << sk)) | (pk << sk);
          if (!wait_spin(v_empty + sv, pv ^ 1u, wc, kSiteAttnKvEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(v_full + sv, kTileBytes);
          load_tile(sV + sv * kTileBytes, &p.tmV, v_full + sv, h, b, j * kKTile);
          v_issued |= 1u << sv;
          v_par = (v_par & ~(1u << sv)) | (pv << sv);
        }
      }
      if (q_issued) wait_drain(q_full, q_par, p.timeout_ns);
      for (int s = 0; s < kDqKStages; ++s)
        if (k_issued & (1u << s)) wait_drain(k_full + s, (k_par >> s) & 1u, p.timeout_ns);
      for (int s = 0; s < kKvStages; ++s)
        if (v_issued & (1u << s)) wait_drain(v_full + s, (v_par >> s) & 1u, p.timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_kk = idesc_bf16_f32(kQTile, kKTile, false, false);  // both K-major
      constexpr uint32_t idesc_mn = idesc_bf16_f32(kQTile, kHd, false, true);       // B MN-major
      const uint32_t q_base = smem_u32(sQ), do_base = smem_u32(sdO);
      bool ok = true;
      int g0 = 0;
      // step j of an item: S_j and dP_j (j < nk), then dQ += dS_{j-1} K_{j-1} (j >= 1); g = running tile count
      for (int it = 0, w = item_of_round(0, snake); ok && w < n_items; ++it, w = item_of_round(it, snake)) {
        int qt, b, h, nk;
        item_of(w, qt, b, h, nk);
        if (!wait_spin(q_full, static_cast<uint32_t>(it) & 1u, wc, kSiteAttnQ)) break;
        tc_fence_after_sync();
        for (int j = 0; ok && j <= nk; ++j) {
          if (j < nk) {
            const int gj = g0 + j;
            const int sk = gj % kDqKStages, sv = gj % kKvStages;
            if (!wait_spin(s_empty, (static_cast<uint32_t>(gj) & 1u) ^ 1u, wc, kSiteAttnSEmpty) ||
                !wait_spin(k_full + sk, static_cast<uint32_t>(gj / kDqKStages) & 1u, wc, kSiteAttnKv) ||
                !wait_spin(v_full + sv, static_cast<uint32_t>(gj / kKvStages) & 1u, wc, kSiteAttnKv)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t k_base = smem_u32(sK + sk * kTileBytes), v_base = smem_u32(sV + sv * kTileBytes);
#pragma unroll
            for (int kk = 0; kk < kHd / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
              umma_bf16(tmem_base, sdesc_sw128(q_base + off, 16, 1024), sdesc_sw128(k_base + off, 16, 1024), idesc_kk,
                        kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < kHd / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
              umma_bf16(tmem_base + 128, sdesc_sw128(do_base + off, 16, 1024), sdesc_sw128(v_base + off, 16, 1024),
                        idesc_kk, kk > 0 ? 1u : 0u);
            }
            umma_commit(s_full);
            umma_commit(v_empty + sv);
            if (j == nk - 1) umma_commit(q_empty);  // the item's last S and dP: Q and dO may be reloaded
          }
          if (j >= 1) {
            const int gj = g0 + j - 1;
            const int st = gj % kDqKStages;
            const int buf = gj & 1;
            // the item's first dQ MMA overwrites dQ: the previous item's epilogue must have read it
            if (j == 1 && it >= 1 && !wait_spin(dq_read, static_cast<uint32_t>(it - 1) & 1u, wc, kSiteAttnOEmpty)) {
              ok = false;
              break;
            }
            if (!wait_spin(ds_full + buf, static_cast<uint32_t>(gj >> 1) & 1u, wc, kSiteAttnP)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t k_base = smem_u32(sK + st * kTileBytes);
#pragma unroll
            for (int kk = 0; kk < kKTile / 16; ++kk)
              umma_bf16_tmem_a(tmem_base + 256, tmem_base + 384 + 64 * buf + 8 * kk,
                               sdesc_sw128(k_base + kk * 2048, kAtom, 1024), idesc_mn, (j > 1 || kk > 0) ? 1u : 0u);
            umma_commit(dq_done + buf);
            umma_commit(k_empty + st);
          }
        }
        g0 += nk;
      }
      umma_commit(drain);
      wait_drain(drain, 0, p.timeout_ns);
    }
  } else {
    const int quad = warp & 3;
    const int quarter = (warp - 2) >> 2;  // keys 32 quarter .. 32 quarter + 31 of every tile
    const int r = quad * 32 + static_cast<int>(lane);
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    bool ok = true;
    int g0 = 0;
    for (int it = 0, w = item_of_round(0, snake); ok && w < n_items; ++it, w = item_of_round(it, snake)) {
      int qt, b, h, nk;
      item_of(w, qt, b, h, nk);
      const int q = qt * kQTile + r;
      const long long stat = (static_cast<long long>(b) * p.H + h) * p.s_pad + q;
      const float neg_lse = q < p.S ? -__ldg(p.lse + stat) : 0.f;
      const float dd = q < p.S ? __ldg(p.delta + stat) : 0.f;
      const int key_end = q < p.S ? (p.causal ? min(p.S, q + 1) : p.S) : 0;  // padding rows: nothing
      for (int j = 0; ok && j < nk; ++j) {
        const int gj = g0 + j;
        int w_ok = 1;
        if (lane == 0) w_ok = wait_spin(s_full, static_cast<uint32_t>(gj) & 1u, wc, kSiteAttnS) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        float sc[32], dp[32];
        tmem_ld32f_nowait(lane_base + static_cast<uint32_t>(32 * quarter), sc);
        tmem_ld32f_nowait(lane_base + 128u + static_cast<uint32_t>(32 * quarter), dp);
        tmem_wait_ld();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty);
        const int key0 = j * kKTile + 32 * quarter;
        if (__all_sync(0xffffffffu, key0 + 32 <= key_end)) {
#pragma unroll
          for (int i = 0; i < 32; ++i) sc[i] = fmaf(sc[i], p.scale_log2, neg_lse);
#pragma unroll
          for (int i = 0; i < 32; ++i) sc[i] = ex2_approx(sc[i]);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            sc[i] = key0 + i < key_end ? ex2_approx(fmaf(sc[i], p.scale_log2, neg_lse)) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) dp[i] = sc[i] * (dp[i] - dd);  // dS
        uint32_t wds[16];
        pack_pairs(dp, wds);
        const int buf = gj & 1;
        // the buffer is free once the dQ MMA of the key tile two before (possibly the previous item's) read it
        if (gj >= 2) {
          if (lane == 0)
            w_ok = wait_spin(dq_done + buf, static_cast<uint32_t>((gj - 2) >> 1) & 1u, wc, kSiteAttnPv) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
        }
        tmem_st16(lane_base + 384u + static_cast<uint32_t>(64 * buf + 16 * quarter), wds);
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(ds_full + buf);
      }
      if (ok && nk > 0) {
        // the item's last dQ commit covers every earlier MMA
        const int pj = g0 + nk - 1;
        int w_ok = 1;
        if (lane == 0)
          w_ok = wait_spin(dq_done + (pj & 1), static_cast<uint32_t>(pj >> 1) & 1u, wc, kSiteAttnPv) ? 1 : 0;
        if (__shfl_sync(0xffffffffu, w_ok, 0)) {
          tc_fence_after_sync();
          float o[32];
          tmem_ld32f_nowait(lane_base + 256u + static_cast<uint32_t>(32 * quarter), o);
          tmem_wait_ld();
          if (q < p.S)
            store_row32_scaled(static_cast<__nv_bfloat16*>(p.dqkv) +
                                   (static_cast<long long>(q) * p.B + b) * (3LL * p.H * kHd) +
                                   static_cast<long long>(h) * kHd + 32 * quarter,
                               o, p.scale);
        } else {
          ok = false;
        }
      }
      // this warp has read the item's dQ: the next item's first dQ MMA may overwrite it
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_read);
      g0 += nk;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 512);
  }
}

// dK and dV, per work item (one 128-key tile of one (batch, head); persistent CTAs walk the items, the first
// key tiles first): per query tile i, S^T_i = K Q_i^T into TMEM columns
// 0..127 and dP^T_i = V dO_i^T into 128..255, each issued as two halves of 64 queries with a barrier of
// their own; the 16 compute warps (four per lane quadrant = key rows, 32 queries each, the first eight on
// the lower half) form P^T = exp2(S^T scale - lse[q]) and dS^T = P^T (dP^T - D[q]) and write both in bf16
// over their own score columns; dV += P^T dO_i and dK += dS^T Q_i take them from TMEM as the A operand (dO,
// Q as the MN-major B), accumulating in columns 256..383 and 384..511, again per half.  The issue order
// (lower-half scores of tile i, upper-half gradients of tile i - 1, upper-half scores of tile i, lower-half
// gradients of tile i) lets one half's math run while the tensor pipe works on the other; a half's score
// columns take new scores once the MMAs that read its P^T and dS^T are done.  Causal attention visits
// query tiles i >= the key tile.
__global__ void __launch_bounds__(kBwdThreads, 1) k_attention_bwd_dkdv(const __grid_constant__ AttnBwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + kTileBytes;
  uint8_t* sQ = sV + kTileBytes;                   // 2 stages
  uint8_t* sdO = sQ + kKvStages * kTileBytes;      // 2 stages
  float* sStat = reinterpret_cast<float*>(sdO + kKvStages * kTileBytes);  // [stage][lse, D][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStat + kKvStages * 2 * kQTile);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = kv_full + 1;                // the item's last S^T and dP^T MMAs have read K and V
  uint64_t* q_full = kv_empty + 1;                 // [stage]: Q_i and dO_i
  uint64_t* q_empty = q_full + kKvStages;
  uint64_t* s_half = q_empty + kKvStages;          // [half]: S^T_i and dP^T_i of one half of the queries in TMEM
  uint64_t* p_half = s_half + 2;                   // [half]: P^T_i and dS^T_i written by the half's compute warps
  uint64_t* pd_half = p_half + 2;                  // [half]: dV and dK MMAs of the half done (its columns free)
  uint64_t* dkdv_read = pd_half + 2;               // the compute warps have read the item's dK and dV
  uint64_t* drain = dkdv_read + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const int bh_count = p.B * p.H;
  const int n_items = p.n_tiles * bh_count;
  const bool snake = p.causal != 0;  // item order: see item_of_round
  // item w: key tile w / (B H) (causal: the first key tiles have the most query tiles), batch-head w % (B H);
  // its query tiles i0 .. n_tiles - 1
  auto item_of = [&](int w, int& kt, int& b, int& h, int& i0, int& nq) {
    kt = w / bh_count;
    const int bh = w % bh_count;
    b = bh % p.B;
    h = bh / p.B;
    i0 = p.causal ? kt : 0;
    nq = p.n_tiles - i0;
  };
  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int s = 0; s < kKvStages; ++s) {
      mbar_init(q_full + s, 1);
      mbar_init(q_empty + s, 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(s_half + x, 1);
      mbar_init(p_half + x, kBwdComputeWarps / 2);
      mbar_init(pd_half + x, 1);
    }
    mbar_init(dkdv_read, kBwdComputeWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;  // S^T [0, 128), dP^T [128, 256), dV [256, 384), dK [384, 512)
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};

  if (warp == 0) {
    if (lane == 0) {
      uint32_t issued = 0, par = 0, kv_par = 0;
      bool kv_issued = false, ok = true;
      int g = 0;  // query tiles issued so far, over all items
      for (int it = 0, w = item_of_round(0, snake); ok && w < n_items; ++it, w = item_of_round(it, snake)) {
        int kt, b, h, i0, nq;
        item_of(w, kt, b, h, i0, nq);
        if (it >= 1 && !wait_spin(kv_empty, static_cast<uint32_t>(it - 1) & 1u, wc, kSiteAttnQEmpty)) break;
        mbar_arrive_expect_tx(kv_full, 2 * kTileBytes);
        load_tile(sK, &p.tmK, kv_full, h, b, kt * kKTile);
        load_tile(sV, &p.tmV, kv_full, h, b, kt * kKTile);
        kv_issued = true;
        kv_par = static_cast<uint32_t>(it) & 1u;
        for (int t = 0; t < nq; ++t, ++g) {
          const int st = g % kKvStages;
          const uint32_t ph = static_cast<uint32_t>(g / kKvStages) & 1u;
          if (!wait_spin(q_empty + st, ph ^ 1u, wc, kSiteAttnKvEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(q_full + st, 2 * kTileBytes + 2 * kQTile * 4);
          load_tile(sQ + st * kTileBytes, &p.tmQ, q_full + st, h, b, (i0 + t) * kQTile);
          load_tile(sdO + st * kTileBytes, &p.tmdO, q_full + st, h, b, (i0 + t) * kQTile);
          // the tile's statistics (512 bytes each, 16-byte aligned: rows of s_pad floats, tiles of 128)
          const long long st0 = (static_cast<long long>(b) * p.H + h) * p.s_pad + (i0 + t) * kQTile;
          bulk_load(sStat + st * 2 * kQTile, p.lse + st0, kQTile * 4, q_full + st);
          bulk_load(sStat + st * 2 * kQTile + kQTile, p.delta + st0, kQTile * 4, q_full + st);
          issued |= 1u << st;
          par = (par & ~(1u << st)) | (ph << st);
        }
      }
      if (kv_issued) wait_drain(kv_full, kv_par, p.timeout_ns);
      for (int s = 0; s < kKvStages; ++s)
        if (issued & (1u << s)) wait_drain(q_full + s, (par >> s) & 1u, p.timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_half = idesc_bf16_f32(kKTile, kQTile / 2, false, false);  // 128 keys x 64 queries
      constexpr uint32_t idesc_mn = idesc_bf16_f32(kKTile, kHd, false, true);
      const uint32_t k_base = smem_u32(sK), v_base = smem_u32(sV);
      // S^T and dP^T of half x (queries 64 x .. 64 x + 63) of the tile in stage st: the half's Q and dO rows
      // start 64 rows (8 KB) into each atom column
      auto issue_scores = [&](int st, int x) {
        const uint32_t q_base = smem_u32(sQ + st * kTileBytes) + static_cast<uint32_t>(x) * 8192u;
        const uint32_t do_base = smem_u32(sdO + st * kTileBytes) + static_cast<uint32_t>(x) * 8192u;
#pragma unroll
        for (int kk = 0; kk < kHd / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
          umma_bf16(tmem_base + 64u * x, sdesc_sw128(k_base + off, 16, 1024), sdesc_sw128(q_base + off, 16, 1024),
                    idesc_half, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < kHd / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
          umma_bf16(tmem_base + 128u + 64u * x, sdesc_sw128(v_base + off, 16, 1024),
                    sdesc_sw128(do_base + off, 16, 1024), idesc_half, kk > 0 ? 1u : 0u);
        }
        umma_commit(s_half + x);
      };
      // dV += P^T dO and dK += dS^T Q over the queries of half x of the item's tile t (stage st); the item's
      // first of them (t = 0, lower half) starts the accumulators
      auto issue_grads = [&](int st, int t, int x) {
        const uint32_t q_base = smem_u32(sQ + st * kTileBytes), do_base = smem_u32(sdO + st * kTileBytes);
#pragma unroll
        for (int j = 0; j < kQTile / 32; ++j) {
          const int kk = 4 * x + j;
          umma_bf16_tmem_a(tmem_base + 256, tmem_base + packed_col(kk), sdesc_sw128(do_base + kk * 2048, kAtom, 1024),
                           idesc_mn, (t | kk) != 0 ? 1u : 0u);
        }
#pragma unroll
        for (int j = 0; j < kQTile / 32; ++j) {
          const int kk = 4 * x + j;
          umma_bf16_tmem_a(tmem_base + 384, tmem_base + 128 + packed_col(kk),
                           sdesc_sw128(q_base + kk * 2048, kAtom, 1024), idesc_mn, (t | kk) != 0 ? 1u : 0u);
        }
        umma_commit(pd_half + x);
        if (x == 1) umma_commit(q_empty + st);  // the tile's last reads of Q and dO
      };
      bool ok = true;
      int g0 = 0;
      for (int it = 0, w = item_of_round(0, snake); ok && w < n_items; ++it, w = item_of_round(it, snake)) {
        int kt, b, h, i0, nq;
        item_of(w, kt, b, h, i0, nq);
        if (!wait_spin(kv_full, static_cast<uint32_t>(it) & 1u, wc, kSiteAttnQ)) break;
        tc_fence_after_sync();
        // Per tile: the lower half's scores, the previous tile's upper-half gradients, this tile's upper-half
        // scores, then its lower-half gradients, so that each half's softmax math runs while the tensor pipe
        // works on the other half.  A half's score columns take new scores only after the MMAs that read
        // its P^T and dS^T have completed.
        for (int t = 0; ok && t < nq; ++t) {
          const int gt = g0 + t;  // running query-tile count: stages, score columns and barrier phases
          const int st = gt % kKvStages;
          const uint32_t prev = static_cast<uint32_t>(gt - 1) & 1u;
          if (!wait_spin(q_full + st, static_cast<uint32_t>(gt / kKvStages) & 1u, wc, kSiteAttnKv) ||
              (gt >= 1 && !wait_spin(pd_half, prev, wc, kSiteAttnSEmpty))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_scores(st, 0);
          if (t >= 1) {
            if (!wait_spin(p_half + 1, prev, wc, kSiteAttnP)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            issue_grads((gt - 1) % kKvStages, t - 1, 1);
          }
          if (gt >= 1 && !wait_spin(pd_half + 1, prev, wc, kSiteAttnSEmpty)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_scores(st, 1);
          if (t == nq - 1) umma_commit(kv_empty);  // the item's last reads of K and V
          // the item's first dV and dK MMAs overwrite them: the previous item's epilogue must have read them
          if ((t == 0 && it >= 1 && !wait_spin(dkdv_read, static_cast<uint32_t>(it - 1) & 1u, wc, kSiteAttnOEmpty)) ||
              !wait_spin(p_half, static_cast<uint32_t>(gt) & 1u, wc, kSiteAttnP)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_grads(st, t, 0);
        }
        if (ok && nq > 0) {  // the item's last tile: its upper half's gradients
          const int gl = g0 + nq - 1;
          if (!wait_spin(p_half + 1, static_cast<uint32_t>(gl) & 1u, wc, kSiteAttnP)) break;
          tc_fence_after_sync();
          issue_grads(gl % kKvStages, nq - 1, 1);
        }
        g0 += nq;
      }
      umma_commit(drain);
      wait_drain(drain, 0, p.timeout_ns);
    }
  } else {
    const int quad = warp & 3;
    const int quarter = (warp - 2) >> 2;  // queries 32 quarter .. 32 quarter + 31 of every tile
    const int half = quarter >> 1;        // the half of the tile's queries (and score barriers) it works on
    const int r = quad * 32 + static_cast<int>(lane);
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    bool ok = true;
    int g0 = 0;
    for (int it = 0, w = item_of_round(0, snake); ok && w < n_items; ++it, w = item_of_round(it, snake)) {
      int kt, b, h, i0, nq;
      item_of(w, kt, b, h, i0, nq);
      const int k = kt * kKTile + r;  // key position
      for (int t = 0; t < nq; ++t) {
        const int gt = g0 + t;
        const int q0 = (i0 + t) * kQTile + 32 * quarter;  // this warp's first query
        int w_ok = 1;
        if (lane == 0) w_ok = wait_spin(s_half + half, static_cast<uint32_t>(gt) & 1u, wc, kSiteAttnS) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        float sc[32], dp[32];
        tmem_ld32f_nowait(lane_base + static_cast<uint32_t>(32 * quarter), sc);
        tmem_ld32f_nowait(lane_base + 128u + static_cast<uint32_t>(32 * quarter), dp);
        tmem_wait_ld();
        // the statistics of this warp's 32 queries, staged with Q and dO (all lanes read the same words)
        const float4* l4 = reinterpret_cast<const float4*>(sStat + (gt % kKvStages) * 2 * kQTile + 32 * quarter);
        const float4* d4 = l4 + kQTile / 4;
        // query q sees key k when q < S and (not causal or k <= q); only the diagonal and the ragged last
        // tile need the test (the condition is the same for the whole warp)
        if (q0 + 32 <= p.S && (!p.causal || q0 >= kt * kKTile + kKTile - 1)) {
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const float4 l = l4[g];
            sc[4 * g] = fmaf(sc[4 * g], p.scale_log2, -l.x);
            sc[4 * g + 1] = fmaf(sc[4 * g + 1], p.scale_log2, -l.y);
            sc[4 * g + 2] = fmaf(sc[4 * g + 2], p.scale_log2, -l.z);
            sc[4 * g + 3] = fmaf(sc[4 * g + 3], p.scale_log2, -l.w);
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) sc[i] = ex2_approx(sc[i]);
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const float4 dd = d4[g];
            dp[4 * g] = sc[4 * g] * (dp[4 * g] - dd.x);
            dp[4 * g + 1] = sc[4 * g + 1] * (dp[4 * g + 1] - dd.y);
            dp[4 * g + 2] = sc[4 * g + 2] * (dp[4 * g + 2] - dd.z);
            dp[4 * g + 3] = sc[4 * g + 3] * (dp[4 * g + 3] - dd.w);
          }
        } else {
          // a query past S reads unwritten statistics: the selects keep them out
          const int q_end = p.causal ? min(p.S, q0 + 32) : p.S;
          const int q_first = p.causal ? k : 0;  // visible: q_first <= q < q_end
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const float4 l = l4[g];
            const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int q = q0 + 4 * g + u;
              const float pv = ex2_approx(fmaf(sc[4 * g + u], p.scale_log2, -lv[u]));
              sc[4 * g + u] = q >= q_first && q < q_end ? pv : 0.f;
            }
          }
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const float4 dd = d4[g];
            const float dv[4] = {dd.x, dd.y, dd.z, dd.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int q = q0 + 4 * g + u;
              dp[4 * g + u] = q >= q_first && q < q_end ? sc[4 * g + u] * (dp[4 * g + u] - dv[u]) : 0.f;
            }
          }
        }
        // P^T and dS^T in bf16 over this quarter's own score columns
        uint32_t w[16];
        pack_pairs(sc, w);
        tmem_st16(lane_base + static_cast<uint32_t>(32 * quarter), w);
        pack_pairs(dp, w);
        tmem_st16(lane_base + 128u + static_cast<uint32_t>(32 * quarter), w);
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_half + half);
      }
      if (ok && nq > 0) {
        // the upper half's gradients of the item's last tile are its last MMAs: their commit covers them all
        int w_ok = 1;
        if (lane == 0) w_ok = wait_spin(pd_half + 1, static_cast<uint32_t>(g0 + nq - 1) & 1u, wc, kSiteAttnPv) ? 1 : 0;
        if (__shfl_sync(0xffffffffu, w_ok, 0)) {
          tc_fence_after_sync();
          __nv_bfloat16* row = static_cast<__nv_bfloat16*>(p.dqkv) +
                               (static_cast<long long>(k) * p.B + b) * (3LL * p.H * kHd) +
                               static_cast<long long>(h) * kHd + 32 * quarter;
          float o[32];
          tmem_ld32f_nowait(lane_base + 384u + static_cast<uint32_t>(32 * quarter), o);  // dK
          tmem_wait_ld();
          if (k < p.S) store_row32_scaled(row + static_cast<long long>(p.H) * kHd, o, p.scale);
          tmem_ld32f_nowait(lane_base + 256u + static_cast<uint32_t>(32 * quarter), o);  // dV
          tmem_wait_ld();
          if (k < p.S) store_row32_scaled(row + 2LL * p.H * kHd, o, 1.f);
        } else {
          ok = false;
        }
      }
      // this warp has read the item's dK and dV: the next item's first dV and dK MMAs may overwrite them
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(dkdv_read);
      g0 += nq;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 attn_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 4-D map over per-head rows of a token-major tensor whose token row (s B + b) holds `ld` elements and
// head h starts at element h hd of `base`: dims (e, h, b, s), boxes of 64 elements x 128 positions.
bool make_head_map(CUtensorMap* m, const void* base, long long ld, int S, int B, int H) {
  auto fn = attn_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHd), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B),
                        static_cast<cuuint64_t>(S)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(kHd) * 2, static_cast<cuuint64_t>(ld) * 2,
                           static_cast<cuuint64_t>(ld) * 2 * static_cast<cuuint64_t>(B)};
  cuuint32_t box[4] = {64, 1, 1, 128};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One part (Q, K or V) of the projection output [S, B, 3, H, hd].
bool make_part_map(CUtensorMap* m, const void* qkv, int part, int S, int B, int H) {
  const long long d = static_cast<long long>(H) * kHd;
  return make_head_map(m, static_cast<const __nv_bfloat16*>(qkv) + part * d, 3 * d, S, B, H);
}

constexpr size_t kAttnSmem = 1024 + (1 + 2 * kFwdKvStages) * kTileBytes + 256;
// dQ: Q, dO, 3 K stages, 2 V stages; dK/dV: K, V, 2 Q and 2 dO stages and the staged statistics
constexpr size_t kAttnDqSmem = 1024 + (2 + kDqKStages + kKvStages) * kTileBytes + 256;
constexpr size_t kAttnDkdvSmem = 1024 + (2 + 2 * kKvStages) * kTileBytes + kKvStages * 2 * kQTile * 4 + 256;

cudaError_t launch_attention(const void* qkv, int S, int B, int H, bool causal, void* out, const DeviceCtx& ctx,
                             cudaStream_t s, float* lse = nullptr) {
  if (S <= 0) return cudaSuccess;
  AttnParams p;
  memset(&p, 0, sizeof(p));
  if (!make_part_map(&p.tmQ, qkv, 0, S, B, H) || !make_part_map(&p.tmK, qkv, 1, S, B, H) ||
      !make_part_map(&p.tmV, qkv, 2, S, B, H))
    return cudaErrorInvalidValue;
  p.out = out;
  p.lse = lse;
  p.S = S;
  p.B = B;
  p.H = H;
  p.n_qtiles = (S + kQTile - 1) / kQTile;
  p.s_pad = p.n_qtiles * kQTile;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kHd)));
  p.err = ctx.err;
  p.timeout_ns = ctx.timeout_ns;
  const long long items = static_cast<long long>(p.n_qtiles) * B * H;
  if (items > INT_MAX) return cudaErrorInvalidValue;
  // persistent: one CTA per SM (the shared memory allows no second), each walking its share of the items
  const int grid = static_cast<int>(items < ctx.sm_count ? items : ctx.sm_count);
  cudaError_t e = cudaFuncSetAttribute(k_attention_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kAttnSmem));
  if (e != cudaSuccess) return e;
  k_attention_fwd<<<grid, kThreads, kAttnSmem, s>>>(p);
  return cudaGetLastError();
}

// Attention backward: D = rowsum(dO O), then dQ (per query tile) and dK, dV (per key tile) into dqkv.
// lse: the forward's [B H x s_pad] statistics; delta: [B H x s_pad] scratch.
cudaError_t launch_attention_bwd(const void* qkv, const void* o, const void* dO, const float* lse, float* delta,
                                 int S, int B, int H, bool causal, void* dqkv, const DeviceCtx& ctx, cudaStream_t s) {
  if (S <= 0) return cudaSuccess;
  AttnBwdParams p;
  memset(&p, 0, sizeof(p));
  if (!make_part_map(&p.tmQ, qkv, 0, S, B, H) || !make_part_map(&p.tmK, qkv, 1, S, B, H) ||
      !make_part_map(&p.tmV, qkv, 2, S, B, H) ||
      !make_head_map(&p.tmdO, dO, static_cast<long long>(H) * kHd, S, B, H))
    return cudaErrorInvalidValue;
  p.lse = lse;
  p.delta = delta;
  p.dqkv = dqkv;
  p.S = S;
  p.B = B;
  p.H = H;
  p.n_tiles = (S + kQTile - 1) / kQTile;
  p.s_pad = p.n_tiles * kQTile;
  p.causal = causal ? 1 : 0;
  p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(kHd)));
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kHd)));
  p.err = ctx.err;
  p.timeout_ns = ctx.timeout_ns;
  const long long grid = static_cast<long long>(p.n_tiles) * B * H;
  const long long warps = static_cast<long long>(S) * B * H;
  if (grid > INT_MAX || warps > INT_MAX / 32) return cudaErrorInvalidValue;
  const long long rows = static_cast<long long>(S) * B;
  k_attention_bwd_delta<<<static_cast<int>((rows * 32 + 255) / 256), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(dO), static_cast<const __nv_bfloat16*>(o), S, B, H, p.s_pad, delta);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_attention_bwd_dq, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kAttnDqSmem));
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM, each walking its share of the (query tile, batch, head) items
  k_attention_bwd_dq<<<static_cast<int>(grid < ctx.sm_count ? grid : ctx.sm_count), kBwdThreads, kAttnDqSmem, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_attention_bwd_dkdv, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kAttnDkdvSmem));
  if (e != cudaSuccess) return e;
  k_attention_bwd_dkdv<<<static_cast<int>(grid < ctx.sm_count ? grid : ctx.sm_count), kBwdThreads, kAttnDkdvSmem,
                         s>>>(p);
  return cudaGetLastError();
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

bool al16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

tpmlp_status attn_check(int64_t S, int64_t B, int64_t H, int64_t head_dim) {
  if (S < 0 || B < 1 || H < 1 || head_dim < 1) return TPMLP_ERR_INVALID_ARG;
  if (head_dim != kHd) return TPMLP_ERR_UNSUPPORTED;
  if (S > INT_MAX / 4 || B > 65535 || H > 65535 || S * B > INT_MAX / 4 || H * kHd > 65536)
    return TPMLP_ERR_UNSUPPORTED;
  return TPMLP_OK;
}

// Backward workspace: D, dO, dQKV, column-sum partials.
struct Bwd {
  size_t delta, dO, dqkv, partial;
};

Bwd bwd_sizes(int64_t S, int64_t B, int64_t H) {
  const size_t T = static_cast<size_t>(S) * static_cast<size_t>(B), d = static_cast<size_t>(H) * kHd;
  const size_t s_pad = (static_cast<size_t>(S) + kQTile - 1) / kQTile * kQTile;
  Bwd z;
  z.delta = align256(static_cast<size_t>(B) * static_cast<size_t>(H) * s_pad * 4);
  z.dO = align256(T * d * 2);
  z.dqkv = align256(T * 3 * d * 2);
  z.partial = align256(column_sum_bf16_scratch_floats(static_cast<int>(T), static_cast<int>(3 * d)) * 4);
  return z;
}

tpmlp_status to_status(cudaError_t e) {
  if (e == cudaSuccess) return TPMLP_OK;
  if (e == cudaErrorNotSupported) return TPMLP_ERR_UNSUPPORTED;
  return TPMLP_ERR_CUDA;
}

}  // namespace
}  // namespace tpmlp

using namespace tpmlp;

extern "C" {

tpmlp_status tpmlp_attention_workspace_size(int64_t S, int64_t B, int64_t H, int64_t head_dim, size_t* bytes) {
  if (bytes == nullptr) return TPMLP_ERR_INVALID_ARG;
  const tpmlp_status st = attn_check(S, B, H, head_dim);
  if (st != TPMLP_OK) return st;
  const size_t T = static_cast<size_t>(S) * static_cast<size_t>(B), d = static_cast<size_t>(H * head_dim);
  *bytes = align256(T * 3 * d * 2) + align256(T * d * 2);
  return TPMLP_OK;
}

tpmlp_status tpmlp_attention_core(const void* QKV, int64_t S, int64_t B, int64_t H, int64_t head_dim, int causal,
                                  void* O, float* LSE, tpmlp_stream_t stream) {
  tpmlp_status st = attn_check(S, B, H, head_dim);
  if (st != TPMLP_OK) return st;
  if (causal != 0 && causal != 1) return TPMLP_ERR_INVALID_ARG;
  if (S == 0) return TPMLP_OK;
  if (!al16(QKV) || !al16(O) || (LSE != nullptr && !al16(LSE))) return TPMLP_ERR_INVALID_ARG;
  DeviceCtx c;
  if (current_device_ctx(&c) != cudaSuccess) return TPMLP_ERR_CUDA;
  return to_status(launch_attention(QKV, static_cast<int>(S), static_cast<int>(B), static_cast<int>(H), causal == 1,
                                    O, c, reinterpret_cast<cudaStream_t>(stream), LSE));
}

tpmlp_status tpmlp_attention_backward_workspace_size(int64_t S, int64_t B, int64_t H, int64_t head_dim,
                                                     size_t* bytes) {
  if (bytes == nullptr) return TPMLP_ERR_INVALID_ARG;
  const tpmlp_status st = attn_check(S, B, H, head_dim);
  if (st != TPMLP_OK) return st;
  const Bwd z = bwd_sizes(S, B, H);
  *bytes = z.delta + z.dO + z.dqkv + z.partial;
  return TPMLP_OK;
}

tpmlp_status tpmlp_attention_core_backward(const void* QKV, const void* O, const void* dO, const float* LSE,
                                           int64_t S, int64_t B, int64_t H, int64_t head_dim, int causal,
                                           void* dQKV, void* workspace, size_t workspace_bytes,
                                           tpmlp_stream_t stream) {
  tpmlp_status st = attn_check(S, B, H, head_dim);
  if (st != TPMLP_OK) return st;
  if (causal != 0 && causal != 1) return TPMLP_ERR_INVALID_ARG;
  if (S == 0) return TPMLP_OK;
  if (!al16(QKV) || !al16(O) || !al16(dO) || !al16(LSE) || !al16(dQKV)) return TPMLP_ERR_INVALID_ARG;
  const Bwd z = bwd_sizes(S, B, H);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < z.delta)
    return TPMLP_ERR_WORKSPACE;
  DeviceCtx c;
  if (current_device_ctx(&c) != cudaSuccess) return TPMLP_ERR_CUDA;
  return to_status(launch_attention_bwd(QKV, O, dO, LSE, static_cast<float*>(workspace), static_cast<int>(S),
                                        static_cast<int>(B), static_cast<int>(H), causal == 1, dQKV, c,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_attention_tp_forward(const void* X, const void* Wqkv, const void* bqkv, const void* Wo,
                                        const void* bo, int64_t S, int64_t B, int64_t H, int32_t n_shards,
                                        int causal, void* Y, void* QKV_out, void* O_out, float* LSE_out,
                                        void* workspace, size_t workspace_bytes, tpmlp_stream_t stream) {
  tpmlp_status st = attn_check(S, B, H, kHd);
  if (st != TPMLP_OK) return st;
  if (n_shards < 1 || H % n_shards != 0 || (causal != 0 && causal != 1)) return TPMLP_ERR_INVALID_ARG;
  if (S == 0) return TPMLP_OK;
  if (!al16(X) || !al16(Wqkv) || !al16(Wo) || !al16(Y) || (bqkv != nullptr && !al16(bqkv)) ||
      (bo != nullptr && !al16(bo)) || (QKV_out != nullptr && !al16(QKV_out)) || (O_out != nullptr && !al16(O_out)) ||
      (LSE_out != nullptr && !al16(LSE_out)))
    return TPMLP_ERR_INVALID_ARG;
  size_t need = 0;
  tpmlp_attention_workspace_size(S, B, H, kHd, &need);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < need)
    return TPMLP_ERR_WORKSPACE;
  DeviceCtx c;
  if (current_device_ctx(&c) != cudaSuccess) return TPMLP_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int T = static_cast<int>(S * B), d = static_cast<int>(H * kHd);
  void* qkv = workspace;
  void* o = static_cast<uint8_t*>(workspace) + align256(static_cast<size_t>(T) * 3 * d * 2);
  if (QKV_out != nullptr) qkv = QKV_out;
  if (O_out != nullptr) o = O_out;
  // column-parallel projection: all shards' Q, K, V columns in one GEMM (bias fused)
  GemmLaunch g1;
  g1.M = T;
  g1.N = 3 * d;
  g1.K = d;
  g1.a = {X, d, false};
  g1.b = {Wqkv, 3 * d, true};
  g1.epi = kEpiBias;
  g1.out0 = qkv;
  g1.ld0 = 3 * d;
  g1.bias = bqkv;
  cudaError_t e = launch_gemm(g1, c, s);
  if (e == cudaSuccess) e = launch_attention(qkv, static_cast<int>(S), static_cast<int>(B), static_cast<int>(H),
                                             causal == 1, o, c, s, LSE_out);
  // row-parallel output projection: the K loop walks the shards' head rows into one accumulator, then
  // the row layer's bias
  if (e == cudaSuccess) {
    GemmLaunch g2;
    g2.M = T;
    g2.N = d;
    g2.K = d;
    g2.a = {o, d, false};
    g2.b = {Wo, d, true};
    g2.epi = kEpiBias;
    g2.out0 = Y;
    g2.ld0 = d;
    g2.bias = bo;
    e = launch_gemm(g2, c, s);
  }
  return to_status(e);
}

tpmlp_status tpmlp_attention_tp_backward(const void* X, const void* Wqkv, const void* Wo, const void* QKV,
                                         const void* O, const float* LSE, const void* dY, int64_t S, int64_t B,
                                         int64_t H, int32_t n_shards, int causal, void* dX, void* dWqkv,
                                         void* dbqkv, void* dWo, void* dbo, void* dQKV_out, void* workspace,
                                         size_t workspace_bytes, tpmlp_stream_t stream) {
  tpmlp_status st = attn_check(S, B, H, kHd);
  if (st != TPMLP_OK) return st;
  if (n_shards < 1 || H % n_shards != 0 || (causal != 0 && causal != 1)) return TPMLP_ERR_INVALID_ARG;
  if (S == 0) return TPMLP_OK;
  if (!al16(X) || !al16(Wqkv) || !al16(Wo) || !al16(QKV) || !al16(O) || !al16(LSE) || !al16(dY) || !al16(dX) ||
      !al16(dWqkv) || !al16(dWo) || (dbqkv != nullptr && !al16(dbqkv)) || (dbo != nullptr && !al16(dbo)) ||
      (dQKV_out != nullptr && !al16(dQKV_out)))
    return TPMLP_ERR_INVALID_ARG;
  const Bwd z = bwd_sizes(S, B, H);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < z.delta + z.dO + z.dqkv + z.partial)
    return TPMLP_ERR_WORKSPACE;
  DeviceCtx c;
  if (current_device_ctx(&c) != cudaSuccess) return TPMLP_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int T = static_cast<int>(S * B), d = static_cast<int>(H * kHd);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  float* delta = reinterpret_cast<float*>(w);
  void* dO = w + z.delta;
  void* dqkv = dQKV_out != nullptr ? dQKV_out : static_cast<void*>(w + z.delta + z.dO);
  float* partial = reinterpret_cast<float*>(w + z.delta + z.dO + z.dqkv);
  // row-parallel output projection: dO_i = dY Wo[rows of shard i]^T for every shard at once,
  // dWo = O^T dY, dbo = column sums of dY
  GemmLaunch g;
  g.M = T;
  g.N = d;
  g.K = d;
  g.a = {dY, d, false};
  g.b = {Wo, d, false};
  g.out0 = dO;
  g.ld0 = d;
  cudaError_t e = launch_gemm(g, c, s);
  if (e == cudaSuccess) {
    GemmLaunch gw;
    gw.M = d;
    gw.N = d;
    gw.K = T;
    gw.a = {O, d, true};
    gw.b = {dY, d, true};
    gw.out0 = dWo;
    gw.ld0 = d;
    e = launch_gemm(gw, c, s);
  }
  if (e == cudaSuccess && dbo != nullptr) e = launch_column_sum_bf16(dY, T, d, d, partial, dbo, s);
  // attention backward of every (batch, head)
  if (e == cudaSuccess)
    e = launch_attention_bwd(QKV, O, dO, LSE, delta, static_cast<int>(S), static_cast<int>(B), static_cast<int>(H),
                             causal == 1, dqkv, c, s);
  // column-parallel projection: dWqkv = X^T dQKV, dbqkv = column sums of dQKV, dX = dQKV Wqkv^T (the K loop
  // walks every shard's columns: the backward shard sum)
  if (e == cudaSuccess) {
    GemmLaunch gw;
    gw.M = d;
    gw.N = 3 * d;
    gw.K = T;
    gw.a = {X, d, true};
    gw.b = {dqkv, 3 * d, true};
    gw.out0 = dWqkv;
    gw.ld0 = 3 * d;
    e = launch_gemm(gw, c, s);
  }
  if (e == cudaSuccess && dbqkv != nullptr) e = launch_column_sum_bf16(dqkv, T, 3 * d, 3 * d, partial, dbqkv, s);
  if (e == cudaSuccess) {
    GemmLaunch gx;
    gx.M = T;
    gx.N = d;
    gx.K = 3 * d;
    gx.a = {dqkv, 3 * d, false};
    gx.b = {Wqkv, 3 * d, false};
    gx.out0 = dX;
    gx.ld0 = d;
    e = launch_gemm(gx, c, s);
  }
  return to_status(e);
}

}  // extern "C"
