// Host launcher of the tcgen05 GEMM: TMA tensor maps, tile grid, and the
// kernel instantiation for each (operand majorness, epilogue) the MLP uses.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>

#include "gemm_tc2.cuh"
#include "launch.h"

namespace tpmlp {
namespace {

constexpr int kStages = 4;       // single CTA: 48 KB per k-block
constexpr int kPairStages = 6;   // CTA pair: 32 KB per CTA per k-block
constexpr int kEpiWarps = 4;
constexpr int kBN = 256;
constexpr int kGroupM = 16;      // raster group, in 128-row blocks
constexpr int kShortK = 2048;    // at or below: the GeLU epilogue runs balanced over all four sub-partitions
// Balanced epilogues (every epilogue warp reads TMEM and does its own math): 10 warps for the bf16 GeLU
// GEMM with a short K and for the row-parallel GEMM's store (measured on GB300, d = 1024: 10 and 14
// warps equal, 6 warps 10% slower), 6 for the FP8 quantising epilogues (10 and 14 measured slower).
constexpr int kBalWarps = 10;
constexpr int kBalFp8 = 6;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 2-D tensor map over a row-major matrix of `outer` rows of `inner` elements
// (`ld` elements apart; bf16, or bytes for E4M3), 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap* m, const void* base, long long inner, long long outer, long long ld, int box_inner,
              int box_outer, bool bytes = false, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * (bytes ? 1 : 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
            dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool AMN, bool BMN, int EPI>
cudaError_t run(const GemmParams& p, int grid, cudaStream_t s) {
  using S = GemmShape<kBN, kStages, kEpiWarps>;
  auto kern = k_gemm_tc<kBN, AMN, BMN, EPI, kStages, kEpiWarps>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, S::kThreads, S::kSmem, s>>>(p);
  return cudaGetLastError();
}

// Largest number of co-resident CTA pairs of `kern` on the current device (cached per device).
template <typename K>
int max_pairs(K kern, int smem, int threads, int dev_cache_slot, std::atomic<int>* cache) {
  const int known = cache[dev_cache_slot].load(std::memory_order_relaxed);
  if (known > 0) return known;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) n = 1;
  cache[dev_cache_slot].store(n, std::memory_order_relaxed);
  return n;
}

// The K-major B map of half tiles was made (the launchers leave it all zero otherwise).
bool half_map_ok(const GemmParams& p) {
  const unsigned char* b = reinterpret_cast<const unsigned char*>(&p.tmB_half);
  for (size_t i = 0; i < sizeof(p.tmB_half); ++i)
    if (b[i] != 0) return true;
  return false;
}

template <int BN, bool AMN, bool BMN, int EPI, bool FP8 = false, int BAL = 0>
cudaError_t run_pair(GemmParams p, cudaStream_t s) {
  using S = PairShape<BN, kPairStages, kEpiWarps, BAL>;
  auto kern = k_gemm_tc2<BN, AMN, BMN, EPI, kPairStages, kEpiWarps, FP8, BAL>;
  constexpr int kThreads = S::kThreads;
  static std::atomic<int> cache[64] = {};  // co-resident pairs per device (concurrent callers store the same value)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmem);
  if (e != cudaSuccess) return e;
  const int pairs = max_pairs(kern, S::kSmem, kThreads, dev & 63, cache);
  const long long tiles = static_cast<long long>(p.m_blocks) * p.n_blocks * p.shards;
  long long units = tiles;
  p.full_units = static_cast<int>(tiles);
  // A last wave of whole tiles that would leave more than half of the pairs idle runs as one round of
  // half-width tiles instead (each pair then finishes its share in half a tile's time).
  const long long rem = tiles % pairs;
  if (BN == kBN && p.shards == 1 && rem != 0 && 2 * rem <= pairs && (BMN || half_map_ok(p))) {
    p.full_units = static_cast<int>(tiles - rem);
    units = tiles + rem;
  }
  const int grid_pairs = static_cast<int>(units < pairs ? units : pairs);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * grid_pairs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = S::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the kernel's set-up overlaps the previous kernel's tail (it waits for
  // that kernel's completion before touching global memory)
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

bool pair_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("TPMLP_GEMM_PAIR");
    return v == nullptr || v[0] != '0';
  }();
  return on;
}

}  // namespace

// E4M3 GEMMs: always the CTA pair (a lone 128-row block leaves the odd CTA's rows to zero fill), both
// operands K-major, 128-element k-blocks.
static cudaError_t launch_gemm_fp8(const GemmLaunch& g, const DeviceCtx& ctx, cudaStream_t s) {
  if (g.a.mn_major || g.b.mn_major || g.shards > 1) return cudaErrorNotSupported;
  if (g.scale_a == nullptr || g.scale_b == nullptr) return cudaErrorInvalidValue;
  if ((g.epi == kEpiBiasGeluQ || g.epi == kEpiDGeluQ) && g.scale_out == nullptr) return cudaErrorInvalidValue;
  if (g.a_fmt < 0 || g.a_fmt > 1 || g.b_fmt < 0 || g.b_fmt > 1) return cudaErrorInvalidValue;
  constexpr int kKb = 128;
  GemmParams p;
  memset(&p, 0, sizeof(p));
  bool ok = make_map(&p.tmA, g.a.ptr, g.K, g.M, g.a.ld, kKb, kBM, true) &&
            make_map(&p.tmB, g.b.ptr, g.K, g.N, g.b.ld, kKb, kBN / 2, true);
  if (!ok) return cudaErrorInvalidValue;
  if (!make_map(&p.tmB_half, g.b.ptr, g.K, g.N, g.b.ld, kKb, kBN / 4, true)) memset(&p.tmB_half, 0, sizeof(p.tmB_half));
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.m_blocks = (g.M + 2 * kBM - 1) / (2 * kBM);
  p.n_blocks = (g.N + kBN - 1) / kBN;
  p.shards = 1;
  p.k_blocks_per_shard = (g.K + kKb - 1) / kKb;
  p.group_m = kGroupM / 2;
  p.out0 = g.out0;
  p.ld0 = g.ld0;
  p.out1 = g.out1;
  p.ld1 = g.ld1;
  p.bias = g.bias;
  p.aux = g.aux;
  p.ld_aux = g.ld_aux;
  p.colsum = g.colsum;
  p.rows_per_chunk = g.rows_per_chunk;
  p.chunks = g.chunks;
  p.tail = g.tail.on && g.rows_per_chunk > 0 && g.epi == kEpiStore ? 1 : 0;
  if (p.tail) p.bias = g.tail.bias2;
  p.drop_scale = g.tail.scale;
  p.drop_seed = g.tail.seed;
  p.drop_offset = g.tail.offset;
  p.drop_thr = g.tail.thr;
  p.drop_mask = g.tail.mask;
  p.res_chunks = g.tail.residual;
  p.a_fmt = g.a_fmt;
  p.b_fmt = g.b_fmt;
  p.scale_a = g.scale_a;
  p.scale_b = g.scale_b;
  p.scale_out = g.scale_out;
  p.amax_out = g.amax_out;
  p.err = ctx.err;
  p.timeout_ns = ctx.timeout_ns;
  switch (g.epi) {
    case kEpiBiasGeluQ: return run_pair<kBN, false, false, kEpiBiasGeluQ, true, kBalFp8>(p, s);
    case kEpiDGeluQ: return run_pair<kBN, false, false, kEpiDGeluQ, true, kBalFp8>(p, s);
    case kEpiStore: return run_pair<kBN, false, false, kEpiStore, true>(p, s);
    default: return cudaErrorNotSupported;
  }
}

cudaError_t gemm_bounds_status(unsigned int* count, unsigned int* site) {
#ifdef TPMLP_DEBUG_BOUNDS
  return bounds_read_and_clear(count, site);
#else
  *count = *site = 0;
  return cudaSuccess;
#endif
}

cudaError_t launch_gemm(const GemmLaunch& g, const DeviceCtx& ctx, cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return cudaSuccess;
  if (g.fp8) return launch_gemm_fp8(g, ctx, s);
  GemmParams p;
  memset(&p, 0, sizeof(p));
  // A operand (the M side): box of 128 rows x 64 k (K-major) or 64 m x 64 k rows (MN-major).
  bool ok = g.a.mn_major ? make_map(&p.tmA, g.a.ptr, g.M, g.K, g.a.ld, 64, kBK)
                         : make_map(&p.tmA, g.a.ptr, g.K, g.M, g.a.ld, kBK, kBM);
  // CTA pairs whenever there are at least two 128-row blocks; each CTA then loads half of B's columns.
  const bool pair = pair_enabled() && g.M > kBM;
  const int b_rows = pair ? kBN / 2 : kBN;
  ok = ok && (g.b.mn_major ? make_map(&p.tmB, g.b.ptr, g.N, g.K, g.b.ld, 64, kBK)
                           : make_map(&p.tmB, g.b.ptr, g.K, g.N, g.b.ld, kBK, b_rows));
  if (!ok) return cudaErrorInvalidValue;
  // K-major B of half-width pair tiles: a quarter tile's columns per CTA
  if (pair && !g.b.mn_major && !make_map(&p.tmB_half, g.b.ptr, g.K, g.N, g.b.ld, kBK, kBN / 4))
    memset(&p.tmB_half, 0, sizeof(p.tmB_half));
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.m_blocks = pair ? (g.M + 2 * kBM - 1) / (2 * kBM) : (g.M + kBM - 1) / kBM;
  p.n_blocks = (g.N + kBN - 1) / kBN;
  p.shards = g.shards < 1 ? 1 : g.shards;
  const int k_blocks = (g.K + kBK - 1) / kBK;
  if (p.shards > 1 && (k_blocks % p.shards != 0 || g.K % (p.shards * kBK) != 0)) return cudaErrorInvalidValue;
  p.k_blocks_per_shard = k_blocks / p.shards;
  p.group_m = pair ? kGroupM / 2 : kGroupM;
  p.out0 = g.out0;
  p.ld0 = g.ld0;
  p.out1 = g.out1;
  p.ld1 = g.ld1;
  p.shard_stride0 = g.shard_stride0;
  p.bias = g.bias;
  p.aux = g.aux;
  p.ld_aux = g.ld_aux;
  p.colsum = g.colsum;
  p.rows_per_chunk = g.rows_per_chunk;
  p.chunks = g.chunks;
  p.tail = g.tail.on && g.rows_per_chunk > 0 && g.epi == kEpiStore ? 1 : 0;
  if (p.tail) p.bias = g.tail.bias2;
  p.drop_scale = g.tail.scale;
  p.drop_seed = g.tail.seed;
  p.drop_offset = g.tail.offset;
  p.drop_thr = g.tail.thr;
  p.drop_mask = g.tail.mask;
  p.res_chunks = g.tail.residual;
  p.err = ctx.err;
  p.timeout_ns = ctx.timeout_ns;
  // bf16 outputs of the pair kernel leave through TMA box stores where a tensor map can describe them (a
  // 16-byte aligned base and row pitch): out0 of the bias (+ GeLU) epilogues and of the plain store, and
  // the pre-activation out1
  p.tma_out = 0;
  if (pair && g.out0 != nullptr &&
      (g.epi == kEpiBiasGelu || g.epi == kEpiBias || (g.epi == kEpiStore && g.rows_per_chunk <= 0 && p.shards == 1))) {
    constexpr CUtensorMapSwizzle kSw = CU_TENSOR_MAP_SWIZZLE_64B;
    if (make_map(&p.tmC0, g.out0, g.N, g.M, g.ld0, 32, 32, false, kSw)) p.tma_out = 1;
    if (p.tma_out && g.epi == kEpiBiasGelu && g.out1 != nullptr)
      p.tma_out = make_map(&p.tmC1, g.out1, g.N, g.M, g.ld1, 32, 32, false, kSw) ? 3 : 0;
  }
  const long long tiles = static_cast<long long>(p.m_blocks) * p.n_blocks * p.shards;
  const int grid = static_cast<int>(tiles < ctx.sm_count ? tiles : ctx.sm_count);

  const bool amn = g.a.mn_major, bmn = g.b.mn_major;
  if (pair) {
    switch (g.epi) {
      case kEpiBiasGelu:
        // with a short K the bias + GeLU epilogue outlasts a tile's MMAs: spread it over all sub-partitions
        if (!amn && bmn && g.K <= kShortK) return run_pair<kBN, false, true, kEpiBiasGelu, false, kBalWarps>(p, s);
        if (!amn && bmn) return run_pair<kBN, false, true, kEpiBiasGelu>(p, s);
        break;
      case kEpiBias:
        if (!amn && bmn) return run_pair<kBN, false, true, kEpiBias>(p, s);
        break;
      case kEpiStore:
        // the row-parallel GEMM: few, long tiles, so the last tile's epilogue is exposed
        if (!amn && bmn) return run_pair<kBN, false, true, kEpiStore, false, kBalWarps>(p, s);
        if (amn && bmn) return run_pair<kBN, true, true, kEpiStore>(p, s);
        if (!amn && !bmn) return run_pair<kBN, false, false, kEpiStore>(p, s);
        break;
      case kEpiDGelu:
        if (!amn && !bmn) return run_pair<kBN, false, false, kEpiDGelu>(p, s);
        break;
      default:
        break;
    }
    return cudaErrorNotSupported;
  }
  switch (g.epi) {
    case kEpiBiasGelu:
      if (!amn && bmn) return run<false, true, kEpiBiasGelu>(p, grid, s);
      break;
    case kEpiBias:
      if (!amn && bmn) return run<false, true, kEpiBias>(p, grid, s);
      break;
    case kEpiStore:
      if (!amn && bmn) return run<false, true, kEpiStore>(p, grid, s);
      if (amn && bmn) return run<true, true, kEpiStore>(p, grid, s);
      if (!amn && !bmn) return run<false, false, kEpiStore>(p, grid, s);
      break;
    case kEpiDGelu:
      if (!amn && !bmn) return run<false, false, kEpiDGelu>(p, grid, s);
      break;
    default:
      break;
  }
  return cudaErrorNotSupported;
}

}  // namespace tpmlp
