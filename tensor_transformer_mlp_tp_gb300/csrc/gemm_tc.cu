// Host launcher of the tcgen05 GEMM: TMA tensor maps, tile grid, and the
// kernel instantiation for each (operand majorness, epilogue) the MLP uses.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "gemm_tc.cuh"
#include "launch.h"

namespace tpmlp {
namespace {

constexpr int kStages = 4;
constexpr int kEpiWarps = 4;
constexpr int kBN = 256;
constexpr int kGroupM = 16;

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

// 2-D bf16 tensor map over a row-major matrix of `outer` rows of `inner`
// elements (`ld` elements apart), 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap* m, const void* base, long long inner, long long outer, long long ld, int box_inner,
              int box_outer) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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

}  // namespace

cudaError_t launch_gemm(const GemmLaunch& g, const DeviceCtx& ctx, cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return cudaSuccess;
  GemmParams p;
  memset(&p, 0, sizeof(p));
  // A operand (the M side): box of 128 rows x 64 k (K-major) or 64 m x 64 k rows (MN-major).
  bool ok = g.a.mn_major ? make_map(&p.tmA, g.a.ptr, g.M, g.K, g.a.ld, 64, kBK)
                         : make_map(&p.tmA, g.a.ptr, g.K, g.M, g.a.ld, kBK, kBM);
  ok = ok && (g.b.mn_major ? make_map(&p.tmB, g.b.ptr, g.N, g.K, g.b.ld, 64, kBK)
                           : make_map(&p.tmB, g.b.ptr, g.K, g.N, g.b.ld, kBK, kBN));
  if (!ok) return cudaErrorInvalidValue;
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.m_blocks = (g.M + kBM - 1) / kBM;
  p.n_blocks = (g.N + kBN - 1) / kBN;
  p.shards = g.shards < 1 ? 1 : g.shards;
  const int k_blocks = (g.K + kBK - 1) / kBK;
  if (p.shards > 1 && (k_blocks % p.shards != 0 || g.K % (p.shards * kBK) != 0)) return cudaErrorInvalidValue;
  p.k_blocks_per_shard = k_blocks / p.shards;
  p.group_m = kGroupM;
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
  p.err = ctx.err;
  p.timeout_ns = ctx.timeout_ns;
  const long long tiles = static_cast<long long>(p.m_blocks) * p.n_blocks * p.shards;
  const int grid = static_cast<int>(tiles < ctx.sm_count ? tiles : ctx.sm_count);

  const bool amn = g.a.mn_major, bmn = g.b.mn_major;
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
