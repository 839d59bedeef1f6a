// tpmlp_layernorm_backward_noalloc: the LayerNorm backward without a caller
// workspace.
//
// The regular tpmlp_layernorm_backward needs scratch for its per-block
// dgamma/dbeta partial sums, and takes it from a workspace the caller
// allocates.  Some callers cannot allocate device memory at the point where
// they run the backward: a host framework whose pool already owns the device
// memory and refuses outside allocations, or latency-critical code that must
// not enter the CUDA allocator (cudaMalloc/cudaFree can synchronise the
// device).  For them this entry point keeps the scratch in a fixed array that
// is part of the library's device image, so the call itself allocates nothing.
//
// Limits and sharing:
//  - The array holds kNoAllocBlocks x 2 x kNoAllocMaxD floats (9.5 MiB): the
//    row statistics and dgamma/dbeta column partials of the backward.  Every
//    GPU that loads the library keeps it until the process exits.
//  - d above kNoAllocMaxD is rejected with TPMLP_ERR_UNSUPPORTED before
//    anything is launched.
//  - All calls on a device share the one array.  Each block writes its whole
//    partial row before the column sum reads it, so nothing has to start at
//    zero, but two calls whose kernels overlap on the GPU (different streams,
//    no ordering between them) race on the array and give wrong dgamma/dbeta.
//  - The first call on a device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call
//    before any stream capture.  The address is cached per device together
//    with the id of the context it belongs to; after a device reset (a new
//    context) the next call looks it up again, so that first call after a
//    reset must also come before any capture.
#include <cstdint>
#include <mutex>

#include "../../include/tpmlp.h"
#include "launch.h"

namespace tpmlp {
namespace {

constexpr int kNoAllocBlocks = 152;
constexpr int kNoAllocMaxD = 8192;
constexpr size_t kNoAllocFloats = static_cast<size_t>(kNoAllocBlocks) * 2 * kNoAllocMaxD;

static __device__ __align__(256) float g_lnbwd_scratch[kNoAllocFloats];

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[64] = {};
unsigned long long g_noalloc_ctx[64] = {};  // context id each cached address belongs to

// Device address of the scratch array on the current device, looked up once per device (and again when
// the device's context has changed since, after a reset).
cudaError_t scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr || current_context_id() != g_noalloc_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_lnbwd_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
    g_noalloc_ctx[dev] = current_context_id();  // the lookup made the device's context current
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace tpmlp

extern "C" tpmlp_status tpmlp_layernorm_backward_noalloc(const void* const* X_chunks, const void* gamma, float eps,
                                                         const void* dXg, const tpmlp_shape* shape,
                                                         void* const* dX_chunks, void* dgamma, void* dbeta,
                                                         tpmlp_stream_t stream) {
  using namespace tpmlp;
  if (shape == nullptr || shape->tokens < 0 || shape->d < 1 || shape->ffn < 1 || shape->n_shards < 1 ||
      shape->n_shards > kMaxShards || shape->dtype != TPMLP_BF16 || shape->ffn % shape->n_shards != 0 ||
      shape->tokens % shape->n_shards != 0 || shape->d % 8 != 0 || (shape->ffn / shape->n_shards) % 8 != 0 ||
      shape->tokens > (1LL << 30))
    return TPMLP_ERR_INVALID_ARG;
  if (shape->d > kNoAllocMaxD) return TPMLP_ERR_UNSUPPORTED;
  if (shape->tokens == 0) return TPMLP_OK;
  if (X_chunks == nullptr || dX_chunks == nullptr || !aligned16(gamma) || !aligned16(dXg) || !aligned16(dgamma) ||
      !aligned16(dbeta) || !(eps >= 0.f))
    return TPMLP_ERR_INVALID_ARG;
  const int n = shape->n_shards;
  for (int i = 0; i < n; ++i)
    if (!aligned16(X_chunks[i]) || !aligned16(dX_chunks[i])) return TPMLP_ERR_INVALID_ARG;
  float* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return TPMLP_ERR_CUDA;
  DeviceCtx ctx;
  if (current_device_ctx(&ctx) != cudaSuccess) return TPMLP_ERR_CUDA;
  RowParams r{};
  for (int i = 0; i < n; ++i) {
    r.in_chunks.p[i] = X_chunks[i];
    r.out_chunks.p[i] = dX_chunks[i];
  }
  r.rows = static_cast<int>(shape->tokens);
  r.d = static_cast<int>(shape->d);
  r.n_chunks = n;
  r.rows_per_chunk = static_cast<int>(shape->tokens / n);
  r.eps = eps;
  r.gamma = gamma;
  r.src = dXg;
  // the launcher lays its statistics and partial sums out within the array's kNoAllocFloats
  const cudaError_t e = launch_layernorm_bwd(r, scratch, kNoAllocFloats, ctx, static_cast<float*>(dgamma),
                                             static_cast<float*>(dbeta), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TPMLP_OK : TPMLP_ERR_CUDA;
}
