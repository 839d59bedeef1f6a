// Debug-build bounds checks on hand-computed global indices.
//
// A build with -DTPMLP_DEBUG_BOUNDS compares each checked index with the extent of the buffer it addresses
// (TPMLP_IN_BOUNDS(index, extent, site)); an index outside [0, extent) is counted in a per-translation-unit
// device word, with the site of the first one, and the access it guards is skipped, so a wrong index never
// reaches memory.  Release builds compile every check to the constant `true`.  Each translation unit that
// includes this header defines its own counters and reads them with bounds_read_and_clear (host code of
// the same unit); the library reports the sum through tpmlp_debug_bounds_status.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tpmlp {

// Sites of the checks (reported as the first failing one).
enum BoundsSite : uint32_t {
  kBoundsInChunk = 101,      // a row of an input chunk (chunk index, row within it)
  kBoundsOutChunk = 102,     // a row of an output chunk
  kBoundsAddChunk = 103,     // a row of an added (residual) chunk
  kBoundsRowStore = 104,     // a row kernel's store into a gathered [rows x d] tensor
  kBoundsRowLoad = 105,      // a row kernel's load from a gathered [rows x d] tensor
  kBoundsPartial = 106,      // a column-partial row [blocks x cols]
  kBoundsShard = 107,        // a shard's slice of the explicit partials [N x rows x d]
  kBoundsGemmChunk = 120,    // the GEMM's chunked store: chunk index
  kBoundsGemmShard = 121,    // the GEMM's per-shard partial store: shard index
  kBoundsGemmColsum = 122,   // the GEMM's column partial sums: partial row
};

#ifdef TPMLP_DEBUG_BOUNDS
namespace {
__device__ unsigned int g_bounds_words[2];  // [0] violations, [1] first site

__device__ __forceinline__ bool in_bounds_dbg(long long index, long long extent, uint32_t site) {
  if (index >= 0 && index < extent) return true;
  atomicAdd(&g_bounds_words[0], 1u);
  atomicCAS(&g_bounds_words[1], 0u, site);
  return false;
}

// Violations counted by this translation unit since the last call, and the first site; clears both.
inline cudaError_t bounds_read_and_clear(unsigned int* count, unsigned int* site) {
  unsigned int w[2] = {0, 0};
  cudaError_t e = cudaMemcpyFromSymbol(w, g_bounds_words, sizeof(w));
  if (e != cudaSuccess) return e;
  *count = w[0];
  *site = w[1];
  const unsigned int zero[2] = {0, 0};
  return cudaMemcpyToSymbol(g_bounds_words, zero, sizeof(zero));
}
}  // namespace
#define TPMLP_IN_BOUNDS(index, extent, site) \
  ::tpmlp::in_bounds_dbg(static_cast<long long>(index), static_cast<long long>(extent), (site))
constexpr bool kBoundsChecked = true;
#else
#define TPMLP_IN_BOUNDS(index, extent, site) true
constexpr bool kBoundsChecked = false;
#endif

}  // namespace tpmlp
