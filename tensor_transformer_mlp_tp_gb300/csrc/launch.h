// Host-side launchers shared by the translation units of libtpmlp (internal).
#pragma once

#include <cuda_runtime.h>

#include "common.h"

namespace tpmlp {

// One operand of C = A * B as it is stored in memory.
//  mn_major == false: stored [MN x K], K contiguous, `ld` elements between rows.
//  mn_major == true : stored [K x MN], M (or N) contiguous, `ld` elements between rows.
struct Operand {
  const void* ptr;
  long long ld;
  bool mn_major;
};

// The rest of the sequence-parallel region after the row-parallel reduction:
// out = residual + keep * (sum + bias2) * scale (philox.cuh decides keep).
struct SpTail {
  bool on = false;
  const void* bias2 = nullptr;    // [d] bf16 or nullptr
  ConstChunkPtrs residual{};      // chunk layout, or residual.p[0] == nullptr
  float scale = 1.f;              // 1 / (1 - p)
  unsigned long long seed = 0, offset = 0;
  unsigned long long thr = 1ull << 32;  // floor((1 - p) 2^32); 2^32 keeps all
  uint8_t* mask = nullptr;        // keep bits: written by the forward tails, read by the dropout backward
};

struct GemmLaunch {
  int M = 0, N = 0, K = 0;
  Operand a{}, b{};
  int epi = kEpiStore;
  int shards = 1;
  void* out0 = nullptr;
  long long ld0 = 0;
  void* out1 = nullptr;
  long long ld1 = 0;
  long long shard_stride0 = 0;
  const void* bias = nullptr;
  const void* aux = nullptr;
  long long ld_aux = 0;
  float* colsum = nullptr;
  int rows_per_chunk = 0;
  ChunkPtrs chunks{};
  SpTail tail{};  // only with the chunked store
  // E4M3 operands (both K-major, row strides multiples of 16 bytes): dequantised by the two scales
  bool fp8 = false;
  const float* scale_a = nullptr;
  const float* scale_b = nullptr;
  const float* scale_out = nullptr;  // kEpiBiasGeluQ, kEpiDGeluQ
  float* amax_out = nullptr;         // kEpiBiasGeluQ, kEpiDGeluQ
  int a_fmt = 0, b_fmt = 0;          // 0 = E4M3, 1 = E5M2
};

struct DeviceCtx {
  unsigned int* err;           // device error words
  unsigned long long timeout_ns;
  int sm_count;
};

// Bounds-check violations counted by the row kernels' / the GEMMs' translation units since the last call
// (zero in release builds, which check nothing), and the first site; both cleared.
cudaError_t rowwise_bounds_status(unsigned int* count, unsigned int* site);
cudaError_t gemm_bounds_status(unsigned int* count, unsigned int* site);

// Returns cudaErrorNotSupported for operand/epilogue combinations without a kernel.
cudaError_t launch_gemm(const GemmLaunch& g, const DeviceCtx& ctx, cudaStream_t s);

cudaError_t launch_layernorm_fwd(const RowParams& r, const DeviceCtx& ctx, cudaStream_t s);
// The RMS norm of the SequenceParallelLayerNorm listing (gamma = the weight; beta unused).
cudaError_t launch_rmsnorm_fwd(const RowParams& r, cudaStream_t s);
// LayerNorm backward using `scratch` (cap_floats floats of dgamma/dbeta block partials, 2 d per block).
// layernorm_bwd_scratch_floats(rows, d) covers the default block count; a smaller scratch runs fewer
// blocks, down to one (2 d floats).
cudaError_t launch_layernorm_bwd(const RowParams& r, float* scratch, size_t cap_floats, const DeviceCtx& ctx,
                                 float* dgamma, float* dbeta, cudaStream_t s);
size_t layernorm_bwd_scratch_floats(int rows, int d);
int layernorm_bwd_blocks(int rows, int max_blocks);
// The device context (error words, SM count, wait budget) of the current device.
cudaError_t current_device_ctx(DeviceCtx* out);
// Process-unique id of the CUDA context current on this thread (the driver's cuCtxGetId), 0 when no
// context is current or the query is unavailable.  A device reset gives the device a new context, and
// with it a new id: addresses of the library's __device__ arrays cached under the old id are stale.
unsigned long long current_context_id();
// Largest d the LayerNorm backward supports (its 2 d fp32 accumulators live in shared memory).
constexpr int kLnBwdMaxD = 16384;
cudaError_t launch_reduce_scatter(const RowParams& r, const DeviceCtx& ctx, cudaStream_t s);
cudaError_t launch_gather_rows(const RowParams& r, const DeviceCtx& ctx, cudaStream_t s);
// Dropout backward: dst [rows x d] (contiguous) = keep * in_chunks * drop_scale; with `partial`
// (dropout_bwd_scratch_floats) also dbias2 [d] bf16 = the column sums of dst before rounding.
cudaError_t launch_dropout_bwd(const RowParams& r, float* partial, void* dbias2, cudaStream_t s);
size_t dropout_bwd_scratch_floats(int rows, int d);
// out[c] = sum_r partial[r * cols + c] over r < rows, fixed order; bf16 or fp32 output.
cudaError_t launch_column_sum(const float* partial, int rows, int cols, void* out, bool out_bf16, cudaStream_t s);
// out[c] (bf16) = sum_r src[r ld + c] for a bf16 matrix [rows x cols] (cols and ld multiples of 8), through
// `partial` (column_sum_bf16_scratch_floats(rows, cols) floats) in a fixed order.
cudaError_t launch_column_sum_bf16(const void* src, int rows, int cols, long long ld, float* partial, void* out,
                                   cudaStream_t s);
size_t column_sum_bf16_scratch_floats(int rows, int cols);
// E4M3 casts.  dst = E4M3(src * (*scale)) for src [rows x cols] bf16 (row-major), written [rows x cols]
// or, with `transpose`, [cols x rows]; *amax is max-combined with max |src|.  Row lengths multiples of 16.
cudaError_t launch_cast_e4m3(const void* src, int rows, int cols, bool transpose, const float* scale, void* dst,
                             float* amax, cudaStream_t s);
// The same cast to E5M2 (fmt 1) or E4M3 (fmt 0).
cudaError_t launch_cast_fp8(const void* src, int rows, int cols, bool transpose, int fmt, const float* scale,
                            void* dst, float* amax, cudaStream_t s);
// dst [cols x rows] bytes = the transpose of src [rows x cols] bytes (rows, cols multiples of 16).
cudaError_t launch_transpose_bytes(const void* src, int rows, int cols, void* dst, cudaStream_t s);
// LayerNorm of every chunk, written as E4M3(LN(x) * (*scale)) into the gathered [T x d] byte buffer
// r.dst; *amax max-combined with max |LN(x)|.
cudaError_t launch_layernorm_fwd_e4m3(const RowParams& r, const float* scale, float* amax, cudaStream_t s);
// Delayed scaling: for each of n tensors, history[i][0..len) shifts by one and takes amax[i];
// scale[i] = fp8_max / mean(history[i]) / 2^margin (1 while the mean is not positive); amax[i] = 0.
cudaError_t launch_fp8_update(float* scale, float* amax, float* history, int n, int len, float fp8_max, int margin,
                              cudaStream_t s);

cudaError_t launch_mlp_fp32(const float* X, const float* A, const float* B, const float* bias, int T, int d, int F,
                            float* H, float* Y, cudaStream_t s);

}  // namespace tpmlp
