/*
 * tpmlp.h -- C ABI of the GB300 tensor-parallel MLP block (libtpmlp.so).
 *
 * The block is the Megatron MLP  Y = GeLU(X A + b) B  with A in R^{d x 4d}
 * split into N column shards and B in R^{4d x d} split into N row shards:
 * shard i computes Y_i = GeLU(X A_i + b_i) B_i and an AllReduce sums the
 * partials, Y = sum_i Y_i.  Sources: "Megatron 架构与 6D 并行完整指南"
 * (walkerchi.com) §3.1 "原理"; "Megatron-LM 심층 아키텍처" (techknowgenie.com),
 * section "열 병렬(Column Parallel)과 행 병렬(Row Parallel)의 결합" and the
 * ColumnParallelLinear / RowParallelLinear listing in "분산 제어 소스코드 구조 패턴".
 * All N shards run on one GPU: the column shards are column ranges of one
 * launch, and the AllReduce is the K loop of the row-parallel GEMM, which
 * accumulates every shard's rows of B into one fp32 accumulator before a
 * single store.
 *
 * Conventions for every call:
 *  - Matrices are row-major.  bf16 is IEEE bfloat16; accumulation is fp32.
 *    X [T x d], A [d x F], B [F x d], bias [F], Y [T x d], with T = tokens,
 *    F = ffn (4d in the pages' model, any multiple of N here).
 *  - Shard i owns FFN columns [i F/N, (i+1) F/N) of A and bias and the same
 *    rows of B; sequence chunk j owns token rows [j T/N, (j+1) T/N).
 *  - Device pointers are owned by the caller and must stay valid until the
 *    work queued on `stream` has finished.  Arrays of chunk pointers
 *    (`X_chunks`, `Y_chunks`, ...) are HOST arrays of N device pointers, read
 *    during the call only.  The library allocates no device memory per call:
 *    scratch comes from the caller's workspace (size: tpmlp_workspace_size).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and never synchronise the host, except
 *    tpmlp_get_device_status.
 *  - Argument errors are returned before anything is launched: NULL where a
 *    pointer is required, tokens < 0, d or ffn < 1, N outside [1, 64],
 *    ffn % N != 0, and for bf16: d % 8 != 0, (ffn / N) % 8 != 0, a device
 *    pointer not 16-byte aligned; for the sequence-parallel calls T % N != 0;
 *    a workspace smaller than required (TPMLP_ERR_WORKSPACE).  tokens == 0 is
 *    a valid empty call: it launches nothing, leaves every output untouched
 *    (weight gradients of an empty batch are the caller's zeros) and accepts
 *    NULL pointers.
 *  - A failed launch returns TPMLP_ERR_CUDA.  Kernels never trap: every wait
 *    inside them is bounded (default 1 s, environment TPMLP_WAIT_TIMEOUT_MS);
 *    a wait that runs out records a device error word and the kernel exits,
 *    reported later by tpmlp_get_device_status as TPMLP_ERR_TIMEOUT.
 *  - Thread-compatible: concurrent calls from several host threads are safe;
 *    the only shared state is the per-device error word and cached device
 *    attributes.
 */
#ifndef TPMLP_H
#define TPMLP_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TPMLP_API __attribute__((visibility("default")))
#else
#define TPMLP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* tpmlp_stream_t; /* identical to cudaStream_t */

typedef enum {
  TPMLP_OK = 0,
  TPMLP_ERR_INVALID_ARG = 1,
  TPMLP_ERR_UNSUPPORTED = 2,
  TPMLP_ERR_CUDA = 3,
  TPMLP_ERR_TIMEOUT = 4,
  TPMLP_ERR_WORKSPACE = 5
} tpmlp_status;

typedef enum { TPMLP_BF16 = 0, TPMLP_FP32 = 1 } tpmlp_dtype;

/* Problem shape.  ffn is the FFN width F (4d on the pages); n_shards is N,
 * the tensor-parallel degree and, for the sequence-parallel calls, the number
 * of sequence chunks, 1 <= N <= 64 (TPMLP_ERR_INVALID_ARG otherwise).  dtype is
 * a tpmlp_dtype. */
typedef struct {
  int64_t tokens;
  int64_t d;
  int64_t ffn;
  int32_t n_shards;
  int32_t dtype;
} tpmlp_shape;

/* Operations whose workspace size can be queried. */
enum {
  TPMLP_OP_FWD = 0,            /* tpmlp_forward */
  TPMLP_OP_SP_FWD = 1,         /* tpmlp_sp_forward, TPMLP_RS_FUSED */
  TPMLP_OP_SP_FWD_PARTIALS = 2,/* tpmlp_sp_forward, TPMLP_RS_PARTIALS */
  TPMLP_OP_BWD = 3,            /* tpmlp_backward */
  TPMLP_OP_SP_BWD = 4,         /* tpmlp_sp_backward */
  TPMLP_OP_DH_GELUPRIME = 5,   /* tpmlp_gemm_dh_geluprime with a dbias output */
  TPMLP_OP_LN_BWD = 6,         /* tpmlp_layernorm_backward, tpmlp_layernorm_backward_add */
  TPMLP_OP_SP_BLOCK_BWD = 7,   /* tpmlp_sp_block_backward */
  TPMLP_OP_DROPOUT_BWD = 8,    /* tpmlp_dropout_backward with a dbias2 output */
  TPMLP_OP_SP_FWD_FP8 = 9,     /* tpmlp_sp_forward_fp8 */
  TPMLP_OP_SP_BWD_FP8 = 10     /* tpmlp_sp_backward_fp8 */
};

/* Dropout of the sequence-parallel region.  The pages name Dropout in the
 * sequence-split region (deep-dive page, section "All-Reduce 통신의 All-Gather
 * 및 Reduce-Scatter 분해"; glossary page, sequence-parallel paragraph) and give
 * neither a rate nor a generator.  p: drop probability in [0, 1), float32.
 * Element (r, c) of the gathered [T x d] output, index e = r d + c, is kept
 * when 32 bits of Philox4x64-10 (Salmon et al., SC 2011) with counter
 * (e / 8, offset, 0, 0) and key (seed, 0) -- word (e % 8) / 2, low half for
 * even e, high half for odd e -- are below floor((1 - p) 2^32); kept elements
  * are scaled by 1 / (1 - p).  The same (p, seed, offset) in the backward
 * regenerates the forward's mask; advance offset per step for a new mask.
 * keep_mask: NULL, or a device buffer of ceil(T d / 8) bytes holding the mask
 * as bits (bit e % 8 of byte e / 8 = element e kept).  With p > 0 the forward
 * calls write it as they apply the dropout; the backward calls read it instead
 * of regenerating the generator's bits (the same p, seed and offset must
 * describe the mask it holds).  No alignment requirement.
 * A NULL tpmlp_dropout pointer means p = 0. */
typedef struct {
  float p;
  uint64_t seed;
  uint64_t offset;
  uint8_t* keep_mask;
} tpmlp_dropout;

/* Reduce-scatter modes of tpmlp_sp_forward. */
enum {
  TPMLP_RS_FUSED = 0,    /* the row-parallel GEMM stores each output row into its chunk */
  TPMLP_RS_PARTIALS = 1  /* per-shard bf16 partials, then tpmlp_reduce_scatter; needs (ffn/N) % 64 == 0 */
};

/* Human-readable name of a status code (static string). */
TPMLP_API const char* tpmlp_status_string(tpmlp_status s);

/* Bytes of workspace `op` needs for `shape` (host arithmetic only, no CUDA
 * call).  The workspace is any 256-byte aligned device buffer of at least that
 * size; its contents need no initialisation and are clobbered. */
TPMLP_API tpmlp_status tpmlp_workspace_size(const tpmlp_shape* shape, int op, size_t* bytes);

/* Synchronise `stream`, then read and clear the current device's error word.
 * Returns TPMLP_ERR_TIMEOUT if a kernel gave up a bounded wait since the last
 * call (and writes the failing wait site to *site when site != NULL),
 * TPMLP_ERR_CUDA if the stream reports a CUDA error, else TPMLP_OK. */
TPMLP_API tpmlp_status tpmlp_get_device_status(tpmlp_stream_t stream, uint32_t* site);

/* Debug builds (compiled with -DTPMLP_DEBUG_BOUNDS; the tests build one
 * beside the release library) check the hand-computed global indices of the
 * row kernels and of the GEMM epilogues' direct stores against the extents of
 * their buffers, count every index found outside, record the site of the
 * first one, and skip (stores) or redirect to the first row (loads) that
 * access.  This call synchronises the device, sets *checked to 1 in such a
 * build and 0 in a release build (which checks nothing), and returns the
 * violations counted since the previous call and the first site (0 if none);
 * it clears both.  There is no counterpart on the pages: it is the library's
 * stand-in for a memory checker. */
TPMLP_API tpmlp_status tpmlp_debug_bounds_status(int32_t* checked, uint32_t* violations, uint32_t* first_site);

/* ------------------------------------------------------------------ block calls */

/* Tensor-parallel MLP forward ("6D" guide §3.1; deep-dive page, column/row
 * parallel section, eq. Output = Z W2 = sum_i Z_i W2_i).
 *   X [T x d], A [d x F], B [F x d], bias [F] or NULL (the column layer's
 *   bias, split with A's columns), Y [T x d] out.
 *   Hpre_out: NULL, or [T x F] receiving the pre-activation X A + b (bf16)
 *   for a later tpmlp_backward.  H_out: NULL, or [T x F] receiving
 *   H = GeLU(X A + b) (otherwise H lives in the workspace); passing it to the
 *   backward saves recomputing it there.
 * bf16: tcgen05 GEMM with bias + exact erf-GeLU in the epilogue into H
 * (workspace), then the row-parallel GEMM summing all N shards in TMEM.
 * fp32 (shape->dtype == TPMLP_FP32): all pointers are fp32, CUDA-core FFMA;
 * Hpre_out must be NULL. */
TPMLP_API tpmlp_status tpmlp_forward(const void* X, const void* A, const void* B, const void* bias,
                                     const tpmlp_shape* shape, void* Y, void* Hpre_out, void* H_out, void* workspace,
                                     size_t workspace_bytes, tpmlp_stream_t stream);

/* Sequence-parallel block forward (deep-dive page, section "All-Reduce 통신의
 * All-Gather 및 Reduce-Scatter 분해"; SequenceParallelLayerNorm in the listing):
 * LayerNorm of every S/N chunk (fp32 statistics, biased variance, eps inside
 * the square root, scale gamma and shift beta), All-Gather of the chunks,
 * the MLP, Reduce-Scatter of the shard partials back to chunks.
 *   X_chunks: host array of N pointers, each [T/N x d]; gamma, beta [d];
 *   Y_chunks: host array of N pointers, each [T/N x d] out; rs_mode:
 *   TPMLP_RS_FUSED or TPMLP_RS_PARTIALS; Hpre_out, H_out: NULL or [T x F]
 *   as in tpmlp_forward; Xg_out: NULL or [T x d] receiving the gathered
 *   LayerNorm output (otherwise it lives in the workspace).  bf16 only. */
TPMLP_API tpmlp_status tpmlp_sp_forward(const void* const* X_chunks, const void* gamma, const void* beta, float eps,
                                        const void* A, const void* B, const void* bias, const tpmlp_shape* shape,
                                        void* const* Y_chunks, int rs_mode, void* Hpre_out, void* H_out,
                                        void* Xg_out, void* workspace, size_t workspace_bytes,
                                        tpmlp_stream_t stream);

/* MLP backward, the chain rule of the forward (the pages name two backward
 * AllReduces per block, glossary page, tensor-parallel section):
 *   Hpre = X A + b (the given Hpre, or recomputed when Hpre == NULL),
 *   H = GeLU(Hpre) (the forward's H when H != NULL and Hpre != NULL, else
 *   derived here), dHpre = (dY B^T) * GeLU'(Hpre), dB = H^T dY, dA = X^T dHpre,
 *   dbias = column sums of dHpre (if dbias != NULL), and
 *   dX = sum_i dHpre_i A_i^T  (the backward AllReduce, as one K loop).
 * Outputs dX [T x d], dA [d x F], dB [F x d], dbias [F] are bf16.  bf16 only. */
TPMLP_API tpmlp_status tpmlp_backward(const void* X, const void* A, const void* B, const void* bias,
                                      const void* Hpre, const void* H, const void* dY, const tpmlp_shape* shape,
                                      void* dX, void* dA, void* dB, void* dbias, void* workspace,
                                      size_t workspace_bytes, tpmlp_stream_t stream);

/* Sequence-parallel block backward: All-Gather of the dY chunks (the mirror
 * of the forward Reduce-Scatter), the MLP backward on the re-normalised
 * gathered input, Reduce-Scatter of the input gradient to chunks (the mirror
 * of the forward All-Gather), LayerNorm backward per chunk.
 *   dX_chunks: host array of N pointers [T/N x d] (bf16) out;
 *   dgamma, dbeta: [d] fp32 out, summed over all chunks; Hpre, H, dA, dB,
 *   dbias as in tpmlp_backward; Xg: NULL (the LayerNorm output is
 *   recomputed) or the forward's Xg_out.  bf16 only. */
TPMLP_API tpmlp_status tpmlp_sp_backward(const void* const* X_chunks, const void* gamma, const void* beta, float eps,
                                         const void* A, const void* B, const void* bias, const void* Hpre,
                                         const void* H, const void* Xg, const void* const* dY_chunks,
                                         const tpmlp_shape* shape,
                                         void* const* dX_chunks, void* dA, void* dB, void* dbias, void* dgamma,
                                         void* dbeta, void* workspace, size_t workspace_bytes,
                                         tpmlp_stream_t stream);

/* The whole sequence-parallel region of the MLP block (deep-dive page:
 * RowParallelLinear in "분산 제어 소스코드 구조 패턴" adds its bias after the
 * reduction; the SP section keeps Dropout in the sequence-split region):
 *   Y_j = X_j + dropout(Z_j + bias2),
 * Z_j chunk j of the reduced MLP output of tpmlp_sp_forward, bias2 [d] the
 * row layer's bias or NULL, X_j the block input chunk (the residual, which
 * the pages do not mention).  With TPMLP_RS_FUSED the row bias, dropout and
 * residual run in the row-parallel GEMM's chunked store; with
 * TPMLP_RS_PARTIALS in the reduce-scatter kernel.  Workspace, Hpre_out,
 * H_out and Xg_out as in tpmlp_sp_forward.  bf16 only. */
TPMLP_API tpmlp_status tpmlp_sp_block_forward(const void* const* X_chunks, const void* gamma, const void* beta,
                                              float eps, const void* A, const void* B, const void* bias,
                                              const void* bias2, const tpmlp_dropout* dropout,
                                              const tpmlp_shape* shape, void* const* Y_chunks, int rs_mode,
                                              void* Hpre_out, void* H_out, void* Xg_out, void* workspace,
                                              size_t workspace_bytes, tpmlp_stream_t stream);

/* Backward of tpmlp_sp_block_forward (chain rule): dZ = dY * keep / (1 - p)
 * gathered to [T x d], dbias2 = column sums of dZ ([d] bf16, or NULL), the
 * MLP and LayerNorm backward of tpmlp_sp_backward driven by dZ, and the
 * residual's gradient dY_j added to dX_j.  `dropout` must equal the
 * forward's.  Workspace: size of TPMLP_OP_SP_BLOCK_BWD.  bf16 only. */
TPMLP_API tpmlp_status tpmlp_sp_block_backward(const void* const* X_chunks, const void* gamma, const void* beta,
                                               float eps, const void* A, const void* B, const void* bias,
                                               const tpmlp_dropout* dropout, const void* Hpre, const void* H,
                                               const void* Xg, const void* const* dY_chunks,
                                               const tpmlp_shape* shape, void* const* dX_chunks, void* dA, void* dB,
                                               void* dbias, void* dbias2, void* dgamma, void* dbeta,
                                               void* workspace, size_t workspace_bytes, tpmlp_stream_t stream);

/* ------------------------------------------------------------------ FP8 (E4M3) forward
 * Deep-dive page, section "FP8 하이브리드 정밀도 및 지연 스케일링(Delayed Scaling)":
 * forward matmul operands in E4M3, each tensor scaled by its factor S before
 * the cast, q = E4M3(x S) (float32 product, round to nearest even, saturating
 * at +-448: the OCP E4M3 format without infinities), and the GEMM's fp32
 * accumulator divided by both scales.  Delayed scaling: the scales a step
 * uses come from the amaxes of earlier steps (the mean of an amax history,
 * the page's moving average); the step records its own amaxes for the next.
 * Scales and amaxes are device memory, so a step needs no host round trip.
 * E4M3 buffers are row-major bytes; d and F must be multiples of 16. */

/* Delayed-scaling state of the FP8 forward, four tensors in the order
 * X (the gathered norm output), A, B, H (the GeLU output):
 *   scale[4]    the factors this step casts with (device, fp32),
 *   amax[4]     this step's max |x| before the casts, max-combined by the
 *               kernels (device, fp32; zero it before the first step),
 *   history[4 x history_len]  earlier amaxes (device, fp32).
 * tpmlp_fp8_update_scales ends a step: each history shifts by one and takes
 * amax[i], scale[i] = 448 / mean(history[i]) / 2^margin (1 while the mean is
 * not positive), amax[i] = 0. */
typedef struct {
  float* scale;
  float* amax;
  float* history;
  int32_t history_len;
  int32_t margin;
} tpmlp_fp8_state;

/* dst = E4M3(src * (*scale)); src [rows x cols] bf16 row-major, dst
 * [rows x cols] bytes, or [cols x rows] with transpose != 0 (the K-major
 * layout the FP8 GEMMs read for a weight stored [K x N]).  *amax is
 * max-combined with max |src|.  rows, cols multiples of 16. */
TPMLP_API tpmlp_status tpmlp_cast_e4m3(const void* src, int64_t rows, int64_t cols, int transpose, const float* scale,
                                       void* dst, float* amax, tpmlp_stream_t stream);

/* tpmlp_layernorm_gather writing E4M3(LN(x) * (*scale)) bytes into Xq
 * [T x d]; *amax max-combined with max |LN(x)|.  d in {256, 512, 1024, 2048,
 * 4096, 8192}. */
TPMLP_API tpmlp_status tpmlp_layernorm_gather_e4m3(const void* const* X_chunks, const void* gamma, const void* beta,
                                                   float eps, const tpmlp_shape* shape, const float* scale, void* Xq,
                                                   float* amax, tpmlp_stream_t stream);

/* Column-parallel GEMM on E4M3 operands: P = (Xq AqT^T) / (sx sa) + bias,
 * Hq = E4M3(GeLU(P) * (*scale_h)), *amax_h max-combined with max |GeLU(P)|;
 * Hpre (NULL or [T x F] bf16) = P.  Xq [T x d], AqT [F x d] (A transposed,
 * from tpmlp_cast_e4m3), Hq [T x F] bytes. */
TPMLP_API tpmlp_status tpmlp_gemm1_e4m3(const void* Xq, const void* AqT, const void* bias, const tpmlp_shape* shape,
                                        const float* scale_x, const float* scale_a, const float* scale_h, void* Hq,
                                        float* amax_h, void* Hpre, tpmlp_stream_t stream);

/* Row-parallel GEMM on E4M3 operands with the in-kernel shard reduction:
 * Y = sum_i (Hq_i BqT_i^T) / (sh sb) in bf16, into Y [T x d] or, with
 * Y_chunks, into the N sequence chunks as tpmlp_gemm2_shard_accum.
 * BqT [d x F] (B transposed). */
TPMLP_API tpmlp_status tpmlp_gemm2_e4m3(const void* Hq, const void* BqT, const tpmlp_shape* shape,
                                        const float* scale_h, const float* scale_b, void* Y, void* const* Y_chunks,
                                        tpmlp_stream_t stream);

/* End of an FP8 step: the delayed-scaling update of `state` (see
 * tpmlp_fp8_state) for its four tensors. */
TPMLP_API tpmlp_status tpmlp_fp8_update_scales(const tpmlp_fp8_state* state, tpmlp_stream_t stream);

/* The sequence-parallel block forward with E4M3 GEMMs: the weights are cast
 * (transposed) with scale[1], scale[2]; the LayerNorm writes E4M3 with
 * scale[0]; GEMM1 dequantises, adds the bias, applies GeLU and casts H with
 * scale[3]; GEMM2 reduces the shards in TMEM and stores bf16 Y chunks.  The
 * scales are not updated here: call tpmlp_fp8_update_scales(state) when the
 * step is over (after tpmlp_sp_backward_fp8, which reads the same scales).
 * Hpre_out ([T x F] bf16), Xq_out ([T x d] E4M3), Hq_out ([T x F] E4M3):
 * NULL, or buffers that keep what the FP8 backward needs (otherwise they live
 * in the workspace).  Workspace: size of TPMLP_OP_SP_FWD_FP8.  bf16 X, gamma,
 * beta, A, B, bias and Y as in tpmlp_sp_forward. */
TPMLP_API tpmlp_status tpmlp_sp_forward_fp8(const void* const* X_chunks, const void* gamma, const void* beta,
                                            float eps, const void* A, const void* B, const void* bias,
                                            const tpmlp_fp8_state* state, const tpmlp_shape* shape,
                                            void* const* Y_chunks, void* Hpre_out, void* Xq_out, void* Hq_out,
                                            void* workspace, size_t workspace_bytes, tpmlp_stream_t stream);

/* ------------------------------------------------------------------ FP8 backward (E5M2 gradients)
 * The page's hybrid: the gradients that enter GEMMs (dY and dHpre) in E5M2
 * (bias 15, 2 mantissa bits, largest finite 57344, same rounding and
 * saturation as the E4M3 casts), the forward's E4M3 operands reused.  Every
 * FP8 GEMM reads both operands K-major; the operands the weight-gradient
 * GEMMs need transposed are byte-transposed copies. */

/* dst = E5M2(src * (*scale)), layouts and amax as tpmlp_cast_e4m3. */
TPMLP_API tpmlp_status tpmlp_cast_e5m2(const void* src, int64_t rows, int64_t cols, int transpose, const float* scale,
                                       void* dst, float* amax, tpmlp_stream_t stream);

/* dst [cols x rows] = the transpose of src [rows x cols], both one byte per
 * element (E4M3 or E5M2 codes); rows, cols multiples of 16. */
TPMLP_API tpmlp_status tpmlp_transpose_bytes(const void* src, int64_t rows, int64_t cols, void* dst,
                                             tpmlp_stream_t stream);

/* The GeLU' GEMM on FP8 operands: g = (dYq Bq^T) / (sdy sb) * GeLU'(Hpre),
 * dHq = E5M2(g * (*scale_g)), *amax_g max-combined with max |g|, dbias
 * (NULL or [F] bf16) = column sums of g (workspace: size of
 * TPMLP_OP_DH_GELUPRIME).  dYq [T x d] E5M2, Bq [F x d] E4M3 (B as stored,
 * from tpmlp_cast_e4m3 without transpose), Hpre [T x F] bf16, dHq [T x F]. */
TPMLP_API tpmlp_status tpmlp_gemm_dh_geluprime_e5m2(const void* dYq, const void* Bq, const void* Hpre,
                                                    const tpmlp_shape* shape, const float* scale_dy,
                                                    const float* scale_b, const float* scale_g, void* dHq,
                                                    float* amax_g, void* dbias, void* workspace,
                                                    size_t workspace_bytes, tpmlp_stream_t stream);

/* C = (A8 B8^T) / ((*scale_a) (*scale_b)) in bf16, one fp32 accumulator over
 * K.  A8 [M x K] and B8 [N x K] row-major bytes in format a_fmt / b_fmt
 * (0 = E4M3, 1 = E5M2); C [M x N] with ldc elements between rows.  K % 16 ==
 * 0, N % 8 == 0, ldc % 8 == 0, ldc >= N.  The weight-gradient and input-
 * gradient GEMMs of the FP8 backward are this call. */
TPMLP_API tpmlp_status tpmlp_gemm_fp8(const void* A8, int a_fmt, const void* B8, int b_fmt, int64_t M, int64_t N,
                                      int64_t K, const float* scale_a, const float* scale_b, void* C, int64_t ldc,
                                      tpmlp_stream_t stream);

/* Backward of tpmlp_sp_forward_fp8: dY gathered and cast to E5M2 (both
 * layouts) with grad->scale[0]; the weights cast to E4M3 as stored with the
 * forward's scale[1], scale[2]; the GeLU' GEMM (dHq in E5M2 with
 * grad->scale[1], dbias); dB = (Hq^T dYq), dA = (Xq^T dHq), dXg = (dHq A^T)
 * on FP8 operands; the LayerNorm backward (bf16) to dX chunks, dgamma,
 * dbeta; then the delayed-scale update of `grad` (two tensors, dY and dHpre,
 * E5M2's largest value 57344 in place of 448).  `fwd` is the forward's state
 * (its scales unchanged since the forward); Hpre, Xq, Hq the forward's saved
 * outputs.  dHq_out: NULL, or [T x F] bytes that receive the E5M2 codes of
 * dHpre the weight- and input-gradient GEMMs read (otherwise they live in
 * the workspace).  T, d, F multiples of 16.  Workspace: size of
 * TPMLP_OP_SP_BWD_FP8. */
TPMLP_API tpmlp_status tpmlp_sp_backward_fp8(const void* const* X_chunks, const void* gamma, float eps, const void* A,
                                             const void* B, const void* Hpre, const void* Xq, const void* Hq,
                                             const void* const* dY_chunks, const tpmlp_fp8_state* fwd,
                                             const tpmlp_fp8_state* grad, const tpmlp_shape* shape,
                                             void* const* dX_chunks, void* dA, void* dB, void* dbias, void* dgamma,
                                             void* dbeta, void* dHq_out, void* workspace, size_t workspace_bytes,
                                             tpmlp_stream_t stream);

/* ------------------------------------------------------------------ single steps (bf16)
 * Each step is one kernel launch (plus a small fixed-order reduction where
 * noted); the block calls above are sequences of these.  They take explicit
 * buffers instead of a workspace. */

/* Column-parallel GEMM of all N shards with bias + exact GeLU fused:
 * H = GeLU(X A + b), optionally Hpre = X A + b.  X [T x d], A [d x F],
 * bias [F] or NULL, H [T x F], Hpre [T x F] or NULL. */
TPMLP_API tpmlp_status tpmlp_gemm1_bias_gelu(const void* X, const void* A, const void* bias, const tpmlp_shape* shape,
                                   void* H, void* Hpre, tpmlp_stream_t stream);

/* Row-parallel GEMM with the in-kernel shard reduction: Y = sum_i H_i B_i.
 * H [T x F], B [F x d].  Y_chunks == NULL: Y [T x d].  Y_chunks != NULL
 * (host array of N pointers, T % N == 0): row r is stored to chunk r / (T/N),
 * the Reduce-Scatter fused into the store; Y is then ignored. */
TPMLP_API tpmlp_status tpmlp_gemm2_shard_accum(const void* H, const void* B, const tpmlp_shape* shape, void* Y,
                                     void* const* Y_chunks, tpmlp_stream_t stream);

/* tpmlp_gemm2_shard_accum into chunks with the rest of the sequence-parallel
 * region in its store: Y_j = R_j + dropout(sum_i H_i B_i + bias2) for the
 * rows of chunk j.  bias2 [d] or NULL; dropout as tpmlp_dropout (NULL: p = 0);
 * R_chunks: host array of N residual chunk pointers [T/N x d], or NULL. */
TPMLP_API tpmlp_status tpmlp_gemm2_bias_dropout_add(const void* H, const void* B, const void* bias2,
                                                    const tpmlp_dropout* dropout, const void* const* R_chunks,
                                                    const tpmlp_shape* shape, void* const* Y_chunks,
                                                    tpmlp_stream_t stream);

/* Per-shard partial outputs of the row-parallel layer, P_i = H_i B_i, as the
 * pages' ranks produce them before their collective.  P [N x T x d] bf16;
 * requires (ffn / N) % 64 == 0. */
TPMLP_API tpmlp_status tpmlp_gemm2_partials(const void* H, const void* B, const tpmlp_shape* shape, void* P,
                                  tpmlp_stream_t stream);

/* Reduce-Scatter of explicit partials: Y_chunk_j = bf16(sum_{i<N} P_i[rows of
 * chunk j]) summed in fp32 in shard order.  P [N x T x d]; Y_chunks host array
 * of N pointers [T/N x d]; T % N == 0. */
TPMLP_API tpmlp_status tpmlp_reduce_scatter(const void* P, const tpmlp_shape* shape, void* const* Y_chunks,
                                  tpmlp_stream_t stream);

/* tpmlp_reduce_scatter with the rest of the sequence-parallel region:
 * Y_j = R_j + dropout(sum_i P_i[rows of chunk j] + bias2), in fp32, one
 * rounding.  bias2, dropout and R_chunks as in tpmlp_gemm2_bias_dropout_add. */
TPMLP_API tpmlp_status tpmlp_reduce_scatter_bias_dropout_add(const void* P, const void* bias2,
                                                             const tpmlp_dropout* dropout,
                                                             const void* const* R_chunks, const tpmlp_shape* shape,
                                                             void* const* Y_chunks, tpmlp_stream_t stream);

/* Dropout backward of the sequence-parallel region, gathering the chunks:
 * dZ[j T/N + r] = dY_chunks[j][r] * keep / (1 - p) ([T x d] bf16); with
 * dbias2 != NULL also dbias2 [d] bf16 = the fixed-order column sums of dZ
 * (before its rounding; workspace: size of TPMLP_OP_DROPOUT_BWD).  dropout
 * as tpmlp_dropout (NULL: p = 0, a plain gather). */
TPMLP_API tpmlp_status tpmlp_dropout_backward(const void* const* dY_chunks, const tpmlp_dropout* dropout,
                                              const tpmlp_shape* shape, void* dZ, void* dbias2, void* workspace,
                                              size_t workspace_bytes, tpmlp_stream_t stream);

/* LayerNorm of every chunk into its row slot of the gathered activation:
 * Xg[j T/N + r] = LN(X_chunks[j][r]).  Xg [T x d]; T % N == 0. */
TPMLP_API tpmlp_status tpmlp_layernorm_gather(const void* const* X_chunks, const void* gamma, const void* beta, float eps,
                                    const tpmlp_shape* shape, void* Xg, tpmlp_stream_t stream);

/* The RMS norm the deep-dive page's SequenceParallelLayerNorm listing
 * computes ("분산 제어 소스코드 구조 패턴"), written into the gathered buffer like
 * tpmlp_layernorm_gather: per row rstd = rsqrt(mean(x^2) + eps) in fp32,
 * n = bf16(x rstd) (the listing's cast back to the input dtype), then
 * Xg = bf16(n * weight).  No mean subtraction, no shift.  weight [d] bf16,
 * Xg [T x d]; T % N == 0. */
TPMLP_API tpmlp_status tpmlp_rmsnorm_gather(const void* const* X_chunks, const void* weight, float eps,
                                            const tpmlp_shape* shape, void* Xg, tpmlp_stream_t stream);

/* dHpre = (dY B^T) * GeLU'(Hpre) in one GEMM epilogue; with H != NULL also
 * H = GeLU(Hpre); with dbias != NULL also dbias = column sums of dHpre
 * (workspace: size of TPMLP_OP_DH_GELUPRIME).  dY [T x d], B [F x d],
 * Hpre/dHpre/H [T x F]. */
TPMLP_API tpmlp_status tpmlp_gemm_dh_geluprime(const void* dY, const void* B, const void* Hpre, const tpmlp_shape* shape,
                                     void* dHpre, void* H, void* dbias, void* workspace, size_t workspace_bytes,
                                     tpmlp_stream_t stream);

/* Weight gradient of the row-parallel layer: dB = H^T dY.  H [T x F], dY [T x d], dB [F x d]. */
TPMLP_API tpmlp_status tpmlp_gemm_wgrad_b(const void* H, const void* dY, const tpmlp_shape* shape, void* dB,
                                tpmlp_stream_t stream);

/* Weight gradient of the column-parallel layer: dA = X^T dHpre.  X [T x d], dHpre [T x F], dA [d x F]. */
TPMLP_API tpmlp_status tpmlp_gemm_wgrad_a(const void* X, const void* dHpre, const tpmlp_shape* shape, void* dA,
                                tpmlp_stream_t stream);

/* Input gradient with the backward shard reduction: dX = sum_i dHpre_i A_i^T.
 * dHpre [T x F], A [d x F], dX [T x d]. */
TPMLP_API tpmlp_status tpmlp_gemm_dx_shard_accum(const void* dHpre, const void* A, const tpmlp_shape* shape, void* dX,
                                       tpmlp_stream_t stream);

/* LayerNorm backward per chunk: with xhat = (x - mean) rstd and g = dXg gamma,
 * dx = rstd (g - mean(g) - xhat mean(g xhat)); dgamma = sum dXg xhat and
 * dbeta = sum dXg over all T rows (fp32 [d]).  X_chunks / dX_chunks host
 * arrays of N pointers [T/N x d]; dXg [T x d] is the gradient of the gathered
 * LayerNorm output.  Workspace: size of TPMLP_OP_LN_BWD. */
TPMLP_API tpmlp_status tpmlp_layernorm_backward(const void* const* X_chunks, const void* gamma, float eps, const void* dXg,
                                      const tpmlp_shape* shape, void* const* dX_chunks, void* dgamma, void* dbeta,
                                      void* workspace, size_t workspace_bytes, tpmlp_stream_t stream);

/* tpmlp_layernorm_backward with its dgamma/dbeta block partials limited to
 * at most max_blocks CTAs (max_blocks >= 1), so that a small workspace of
 * max_blocks * 2 * d floats serves (workspace_bytes below that, or
 * max_blocks < 1, returns TPMLP_ERR_WORKSPACE / TPMLP_ERR_INVALID_ARG).
 * The results equal tpmlp_layernorm_backward's up to the order of the
 * dgamma/dbeta sums; fewer CTAs take longer. */
TPMLP_API tpmlp_status tpmlp_layernorm_backward_blocks(const void* const* X_chunks, const void* gamma, float eps,
                                                       const void* dXg, const tpmlp_shape* shape,
                                                       void* const* dX_chunks, void* dgamma, void* dbeta,
                                                       int32_t max_blocks, void* workspace, size_t workspace_bytes,
                                                       tpmlp_stream_t stream);

/* tpmlp_layernorm_backward with the residual's gradient added to the input
 * gradient: dX_chunks[j] = LN backward(dXg rows of chunk j) + R_chunks[j]
 * (R_chunks: host array of N pointers [T/N x d]).  Workspace: size of
 * TPMLP_OP_LN_BWD. */
TPMLP_API tpmlp_status tpmlp_layernorm_backward_add(const void* const* X_chunks, const void* gamma, float eps,
                                                    const void* dXg, const void* const* R_chunks,
                                                    const tpmlp_shape* shape, void* const* dX_chunks, void* dgamma,
                                                    void* dbeta, void* workspace, size_t workspace_bytes,
                                                    tpmlp_stream_t stream);

/* LayerNorm backward exactly as tpmlp_layernorm_backward, for callers that
 * cannot allocate device memory: it takes no workspace.  (This entry point
 * has no counterpart on the pages; it is an interface convenience.)  The
 * per-block dgamma/dbeta partial sums live in a fixed 9.5 MiB array inside
 * the library's device image, which every GPU that loads the library keeps
 * until the process exits.  d > 8192 returns TPMLP_ERR_UNSUPPORTED before
 * anything is launched.  All calls on a device share that array: calls whose
 * kernels overlap on the GPU (e.g. on unordered streams) race on it and give
 * wrong dgamma/dbeta.  The first call on a device looks the array up with
 * that device current; make it before any stream capture.  After a device
 * reset (cudaDeviceReset, or another runtime in the process resetting the
 * primary context) the device has a new context and the next call looks
 * the array up again: that call, too, must come before any capture. */
TPMLP_API tpmlp_status tpmlp_layernorm_backward_noalloc(const void* const* X_chunks, const void* gamma, float eps,
                                                        const void* dXg, const tpmlp_shape* shape,
                                                        void* const* dX_chunks, void* dgamma, void* dbeta,
                                                        tpmlp_stream_t stream);

/* ------------------------------------------------------------------ tensor-parallel attention
 * "6D" guide §3.2 (attention TP splits by heads: 32 heads at TP = 8 give each
 * GPU 4 heads), the glossary page's tensor-parallel section and the deep-dive
 * page's multi-head attention paragraph: the Q, K, V projections are split by
 * columns along heads, every shard computes complete attention for its heads,
 * the output projection is split by rows and the shards' partial outputs are
 * summed.  Here all N shards run on one GPU: one GEMM projects every head, the
 * attention core handles every (batch, head), and the output projection's K
 * loop walks the shards' head rows into one TMEM accumulator.
 * Layout: tokens sequence-major, row s B + b (the listing's [S, batch, hidden]);
 * QKV [T x 3d] with columns Q | K | V, head h at columns h hd .. (h+1) hd of
 * each part; O [T x d] heads side by side; d = H hd.  Head dimension 128. */

/* Bytes of workspace tpmlp_attention_tp_forward needs (QKV and O buffers).
 * head_dim other than 128 returns TPMLP_ERR_UNSUPPORTED. */
TPMLP_API tpmlp_status tpmlp_attention_workspace_size(int64_t S, int64_t B, int64_t H, int64_t head_dim,
                                                      size_t* bytes);

/* Attention core: for every batch element b and head h,
 * O[:, h] = softmax(Q_h K_h^T / sqrt(hd)) V_h over that batch element's S
 * positions, causal (position s sees keys <= s) when causal == 1.  fp32
 * scores and accumulation, bf16 in and out.  QKV [S B x 3 H hd], O [S B x H hd].
 * LSE: NULL, or fp32 [B H x S_pad] with S_pad = 128 ceil(S / 128) (16-byte
 * aligned): row (b H + h) entry s = log2 of sum_k exp2(q_s . k_k log2(e) /
 * sqrt(hd)) over the keys s sees, the statistics the backward re-uses;
 * entries S .. S_pad - 1 are left unwritten. */
TPMLP_API tpmlp_status tpmlp_attention_core(const void* QKV, int64_t S, int64_t B, int64_t H, int64_t head_dim,
                                            int causal, void* O, float* LSE, tpmlp_stream_t stream);

/* Bytes of workspace for tpmlp_attention_core_backward (the first part:
 * B H S_pad floats) and tpmlp_attention_tp_backward (all of it: also dO,
 * dQKV and column-sum partials). */
TPMLP_API tpmlp_status tpmlp_attention_backward_workspace_size(int64_t S, int64_t B, int64_t H, int64_t head_dim,
                                                               size_t* bytes);

/* Attention core backward (the chain rule through softmax, per batch element
 * and head): with P = softmax(Q K^T / sqrt(hd)) re-formed from LSE,
 * D = rowsum(dO . O), dV = P^T dO, dS = P . (dO V^T - D),
 * dQ = dS K / sqrt(hd), dK = dS^T Q / sqrt(hd).  QKV, O, LSE: the forward's
 * (LSE as tpmlp_attention_core writes it); dO [S B x H hd]; dQKV [S B x 3 H hd]
 * receives dQ | dK | dV in QKV's layout.  fp32 accumulation; deterministic
 * (no atomics).  Workspace 256-byte aligned. */
TPMLP_API tpmlp_status tpmlp_attention_core_backward(const void* QKV, const void* O, const void* dO,
                                                     const float* LSE, int64_t S, int64_t B, int64_t H,
                                                     int64_t head_dim, int causal, void* dQKV, void* workspace,
                                                     size_t workspace_bytes, tpmlp_stream_t stream);

/* The attention block: QKV = X Wqkv + bqkv (bqkv [3d] or NULL), O = attention
 * core, Y = O Wo + bo (Wo [d x d] row-split by heads, bo [d] or NULL, added
 * after the shard sum).  X, Y [S B x d]; Wqkv [d x 3d]; H % n_shards == 0.
 * QKV_out, O_out, LSE_out: NULL or buffers that keep the intermediates (what
 * tpmlp_attention_tp_backward needs).  Workspace: tpmlp_attention_workspace_size. */
TPMLP_API tpmlp_status tpmlp_attention_tp_forward(const void* X, const void* Wqkv, const void* bqkv, const void* Wo,
                                                  const void* bo, int64_t S, int64_t B, int64_t H, int32_t n_shards,
                                                  int causal, void* Y, void* QKV_out, void* O_out, float* LSE_out,
                                                  void* workspace, size_t workspace_bytes, tpmlp_stream_t stream);

/* Backward of the attention block (the same glossary and deep-dive sections:
 * the conjugate of the forward's column/row split).  Row-parallel output
 * projection: dO = dY Wo^T (every shard's rows of Wo), dWo = O^T dY,
 * dbo = column sums of dY; the core backward into dQKV; column-parallel
 * projection: dWqkv = X^T dQKV, dbqkv = column sums of dQKV, and
 * dX = dQKV Wqkv^T, whose K loop over the 3d columns adds every shard's
 * contribution (the backward all-reduce).  QKV, O, LSE: saved by
 * tpmlp_attention_tp_forward.  dbqkv, dbo: NULL to skip.  dQKV_out: NULL, or a
 * [S B x 3d] buffer that receives dQKV.  bf16 outputs, fp32 accumulation.
 * Workspace: tpmlp_attention_backward_workspace_size, 256-byte aligned. */
TPMLP_API tpmlp_status tpmlp_attention_tp_backward(const void* X, const void* Wqkv, const void* Wo, const void* QKV,
                                                   const void* O, const float* LSE, const void* dY, int64_t S,
                                                   int64_t B, int64_t H, int32_t n_shards, int causal, void* dX,
                                                   void* dWqkv, void* dbqkv, void* dWo, void* dbo, void* dQKV_out,
                                                   void* workspace, size_t workspace_bytes, tpmlp_stream_t stream);

/* Failure-detection self test: launches one CTA that waits on a barrier no
 * thread ever arrives at, with a limit of `budget_us` microseconds (1 to
 * 1000000).  The wait runs out, the kernel records the timeout and exits;
 * tpmlp_get_device_status then returns TPMLP_ERR_TIMEOUT.  Nothing traps. */
TPMLP_API tpmlp_status tpmlp_selftest_wait_timeout(uint32_t budget_us, tpmlp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TPMLP_H */
