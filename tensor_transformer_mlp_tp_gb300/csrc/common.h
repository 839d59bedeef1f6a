// Constants and kernel-parameter structs shared by the host launchers and
// the kernels of libtpmlp.  No torch types, no allocation.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace tpmlp {

constexpr int kMaxShards = 64;  // N, the number of column/row shards (and of SP chunks)

// Device error words: [0] = OR of error bits, [1] = first failing wait site.
constexpr int kErrWords = 4;
constexpr uint32_t kErrTimeout = 1u;
// A kernel refused a launch configuration it cannot run safely (and touched no memory).
constexpr uint32_t kErrConfig = 2u;

// Wait sites reported in error word [1] (one id per wait in the GEMM kernel).
enum WaitSite : uint32_t {
  kSiteProducerEmpty = 1,
  kSiteMmaFull = 2,
  kSiteMmaTmemEmpty = 3,
  kSiteEpiTmemFull = 4,
  kSiteEpiStageDrained = 5,
  kSiteEpiStageFilled = 6,
};

// GEMM tile: BM x BN output, BK-deep k-blocks (64 bf16 = one 128-byte swizzle row).
constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kUmmaK = 16;

// Epilogues of the tcgen05 GEMM.
enum Epilogue : int {
  kEpiBiasGelu = 0,   // out0 = bf16(GeLU(acc + bias)); out1 (optional) = bf16(acc + bias)
  kEpiBias = 1,       // out0 = bf16(acc + bias)
  kEpiStore = 2,      // out0 = bf16(acc), optional row -> chunk remap, optional per-shard partials
  kEpiDGelu = 3,      // out0 = bf16(acc * GeLU'(aux)); out1 = bf16(GeLU(aux)); optional column sums
  kEpiBiasGeluQ = 4,  // out0 = E4M3(GeLU(acc + bias) * scale_out), amax_out = max |GeLU(acc + bias)|;
                      // out1 (optional) = bf16(acc + bias)
  kEpiDGeluQ = 5,     // g = acc * GeLU'(aux): out0 = E5M2(g * scale_out), amax_out = max |g|, optional
                      // column sums of g
};

struct ChunkPtrs {
  void* p[kMaxShards];
};

struct ConstChunkPtrs {
  const void* p[kMaxShards];
};

// Parameters of one tcgen05 GEMM launch: C[M x N] = sum_k A[m, k] * B[k, n].
// A and B are read through TMA tensor maps.  A "K-major" operand has k as
// its contiguous dimension; an "MN-major" one has m (or n) contiguous.
struct GemmParams {
  CUtensorMap tmA;
  CUtensorMap tmB;
  CUtensorMap tmC0;         // out0 / out1 as [M x N] bf16, 32 x 32 boxes, 64-byte swizzle (tma_out bits 0 / 1)
  CUtensorMap tmC1;
  CUtensorMap tmB_half;     // K-major B with boxes of a quarter tile's columns (half tiles of the pair kernel)
  int tma_out;              // bit 0: out0 rows leave through TMA box stores, bit 1: out1 too
  int M, N, K;
  int m_blocks, n_blocks;
  int k_blocks_per_shard;   // k-blocks summed into one accumulator
  int shards;               // >1: per-shard partial outputs (tile space x shards, K split evenly)
  int group_m;              // raster: tiles walk group_m row blocks before the next column block
  // CTA-pair kernel: tiles from full_units on are each split into two half-width tiles (the two halves of
  // its columns), so that a last wave of fewer than half the pairs' tiles runs as one round of halves.
  // Work unit u < full_units is tile u; unit full_units + 2 j + h is half h of tile full_units + j.
  int full_units;
  void* out0;
  long long ld0;
  void* out1;
  long long ld1;
  long long shard_stride0;  // elements between consecutive shards' partial outputs
  const void* bias;         // [N] bf16 or nullptr
  const void* aux;          // [M x N] bf16 (pre-activation) for kEpiDGelu
  long long ld_aux;
  float* colsum;            // [4 * m_blocks x N] fp32 column partial sums, or nullptr
  int rows_per_chunk;       // >0: row r of C goes to chunk r / rows_per_chunk
  ChunkPtrs chunks;
  // Sequence-parallel tail of the chunked store (kEpiStore with rows_per_chunk > 0 and tail != 0):
  // out = res + keep * (acc + bias) * drop_scale, bias = the row layer's [N] bias or nullptr,
  // res = the residual rows in chunk layout (res_chunks.p[0] == nullptr: none), keep from philox.cuh.
  int tail;
  float drop_scale;
  unsigned long long drop_seed, drop_offset, drop_thr;  // drop_thr = 2^32 keeps every element
  uint8_t* drop_mask;  // nullptr, or the keep bits (one byte per 8 elements) written as they are drawn
  ConstChunkPtrs res_chunks;
  // FP8 operands: the accumulator is divided by (*scale_a) (*scale_b); kEpiBiasGeluQ quantises with
  // *scale_out and max-combines its amax into *amax_out.
  const float* scale_a;
  const float* scale_b;
  const float* scale_out;
  float* amax_out;
  int a_fmt, b_fmt;           // 8-bit operand formats (0 = E4M3, 1 = E5M2)
  unsigned int* err;
  unsigned long long timeout_ns;
};

// Row-wise kernels (LayerNorm forward/backward, reduce-scatter).
struct RowParams {
  ConstChunkPtrs in_chunks;   // N chunk pointers, each [rows_per_chunk x d] bf16
  ChunkPtrs out_chunks;
  int rows;                   // total rows T
  int d;
  int n_chunks;
  int rows_per_chunk;
  float eps;
  const void* gamma;          // [d] bf16
  const void* beta;           // [d] bf16
  const void* src;            // contiguous [rows x d] bf16 input (gathered tensor / partials)
  void* dst;                  // contiguous [rows x d] bf16 output
  float* partial;             // column partial sums [blocks x 2d] fp32 (LayerNorm backward)
  long long shard_stride;     // elements between partials (reduce-scatter)
  float* stats;               // [rows x 2] fp32 mean, rstd (LayerNorm backward)
  int rows_per_block;         // rows summed by one column-partial block (LayerNorm backward)
  int slots;                  // shared-memory row slots of the streaming kernels
  // Sequence-parallel tail (reduce-scatter: out = add + keep * (sum + bias2) * drop_scale;
  // dropout backward: dst = keep * in * drop_scale; LayerNorm backward: dx += add)
  int tail;                   // nonzero: apply the tail below
  const void* bias2;          // [d] bf16 or nullptr
  ConstChunkPtrs add_chunks;  // N chunk pointers [rows_per_chunk x d] bf16, or p[0] == nullptr
  float drop_scale;
  unsigned long long drop_seed, drop_offset, drop_thr;
  uint8_t* drop_mask;  // reduce-scatter tail: keep bits written; dropout backward: keep bits read
  const float* qscale;        // E4M3 outputs: quantisation scale (device), and the amax they max-combine into
  float* amax;
  unsigned int* err;          // device error words
  unsigned long long timeout_ns;
};

// Wait sites of the row-streaming kernels.
constexpr uint32_t kSiteRowProducer = 16;
constexpr uint32_t kSiteRowConsumer = 17;
constexpr uint32_t kSiteRowConfig = 18;

}  // namespace tpmlp
