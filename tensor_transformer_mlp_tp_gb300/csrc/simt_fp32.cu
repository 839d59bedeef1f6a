// fp32 path of the block: Y = GeLU(X A + b) B with fp32 inputs, fp32 FFMA
// accumulation on the CUDA cores and fp32 outputs.  Used when the caller
// asks for fp32 arithmetic (tensor-core TF32 would round the inputs to 10
// mantissa bits).  Two launches: the column-parallel GEMM with bias and
// GeLU into H, then the row-parallel GEMM whose K loop runs over all shards'
// rows of B in order (the shard sum is the K loop).
#include "launch.h"
#include "ptx.cuh"

namespace tpmlp {
namespace {

constexpr int kT = 64;   // output tile kT x kT
constexpr int kKB = 16;  // k-slab

// C[M x N] = A[M x K] B[K x N] (+ bias, GeLU), row-major, 256 threads, 4 x 4 outputs each.
template <bool BIAS_GELU>
__global__ void __launch_bounds__(256) k_sgemm(int M, int N, int K, const float* __restrict__ A,
                                               const float* __restrict__ B, const float* __restrict__ bias,
                                               float* __restrict__ C) {
  __shared__ float sA[kKB][kT + 1];
  __shared__ float sB[kKB][kT];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * kT, n0 = blockIdx.x * kT;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kKB) {
    for (int i = threadIdx.x; i < kT * kKB; i += 256) {
      const int r = i / kKB, c = i % kKB;  // A tile: rows m, cols k
      const int gm = m0 + r, gk = k0 + c;
      sA[c][r] = (gm < M && gk < K) ? A[static_cast<long long>(gm) * K + gk] : 0.f;
      const int br = i / kT, bc = i % kT;  // B tile: rows k, cols n
      const int bk = k0 + br, bn = n0 + bc;
      sB[br][bc] = (bk < K && bn < N) ? B[static_cast<long long>(bk) * N + bn] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kKB; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = sA[k][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = sB[k][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= N) continue;
      float v = acc[i][j];
      if constexpr (BIAS_GELU) {
        if (bias != nullptr) v += bias[gn];
        v = gelu_f(v);
      }
      C[static_cast<long long>(gm) * N + gn] = v;
    }
  }
}

}  // namespace

cudaError_t launch_mlp_fp32(const float* X, const float* A, const float* B, const float* bias, int T, int d, int F,
                            float* H, float* Y, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  dim3 g1((F + kT - 1) / kT, (T + kT - 1) / kT);
  k_sgemm<true><<<g1, 256, 0, s>>>(T, F, d, X, A, bias, H);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 g2((d + kT - 1) / kT, (T + kT - 1) / kT);
  k_sgemm<false><<<g2, 256, 0, s>>>(T, d, F, H, B, nullptr, Y);
  return cudaGetLastError();
}

}  // namespace tpmlp
