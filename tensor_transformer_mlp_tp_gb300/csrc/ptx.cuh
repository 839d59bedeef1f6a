// Inline-PTX building blocks for sm_103a kernels: mbarriers, TMA tensor
// copies, tcgen05 (TMEM allocation, UMMA issue/commit, TMEM loads) and the
// bounded waits every kernel of this library uses.
//
// Encodings follow the public PTX ISA for tcgen05 ("Shared memory
// descriptor", "Instruction descriptor" for .kind::f16) and for
// cp.async.bulk.tensor.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "common.h"

namespace tpmlp {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lane_id() {
  uint32_t l;
  asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
  return l;
}

// ----------------------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// try_wait with a suspend-time hint: the thread sleeps until the phase
// completes or about kSuspendHintNs elapse, instead of spinning on the barrier.
constexpr uint32_t kSuspendHintNs = 200000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// State shared by the bounded waits of one CTA: a CTA-wide abort flag in
// shared memory, the library's device error words and the time budget.
struct WaitCtx {
  volatile int* abort;   // shared memory; set once any wait of the CTA gives up
  unsigned int* err;     // device error words (kErrWords entries)
  uint64_t budget_ns;    // per-wait limit
};

__device__ __forceinline__ void record_error(const WaitCtx& w, uint32_t bit, uint32_t site) {
  *w.abort = 1;
  atomicOr(w.err + 0, bit);
  atomicCAS(w.err + 1, 0u, site);
}

// Wait until the phase with parity `parity` of `bar` has completed, for at
// most the budget.  Returns false (and raises the CTA abort flag and the
// device error word) on timeout, or if another thread of the CTA already
// aborted.  Never traps, never spins without limit.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, const WaitCtx& w, uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*w.abort) return false;
    if (global_timer_ns() - t0 > w.budget_ns) {
      record_error(w, kErrTimeout, site);
      return false;
    }
  }
}

// Teardown wait: same limit, but ignores the abort flag (used to drain
// copies or MMAs still in flight before shared memory or TMEM is released).
__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity, uint64_t budget_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > budget_ns) return false;
  }
  return true;
}

// ----------------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch: the next kernel of the stream (launched with programmatic stream
// serialisation) may begin launching; wait until the previous kernel has completed and its memory
// operations are visible (a no-op for a kernel launched without the attribute).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// 2-D tiled store shared -> global, tracked as a bulk group of the issuing thread.  c0 is the innermost
// coordinate (a multiple of 16 bytes), c1 >= 0; elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the thread's committed bulk stores have finished reading shared memory / have completed
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// 2-D tiled load global -> shared; completion is signalled as transaction
// bytes on `bar`.  c0 is the innermost coordinate (its byte offset must be a
// multiple of 16, which the host guarantees by requiring 8-element multiples).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            uint64_t cache_hint) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(cache_hint)
      : "memory");
}

// 1-D bulk copy global -> shared (both 16-byte aligned, `bytes` a multiple of 16), counted on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Bring `bytes` (a multiple of 16) at a 16-byte aligned global address into L2, asynchronously.
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}

// L2 cache-policy constants for the .L2::cache_hint operand (createpolicy
// fractions are not needed: one policy per operand class).
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ----------------------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, fp32 accumulator, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One 128 x N x 16 UMMA with A in tensor memory: A(m, k) at lane m, column a_tmem + k / 2 (two bf16 per
// 32-bit column, the lower k in the low half); B from shared memory through its descriptor.
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread t gets row (lane base + t),
// columns [col, col+32).  Load and wait are one asm statement so no use of
// the registers can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_load_32cols(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor (tcgen05 format), 128-byte swizzle.
//  bits  0-13  start address >> 4
//  bits 16-29  leading-dimension byte offset >> 4
//  bits 32-45  stride-dimension byte offset >> 4
//  bits 46-47  descriptor version (1 for tcgen05)
//  bits 49-51  base offset (0: every tile starts on a 1024-byte boundary)
//  bits 61-63  layout: 2 = 128-byte swizzle
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, .kind::f16 with bf16 A/B and fp32 D.
//  bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format (1 = bf16),
//  bit 15 A major (0 = K, 1 = MN), bit 16 B major, bits 17-22 N >> 3, bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor, .kind::f8f6f4 with fp32 D: A/B formats in bits 7-9 / 10-12
// (E4M3 = 0, E5M2 = 1), majors in bits 15/16, N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kFmtE4M3 = 0, kFmtE5M2 = 1;
__host__ __device__ constexpr uint32_t idesc_f8_f32(int M, int N, uint32_t a_fmt, uint32_t b_fmt, bool a_mn, bool b_mn) {
  return (1u << 4) | (a_fmt << 7) | (b_fmt << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ----------------------------------------------------------------------------- small math

// Exact GeLU x * Phi(x) and its derivative Phi(x) + x * phi(x), in fp32.
// Phi(x) = (1 + erf(x / sqrt 2)) / 2 with erf from Abramowitz & Stegun,
// Handbook of Mathematical Functions, eq. 7.1.26 (Hastings' rational
// approximation, |error in erf| <= 1.5e-7 for all real arguments):
//   erf(z) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-z^2),  t = 1 / (1 + p z),  z >= 0,
// and erf(-z) = -erf(z).  With z = |x| / sqrt 2, exp(-z^2) = exp(-x^2 / 2) is
// also what the normal density phi(x) needs, so GeLU' costs one exponential.
struct NormalCdfPdf {
  float cdf, pdf;
};

// Abramowitz & Stegun eq. 7.1.26: erf(z) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2),
// t = 1 / (1 + p z), |error| <= 1.5e-7.
constexpr float kP = 0.3275911f, kA1 = 0.254829592f, kA2 = -0.284496736f, kA3 = 1.421413741f,
                kA4 = -1.453152027f, kA5 = 1.061405429f;

__device__ __forceinline__ NormalCdfPdf normal_cdf_pdf(float x) {
  const float e = __expf(-0.5f * x * x);                               // exp(-z^2)
  const float t = __fdividef(1.0f, fmaf(kP * 0.70710678118654752f, fabsf(x), 1.0f));
  const float poly = t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, kA5, kA4), kA3), kA2), kA1);
  const float tail = 0.5f * poly * e;                                  // Phi(-|x|)
  return {x >= 0.f ? 1.0f - tail : tail, 0.39894228040143268f * e};
}

__device__ __forceinline__ float gelu_f(float x) { return x * normal_cdf_pdf(x).cdf; }

// 2^x and 1/x with the hardware's approximate instructions (subnormal results flush to zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The pair forms below follow the same eq. 7.1.26 with the 1/2 of Phi(-|x|) = (1 - erf(|x| / sqrt 2)) / 2
// folded into the coefficients: Phi(-|x|) = t (a1/2 + t (a2/2 + ...)) exp(-x^2 / 2), t = 1 / (1 + p |x| / sqrt 2),
// exp(-x^2 / 2) = 2^(-x^2 log2(e) / 2).  Polynomial and products on float pairs (the packed fp32
// instructions), the exponential and the reciprocal per element.
constexpr float kP2 = kP * 0.70710678118654752f;
constexpr float kNegHalfLog2e = -0.72134752044448170f;  // -log2(e) / 2
constexpr float kInvSqrt2Pi = 0.39894228040143268f;

// Phi(-|x|) and exp(-x^2 / 2) of two values; `nax` = -|x|.
__device__ __forceinline__ void normal_tail2(float2 x, float2 nax, float2& tail, float2& e) {
  const float2 den = __ffma2_rn(make_float2(-kP2, -kP2), nax, make_float2(1.f, 1.f));
  const float2 t = make_float2(rcp_approx(den.x), rcp_approx(den.y));
  const float2 m = __fmul2_rn(__fmul2_rn(make_float2(kNegHalfLog2e, kNegHalfLog2e), x), x);
  e = make_float2(ex2_approx(m.x), ex2_approx(m.y));
  float2 poly = __ffma2_rn(t, make_float2(0.5f * kA5, 0.5f * kA5), make_float2(0.5f * kA4, 0.5f * kA4));
  poly = __ffma2_rn(t, poly, make_float2(0.5f * kA3, 0.5f * kA3));
  poly = __ffma2_rn(t, poly, make_float2(0.5f * kA2, 0.5f * kA2));
  poly = __ffma2_rn(t, poly, make_float2(0.5f * kA1, 0.5f * kA1));
  tail = __fmul2_rn(__fmul2_rn(t, poly), e);
}

struct NormalCdfPdf2 {
  float2 cdf, pdf;
};
__device__ __forceinline__ NormalCdfPdf2 normal_cdf_pdf2(float2 x) {
  float2 tail, e;
  normal_tail2(x, make_float2(-fabsf(x.x), -fabsf(x.y)), tail, e);
  return {make_float2(x.x >= 0.f ? 1.0f - tail.x : tail.x, x.y >= 0.f ? 1.0f - tail.y : tail.y),
          __fmul2_rn(make_float2(kInvSqrt2Pi, kInvSqrt2Pi), e)};
}

// GeLU of two values: x Phi(x) = max(x, 0) - |x| Phi(-|x|) (for x < 0, Phi(x) = Phi(-|x|); for x >= 0,
// x Phi(x) = x - x Phi(-x)), one fused multiply-add after the tail instead of a select and a product.
__device__ __forceinline__ float2 gelu2(float2 x) {
  const float2 nax = make_float2(-fabsf(x.x), -fabsf(x.y));
  float2 tail, e;
  normal_tail2(x, nax, tail, e);
  return __ffma2_rn(nax, tail, make_float2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)));
}

__device__ __forceinline__ float gelu_prime_f(float x) {
  const NormalCdfPdf n = normal_cdf_pdf(x);
  return n.cdf + x * n.pdf;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(v);
}

}  // namespace tpmlp

// ----------------------------------------------------------------------------- CTA pairs (cta_group::2)

namespace tpmlp {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of the variable at shared::cta address `saddr` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Tiled load into this CTA's shared memory whose completion is counted on an
// mbarrier that may live in the peer CTA of the pair (`bar_cluster` is a
// shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster, int c0,
                                                 int c1, uint64_t cache_hint) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "l"(cache_hint)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 256 x N x 16 MMA over the CTA pair: rows 0-127 of A and columns 0..N/2-1 of
// B come from the even CTA's shared memory, the rest from the odd CTA's (same
// offsets); each CTA's TMEM receives its 128 rows of D.  Issued by the even CTA.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One 256 x N x 32 UMMA of the CTA pair, .kind::f8f6f4 (8-bit A and B, fp32 D in TMEM).
__device__ __forceinline__ void umma_f8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the barrier at the same offset in every CTA of `cta_mask`
// when all tcgen05 ops issued so far by this thread have completed.
__device__ __forceinline__ void umma_commit_pair_multicast(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

}  // namespace tpmlp
