// C ABI of libtpmlp: argument validation, workspace carving and the launch
// sequences of the block calls.  Everything here is host code except the
// device error words and the wait-timeout self test.
#include <climits>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <utility>

#include "../../include/tpmlp.h"
#include "launch.h"
#include "ptx.cuh"

namespace tpmlp {

__device__ unsigned int g_err_words[kErrWords];

namespace {

// One CTA waits on a barrier nobody arrives at; the bounded wait gives up,
// records kErrTimeout and the kernel returns.
__global__ void k_wait_timeout_selftest(unsigned int* err, unsigned long long budget_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtx wc{&abort_flag, err, budget_ns};
    (void)wait_bounded(&bar, 0, wc, 99u);
  }
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct DevState {
  bool init = false;
  unsigned long long ctx_id = 0;  // the context the cached addresses belong to
  DeviceCtx ctx{};
};
std::mutex g_mu;
DevState g_dev[64];

unsigned long long timeout_ns_from_env() {
  const char* s = std::getenv("TPMLP_WAIT_TIMEOUT_MS");
  if (s != nullptr) {
    const long long ms = std::atoll(s);
    if (ms > 0) return static_cast<unsigned long long>(ms) * 1000000ull;
  }
  return 1000000000ull;
}

tpmlp_status device_ctx(DeviceCtx* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TPMLP_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DevState& st = g_dev[dev];
  // a reset device (cudaDeviceReset, or another runtime in the process resetting the primary context)
  // comes back as a new context with the module loaded afresh: look the addresses up again
  if (!st.init || current_context_id() != st.ctx_id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_err_words) != cudaSuccess) return TPMLP_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return TPMLP_ERR_CUDA;
    st.ctx.err = static_cast<unsigned int*>(p);
    st.ctx.sm_count = sms;
    st.ctx.timeout_ns = timeout_ns_from_env();
    st.ctx_id = current_context_id();  // the lookup above made the device's context current
    st.init = true;
  }
  *out = st.ctx;
  return TPMLP_OK;
}

}  // namespace

unsigned long long current_context_id() {
  using GetCurrent = int (*)(void**);
  using GetId = int (*)(void*, unsigned long long*);
  // the two driver calls through the runtime's entry-point query (the library links no driver library);
  // resolved once, both or neither
  static const std::pair<GetCurrent, GetId> fns = [] {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa{}, qb{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) != cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) != cudaSuccess ||
        qa != cudaDriverEntryPointSuccess || qb != cudaDriverEntryPointSuccess || a == nullptr || b == nullptr)
      return std::pair<GetCurrent, GetId>(nullptr, nullptr);
    return std::pair<GetCurrent, GetId>(reinterpret_cast<GetCurrent>(a), reinterpret_cast<GetId>(b));
  }();
  if (fns.first == nullptr) return 0;
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (fns.first(&ctx) != 0 || ctx == nullptr || fns.second(ctx, &id) != 0) return 0;
  return id;
}

cudaError_t current_device_ctx(DeviceCtx* out) {
  return device_ctx(out) == TPMLP_OK ? cudaSuccess : cudaErrorUnknown;
}

namespace {

tpmlp_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return TPMLP_OK;
  if (e == cudaErrorNotSupported) return TPMLP_ERR_UNSUPPORTED;
  return TPMLP_ERR_CUDA;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks common to every call.  `sp` adds T % N == 0.
tpmlp_status check_shape(const tpmlp_shape* s, bool sp, bool bf16_only) {
  if (s == nullptr) return TPMLP_ERR_INVALID_ARG;
  if (s->tokens < 0 || s->d < 1 || s->ffn < 1 || s->n_shards < 1 || s->n_shards > kMaxShards)
    return TPMLP_ERR_INVALID_ARG;
  if (s->dtype != TPMLP_BF16 && s->dtype != TPMLP_FP32) return TPMLP_ERR_INVALID_ARG;
  if (s->ffn % s->n_shards != 0) return TPMLP_ERR_INVALID_ARG;
  if (sp && s->tokens % s->n_shards != 0) return TPMLP_ERR_INVALID_ARG;
  if (s->tokens > INT_MAX / 2 || s->d > INT_MAX / 2 || s->ffn > INT_MAX / 2) return TPMLP_ERR_UNSUPPORTED;
  if (s->dtype == TPMLP_BF16) {
    if (s->d % 8 != 0 || (s->ffn / s->n_shards) % 8 != 0) return TPMLP_ERR_INVALID_ARG;
  } else if (bf16_only) {
    return TPMLP_ERR_UNSUPPORTED;
  }
  return TPMLP_OK;
}

bool ptrs_ok(std::initializer_list<const void*> required) {
  for (const void* p : required)
    if (p == nullptr || !al16(p)) return false;
  return true;
}

bool opt_ok(const void* p) { return p == nullptr || al16(p); }

bool chunks_ok(const void* const* c, int n) {
  if (c == nullptr) return false;
  for (int i = 0; i < n; ++i)
    if (c[i] == nullptr || !al16(c[i])) return false;
  return true;
}

// Sizes of the workspace regions (bytes, each 256-aligned).
struct Sizes {
  size_t td, tf, ptd, colsum, lnbwd, dropcol, td8, tf8, df8;
};


Sizes sizes_of(const tpmlp_shape* s) {
  const size_t T = static_cast<size_t>(s->tokens), d = static_cast<size_t>(s->d), F = static_cast<size_t>(s->ffn);
  const size_t el = s->dtype == TPMLP_FP32 ? 4 : 2;
  Sizes z;
  z.td = align_up(T * d * el);
  z.tf = align_up(T * F * el);
  z.ptd = align_up(static_cast<size_t>(s->n_shards) * T * d * 2);
  const size_t m_blocks = (T + kBM - 1) / kBM;
  z.colsum = align_up(4 * m_blocks * F * 4);
  z.lnbwd = align_up(layernorm_bwd_scratch_floats(static_cast<int>(T), static_cast<int>(d)) * 4);
  z.dropcol = align_up(dropout_bwd_scratch_floats(static_cast<int>(T), static_cast<int>(d)) * 4);
  z.td8 = align_up(T * d);
  z.tf8 = align_up(T * F);
  z.df8 = align_up(d * F);
  return z;
}

size_t ws_bytes(const tpmlp_shape* s, int op) {
  const Sizes z = sizes_of(s);
  switch (op) {
    case TPMLP_OP_FWD: return z.tf;
    case TPMLP_OP_SP_FWD: return z.td + z.tf;
    case TPMLP_OP_SP_FWD_PARTIALS: return z.td + z.tf + z.ptd;
    case TPMLP_OP_BWD: return 3 * z.tf + z.colsum;
    case TPMLP_OP_SP_BWD: return 3 * z.tf + z.colsum + 3 * z.td + z.lnbwd;
    case TPMLP_OP_DH_GELUPRIME: return z.colsum;
    case TPMLP_OP_LN_BWD: return z.lnbwd;
    case TPMLP_OP_SP_BLOCK_BWD: return 3 * z.tf + z.colsum + 3 * z.td + z.lnbwd + z.dropcol;
    case TPMLP_OP_DROPOUT_BWD: return z.dropcol;
    case TPMLP_OP_SP_FWD_FP8: return 2 * z.df8 + z.td8 + z.tf8;
    case TPMLP_OP_SP_BWD_FP8: return 2 * z.td + 3 * z.td8 + 2 * z.df8 + 3 * z.tf8 + z.colsum + z.lnbwd;
    default: return 0;
  }
}

// Bump allocator over the caller's workspace.
struct Carve {
  uint8_t* base;
  size_t used = 0;
  explicit Carve(void* p) : base(static_cast<uint8_t*>(p)) {}
  void* take(size_t bytes) {
    void* p = base + used;
    used += bytes;
    return p;
  }
};

ChunkPtrs to_chunks(void* const* c, int n) {
  ChunkPtrs r{};
  for (int i = 0; i < n; ++i) r.p[i] = c[i];
  return r;
}

ConstChunkPtrs to_const_chunks(const void* const* c, int n) {
  ConstChunkPtrs r{};
  for (int i = 0; i < n; ++i) r.p[i] = c[i];
  return r;
}

// The rest of the sequence-parallel region: row bias, dropout (p in [0, 1), float32) and residual chunks.
tpmlp_status make_tail(const void* bias2, const tpmlp_dropout* drop, const void* const* R_chunks, int n, SpTail* t) {
  if (!opt_ok(bias2)) return TPMLP_ERR_INVALID_ARG;
  const float p = drop != nullptr ? drop->p : 0.f;
  if (!(p >= 0.f && p < 1.f)) return TPMLP_ERR_INVALID_ARG;
  if (R_chunks != nullptr && !chunks_ok(R_chunks, n)) return TPMLP_ERR_INVALID_ARG;
  *t = SpTail{};
  t->on = true;
  t->bias2 = bias2;
  if (R_chunks != nullptr) t->residual = to_const_chunks(R_chunks, n);
  const double keep = 1.0 - static_cast<double>(p);
  t->thr = static_cast<unsigned long long>(std::floor(keep * 4294967296.0));
  t->scale = static_cast<float>(1.0 / keep);
  t->seed = drop != nullptr ? drop->seed : 0;
  t->offset = drop != nullptr ? drop->offset : 0;
  t->mask = drop != nullptr ? drop->keep_mask : nullptr;
  return TPMLP_OK;
}

void apply_tail(RowParams& r, const SpTail& t) {
  r.tail = 1;
  r.bias2 = t.bias2;
  r.add_chunks = t.residual;
  r.drop_scale = t.scale;
  r.drop_seed = t.seed;
  r.drop_offset = t.offset;
  r.drop_thr = t.thr;
  r.drop_mask = t.mask;
}

// ------------------------------------------------------------------ step implementations (validated inputs)

cudaError_t do_gemm1(const DeviceCtx& c, const void* X, const void* A, const void* bias, const tpmlp_shape* s,
                     void* H, void* Hpre, int epi, cudaStream_t st) {
  GemmLaunch g;
  g.M = static_cast<int>(s->tokens);
  g.N = static_cast<int>(s->ffn);
  g.K = static_cast<int>(s->d);
  g.a = {X, s->d, false};
  g.b = {A, s->ffn, true};
  g.epi = epi;
  g.out0 = H;
  g.ld0 = s->ffn;
  g.out1 = Hpre;
  g.ld1 = s->ffn;
  g.bias = bias;
  return launch_gemm(g, c, st);
}

cudaError_t do_gemm2(const DeviceCtx& c, const void* H, const void* B, const tpmlp_shape* s, void* Y,
                     void* const* Y_chunks, cudaStream_t st, const SpTail* tail = nullptr) {
  GemmLaunch g;
  g.M = static_cast<int>(s->tokens);
  g.N = static_cast<int>(s->d);
  g.K = static_cast<int>(s->ffn);
  g.a = {H, s->ffn, false};
  g.b = {B, s->d, true};
  g.epi = kEpiStore;
  g.out0 = Y;
  g.ld0 = s->d;
  if (Y_chunks != nullptr) {
    g.rows_per_chunk = static_cast<int>(s->tokens / s->n_shards);
    g.chunks = to_chunks(Y_chunks, s->n_shards);
    if (tail != nullptr) g.tail = *tail;
  }
  return launch_gemm(g, c, st);
}

cudaError_t do_gemm2_partials(const DeviceCtx& c, const void* H, const void* B, const tpmlp_shape* s, void* P,
                              cudaStream_t st) {
  GemmLaunch g;
  g.M = static_cast<int>(s->tokens);
  g.N = static_cast<int>(s->d);
  g.K = static_cast<int>(s->ffn);
  g.a = {H, s->ffn, false};
  g.b = {B, s->d, true};
  g.epi = kEpiStore;
  g.shards = s->n_shards;
  g.out0 = P;
  g.ld0 = s->d;
  g.shard_stride0 = s->tokens * s->d;
  return launch_gemm(g, c, st);
}

cudaError_t do_reduce_scatter(const DeviceCtx& c, const void* P, const tpmlp_shape* s, void* const* Y_chunks,
                              cudaStream_t st, const SpTail* tail = nullptr) {
  RowParams r{};
  r.out_chunks = to_chunks(Y_chunks, s->n_shards);
  r.rows = static_cast<int>(s->tokens);
  r.d = static_cast<int>(s->d);
  r.n_chunks = s->n_shards;
  r.rows_per_chunk = static_cast<int>(s->tokens / s->n_shards);
  r.src = P;
  r.shard_stride = s->tokens * s->d;
  if (tail != nullptr) apply_tail(r, *tail);
  return launch_reduce_scatter(r, c, st);
}

cudaError_t do_layernorm(const DeviceCtx& c, const void* const* X_chunks, const void* gamma, const void* beta,
                         float eps, const tpmlp_shape* s, void* Xg, cudaStream_t st) {
  RowParams r{};
  r.in_chunks = to_const_chunks(X_chunks, s->n_shards);
  r.rows = static_cast<int>(s->tokens);
  r.d = static_cast<int>(s->d);
  r.n_chunks = s->n_shards;
  r.rows_per_chunk = static_cast<int>(s->tokens / s->n_shards);
  r.eps = eps;
  r.gamma = gamma;
  r.beta = beta;
  r.dst = Xg;
  return launch_layernorm_fwd(r, c, st);
}

cudaError_t do_dh(const DeviceCtx& c, const void* dY, const void* B, const void* Hpre, const tpmlp_shape* s,
                  void* dHpre, void* H, void* dbias, float* colsum, cudaStream_t st) {
  GemmLaunch g;
  g.M = static_cast<int>(s->tokens);
  g.N = static_cast<int>(s->ffn);
  g.K = static_cast<int>(s->d);
  g.a = {dY, s->d, false};
  g.b = {B, s->d, false};
  g.epi = kEpiDGelu;
  g.out0 = dHpre;
  g.ld0 = s->ffn;
  g.out1 = H;
  g.ld1 = s->ffn;
  g.aux = Hpre;
  g.ld_aux = s->ffn;
  g.colsum = dbias != nullptr ? colsum : nullptr;
  cudaError_t e = launch_gemm(g, c, st);
  if (e != cudaSuccess || dbias == nullptr) return e;
  const int m_blocks = static_cast<int>((s->tokens + kBM - 1) / kBM);
  return launch_column_sum(colsum, 4 * m_blocks, static_cast<int>(s->ffn), dbias, true, st);
}

cudaError_t do_wgrad_b(const DeviceCtx& c, const void* H, const void* dY, const tpmlp_shape* s, void* dB,
                       cudaStream_t st) {
  GemmLaunch g;
  g.M = static_cast<int>(s->ffn);
  g.N = static_cast<int>(s->d);
  g.K = static_cast<int>(s->tokens);
  g.a = {H, s->ffn, true};
  g.b = {dY, s->d, true};
  g.epi = kEpiStore;
  g.out0 = dB;
  g.ld0 = s->d;
  return launch_gemm(g, c, st);
}

cudaError_t do_wgrad_a(const DeviceCtx& c, const void* X, const void* dHpre, const tpmlp_shape* s, void* dA,
                       cudaStream_t st) {
  GemmLaunch g;
  g.M = static_cast<int>(s->d);
  g.N = static_cast<int>(s->ffn);
  g.K = static_cast<int>(s->tokens);
  g.a = {X, s->d, true};
  g.b = {dHpre, s->ffn, true};
  g.epi = kEpiStore;
  g.out0 = dA;
  g.ld0 = s->ffn;
  return launch_gemm(g, c, st);
}

cudaError_t do_dx(const DeviceCtx& c, const void* dHpre, const void* A, const tpmlp_shape* s, void* dX,
                  cudaStream_t st) {
  GemmLaunch g;
  g.M = static_cast<int>(s->tokens);
  g.N = static_cast<int>(s->d);
  g.K = static_cast<int>(s->ffn);
  g.a = {dHpre, s->ffn, false};
  g.b = {A, s->ffn, false};
  g.epi = kEpiStore;
  g.out0 = dX;
  g.ld0 = s->d;
  return launch_gemm(g, c, st);
}

cudaError_t do_ln_bwd(const DeviceCtx& c, const void* const* X_chunks, const void* gamma, float eps, const void* dXg,
                      const tpmlp_shape* s, void* const* dX_chunks, void* dgamma, void* dbeta, float* partial,
                      cudaStream_t st, const void* const* add_chunks = nullptr) {
  RowParams r{};
  if (add_chunks != nullptr) r.add_chunks = to_const_chunks(add_chunks, s->n_shards);
  r.in_chunks = to_const_chunks(X_chunks, s->n_shards);
  r.out_chunks = to_chunks(dX_chunks, s->n_shards);
  r.rows = static_cast<int>(s->tokens);
  r.d = static_cast<int>(s->d);
  r.n_chunks = s->n_shards;
  r.rows_per_chunk = static_cast<int>(s->tokens / s->n_shards);
  r.eps = eps;
  r.gamma = gamma;
  r.src = dXg;
  return launch_layernorm_bwd(r, partial, layernorm_bwd_scratch_floats(r.rows, r.d), c, static_cast<float*>(dgamma),
                              static_cast<float*>(dbeta), st);
}

// dZ = keep * dY / (1 - p) gathered to [T x d]; dbias2 (optional) = column sums through `partial`.
cudaError_t do_dropout_bwd(const void* const* dY_chunks, const SpTail& t, const tpmlp_shape* s, void* dZ,
                           void* dbias2, float* partial, cudaStream_t st) {
  RowParams r{};
  r.in_chunks = to_const_chunks(dY_chunks, s->n_shards);
  r.rows = static_cast<int>(s->tokens);
  r.d = static_cast<int>(s->d);
  r.n_chunks = s->n_shards;
  r.rows_per_chunk = static_cast<int>(s->tokens / s->n_shards);
  r.dst = dZ;
  apply_tail(r, t);
  return launch_dropout_bwd(r, partial, dbias2, st);
}

// FP8 shape rule on top of check_shape: byte rows of E4M3 tensors are multiples of 16 bytes.
tpmlp_status check_fp8(const tpmlp_shape* s) {
  return s->d % 16 == 0 && s->ffn % 16 == 0 ? TPMLP_OK : TPMLP_ERR_INVALID_ARG;
}

bool fp8_ln_width(int64_t d) { return d == 256 || d == 512 || d == 1024 || d == 2048 || d == 4096 || d == 8192; }

cudaError_t do_ln_e4m3(const void* const* X_chunks, const void* gamma, const void* beta, float eps,
                       const tpmlp_shape* s, const float* scale, void* Xq, float* amax, cudaStream_t st) {
  RowParams r{};
  r.in_chunks = to_const_chunks(X_chunks, s->n_shards);
  r.rows = static_cast<int>(s->tokens);
  r.d = static_cast<int>(s->d);
  r.n_chunks = s->n_shards;
  r.rows_per_chunk = static_cast<int>(s->tokens / s->n_shards);
  r.eps = eps;
  r.gamma = gamma;
  r.beta = beta;
  r.dst = Xq;
  return launch_layernorm_fwd_e4m3(r, scale, amax, st);
}

cudaError_t do_gemm1_e4m3(const DeviceCtx& c, const void* Xq, const void* AqT, const void* bias, const tpmlp_shape* s,
                          const float* sx, const float* sa, const float* sh, void* Hq, float* amax_h, void* Hpre,
                          cudaStream_t st) {
  GemmLaunch g;
  g.M = static_cast<int>(s->tokens);
  g.N = static_cast<int>(s->ffn);
  g.K = static_cast<int>(s->d);
  g.a = {Xq, s->d, false};
  g.b = {AqT, s->d, false};
  g.epi = kEpiBiasGeluQ;
  g.fp8 = true;
  g.scale_a = sx;
  g.scale_b = sa;
  g.scale_out = sh;
  g.amax_out = amax_h;
  g.out0 = Hq;
  g.ld0 = s->ffn;
  g.out1 = Hpre;
  g.ld1 = s->ffn;
  g.bias = bias;
  return launch_gemm(g, c, st);
}

cudaError_t do_gemm2_e4m3(const DeviceCtx& c, const void* Hq, const void* BqT, const tpmlp_shape* s, const float* sh,
                          const float* sb, void* Y, void* const* Y_chunks, cudaStream_t st) {
  GemmLaunch g;
  g.M = static_cast<int>(s->tokens);
  g.N = static_cast<int>(s->d);
  g.K = static_cast<int>(s->ffn);
  g.a = {Hq, s->ffn, false};
  g.b = {BqT, s->ffn, false};
  g.epi = kEpiStore;
  g.fp8 = true;
  g.scale_a = sh;
  g.scale_b = sb;
  g.out0 = Y;
  g.ld0 = s->d;
  if (Y_chunks != nullptr) {
    g.rows_per_chunk = static_cast<int>(s->tokens / s->n_shards);
    g.chunks = to_chunks(Y_chunks, s->n_shards);
  }
  return launch_gemm(g, c, st);
}

cudaError_t do_dh_e5m2(const DeviceCtx& c, const void* dYq, const void* Bq, const void* Hpre, const tpmlp_shape* s,
                       const float* sdy, const float* sb, const float* sg, void* dHq, float* amax_g, void* dbias,
                       float* colsum, cudaStream_t st) {
  GemmLaunch g;
  g.M = static_cast<int>(s->tokens);
  g.N = static_cast<int>(s->ffn);
  g.K = static_cast<int>(s->d);
  g.a = {dYq, s->d, false};
  g.b = {Bq, s->d, false};
  g.epi = kEpiDGeluQ;
  g.fp8 = true;
  g.a_fmt = 1;
  g.b_fmt = 0;
  g.scale_a = sdy;
  g.scale_b = sb;
  g.scale_out = sg;
  g.amax_out = amax_g;
  g.out0 = dHq;
  g.ld0 = s->ffn;
  g.aux = Hpre;
  g.ld_aux = s->ffn;
  g.colsum = dbias != nullptr ? colsum : nullptr;
  cudaError_t e = launch_gemm(g, c, st);
  if (e != cudaSuccess || dbias == nullptr) return e;
  const int m_blocks = static_cast<int>((s->tokens + kBM - 1) / kBM);  // 4 partial rows per 128-row block
  return launch_column_sum(colsum, 4 * m_blocks, static_cast<int>(s->ffn), dbias, true, st);
}

cudaError_t do_gemm_fp8(const DeviceCtx& c, const void* A8, int a_fmt, const void* B8, int b_fmt, int M, int N, int K,
                        const float* sa, const float* sb, void* C, long long ldc, cudaStream_t st) {
  GemmLaunch g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.a = {A8, K, false};
  g.b = {B8, K, false};
  g.epi = kEpiStore;
  g.fp8 = true;
  g.a_fmt = a_fmt;
  g.b_fmt = b_fmt;
  g.scale_a = sa;
  g.scale_b = sb;
  g.out0 = C;
  g.ld0 = ldc;
  return launch_gemm(g, c, st);
}

bool fp8_state_ok(const tpmlp_fp8_state* f) {
  return f != nullptr && f->scale != nullptr && f->amax != nullptr && f->history != nullptr &&
         f->history_len >= 1 && f->history_len <= (1 << 20) && f->margin >= 0 && f->margin <= 64 &&
         (reinterpret_cast<uintptr_t>(f->scale) & 3u) == 0 && (reinterpret_cast<uintptr_t>(f->amax) & 3u) == 0 &&
         (reinterpret_cast<uintptr_t>(f->history) & 3u) == 0;
}

// Backward core shared by tpmlp_backward and tpmlp_sp_backward.  With Hpre
// and H from the forward only the four backward GEMMs run; without Hpre, one
// GEMM1 recomputes both.
cudaError_t backward_core(const DeviceCtx& c, const void* X, const void* A, const void* B, const void* bias,
                          const void* Hpre, const void* H, const void* dY, const tpmlp_shape* s, void* dX, void* dA,
                          void* dB, void* dbias, Carve& ws, cudaStream_t st) {
  const Sizes z = sizes_of(s);
  void* hpre_ws = ws.take(z.tf);
  void* dhpre = ws.take(z.tf);
  void* h_ws = ws.take(z.tf);
  float* colsum = static_cast<float*>(ws.take(z.colsum));
  cudaError_t e = cudaSuccess;
  void* h_out = nullptr;  // H emitted by the GeLU' epilogue only when nobody supplied it
  if (Hpre == nullptr) {
    e = do_gemm1(c, X, A, bias, s, h_ws, hpre_ws, kEpiBiasGelu, st);
    if (e != cudaSuccess) return e;
    Hpre = hpre_ws;
    H = h_ws;
  } else if (H == nullptr) {
    h_out = h_ws;
    H = h_ws;
  }
  if ((e = do_dh(c, dY, B, Hpre, s, dhpre, h_out, dbias, colsum, st)) != cudaSuccess) return e;
  if ((e = do_wgrad_b(c, H, dY, s, dB, st)) != cudaSuccess) return e;
  if ((e = do_wgrad_a(c, X, dhpre, s, dA, st)) != cudaSuccess) return e;
  return do_dx(c, dhpre, A, s, dX, st);
}

}  // namespace
}  // namespace tpmlp

using namespace tpmlp;

extern "C" {

const char* tpmlp_status_string(tpmlp_status s) {
  switch (s) {
    case TPMLP_OK: return "ok";
    case TPMLP_ERR_INVALID_ARG: return "invalid argument";
    case TPMLP_ERR_UNSUPPORTED: return "unsupported shape or option";
    case TPMLP_ERR_CUDA: return "CUDA error";
    case TPMLP_ERR_TIMEOUT: return "device wait timed out";
    case TPMLP_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

tpmlp_status tpmlp_workspace_size(const tpmlp_shape* shape, int op, size_t* bytes) {
  if (bytes == nullptr) return TPMLP_ERR_INVALID_ARG;
  const bool sp = op == TPMLP_OP_SP_FWD || op == TPMLP_OP_SP_FWD_PARTIALS || op == TPMLP_OP_SP_BWD ||
                  op == TPMLP_OP_LN_BWD || op == TPMLP_OP_SP_BLOCK_BWD || op == TPMLP_OP_DROPOUT_BWD ||
                  op == TPMLP_OP_SP_FWD_FP8 || op == TPMLP_OP_SP_BWD_FP8;
  const bool bf16_only = op != TPMLP_OP_FWD;
  tpmlp_status st = check_shape(shape, sp, bf16_only);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (op < TPMLP_OP_FWD || op > TPMLP_OP_SP_BWD_FP8) return TPMLP_ERR_INVALID_ARG;
  if ((op == TPMLP_OP_SP_FWD_FP8 || op == TPMLP_OP_SP_BWD_FP8) && (shape->d % 16 != 0 || shape->ffn % 16 != 0))
    return TPMLP_ERR_INVALID_ARG;
  if (op == TPMLP_OP_SP_BWD_FP8 && shape->tokens % 16 != 0) return TPMLP_ERR_INVALID_ARG;
  *bytes = ws_bytes(shape, op);
  return TPMLP_OK;
}

tpmlp_status tpmlp_get_device_status(tpmlp_stream_t stream, uint32_t* site) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return TPMLP_ERR_CUDA;
  unsigned int w[kErrWords];
  if (cudaMemcpyFromSymbol(w, g_err_words, sizeof(w)) != cudaSuccess) return TPMLP_ERR_CUDA;
  if (site != nullptr) *site = w[1];
  if (w[0] == 0) return TPMLP_OK;
  unsigned int zero[kErrWords] = {0, 0, 0, 0};
  if (cudaMemcpyToSymbol(g_err_words, zero, sizeof(zero)) != cudaSuccess) return TPMLP_ERR_CUDA;
  return (w[0] & kErrTimeout) ? TPMLP_ERR_TIMEOUT : TPMLP_ERR_CUDA;
}

tpmlp_status tpmlp_debug_bounds_status(int32_t* checked, uint32_t* violations, uint32_t* first_site) {
  if (checked == nullptr || violations == nullptr || first_site == nullptr) return TPMLP_ERR_INVALID_ARG;
  unsigned int c[2] = {0, 0}, site[2] = {0, 0};
  if (cudaDeviceSynchronize() != cudaSuccess) return TPMLP_ERR_CUDA;
  if (rowwise_bounds_status(&c[0], &site[0]) != cudaSuccess || gemm_bounds_status(&c[1], &site[1]) != cudaSuccess)
    return TPMLP_ERR_CUDA;
#ifdef TPMLP_DEBUG_BOUNDS
  *checked = 1;
#else
  *checked = 0;
#endif
  *violations = c[0] + c[1];
  *first_site = site[0] != 0 ? site[0] : site[1];
  return TPMLP_OK;
}

tpmlp_status tpmlp_selftest_wait_timeout(uint32_t budget_us, tpmlp_stream_t stream) {
  if (budget_us < 1 || budget_us > 1000000) return TPMLP_ERR_INVALID_ARG;
  DeviceCtx c;
  tpmlp_status st = device_ctx(&c);
  if (st != TPMLP_OK) return st;
  k_wait_timeout_selftest<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      c.err, static_cast<unsigned long long>(budget_us) * 1000ull);
  return cuda_status(cudaGetLastError());
}

tpmlp_status tpmlp_forward(const void* X, const void* A, const void* B, const void* bias, const tpmlp_shape* shape,
                           void* Y, void* Hpre_out, void* H_out, void* workspace, size_t workspace_bytes,
                           tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, false, false);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({X, A, B, Y}) || !opt_ok(bias) || !opt_ok(Hpre_out) || !opt_ok(H_out)) return TPMLP_ERR_INVALID_ARG;
  if (shape->dtype == TPMLP_FP32 && (Hpre_out != nullptr || H_out != nullptr)) return TPMLP_ERR_UNSUPPORTED;
  if (workspace == nullptr || !al16(workspace) || workspace_bytes < ws_bytes(shape, TPMLP_OP_FWD))
    return TPMLP_ERR_WORKSPACE;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (shape->dtype == TPMLP_FP32) {
    return cuda_status(launch_mlp_fp32(static_cast<const float*>(X), static_cast<const float*>(A),
                                       static_cast<const float*>(B), static_cast<const float*>(bias),
                                       static_cast<int>(shape->tokens), static_cast<int>(shape->d),
                                       static_cast<int>(shape->ffn), static_cast<float*>(workspace),
                                       static_cast<float*>(Y), s));
  }
  void* H = H_out != nullptr ? H_out : workspace;
  cudaError_t e = do_gemm1(c, X, A, bias, shape, H, Hpre_out, kEpiBiasGelu, s);
  if (e == cudaSuccess) e = do_gemm2(c, H, B, shape, Y, nullptr, s);
  return cuda_status(e);
}

// tpmlp_sp_forward, and with `tail` (validated, residual = X_chunks) tpmlp_sp_block_forward.
static tpmlp_status sp_forward_impl(const void* const* X_chunks, const void* gamma, const void* beta, float eps,
                                    const void* A, const void* B, const void* bias, const tpmlp_shape* shape,
                                    void* const* Y_chunks, int rs_mode, void* Hpre_out, void* H_out, void* Xg_out,
                                    void* workspace, size_t workspace_bytes, tpmlp_stream_t stream,
                                    const SpTail* tail) {
  tpmlp_status st = check_shape(shape, true, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({gamma, beta, A, B}) || !opt_ok(bias) || !opt_ok(Hpre_out) || !opt_ok(H_out) || !opt_ok(Xg_out))
    return TPMLP_ERR_INVALID_ARG;
  if (!chunks_ok(X_chunks, shape->n_shards) || !chunks_ok(Y_chunks, shape->n_shards)) return TPMLP_ERR_INVALID_ARG;
  if (!(eps >= 0.f)) return TPMLP_ERR_INVALID_ARG;
  if (rs_mode != TPMLP_RS_FUSED && rs_mode != TPMLP_RS_PARTIALS) return TPMLP_ERR_INVALID_ARG;
  if (rs_mode == TPMLP_RS_PARTIALS && (shape->ffn / shape->n_shards) % kBK != 0) return TPMLP_ERR_UNSUPPORTED;
  const int op = rs_mode == TPMLP_RS_FUSED ? TPMLP_OP_SP_FWD : TPMLP_OP_SP_FWD_PARTIALS;
  if (workspace == nullptr || !al16(workspace) || workspace_bytes < ws_bytes(shape, op)) return TPMLP_ERR_WORKSPACE;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const Sizes z = sizes_of(shape);
  Carve ws(workspace);
  void* Xg = ws.take(z.td);
  void* H = ws.take(z.tf);
  if (H_out != nullptr) H = H_out;
  if (Xg_out != nullptr) Xg = Xg_out;
  cudaError_t e = do_layernorm(c, X_chunks, gamma, beta, eps, shape, Xg, s);
  if (e == cudaSuccess) e = do_gemm1(c, Xg, A, bias, shape, H, Hpre_out, kEpiBiasGelu, s);
  if (e == cudaSuccess) {
    if (rs_mode == TPMLP_RS_FUSED) {
      e = do_gemm2(c, H, B, shape, nullptr, Y_chunks, s, tail);
    } else {
      void* P = ws.take(z.ptd);
      e = do_gemm2_partials(c, H, B, shape, P, s);
      if (e == cudaSuccess) e = do_reduce_scatter(c, P, shape, Y_chunks, s, tail);
    }
  }
  return cuda_status(e);
}

tpmlp_status tpmlp_sp_forward(const void* const* X_chunks, const void* gamma, const void* beta, float eps,
                              const void* A, const void* B, const void* bias, const tpmlp_shape* shape,
                              void* const* Y_chunks, int rs_mode, void* Hpre_out, void* H_out, void* Xg_out,
                              void* workspace, size_t workspace_bytes, tpmlp_stream_t stream) {
  return sp_forward_impl(X_chunks, gamma, beta, eps, A, B, bias, shape, Y_chunks, rs_mode, Hpre_out, H_out, Xg_out,
                         workspace, workspace_bytes, stream, nullptr);
}

tpmlp_status tpmlp_sp_block_forward(const void* const* X_chunks, const void* gamma, const void* beta, float eps,
                                    const void* A, const void* B, const void* bias, const void* bias2,
                                    const tpmlp_dropout* dropout, const tpmlp_shape* shape, void* const* Y_chunks,
                                    int rs_mode, void* Hpre_out, void* H_out, void* Xg_out, void* workspace,
                                    size_t workspace_bytes, tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, true, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!chunks_ok(X_chunks, shape->n_shards)) return TPMLP_ERR_INVALID_ARG;
  SpTail tail;
  if ((st = make_tail(bias2, dropout, X_chunks, shape->n_shards, &tail)) != TPMLP_OK) return st;
  return sp_forward_impl(X_chunks, gamma, beta, eps, A, B, bias, shape, Y_chunks, rs_mode, Hpre_out, H_out, Xg_out,
                         workspace, workspace_bytes, stream, &tail);
}

tpmlp_status tpmlp_backward(const void* X, const void* A, const void* B, const void* bias, const void* Hpre,
                            const void* H, const void* dY, const tpmlp_shape* shape, void* dX, void* dA, void* dB,
                            void* dbias, void* workspace, size_t workspace_bytes, tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, false, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({X, A, B, dY, dX, dA, dB}) || !opt_ok(bias) || !opt_ok(Hpre) || !opt_ok(H) || !opt_ok(dbias))
    return TPMLP_ERR_INVALID_ARG;
  if (workspace == nullptr || !al16(workspace) || workspace_bytes < ws_bytes(shape, TPMLP_OP_BWD))
    return TPMLP_ERR_WORKSPACE;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  Carve ws(workspace);
  return cuda_status(backward_core(c, X, A, B, bias, Hpre, H, dY, shape, dX, dA, dB, dbias, ws,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

// tpmlp_sp_backward, and with `tail` (validated) tpmlp_sp_block_backward.
static tpmlp_status sp_backward_impl(const void* const* X_chunks, const void* gamma, const void* beta, float eps,
                                     const void* A, const void* B, const void* bias, const void* Hpre, const void* H,
                                     const void* Xg_saved, const void* const* dY_chunks, const tpmlp_shape* shape,
                                     void* const* dX_chunks, void* dA, void* dB, void* dbias, void* dgamma,
                                     void* dbeta, void* workspace, size_t workspace_bytes, tpmlp_stream_t stream,
                                     const SpTail* tail, void* dbias2) {
  tpmlp_status st = check_shape(shape, true, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({gamma, beta, A, B, dA, dB, dgamma, dbeta}) || !opt_ok(bias) || !opt_ok(Hpre) || !opt_ok(H) ||
      !opt_ok(Xg_saved) || !opt_ok(dbias))
    return TPMLP_ERR_INVALID_ARG;
  const int n = shape->n_shards;
  if (!chunks_ok(X_chunks, n) || !chunks_ok(dY_chunks, n) || !chunks_ok(dX_chunks, n)) return TPMLP_ERR_INVALID_ARG;
  if (shape->d > kLnBwdMaxD) return TPMLP_ERR_UNSUPPORTED;
  if (!(eps >= 0.f)) return TPMLP_ERR_INVALID_ARG;
  if (!opt_ok(dbias2)) return TPMLP_ERR_INVALID_ARG;
  const int op = tail != nullptr ? TPMLP_OP_SP_BLOCK_BWD : TPMLP_OP_SP_BWD;
  if (workspace == nullptr || !al16(workspace) || workspace_bytes < ws_bytes(shape, op)) return TPMLP_ERR_WORKSPACE;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const Sizes z = sizes_of(shape);
  Carve ws(workspace);
  void* Xg = ws.take(z.td);
  void* dYg = ws.take(z.td);
  void* dXg = ws.take(z.td);
  float* lnpart = static_cast<float*>(ws.take(z.lnbwd));
  cudaError_t e = cudaSuccess;
  if (Xg_saved != nullptr) {
    Xg = const_cast<void*>(Xg_saved);
  } else {
    e = do_layernorm(c, X_chunks, gamma, beta, eps, shape, Xg, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  const void* dY = dY_chunks[0];
  if (tail != nullptr) {
    // the dropout backward gathers dZ = keep * dY / (1 - p) (and dbias2); the MLP backward runs on dZ and
    // the residual's gradient dY joins the input gradient in the LayerNorm backward
    float* dropcol = static_cast<float*>(ws.take(z.dropcol));
    if ((e = do_dropout_bwd(dY_chunks, *tail, shape, dYg, dbias2, dropcol, s)) != cudaSuccess) return cuda_status(e);
    dY = dYg;
  } else {
    // The All-Gather of dY is free when the chunks already lie back to back.
    const size_t chunk_bytes = static_cast<size_t>(shape->tokens / n) * shape->d * 2;
    bool contiguous = true;
    for (int j = 1; j < n; ++j)
      contiguous = contiguous && static_cast<const uint8_t*>(dY_chunks[j]) ==
                                     static_cast<const uint8_t*>(dY_chunks[0]) + j * chunk_bytes;
    if (!contiguous) {
      RowParams r{};
      r.in_chunks = to_const_chunks(dY_chunks, n);
      r.rows = static_cast<int>(shape->tokens);
      r.d = static_cast<int>(shape->d);
      r.n_chunks = n;
      r.rows_per_chunk = static_cast<int>(shape->tokens / n);
      r.dst = dYg;
      if ((e = launch_gather_rows(r, c, s)) != cudaSuccess) return cuda_status(e);
      dY = dYg;
    }
  }
  e = backward_core(c, Xg, A, B, bias, Hpre, H, dY, shape, dXg, dA, dB, dbias, ws, s);
  if (e == cudaSuccess)
    e = do_ln_bwd(c, X_chunks, gamma, eps, dXg, shape, dX_chunks, dgamma, dbeta, lnpart, s,
                  tail != nullptr ? dY_chunks : nullptr);
  return cuda_status(e);
}

tpmlp_status tpmlp_sp_backward(const void* const* X_chunks, const void* gamma, const void* beta, float eps,
                               const void* A, const void* B, const void* bias, const void* Hpre, const void* H,
                               const void* Xg_saved, const void* const* dY_chunks, const tpmlp_shape* shape,
                               void* const* dX_chunks, void* dA, void* dB, void* dbias, void* dgamma, void* dbeta,
                               void* workspace, size_t workspace_bytes, tpmlp_stream_t stream) {
  return sp_backward_impl(X_chunks, gamma, beta, eps, A, B, bias, Hpre, H, Xg_saved, dY_chunks, shape, dX_chunks, dA,
                          dB, dbias, dgamma, dbeta, workspace, workspace_bytes, stream, nullptr, nullptr);
}

tpmlp_status tpmlp_sp_block_backward(const void* const* X_chunks, const void* gamma, const void* beta, float eps,
                                     const void* A, const void* B, const void* bias, const tpmlp_dropout* dropout,
                                     const void* Hpre, const void* H, const void* Xg, const void* const* dY_chunks,
                                     const tpmlp_shape* shape, void* const* dX_chunks, void* dA, void* dB,
                                     void* dbias, void* dbias2, void* dgamma, void* dbeta, void* workspace,
                                     size_t workspace_bytes, tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, true, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  SpTail tail;
  if ((st = make_tail(nullptr, dropout, nullptr, shape->n_shards, &tail)) != TPMLP_OK) return st;
  return sp_backward_impl(X_chunks, gamma, beta, eps, A, B, bias, Hpre, H, Xg, dY_chunks, shape, dX_chunks, dA, dB,
                          dbias, dgamma, dbeta, workspace, workspace_bytes, stream, &tail, dbias2);
}

// ------------------------------------------------------------------ single steps

tpmlp_status tpmlp_gemm1_bias_gelu(const void* X, const void* A, const void* bias, const tpmlp_shape* shape, void* H,
                                   void* Hpre, tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, false, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({X, A, H}) || !opt_ok(bias) || !opt_ok(Hpre)) return TPMLP_ERR_INVALID_ARG;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  return cuda_status(do_gemm1(c, X, A, bias, shape, H, Hpre, kEpiBiasGelu, reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_gemm2_shard_accum(const void* H, const void* B, const tpmlp_shape* shape, void* Y,
                                     void* const* Y_chunks, tpmlp_stream_t stream) {
  const bool chunked = Y_chunks != nullptr;
  tpmlp_status st = check_shape(shape, chunked, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({H, B})) return TPMLP_ERR_INVALID_ARG;
  if (chunked ? !chunks_ok(Y_chunks, shape->n_shards) : !ptrs_ok({Y})) return TPMLP_ERR_INVALID_ARG;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  return cuda_status(do_gemm2(c, H, B, shape, Y, Y_chunks, reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_gemm2_partials(const void* H, const void* B, const tpmlp_shape* shape, void* P,
                                  tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, false, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({H, B, P})) return TPMLP_ERR_INVALID_ARG;
  if ((shape->ffn / shape->n_shards) % kBK != 0) return TPMLP_ERR_UNSUPPORTED;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  return cuda_status(do_gemm2_partials(c, H, B, shape, P, reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_reduce_scatter(const void* P, const tpmlp_shape* shape, void* const* Y_chunks,
                                  tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, true, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({P}) || !chunks_ok(Y_chunks, shape->n_shards)) return TPMLP_ERR_INVALID_ARG;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  return cuda_status(do_reduce_scatter(c, P, shape, Y_chunks, reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_layernorm_gather(const void* const* X_chunks, const void* gamma, const void* beta, float eps,
                                    const tpmlp_shape* shape, void* Xg, tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, true, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({gamma, beta, Xg}) || !chunks_ok(X_chunks, shape->n_shards) || !(eps >= 0.f))
    return TPMLP_ERR_INVALID_ARG;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  return cuda_status(do_layernorm(c, X_chunks, gamma, beta, eps, shape, Xg, reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_rmsnorm_gather(const void* const* X_chunks, const void* weight, float eps,
                                  const tpmlp_shape* shape, void* Xg, tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, true, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({weight, Xg}) || !chunks_ok(X_chunks, shape->n_shards) || !(eps >= 0.f))
    return TPMLP_ERR_INVALID_ARG;
  RowParams r{};
  r.in_chunks = to_const_chunks(X_chunks, shape->n_shards);
  r.rows = static_cast<int>(shape->tokens);
  r.d = static_cast<int>(shape->d);
  r.n_chunks = shape->n_shards;
  r.rows_per_chunk = static_cast<int>(shape->tokens / shape->n_shards);
  r.eps = eps;
  r.gamma = weight;
  r.dst = Xg;
  return cuda_status(launch_rmsnorm_fwd(r, reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_gemm_dh_geluprime(const void* dY, const void* B, const void* Hpre, const tpmlp_shape* shape,
                                     void* dHpre, void* H, void* dbias, void* workspace, size_t workspace_bytes,
                                     tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, false, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({dY, B, Hpre, dHpre}) || !opt_ok(H) || !opt_ok(dbias)) return TPMLP_ERR_INVALID_ARG;
  if (dbias != nullptr && (workspace == nullptr || !al16(workspace) ||
                           workspace_bytes < ws_bytes(shape, TPMLP_OP_DH_GELUPRIME)))
    return TPMLP_ERR_WORKSPACE;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  return cuda_status(do_dh(c, dY, B, Hpre, shape, dHpre, H, dbias, static_cast<float*>(workspace),
                           reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_gemm_wgrad_b(const void* H, const void* dY, const tpmlp_shape* shape, void* dB,
                                tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, false, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({H, dY, dB})) return TPMLP_ERR_INVALID_ARG;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  return cuda_status(do_wgrad_b(c, H, dY, shape, dB, reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_gemm_wgrad_a(const void* X, const void* dHpre, const tpmlp_shape* shape, void* dA,
                                tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, false, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({X, dHpre, dA})) return TPMLP_ERR_INVALID_ARG;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  return cuda_status(do_wgrad_a(c, X, dHpre, shape, dA, reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_gemm_dx_shard_accum(const void* dHpre, const void* A, const tpmlp_shape* shape, void* dX,
                                       tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, false, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({dHpre, A, dX})) return TPMLP_ERR_INVALID_ARG;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  return cuda_status(do_dx(c, dHpre, A, shape, dX, reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_layernorm_backward(const void* const* X_chunks, const void* gamma, float eps, const void* dXg,
                                      const tpmlp_shape* shape, void* const* dX_chunks, void* dgamma, void* dbeta,
                                      void* workspace, size_t workspace_bytes, tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, true, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({gamma, dXg, dgamma, dbeta}) || !chunks_ok(X_chunks, shape->n_shards) ||
      !chunks_ok(dX_chunks, shape->n_shards) || !(eps >= 0.f))
    return TPMLP_ERR_INVALID_ARG;
  if (shape->d > kLnBwdMaxD) return TPMLP_ERR_UNSUPPORTED;
  if (workspace == nullptr || !al16(workspace) || workspace_bytes < ws_bytes(shape, TPMLP_OP_LN_BWD))
    return TPMLP_ERR_WORKSPACE;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  return cuda_status(do_ln_bwd(c, X_chunks, gamma, eps, dXg, shape, dX_chunks, dgamma, dbeta,
                               static_cast<float*>(workspace), reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_layernorm_backward_blocks(const void* const* X_chunks, const void* gamma, float eps,
                                             const void* dXg, const tpmlp_shape* shape, void* const* dX_chunks,
                                             void* dgamma, void* dbeta, int32_t max_blocks, void* workspace,
                                             size_t workspace_bytes, tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, true, true);
  if (st != TPMLP_OK) return st;
  if (max_blocks < 1) return TPMLP_ERR_INVALID_ARG;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({gamma, dXg, dgamma, dbeta}) || !chunks_ok(X_chunks, shape->n_shards) ||
      !chunks_ok(dX_chunks, shape->n_shards) || !(eps >= 0.f))
    return TPMLP_ERR_INVALID_ARG;
  if (shape->d > kLnBwdMaxD) return TPMLP_ERR_UNSUPPORTED;
  const size_t cap = static_cast<size_t>(max_blocks) * 2 * static_cast<size_t>(shape->d);
  if (workspace == nullptr || !al16(workspace) || workspace_bytes < cap * sizeof(float)) return TPMLP_ERR_WORKSPACE;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  RowParams r{};
  r.in_chunks = to_const_chunks(X_chunks, shape->n_shards);
  r.out_chunks = to_chunks(dX_chunks, shape->n_shards);
  r.rows = static_cast<int>(shape->tokens);
  r.d = static_cast<int>(shape->d);
  r.n_chunks = shape->n_shards;
  r.rows_per_chunk = static_cast<int>(shape->tokens / shape->n_shards);
  r.eps = eps;
  r.gamma = gamma;
  r.src = dXg;
  return cuda_status(launch_layernorm_bwd(r, static_cast<float*>(workspace), cap, c, static_cast<float*>(dgamma),
                                          static_cast<float*>(dbeta), reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_gemm2_bias_dropout_add(const void* H, const void* B, const void* bias2, const tpmlp_dropout* dropout,
                                          const void* const* R_chunks, const tpmlp_shape* shape,
                                          void* const* Y_chunks, tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, true, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({H, B}) || !chunks_ok(Y_chunks, shape->n_shards)) return TPMLP_ERR_INVALID_ARG;
  SpTail tail;
  if ((st = make_tail(bias2, dropout, R_chunks, shape->n_shards, &tail)) != TPMLP_OK) return st;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  return cuda_status(do_gemm2(c, H, B, shape, nullptr, Y_chunks, reinterpret_cast<cudaStream_t>(stream), &tail));
}

tpmlp_status tpmlp_reduce_scatter_bias_dropout_add(const void* P, const void* bias2, const tpmlp_dropout* dropout,
                                                   const void* const* R_chunks, const tpmlp_shape* shape,
                                                   void* const* Y_chunks, tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, true, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({P}) || !chunks_ok(Y_chunks, shape->n_shards)) return TPMLP_ERR_INVALID_ARG;
  SpTail tail;
  if ((st = make_tail(bias2, dropout, R_chunks, shape->n_shards, &tail)) != TPMLP_OK) return st;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  return cuda_status(do_reduce_scatter(c, P, shape, Y_chunks, reinterpret_cast<cudaStream_t>(stream), &tail));
}

tpmlp_status tpmlp_dropout_backward(const void* const* dY_chunks, const tpmlp_dropout* dropout,
                                    const tpmlp_shape* shape, void* dZ, void* dbias2, void* workspace,
                                    size_t workspace_bytes, tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, true, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({dZ}) || !opt_ok(dbias2) || !chunks_ok(dY_chunks, shape->n_shards)) return TPMLP_ERR_INVALID_ARG;
  SpTail tail;
  if ((st = make_tail(nullptr, dropout, nullptr, shape->n_shards, &tail)) != TPMLP_OK) return st;
  if (dbias2 != nullptr && (workspace == nullptr || !al16(workspace) ||
                            workspace_bytes < ws_bytes(shape, TPMLP_OP_DROPOUT_BWD)))
    return TPMLP_ERR_WORKSPACE;
  return cuda_status(do_dropout_bwd(dY_chunks, tail, shape, dZ, dbias2, static_cast<float*>(workspace),
                                    reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_layernorm_backward_add(const void* const* X_chunks, const void* gamma, float eps, const void* dXg,
                                          const void* const* R_chunks, const tpmlp_shape* shape,
                                          void* const* dX_chunks, void* dgamma, void* dbeta, void* workspace,
                                          size_t workspace_bytes, tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, true, true);
  if (st != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({gamma, dXg, dgamma, dbeta}) || !chunks_ok(X_chunks, shape->n_shards) ||
      !chunks_ok(dX_chunks, shape->n_shards) || !chunks_ok(R_chunks, shape->n_shards) || !(eps >= 0.f))
    return TPMLP_ERR_INVALID_ARG;
  if (shape->d > kLnBwdMaxD) return TPMLP_ERR_UNSUPPORTED;
  if (workspace == nullptr || !al16(workspace) || workspace_bytes < ws_bytes(shape, TPMLP_OP_LN_BWD))
    return TPMLP_ERR_WORKSPACE;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  return cuda_status(do_ln_bwd(c, X_chunks, gamma, eps, dXg, shape, dX_chunks, dgamma, dbeta,
                               static_cast<float*>(workspace), reinterpret_cast<cudaStream_t>(stream), R_chunks));
}

// ------------------------------------------------------------------ FP8 forward

tpmlp_status tpmlp_cast_e4m3(const void* src, int64_t rows, int64_t cols, int transpose, const float* scale, void* dst,
                             float* amax, tpmlp_stream_t stream) {
  if (rows < 0 || cols < 0 || rows % 16 != 0 || cols % 16 != 0 || rows > INT_MAX / 2 || cols > INT_MAX / 2)
    return TPMLP_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return TPMLP_OK;
  if (!ptrs_ok({src, dst}) || scale == nullptr || amax == nullptr) return TPMLP_ERR_INVALID_ARG;
  if (transpose && (rows + 63) / 64 > 65535) return TPMLP_ERR_UNSUPPORTED;
  return cuda_status(launch_cast_e4m3(src, static_cast<int>(rows), static_cast<int>(cols), transpose != 0, scale, dst,
                                      amax, reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_layernorm_gather_e4m3(const void* const* X_chunks, const void* gamma, const void* beta, float eps,
                                         const tpmlp_shape* shape, const float* scale, void* Xq, float* amax,
                                         tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, true, true);
  if (st != TPMLP_OK) return st;
  if ((st = check_fp8(shape)) != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({gamma, beta, Xq}) || !chunks_ok(X_chunks, shape->n_shards) || !(eps >= 0.f) || scale == nullptr ||
      amax == nullptr)
    return TPMLP_ERR_INVALID_ARG;
  if (!fp8_ln_width(shape->d)) return TPMLP_ERR_UNSUPPORTED;
  return cuda_status(do_ln_e4m3(X_chunks, gamma, beta, eps, shape, scale, Xq, amax,
                                reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_gemm1_e4m3(const void* Xq, const void* AqT, const void* bias, const tpmlp_shape* shape,
                              const float* scale_x, const float* scale_a, const float* scale_h, void* Hq,
                              float* amax_h, void* Hpre, tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, false, true);
  if (st != TPMLP_OK) return st;
  if ((st = check_fp8(shape)) != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({Xq, AqT, Hq}) || !opt_ok(bias) || !opt_ok(Hpre) || scale_x == nullptr || scale_a == nullptr ||
      scale_h == nullptr)
    return TPMLP_ERR_INVALID_ARG;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  return cuda_status(do_gemm1_e4m3(c, Xq, AqT, bias, shape, scale_x, scale_a, scale_h, Hq, amax_h, Hpre,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_gemm2_e4m3(const void* Hq, const void* BqT, const tpmlp_shape* shape, const float* scale_h,
                              const float* scale_b, void* Y, void* const* Y_chunks, tpmlp_stream_t stream) {
  const bool chunked = Y_chunks != nullptr;
  tpmlp_status st = check_shape(shape, chunked, true);
  if (st != TPMLP_OK) return st;
  if ((st = check_fp8(shape)) != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({Hq, BqT}) || scale_h == nullptr || scale_b == nullptr) return TPMLP_ERR_INVALID_ARG;
  if (chunked ? !chunks_ok(Y_chunks, shape->n_shards) : !ptrs_ok({Y})) return TPMLP_ERR_INVALID_ARG;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  return cuda_status(do_gemm2_e4m3(c, Hq, BqT, shape, scale_h, scale_b, Y, Y_chunks,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_fp8_update_scales(const tpmlp_fp8_state* state, tpmlp_stream_t stream) {
  if (!fp8_state_ok(state)) return TPMLP_ERR_INVALID_ARG;
  return cuda_status(launch_fp8_update(state->scale, state->amax, state->history, 4, state->history_len, 448.f,
                                       state->margin, reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_sp_forward_fp8(const void* const* X_chunks, const void* gamma, const void* beta, float eps,
                                  const void* A, const void* B, const void* bias, const tpmlp_fp8_state* state,
                                  const tpmlp_shape* shape, void* const* Y_chunks, void* Hpre_out, void* Xq_out,
                                  void* Hq_out, void* workspace, size_t workspace_bytes, tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, true, true);
  if (st != TPMLP_OK) return st;
  if ((st = check_fp8(shape)) != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({gamma, beta, A, B}) || !opt_ok(bias) || !chunks_ok(X_chunks, shape->n_shards) ||
      !chunks_ok(Y_chunks, shape->n_shards) || !(eps >= 0.f) || !fp8_state_ok(state) || !opt_ok(Hpre_out) ||
      !opt_ok(Xq_out) || !opt_ok(Hq_out))
    return TPMLP_ERR_INVALID_ARG;
  if (!fp8_ln_width(shape->d) || (shape->ffn + 63) / 64 > 65535 || (shape->d + 63) / 64 > 65535)
    return TPMLP_ERR_UNSUPPORTED;
  if (workspace == nullptr || !al16(workspace) || workspace_bytes < ws_bytes(shape, TPMLP_OP_SP_FWD_FP8))
    return TPMLP_ERR_WORKSPACE;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const Sizes z = sizes_of(shape);
  Carve ws(workspace);
  void* AqT = ws.take(z.df8);
  void* BqT = ws.take(z.df8);
  void* Xq = ws.take(z.td8);
  void* Hq = ws.take(z.tf8);
  if (Xq_out != nullptr) Xq = Xq_out;
  if (Hq_out != nullptr) Hq = Hq_out;
  float* sc = state->scale;
  float* am = state->amax;
  const int d = static_cast<int>(shape->d), F = static_cast<int>(shape->ffn);
  cudaError_t e = launch_cast_e4m3(A, d, F, true, sc + 1, AqT, am + 1, s);
  if (e == cudaSuccess) e = launch_cast_e4m3(B, F, d, true, sc + 2, BqT, am + 2, s);
  if (e == cudaSuccess) e = do_ln_e4m3(X_chunks, gamma, beta, eps, shape, sc + 0, Xq, am + 0, s);
  if (e == cudaSuccess) e = do_gemm1_e4m3(c, Xq, AqT, bias, shape, sc + 0, sc + 1, sc + 3, Hq, am + 3, Hpre_out, s);
  if (e == cudaSuccess) e = do_gemm2_e4m3(c, Hq, BqT, shape, sc + 3, sc + 2, nullptr, Y_chunks, s);
  return cuda_status(e);
}

tpmlp_status tpmlp_cast_e5m2(const void* src, int64_t rows, int64_t cols, int transpose, const float* scale, void* dst,
                             float* amax, tpmlp_stream_t stream) {
  if (rows < 0 || cols < 0 || rows % 16 != 0 || cols % 16 != 0 || rows > INT_MAX / 2 || cols > INT_MAX / 2)
    return TPMLP_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return TPMLP_OK;
  if (!ptrs_ok({src, dst}) || scale == nullptr || amax == nullptr) return TPMLP_ERR_INVALID_ARG;
  if (transpose && (rows + 63) / 64 > 65535) return TPMLP_ERR_UNSUPPORTED;
  return cuda_status(launch_cast_fp8(src, static_cast<int>(rows), static_cast<int>(cols), transpose != 0, 1, scale,
                                     dst, amax, reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_transpose_bytes(const void* src, int64_t rows, int64_t cols, void* dst, tpmlp_stream_t stream) {
  if (rows < 0 || cols < 0 || rows % 16 != 0 || cols % 16 != 0 || rows > INT_MAX / 2 || cols > INT_MAX / 2)
    return TPMLP_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return TPMLP_OK;
  if (!ptrs_ok({src, dst})) return TPMLP_ERR_INVALID_ARG;
  if ((rows + 63) / 64 > 65535) return TPMLP_ERR_UNSUPPORTED;
  return cuda_status(launch_transpose_bytes(src, static_cast<int>(rows), static_cast<int>(cols), dst,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_gemm_dh_geluprime_e5m2(const void* dYq, const void* Bq, const void* Hpre, const tpmlp_shape* shape,
                                          const float* scale_dy, const float* scale_b, const float* scale_g,
                                          void* dHq, float* amax_g, void* dbias, void* workspace,
                                          size_t workspace_bytes, tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, false, true);
  if (st != TPMLP_OK) return st;
  if ((st = check_fp8(shape)) != TPMLP_OK) return st;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  if (!ptrs_ok({dYq, Bq, Hpre, dHq}) || !opt_ok(dbias) || scale_dy == nullptr || scale_b == nullptr ||
      scale_g == nullptr)
    return TPMLP_ERR_INVALID_ARG;
  if (dbias != nullptr && (workspace == nullptr || !al16(workspace) ||
                           workspace_bytes < ws_bytes(shape, TPMLP_OP_DH_GELUPRIME)))
    return TPMLP_ERR_WORKSPACE;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  return cuda_status(do_dh_e5m2(c, dYq, Bq, Hpre, shape, scale_dy, scale_b, scale_g, dHq, amax_g, dbias,
                                static_cast<float*>(workspace), reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_gemm_fp8(const void* A8, int a_fmt, const void* B8, int b_fmt, int64_t M, int64_t N, int64_t K,
                            const float* scale_a, const float* scale_b, void* C, int64_t ldc, tpmlp_stream_t stream) {
  if (M < 0 || N < 0 || K < 0 || M > INT_MAX / 2 || N > INT_MAX / 2 || K > INT_MAX / 2 || K % 16 != 0 ||
      N % 8 != 0 || ldc < N || ldc % 8 != 0 || (a_fmt != 0 && a_fmt != 1) || (b_fmt != 0 && b_fmt != 1))
    return TPMLP_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return TPMLP_OK;
  if (!ptrs_ok({A8, B8, C}) || scale_a == nullptr || scale_b == nullptr || K == 0) return TPMLP_ERR_INVALID_ARG;
  DeviceCtx c;
  tpmlp_status st;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  return cuda_status(do_gemm_fp8(c, A8, a_fmt, B8, b_fmt, static_cast<int>(M), static_cast<int>(N),
                                 static_cast<int>(K), scale_a, scale_b, C, ldc,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

tpmlp_status tpmlp_sp_backward_fp8(const void* const* X_chunks, const void* gamma, float eps, const void* A,
                                   const void* B, const void* Hpre, const void* Xq, const void* Hq,
                                   const void* const* dY_chunks, const tpmlp_fp8_state* fwd,
                                   const tpmlp_fp8_state* grad, const tpmlp_shape* shape, void* const* dX_chunks,
                                   void* dA, void* dB, void* dbias, void* dgamma, void* dbeta, void* dHq_out,
                                   void* workspace, size_t workspace_bytes, tpmlp_stream_t stream) {
  tpmlp_status st = check_shape(shape, true, true);
  if (st != TPMLP_OK) return st;
  if ((st = check_fp8(shape)) != TPMLP_OK) return st;
  if (shape->tokens % 16 != 0) return TPMLP_ERR_INVALID_ARG;
  if (shape->tokens == 0) return TPMLP_OK;  // empty batch: nothing to launch, pointers may be NULL
  const int n = shape->n_shards;
  if (!ptrs_ok({gamma, A, B, Hpre, Xq, Hq, dA, dB, dgamma, dbeta}) || !opt_ok(dbias) || !opt_ok(dHq_out) ||
      !chunks_ok(X_chunks, n) ||
      !chunks_ok(dY_chunks, n) || !chunks_ok(dX_chunks, n) || !(eps >= 0.f) || !fp8_state_ok(fwd) ||
      !fp8_state_ok(grad))
    return TPMLP_ERR_INVALID_ARG;
  if (shape->d > kLnBwdMaxD) return TPMLP_ERR_UNSUPPORTED;
  const int T = static_cast<int>(shape->tokens), d = static_cast<int>(shape->d), F = static_cast<int>(shape->ffn);
  if ((T + 63) / 64 > 65535 || (F + 63) / 64 > 65535 || (d + 63) / 64 > 65535) return TPMLP_ERR_UNSUPPORTED;
  if (workspace == nullptr || !al16(workspace) || workspace_bytes < ws_bytes(shape, TPMLP_OP_SP_BWD_FP8))
    return TPMLP_ERR_WORKSPACE;
  DeviceCtx c;
  if ((st = device_ctx(&c)) != TPMLP_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const Sizes z = sizes_of(shape);
  Carve ws(workspace);
  void* dYg = ws.take(z.td);
  void* dXg = ws.take(z.td);
  void* dYq = ws.take(z.td8);
  void* dYqT = ws.take(z.td8);
  void* XqT = ws.take(z.td8);
  void* Aq = ws.take(z.df8);
  void* Bq = ws.take(z.df8);
  void* dHq = ws.take(z.tf8);
  if (dHq_out != nullptr) dHq = dHq_out;  // the caller keeps the E5M2 dHpre
  void* HqT = ws.take(z.tf8);
  void* dHqT = ws.take(z.tf8);
  float* colsum = static_cast<float*>(ws.take(z.colsum));
  float* lnpart = static_cast<float*>(ws.take(z.lnbwd));
  const float* fs = fwd->scale;
  float* fa = fwd->amax;
  const float* gs = grad->scale;
  float* ga = grad->amax;
  // dY gathered (free when the chunks lie back to back), then E5M2 in both layouts
  cudaError_t e = cudaSuccess;
  const void* dY = dY_chunks[0];
  const size_t chunk_bytes = static_cast<size_t>(T / n) * d * 2;
  bool contiguous = true;
  for (int j = 1; j < n; ++j)
    contiguous = contiguous && static_cast<const uint8_t*>(dY_chunks[j]) ==
                                   static_cast<const uint8_t*>(dY_chunks[0]) + j * chunk_bytes;
  if (!contiguous) {
    RowParams r{};
    r.in_chunks = to_const_chunks(dY_chunks, n);
    r.rows = T;
    r.d = d;
    r.n_chunks = n;
    r.rows_per_chunk = T / n;
    r.dst = dYg;
    if ((e = launch_gather_rows(r, c, s)) != cudaSuccess) return cuda_status(e);
    dY = dYg;
  }
  if (e == cudaSuccess) e = launch_cast_fp8(dY, T, d, false, 1, gs + 0, dYq, ga + 0, s);
  if (e == cudaSuccess) e = launch_cast_fp8(dY, T, d, true, 1, gs + 0, dYqT, ga + 0, s);
  // the weights as stored, E4M3 with the forward's scales
  if (e == cudaSuccess) e = launch_cast_fp8(A, d, F, false, 0, fs + 1, Aq, fa + 1, s);
  if (e == cudaSuccess) e = launch_cast_fp8(B, F, d, false, 0, fs + 2, Bq, fa + 2, s);
  // dHpre = (dY B^T) * GeLU'(Hpre) in E5M2, and db
  if (e == cudaSuccess) e = do_dh_e5m2(c, dYq, Bq, Hpre, shape, gs + 0, fs + 2, gs + 1, dHq, ga + 1, dbias, colsum, s);
  // K-major copies for the weight gradients (K = T)
  if (e == cudaSuccess) e = launch_transpose_bytes(Hq, T, F, HqT, s);
  if (e == cudaSuccess) e = launch_transpose_bytes(Xq, T, d, XqT, s);
  if (e == cudaSuccess) e = launch_transpose_bytes(dHq, T, F, dHqT, s);
  // dB = H^T dY [F x d]; dA = Xg^T dHpre [d x F]; dXg = dHpre A^T [T x d] (the backward shard sum over K = F)
  if (e == cudaSuccess) e = do_gemm_fp8(c, HqT, 0, dYqT, 1, F, d, T, fs + 3, gs + 0, dB, d, s);
  if (e == cudaSuccess) e = do_gemm_fp8(c, XqT, 0, dHqT, 1, d, F, T, fs + 0, gs + 1, dA, F, s);
  if (e == cudaSuccess) e = do_gemm_fp8(c, dHq, 1, Aq, 0, T, d, F, gs + 1, fs + 1, dXg, d, s);
  if (e == cudaSuccess) e = do_ln_bwd(c, X_chunks, gamma, eps, dXg, shape, dX_chunks, dgamma, dbeta, lnpart, s);
  if (e == cudaSuccess)
    e = launch_fp8_update(grad->scale, grad->amax, grad->history, 2, grad->history_len, 57344.f, grad->margin, s);
  return cuda_status(e);
}

}  // extern "C"
