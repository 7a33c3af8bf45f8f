// csa_api.cu -- host side of the C ABI: context and workspaces, argument validation, the RoPE
// tables, and the layer forward ("DeepSeek V4.1 - Compressed sparse attention", Attention.forward
// excerpt; "metrale_model_arch::attn_v41" AttnV41 and its "Invariants").
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "csa_internal.cuh"

using csa::bf16;

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char *where) {
  return fail(CSA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

#define CSA_CUDA(call, where)                         \
  do {                                                \
    cudaError_t e_ = (call);                          \
    if (e_ != cudaSuccess) return cuda_fail(e_, where); \
  } while (0)

}  // namespace

int csa::set_error(int code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

struct csa_ctx {
  csa_cfg cfg;
  int device = 0;
  int num_sms = 0;
  int max_nt = 0;
  int tab_rows = 0;
  float *tab_plain = nullptr, *tab_comp = nullptr;
  bf16 *qr_raw = nullptr, *qr = nullptr, *q = nullptr, *kv_raw = nullptr, *kv = nullptr, *qI = nullptr,
       *iw_raw = nullptr, *o = nullptr, *o_rot = nullptr, *og = nullptr, *x_stage = nullptr, *out_stage = nullptr;
  float *wI = nullptr, *scores = nullptr;
  float *xpart = nullptr;  // split-K partials of the x projections [S][NT][q_rank + hd + Hi]
  int xpart_rows = 0;
  int32_t *idx_win = nullptr;
  int *status = nullptr;
  float *ws = nullptr;  // Stream-K counters and partials, the attention's split shares, the compressor's partials
  size_t ws_bytes = 0;
  size_t gemm_ws_bytes() const { return ws_bytes; }
  // the compressor's partial products: past the projections' arrival counters, which must stay zero
  float *comp_ws() const { return ws + csa::kGemmCounterBytes / sizeof(float); }
  size_t comp_ws_bytes() const { return ws_bytes - csa::kGemmCounterBytes; }
  int scores_stride = 0;
  size_t bytes = 0;
  std::vector<void *> allocs;
  // tracing: one event pair per stage of the last forward (mode 1) or of every forward since
  // tracing was enabled (mode 2), when enabled
  static constexpr int kTraceStages = 64;
  struct Stage {
    const char *name;
    cudaEvent_t a, b;
  };
  int trace = 0;
  std::vector<Stage> stages;
  int n_stages = 0;
  int launches = 0;

  template <class T>
  cudaError_t alloc(T **p, size_t n) {
    void *v = nullptr;
    size_t b = n * sizeof(T);
    if (b == 0) b = 16;
    cudaError_t e = cudaMalloc(&v, b);
    if (e != cudaSuccess) return e;
    allocs.push_back(v);
    bytes += b;
    *p = static_cast<T *>(v);
    return cudaSuccess;
  }
  void release() {
    for (void *p : allocs) cudaFree(p);
    allocs.clear();
    for (auto &st : stages) {
      cudaEventDestroy(st.a);
      cudaEventDestroy(st.b);
    }
    stages.clear();
  }
};

namespace {

// A context's workspaces live on the device that was current at csa_create: the calls that launch
// work with them, or wait for it, must find that device current.
int check_device(const csa_ctx *ctx, const char *where) {
  int dev = -1;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, where);
  if (dev != ctx->device)
    return fail(CSA_ERR_ARG, "%s: the context lives on device %d, the current device is %d", where, ctx->device, dev);
  return CSA_OK;
}

}  // namespace

namespace csa {

// RoPE table, "deepseek_v41_ref::attn" freqs_cis: [max_seq][rd/2] of (cos, sin) with pair i at
// frequency theta^(-2i/rd), angle p * f_i, taken in double and rounded to f32.  With YaRN
// (Peng et al., 2023, frequency interpolation by parts) when max_seq exceeds the original length:
// pairs that complete more than beta_fast turns over the original length keep f_i, those with
// fewer than beta_slow turns use f_i / factor, with a linear ramp over the pair index between
// floor(d(beta_fast)) and ceil(d(beta_slow)), d(n) = rd ln(L / (2 pi n)) / (2 ln theta).
void build_rope_table(int rd, int max_seq, double theta, int orig_seq, double factor, double beta_fast,
                      double beta_slow, float *tab) {
  const int half = rd / 2;
  std::vector<double> f(half);
  for (int i = 0; i < half; ++i) f[i] = std::pow(theta, -2.0 * i / (double)rd);
  if (orig_seq > 0 && max_seq > orig_seq) {
    const double two_pi = 2.0 * 3.14159265358979323846264338327950288;
    auto turns_to_index = [&](double n) { return rd * std::log(orig_seq / (two_pi * n)) / (2.0 * std::log(theta)); };
    double lo = std::max(std::floor(turns_to_index(beta_fast)), 0.0);
    double hi = std::min(std::ceil(turns_to_index(beta_slow)), (double)(rd - 1));
    if (hi == lo) hi += 0.001;
    for (int i = 0; i < half; ++i) {
      const double ramp = std::min(std::max((i - lo) / (hi - lo), 0.0), 1.0);
      f[i] = f[i] * (1.0 - ramp) + f[i] / factor * ramp;
    }
  }
  for (int64_t p = 0; p < max_seq; ++p)
    for (int i = 0; i < half; ++i) {
      const double a = (double)p * f[i];
      tab[(p * half + i) * 2] = (float)std::cos(a);
      tab[(p * half + i) * 2 + 1] = (float)std::sin(a);
    }
}

}  // namespace csa

extern "C" {

const char *attn_v41_last_error(void) { return g_err; }

static int check_cfg(const csa_cfg *c) {
  if (!c) return fail(CSA_ERR_ARG, "cfg is NULL");
  if (c->dim <= 0 || c->n_heads <= 0 || c->head_dim <= 0 || c->q_rank <= 0 || c->o_rank <= 0 || c->groups <= 0 ||
      c->window <= 0 || c->max_seq <= 0 || c->max_tokens <= 0 || c->max_batch <= 0)
    return fail(CSA_ERR_ARG, "cfg: non-positive dimension");
  if (c->head_dim % 64 != 0 || c->head_dim > 1024) return fail(CSA_ERR_ARG, "cfg: head_dim must be a multiple of 64, <= 1024");
  if (c->rope_dim <= 0 || c->rope_dim % 2 || c->rope_dim > c->head_dim || (c->head_dim - c->rope_dim) % 2)
    return fail(CSA_ERR_ARG, "cfg: rope_dim must be even and <= head_dim");
  if ((c->n_heads * c->head_dim) % c->groups) return fail(CSA_ERR_ARG, "cfg: groups must divide n_heads*head_dim");
  if (c->index_heads < 0 || c->index_hd < 0 || c->index_topk < 0) return fail(CSA_ERR_ARG, "cfg: negative indexer size");
  if (c->index_heads > 0 && c->index_hd != 32 && c->index_hd != 64 && c->index_hd != 128)
    return fail(CSA_ERR_ARG, "cfg: index_hd must be 32, 64 or 128");
  if (c->index_topk > 2048) return fail(CSA_ERR_ARG, "cfg: index_topk above 2048");
  if (c->cand_block <= 0) return fail(CSA_ERR_ARG, "cfg: cand_block must be positive");
  return CSA_OK;
}

int csa_create(const csa_cfg *cfg, csa_ctx **out) {
  if (!out) return fail(CSA_ERR_ARG, "out is NULL");
  *out = nullptr;
  int rc = check_cfg(cfg);
  if (rc) return rc;
  csa_ctx *c = new (std::nothrow) csa_ctx();
  if (!c) return fail(CSA_ERR_NOMEM, "host allocation failed");
  c->cfg = *cfg;
  cudaError_t e = cudaGetDevice(&c->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
  if (e != cudaSuccess) {
    delete c;
    return cuda_fail(e, "csa_create: device query");
  }
  const csa_cfg &g = *cfg;
  const size_t nt = (size_t)g.max_batch * g.max_tokens;
  c->max_nt = (int)nt;
  const size_t H = g.n_heads, hd = g.head_dim;
  const size_t Hi = g.index_heads, dI = g.index_hd;
  c->tab_rows = g.max_seq;
  c->scores_stride = g.max_seq;
  const size_t tab_n = (size_t)g.max_seq * g.rope_dim;
  c->ws_bytes = (size_t)128 << 20;
#define ALLOC(ptr, n)                                            \
  if (e == cudaSuccess) e = c->alloc(&c->ptr, (n));
  ALLOC(tab_plain, tab_n);
  ALLOC(tab_comp, tab_n);
  ALLOC(qr_raw, nt * g.q_rank);
  ALLOC(qr, nt * g.q_rank);
  ALLOC(q, nt * H * hd);
  ALLOC(kv_raw, nt * hd);
  ALLOC(kv, nt * hd);
  ALLOC(qI, nt * Hi * dI);
  ALLOC(iw_raw, nt * Hi);
  ALLOC(wI, nt * Hi);
  ALLOC(scores, nt * (size_t)c->scores_stride);
  ALLOC(idx_win, nt * (size_t)g.window);
  c->xpart_rows = (int)std::max<size_t>(nt, 16 * std::min<size_t>(nt, 256));
  ALLOC(xpart, (size_t)c->xpart_rows * (g.q_rank + g.head_dim + g.index_heads));
  ALLOC(o, nt * H * hd);
  ALLOC(o_rot, nt * H * hd);
  ALLOC(og, nt * (size_t)g.groups * g.o_rank);
  ALLOC(x_stage, nt * g.dim);
  ALLOC(out_stage, nt * g.dim);
  ALLOC(status, 4);
  {
    float *w = nullptr;
    if (e == cudaSuccess) e = c->alloc(&w, c->ws_bytes / sizeof(float));
    c->ws = w;
  }
#undef ALLOC
  if (e == cudaSuccess) e = cudaMemset(c->status, 0, 4 * sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(c->ws, 0, csa::kGemmCounterBytes);  // Stream-K arrival counters
  if (e != cudaSuccess) {
    c->release();
    delete c;
    return fail(CSA_ERR_NOMEM, "csa_create: workspace allocation: %s", cudaGetErrorString(e));
  }
  std::vector<float> tab(tab_n);
  csa::build_rope_table(g.rope_dim, g.max_seq, g.rope_theta, 0, 1.0, g.beta_fast, g.beta_slow, tab.data());
  e = cudaMemcpy(c->tab_plain, tab.data(), tab_n * sizeof(float), cudaMemcpyHostToDevice);
  csa::build_rope_table(g.rope_dim, g.max_seq, g.compress_rope_theta, g.orig_seq, g.rope_factor, g.beta_fast,
                        g.beta_slow, tab.data());
  if (e == cudaSuccess) e = cudaMemcpy(c->tab_comp, tab.data(), tab_n * sizeof(float), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    c->release();
    delete c;
    return cuda_fail(e, "csa_create: table upload");
  }
  *out = c;
  return CSA_OK;
}

int csa_destroy(csa_ctx *ctx) {
  if (!ctx) return CSA_OK;
  // wait for and free on the context's own device, then give the caller back its current device
  int cur = -1;
  const bool other = cudaGetDevice(&cur) == cudaSuccess && cur != ctx->device;
  if (other) cudaSetDevice(ctx->device);
  cudaDeviceSynchronize();
  ctx->release();
  if (other) cudaSetDevice(cur);
  delete ctx;
  return CSA_OK;
}

size_t csa_workspace_bytes(const csa_ctx *ctx) { return ctx ? ctx->bytes : 0; }

int csa_trace_enable(csa_ctx *ctx, int enable) {
  constexpr int kTraceStages = csa_ctx::kTraceStages;
  if (!ctx) return fail(CSA_ERR_ARG, "csa_trace_enable: NULL context");
  if (int rc = check_device(ctx, "csa_trace_enable")) return rc;
  if (enable && ctx->stages.empty()) {
    ctx->stages.resize(kTraceStages);
    for (auto &st : ctx->stages) {
      CSA_CUDA(cudaEventCreate(&st.a), "csa_trace_enable");
      CSA_CUDA(cudaEventCreate(&st.b), "csa_trace_enable");
    }
  }
  ctx->trace = enable == 2 ? 2 : (enable ? 1 : 0);
  ctx->n_stages = 0;
  return CSA_OK;
}

int csa_trace_read(csa_ctx *ctx, int max, const char **names, float *ms) {
  if (!ctx || (max > 0 && (!names || !ms))) return fail(CSA_ERR_ARG, "csa_trace_read: bad argument");
  const int n = std::min(max, ctx->n_stages);
  for (int i = 0; i < n; ++i) {
    CSA_CUDA(cudaEventSynchronize(ctx->stages[i].b), "csa_trace_read");
    names[i] = ctx->stages[i].name;
    CSA_CUDA(cudaEventElapsedTime(&ms[i], ctx->stages[i].a, ctx->stages[i].b), "csa_trace_read");
  }
  return ctx->n_stages;
}

int csa_last_launches(const csa_ctx *ctx) { return ctx ? ctx->launches : 0; }

int csa_rope_table_get(const csa_ctx *ctx, int ratio_class, float *tab_host) {
  if (!ctx || !tab_host) return fail(CSA_ERR_ARG, "csa_rope_table_get: NULL argument");
  const float *src = ratio_class ? ctx->tab_comp : ctx->tab_plain;
  CSA_CUDA(cudaMemcpy(tab_host, src, sizeof(float) * (size_t)ctx->tab_rows * ctx->cfg.rope_dim, cudaMemcpyDeviceToHost),
           "csa_rope_table_get");
  return CSA_OK;
}

int csa_status(csa_ctx *ctx, int clear) {
  if (!ctx) return fail(CSA_ERR_ARG, "csa_status: NULL context");
  if (int rc = check_device(ctx, "csa_status")) return rc;
  int st = 0;
  CSA_CUDA(cudaDeviceSynchronize(), "csa_status: synchronize");
  CSA_CUDA(cudaMemcpy(&st, ctx->status, sizeof(int), cudaMemcpyDeviceToHost), "csa_status: read");
  if (clear) {
    CSA_CUDA(cudaMemset(ctx->status, 0, sizeof(int)), "csa_status: clear");
    // a projection that gave up may have left Stream-K arrival counters raised: start them at zero
    if (st & csa::kStatusTimeout) CSA_CUDA(cudaMemset(ctx->ws, 0, csa::kGemmCounterBytes), "csa_status: counters");
    CSA_CUDA(cudaDeviceSynchronize(), "csa_status: clear");
  }
  if (st & csa::kStatusTimeout) return fail(CSA_ERR_DEVICE_TIMEOUT, "a bounded device-side wait ran out");
  if (st & csa::kStatusBadIndex) return fail(CSA_ERR_ARG, "a selection index was outside [-1, rows)");
  return CSA_OK;
}

int csa_debug_stall(unsigned long long ns) {
  CSA_CUDA(csa::set_gemm_stall(ns), "csa_debug_stall");
  return CSA_OK;
}

int csa_state_init(csa_ctx *ctx, csa_layer_state *state, int batch, csa_stream stream) {
  if (!ctx || !state || !state->window) return fail(CSA_ERR_ARG, "csa_state_init: NULL argument");
  if (batch <= 0 || batch > ctx->cfg.max_batch) return fail(CSA_ERR_SHAPE, "csa_state_init: batch %d", batch);
  if ((state->comp_kv || state->comp_score) && (!state->comp_kv || !state->comp_score || state->comp_ratio <= 0))
    return fail(CSA_ERR_ARG, "csa_state_init: a compressor state needs comp_kv, comp_score and comp_ratio");
  if (int rc = check_device(ctx, "csa_state_init")) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  CSA_CUDA(cudaMemsetAsync(state->window, 0, sizeof(bf16) * (size_t)batch * ctx->cfg.window * ctx->cfg.head_dim, s),
           "csa_state_init");
  if (state->comp_kv) {
    const int64_t n = (int64_t)batch * state->comp_ratio * ctx->cfg.head_dim;
    CSA_CUDA(cudaMemsetAsync(state->comp_kv, 0, sizeof(float) * (size_t)n, s), "csa_state_init");
    CSA_CUDA(csa::launch_fill_f32(state->comp_score, n, -INFINITY, s), "csa_state_init");
  }
  return CSA_OK;
}

// The compressor's arguments of a kv-source layer (validated); CSA_OK or an error code.
static int compress_args(const csa_ctx *ctx, const csa_layer_weights *w, const csa_layer_state *st, const void *x,
                         int B, int T, int start_pos, csa_bf16 *y_dbg, csa::CompressArgs *a, const char *who) {
  const csa_cfg &g = ctx->cfg;
  const int ratio = w->role.ratio;
  if (ratio < 1 || ratio > 16) return fail(CSA_ERR_ARG, "%s: a kv source needs a ratio in 1..16", who);
  if (!w->comp_wkv || !w->comp_norm || (ratio > 1 && !w->comp_wgate))
    return fail(CSA_ERR_ARG, "%s: compressor weights missing", who);
  if (w->idx_wk && (!w->idx_k_norm || g.index_hd <= 0 || g.index_hd > 256))
    return fail(CSA_ERR_ARG, "%s: index-key weights need idx_k_norm and index_hd in 1..256", who);
  if (!st->comp_kv || !st->comp_score || st->comp_ratio != ratio || !st->latent || (w->idx_wk && !st->index_keys))
    return fail(CSA_ERR_ARG, "%s: the state lacks the compressor's partial group or caches for ratio %d", who, ratio);
  if (B <= 0 || B > g.max_batch || T <= 0 || T > g.max_tokens || start_pos < 0 || (int64_t)start_pos + T > g.max_seq)
    return fail(CSA_ERR_SHAPE, "%s: batch %d, T %d at %d", who, B, T, start_pos);
  if (start_pos > 0 && T != 1) return fail(CSA_ERR_SHAPE, "%s: decode takes one token per sequence", who);
  if ((start_pos + T) / ratio > st->cache_rows)
    return fail(CSA_ERR_SHAPE, "%s: cache_rows %d below the groups written", who, st->cache_rows);
  a->x = (const bf16 *)x;
  a->B = B;
  a->T = T;
  a->start_pos = start_pos;
  a->ratio = ratio;
  a->dim = g.dim;
  a->hd = g.head_dim;
  a->rd = g.rope_dim;
  a->dI = g.index_hd;
  a->wkv = w->comp_wkv;
  a->wgate = w->comp_wgate;
  a->norm = w->comp_norm;
  a->wk = (const bf16 *)w->idx_wk;
  a->k_norm = w->idx_k_norm;
  a->st_kv = st->comp_kv;
  a->st_score = st->comp_score;
  a->Z = (bf16 *)st->latent;
  a->KI = (bf16 *)st->index_keys;
  a->y_dbg = (bf16 *)y_dbg;
  a->Lstride = st->cache_rows;
  a->tab = ctx->tab_comp;
  a->eps = g.eps;
  if (!csa::compress_supported(*a))
    return fail(CSA_ERR_ARG, "%s: head_dim a multiple of 64 (<= 1024), dim of 8, x 16-byte aligned", who);
  return CSA_OK;
}

// A kv source's caches as the shared slots later layers read ([attn_v41] SharedV41: compress_len
// only grows).
static void publish_caches(const csa_layer_weights *w, const csa_layer_state *st, int T, int start_pos,
                           csa_shared *sh) {
  if (!sh) return;
  sh->compress_kv = st->latent;
  if (w->idx_wk) sh->index_k = st->index_keys;
  sh->compress_stride = st->cache_rows;
  sh->compress_len = std::max(sh->compress_len, (start_pos + T) / w->role.ratio);
}

int csa_compress(csa_ctx *ctx, const csa_layer_weights *w, csa_layer_state *st, const csa_bf16 *x, int B, int T,
                 int start_pos, csa_shared *sh, csa_bf16 *y_dbg, csa_stream stream) {
  if (!ctx || !w || !st || !x) return fail(CSA_ERR_ARG, "csa_compress: NULL argument");
  if (int rc = check_device(ctx, "csa_compress")) return rc;
  csa::CompressArgs a;
  if (int rc = compress_args(ctx, w, st, x, B, T, start_pos, y_dbg, &a, "csa_compress")) return rc;
  CSA_CUDA(csa::launch_compress(a, ctx->comp_ws(), ctx->comp_ws_bytes(), ctx->num_sms, (cudaStream_t)stream),
           "csa_compress");
  publish_caches(w, st, T, start_pos, sh);
  return CSA_OK;
}

// ---------------------------------------------------------------------------------------------
// per-step entry points
// ---------------------------------------------------------------------------------------------

int csa_linear(csa_ctx *ctx, const csa_bf16 *x, int M, int K, int ldx, const csa_bf16 *W, int N, int ldw, csa_bf16 *y,
               int ldy, int groups, csa_stream stream) {
  if (!ctx || !x || !W || !y) return fail(CSA_ERR_ARG, "csa_linear: NULL argument");
  if (M < 0 || K <= 0 || N <= 0 || groups <= 0 || ldx < K * groups || ldw < K || ldy < N * groups)
    return fail(CSA_ERR_ARG, "csa_linear: bad shape M=%d K=%d N=%d groups=%d", M, K, N, groups);
  if (int rc = check_device(ctx, "csa_linear")) return rc;
  csa::LinearProblem pr{(const bf16 *)x, M, K, ldx, (const bf16 *)W, N, ldw, (bf16 *)y, ldy, groups};
  int kernels = 0;  // (counted, so that a paired launch may split its last wave)
  CSA_CUDA(csa::launch_linear(&pr, 1, ctx->ws, ctx->gemm_ws_bytes(), ctx->num_sms, ctx->status, (cudaStream_t)stream,
                              &kernels),
           "csa_linear");
  return CSA_OK;
}

int csa_linear_fp8w(csa_ctx *ctx, const csa_bf16 *x, int M, int K, int ldx, const uint8_t *W8, const float *scale,
                    int N, int ldw8, csa_bf16 *y, int ldy, int groups, csa_stream stream) {
  if (!ctx || !x || !W8 || !scale || !y) return fail(CSA_ERR_ARG, "csa_linear_fp8w: NULL argument");
  if (M < 0 || K <= 0 || N <= 0 || groups <= 0 || ldx < K * groups || ldw8 < K || ldy < N * groups)
    return fail(CSA_ERR_ARG, "csa_linear_fp8w: bad shape M=%d K=%d N=%d groups=%d", M, K, N, groups);
  if (int rc = check_device(ctx, "csa_linear_fp8w")) return rc;
  csa::LinearProblem pr{(const bf16 *)x, M, K, ldx, nullptr, N, ldw8, (bf16 *)y, ldy, groups};
  pr.W8 = W8;
  pr.w8_scale = scale;
  if (M == 0) return CSA_OK;
  if (!csa::gemm_tc_supported(pr))
    return fail(CSA_ERR_ARG, "csa_linear_fp8w: x and W8 16-byte aligned, ldx a multiple of 8, ldw8 and K of 16 "
                             "(K of 64 with groups)");
  CSA_CUDA(csa::launch_linear(&pr, 1, ctx->ws, ctx->gemm_ws_bytes(), ctx->num_sms, ctx->status, (cudaStream_t)stream),
           "csa_linear_fp8w");
  return CSA_OK;
}

int csa_rmsnorm(const csa_bf16 *x, int M, int N, const float *w, float eps, csa_bf16 *y, csa_stream stream) {
  if (!x || !w || !y || M < 0 || N <= 0) return fail(CSA_ERR_ARG, "csa_rmsnorm: bad argument");
  CSA_CUDA(csa::launch_rmsnorm((const bf16 *)x, M, N, w, eps, (bf16 *)y, (cudaStream_t)stream), "csa_rmsnorm");
  return CSA_OK;
}

int csa_rope(csa_bf16 *x, int64_t rows, int row_len, int rd, const int32_t *pos, int rows_per_pos, const float *tab,
             int tab_rows, int inverse, csa_stream stream) {
  if (!x || !pos || !tab || rows < 0 || rd <= 0 || rd % 2 || rd > row_len || (row_len - rd) % 2 || rows_per_pos <= 0 ||
      tab_rows <= 0)
    return fail(CSA_ERR_ARG, "csa_rope: bad argument");
  csa::PosSpec ps{pos, 0, 1, rows_per_pos};
  CSA_CUDA(csa::launch_rope((bf16 *)x, rows, row_len, rd, ps, tab, tab_rows, inverse, nullptr, (cudaStream_t)stream),
           "csa_rope");
  return CSA_OK;
}

int csa_act_quant(csa_bf16 *x, int64_t n, uint8_t *codes, int8_t *scale_exp, csa_stream stream) {
  if (!x || n < 0 || n % 32) return fail(CSA_ERR_ARG, "csa_act_quant: n must be a multiple of 32");
  CSA_CUDA(csa::launch_act_quant((bf16 *)x, n, codes, scale_exp, (cudaStream_t)stream), "csa_act_quant");
  return CSA_OK;
}

int csa_kv_finish(const csa_bf16 *kv_in, csa_bf16 *kv_out, int B, int T, int start_pos, int hd, int rd,
                  const float *tab, int tab_rows, csa_bf16 *ring, int W, int32_t *win_idx, int idx_stride,
                  uint8_t *codes, int8_t *scales, csa_stream stream) {
  if (!kv_in || !kv_out || !tab || !ring || B <= 0 || T <= 0 || start_pos < 0 || W <= 0)
    return fail(CSA_ERR_ARG, "csa_kv_finish: bad argument");
  if (hd % 32 || hd > 1024 || rd <= 0 || rd % 2 || rd > hd || (hd - rd) % 2)
    return fail(CSA_ERR_ARG, "csa_kv_finish: hd must be a multiple of 32 (<= 1024), rd even");
  if (start_pos > 0 && T != 1) return fail(CSA_ERR_SHAPE, "csa_kv_finish: decode takes one token per sequence");
  if (start_pos + T > tab_rows) return fail(CSA_ERR_SHAPE, "csa_kv_finish: position beyond the table");
  if (win_idx && idx_stride < W) return fail(CSA_ERR_ARG, "csa_kv_finish: idx_stride < W");
  CSA_CUDA(csa::launch_kv_finish((const bf16 *)kv_in, (bf16 *)kv_out, B, T, start_pos, hd, rd, tab, (bf16 *)ring, W,
                                 win_idx, idx_stride, codes, scales, (cudaStream_t)stream),
           "csa_kv_finish");
  return CSA_OK;
}

int csa_index_scores(const csa_bf16 *qI, const float *wI, const csa_bf16 *KI, int B, int T, int start_pos, int Hi,
                     int dI, int Lstride, int compress_len, int ratio, const uint8_t *cand, int cand_width,
                     int cand_block, float *S, csa_stream stream) {
  if (!qI || !wI || !KI || !S || B <= 0 || T <= 0 || start_pos < 0 || Hi <= 0 || ratio <= 0 || Lstride <= 0 ||
      compress_len < 0 || compress_len > Lstride)
    return fail(CSA_ERR_ARG, "csa_index_scores: bad argument");
  if (dI != 32 && dI != 64 && dI != 128) return fail(CSA_ERR_ARG, "csa_index_scores: dI must be 32, 64 or 128");
  if (cand && (cand_block <= 0 || (int64_t)cand_width * cand_block < compress_len))
    return fail(CSA_ERR_ARG, "csa_index_scores: candidate mask narrower than the cache");
  CSA_CUDA(csa::launch_index_scores((const bf16 *)qI, wI, (const bf16 *)KI, B, T, start_pos, Hi, dI, Lstride,
                                    compress_len, ratio, cand, cand_width, cand_block, S, (cudaStream_t)stream),
           "csa_index_scores");
  return CSA_OK;
}

int csa_candidate_blocks(const float *S, int B, int T, int start_pos, int Lstride, int compress_len, int ratio,
                         int cand_block, int K, uint8_t *mask, int cand_width, csa_stream stream) {
  if (!S || !mask || B <= 0 || T <= 0 || start_pos < 0 || ratio <= 0 || Lstride <= 0 || compress_len < 0 ||
      compress_len > Lstride || cand_block <= 0 || K <= 0 || K > 2048 || cand_width <= 0 || cand_width > 25600)
    return fail(CSA_ERR_ARG, "csa_candidate_blocks: bad argument");
  if ((int64_t)cand_width * cand_block < compress_len)
    return fail(CSA_ERR_ARG, "csa_candidate_blocks: the mask is narrower than the cache");
  CSA_CUDA(csa::launch_cand_blocks(S, B, T, start_pos, Lstride, compress_len, ratio, cand_block, K, mask, cand_width,
                                   (cudaStream_t)stream),
           "csa_candidate_blocks");
  return CSA_OK;
}

int csa_index_topk(const float *S, int B, int T, int start_pos, int Lstride, int compress_len, int ratio,
                   const uint8_t *cand, int cand_width, int cand_block, int K, int offset, int32_t *out,
                   csa_stream stream) {
  if (!S || !out || B <= 0 || T <= 0 || start_pos < 0 || ratio <= 0 || Lstride <= 0 || compress_len < 0 ||
      compress_len > Lstride || K <= 0 || K > 2048)
    return fail(CSA_ERR_ARG, "csa_index_topk: bad argument");
  if (cand && (cand_block <= 0 || (int64_t)cand_width * cand_block < compress_len))
    return fail(CSA_ERR_ARG, "csa_index_topk: candidate mask narrower than the cache");
  CSA_CUDA(csa::launch_index_topk(S, B, T, start_pos, Lstride, compress_len, ratio, cand, cand_width, cand_block, K,
                                  offset, out, (cudaStream_t)stream),
           "csa_index_topk");
  return CSA_OK;
}

int csa_sparse_attn(csa_ctx *ctx, const csa_bf16 *q, int B, int T, int H, int hd, const csa_bf16 *rows_a,
                    int64_t a_seq_stride, int a_len, const csa_bf16 *rows_b, int64_t b_seq_stride, int b_len,
                    const int32_t *idx_a, int na, const int32_t *idx_b, int nb, const float *sink, float scale,
                    csa_bf16 *o, csa_bf16 *o_rot, int rd, int start_pos, const float *tab, int tab_rows,
                    csa_stream stream) {
  if (!ctx || !q || !rows_a || !idx_a || !sink || B <= 0 || T <= 0 || H <= 0 || a_len < 0 || b_len < 0 || na < 0 ||
      nb < 0)
    return fail(CSA_ERR_ARG, "csa_sparse_attn: bad argument");
  if (hd % 64 || hd > 1024) return fail(CSA_ERR_ARG, "csa_sparse_attn: hd must be a multiple of 64, <= 1024");
  if (nb > 0 && (!idx_b)) return fail(CSA_ERR_ARG, "csa_sparse_attn: idx_b is NULL");
  if (b_len > 0 && !rows_b) return fail(CSA_ERR_ARG, "csa_sparse_attn: rows_b is NULL");
  if (na + nb > 2048) return fail(CSA_ERR_TOO_WIDE, "csa_sparse_attn: selection of %d rows above 2048", na + nb);
  if ((int64_t)a_len * hd > a_seq_stride && B > 1) return fail(CSA_ERR_ARG, "csa_sparse_attn: a_len rows exceed a_seq_stride");
  if ((int64_t)b_len * hd > b_seq_stride && B > 1 && b_len > 0)
    return fail(CSA_ERR_ARG, "csa_sparse_attn: b_len rows exceed b_seq_stride");
  if (a_seq_stride % hd || (b_len > 0 && b_seq_stride % hd))
    return fail(CSA_ERR_ARG, "csa_sparse_attn: sequence strides must be whole rows");
  if (o_rot && (!tab || rd <= 0 || rd % 2 || rd > hd || start_pos < 0 || start_pos + T > tab_rows))
    return fail(CSA_ERR_ARG, "csa_sparse_attn: inverse rotation needs a table covering the positions");
  if (int rc = check_device(ctx, "csa_sparse_attn")) return rc;
  csa::AttnArgs a{(const bf16 *)q, B, T, H, hd, (const bf16 *)rows_a, a_seq_stride, a_len, (const bf16 *)rows_b,
                  b_seq_stride, b_len, idx_a, na, idx_b, nb, sink, scale, (bf16 *)o, (bf16 *)o_rot, rd, start_pos,
                  tab, ctx->status};
  CSA_CUDA(csa::launch_sparse_attn(a, ctx->ws, ctx->ws_bytes, ctx->num_sms, (cudaStream_t)stream), "csa_sparse_attn");
  return CSA_OK;
}

// ---------------------------------------------------------------------------------------------
// the layer
// ---------------------------------------------------------------------------------------------

static int check_forward(const csa_ctx *ctx, const csa_layer_weights *w, const csa_layer_state *st, const void *x,
                         int B, int T, int start_pos, const csa_shared *sh, const void *out) {
  if (!ctx || !w || !st || !st->window || !x || !out) return fail(CSA_ERR_ARG, "attn_v41_forward: NULL argument");
  if (int rc = check_device(ctx, "attn_v41_forward")) return rc;
  const csa_cfg &g = ctx->cfg;
  const csa_role &r = w->role;
  if (!w->sink || !w->q_norm || !w->kv_norm || !w->wq_a || !w->wq_b || !w->wkv || !w->wo_b ||
      (!w->wo_a && !w->wo_a_fp8))
    return fail(CSA_ERR_ARG, "attn_v41_forward: a weight pointer is NULL");
  if (w->wo_a_fp8) {
    const int gw = g.n_heads * g.head_dim / g.groups;
    if (!w->wo_a_scale || ((uintptr_t)w->wo_a_fp8 & 15) || gw % 64)
      return fail(CSA_ERR_ARG, "attn_v41_forward: fp8 wo_a needs its scales, 16-byte alignment and gw a multiple of 64");
  }
  if (r.ratio < 0) return fail(CSA_ERR_ARG, "attn_v41_forward: negative ratio");
  {
    const void *al[] = {x, out, w->wq_a, w->wq_b, w->wkv, w->wo_a, w->wo_b, w->idx_wq_b, w->idx_wproj};
    for (const void *p : al)
      if ((uintptr_t)p & 15) return fail(CSA_ERR_ARG, "attn_v41_forward: tensors must be 16-byte aligned");
    if (g.dim % 8 || g.q_rank % 8 || g.o_rank % 8 || (g.n_heads * g.head_dim / g.groups) % 64)
      return fail(CSA_ERR_ARG, "attn_v41_forward: dim, q_rank, o_rank must be multiples of 8, the group width of 64");
  }
  if (r.is_candidate_source) {
    if (r.ratio <= 0 || !r.is_index_source || r.uses_candidates)
      return fail(CSA_ERR_ARG, "attn_v41_forward: a candidate source is an index source at ratio > 0 that applies no mask");
    if (!sh || !sh->candidates || g.cand_topk_blocks <= 0 || g.cand_topk_blocks > 2048 || sh->cand_width > 25600)
      return fail(CSA_ERR_ARG, "attn_v41_forward: a candidate source needs shared->candidates and cand_topk_blocks in 1..2048");
  }
  if (r.is_kv_source) {
    if (r.ratio <= 0) return fail(CSA_ERR_ARG, "attn_v41_forward: a kv source compresses at ratio > 0");
    if (!sh) return fail(CSA_ERR_ARG, "attn_v41_forward: a kv source publishes through shared, which is NULL");
    csa::CompressArgs a;
    if (int rc = compress_args(ctx, w, st, x, B, T, start_pos, nullptr, &a, "attn_v41_forward")) return rc;
  }
  if (B <= 0 || B > g.max_batch) return fail(CSA_ERR_SHAPE, "attn_v41_forward: batch %d outside [1, %d]", B, g.max_batch);
  if (T <= 0 || T > g.max_tokens) return fail(CSA_ERR_SHAPE, "attn_v41_forward: T %d outside [1, %d]", T, g.max_tokens);
  if (start_pos < 0 || (int64_t)start_pos + T > g.max_seq)
    return fail(CSA_ERR_SHAPE, "attn_v41_forward: positions [%d, %d) beyond max_seq %d", start_pos, start_pos + T, g.max_seq);
  if (start_pos > 0 && T != 1) return fail(CSA_ERR_SHAPE, "attn_v41_forward: decode takes one token per sequence");
  csa_shared pub;  // a kv source publishes its own caches before it attends
  if (r.ratio > 0 && r.is_kv_source && sh) {
    pub = *sh;
    publish_caches(w, st, T, start_pos, &pub);
    sh = &pub;
  }
  if (r.ratio > 0) {
    if (!sh || !sh->compress_kv) return fail(CSA_ERR_NO_KV_SOURCE, "attn_v41_forward: ratio > 0 and no latent cache published");
    if (sh->compress_len < 0 || sh->compress_stride < sh->compress_len || sh->compress_stride <= 0)
      return fail(CSA_ERR_ARG, "attn_v41_forward: compress_len / compress_stride");
    if (!sh->topk_idxs) return fail(CSA_ERR_ARG, "attn_v41_forward: shared topk_idxs buffer is NULL");
    if (sh->topk != g.index_topk) return fail(CSA_ERR_ARG, "attn_v41_forward: shared topk %d != index_topk %d", sh->topk, g.index_topk);
    const int width = g.window + g.index_topk;
    if (width > 2048) return fail(CSA_ERR_TOO_WIDE, "attn_v41_forward: selection of %d rows above 2048", width);
    if (r.is_index_source) {
      if (!w->idx_wq_b || !w->idx_wproj) return fail(CSA_ERR_ARG, "attn_v41_forward: index source without indexer weights");
      if (!sh->index_k) return fail(CSA_ERR_NO_KV_SOURCE, "attn_v41_forward: index source and no index keys published");
      if (g.index_heads <= 0) return fail(CSA_ERR_ARG, "attn_v41_forward: cfg has no indexer");
      if (sh->compress_stride > ctx->scores_stride) return fail(CSA_ERR_SHAPE, "attn_v41_forward: compress_stride above max_seq");
      if (r.uses_candidates && (!sh->candidates || (int64_t)sh->cand_width * g.cand_block < sh->compress_len))
        return fail(CSA_ERR_ARG, "attn_v41_forward: candidate mask missing or narrower than the cache");
    } else if (!sh->has_topk) {
      return fail(CSA_ERR_NO_SELECTION, "attn_v41_forward: reuse layer and no selection published");
    }
  }
  return CSA_OK;
}

int attn_v41_forward(csa_ctx *ctx, const csa_layer_weights *w, csa_layer_state *st, const csa_bf16 *x_, int B, int T,
                     int start_pos, csa_shared *sh, csa_bf16 *out_, const csa_debug *dbg, csa_stream stream_) {
  int rc = check_forward(ctx, w, st, x_, B, T, start_pos, sh, out_);
  if (rc) return rc;
  const csa_cfg &g = ctx->cfg;
  const csa_role &r = w->role;
  cudaStream_t s = (cudaStream_t)stream_;
  const bf16 *x = (const bf16 *)x_;
  bf16 *out = (bf16 *)out_;
  const int NT = B * T, H = g.n_heads, hd = g.head_dim, rd = g.rope_dim, W = g.window;
  const int G = g.groups, gw = H * hd / G;
  const bool decode = start_pos > 0;
  const float *tab = r.ratio > 0 ? ctx->tab_comp : ctx->tab_plain;
  const csa::PosSpec pos_q{nullptr, start_pos, T, H};
  bf16 *q = dbg && dbg->q ? (bf16 *)dbg->q : ctx->q;
  bf16 *kv = dbg && dbg->kv ? (bf16 *)dbg->kv : ctx->kv;
  bf16 *qr = dbg && dbg->qr ? (bf16 *)dbg->qr : ctx->qr;
  bf16 *o = dbg && dbg->o ? (bf16 *)dbg->o : nullptr;
  bf16 *og = dbg && dbg->og ? (bf16 *)dbg->og : ctx->og;
  int32_t *win_idx = ctx->idx_win;
  int idx_stride = W;
  if (dbg && dbg->idx) {
    win_idx = dbg->idx;
    idx_stride = W + (r.ratio > 0 ? g.index_topk : 0);
  }
  if (ctx->trace != 2) ctx->n_stages = 0;
  ctx->launches = 0;
  // while the stream is being captured, a traced stage's events become event-record nodes of the
  // graph; outside a capture they are plain records
  unsigned ev_flags = cudaEventRecordDefault;
  if (ctx->trace) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
      ev_flags = cudaEventRecordExternal;
  }
  // one traced stage: events around it when tracing is on (recorded as event nodes when the stream
  // is being captured, so a replayed graph times its stages too); counts the kernels it launches
#define STAGE(call, what, kernels)                                                             \
  do {                                                                                         \
    csa_ctx::Stage *st_ = nullptr;                                                             \
    if (ctx->trace && ctx->n_stages < (int)ctx->stages.size()) {                               \
      st_ = &ctx->stages[ctx->n_stages++];                                                     \
      st_->name = what;                                                                        \
      cudaEventRecordWithFlags(st_->a, s, ev_flags);                                           \
    }                                                                                          \
    cudaError_t e_ = (call);                                                                   \
    if (e_ != cudaSuccess) return cuda_fail(e_, what);                                         \
    if (st_) cudaEventRecordWithFlags(st_->b, s, ev_flags);                                    \
    ctx->launches += (kernels);                                                                \
  } while (0)
#define STEP(call, what) STAGE(call, what, 1)
#define COPY(call, what) STAGE(call, what, 0)
  // a kv source first compresses this call's tokens and publishes its caches ([atlas] the excerpt's
  // _compress_kv precedes the selection and the attention)
  if (r.is_kv_source) {
    csa::CompressArgs ca;
    if (int rc2 = compress_args(ctx, w, st, x_, B, T, start_pos, nullptr, &ca, "attn_v41_forward")) return rc2;
    STAGE(csa::launch_compress(ca, ctx->comp_ws(), ctx->comp_ws_bytes(), ctx->num_sms, s), "compress", 2);
    publish_caches(w, st, T, start_pos, sh);
  }
  const bool idx_src = r.ratio > 0 && r.is_index_source;
  const int Hi = g.index_heads, dI = g.index_hd;
  bf16 *qI = dbg && dbg->qI ? (bf16 *)dbg->qI : ctx->qI;
  auto lin = [&](const bf16 *xx, int K, int ldx, const csa_bf16 *Wt, int N, bf16 *y, int ldy, int groups) {
    return csa::LinearProblem{xx, NT, K, ldx, (const bf16 *)Wt, N, K, y, ldy, groups};
  };
  // projections of x: wq_a, wkv and (index sources) the indexer's head weights, one split-K launch
  // writing f32 partials; one fused kernel reduces them into qr (RMSNorm), the window row (RMSNorm,
  // RoPE, fp8, ring, window selection) and w^I
  const int ldp = g.q_rank + hd + (idx_src ? Hi : 0);
  float *wI = dbg && dbg->wI ? dbg->wI : ctx->wI;
  {
    csa::LinearProblem px[3] = {lin(x, g.dim, g.dim, w->wq_a, g.q_rank, nullptr, 0, 1),
                                lin(x, g.dim, g.dim, w->wkv, hd, nullptr, 0, 1),
                                lin(x, g.dim, g.dim, w->idx_wproj, Hi, nullptr, 0, 1)};
    px[0].part = ctx->xpart;
    px[1].part = ctx->xpart + g.q_rank;
    px[2].part = ctx->xpart + g.q_rank + hd;
    for (auto &p : px) p.ldp = ldp;
    const int np = idx_src ? 3 : 2;
    const int S = csa::gemm_tc_split_count(px, np, ctx->num_sms, std::max(1, ctx->xpart_rows / NT));
    // x finish, next, is a programmatic dependent that reads the slices only after its dependency wait
    for (int i = 0; i < np; ++i) px[i].early_dependents = 1;
    // and it is itself one of the kernel before (the layer's input is read after the wait)
    for (int i = 0; i < np; ++i) px[i].pdl = 1;
    // many tokens and one slice: the paired-CTA kernel writes the f32 slice itself
    bool paired = S == 1 && NT >= 2048;
    for (int i = 0; i < np; ++i) paired = paired && csa::gemm_tc_supported(px[i]);
    if (paired)
      STEP(csa::launch_gemm_tc(px, np, ctx->ws, ctx->gemm_ws_bytes(), ctx->num_sms, ctx->status, s), "proj x");
    else
      STEP(csa::launch_gemm_tc_split(px, np, S, ctx->status, s), "proj x");
    csa::XFinishArgs xa{ctx->xpart, S, ldp, g.q_rank, hd, idx_src ? Hi : 0, w->q_norm, w->kv_norm, g.eps, qr, kv, B,
                        T, start_pos, rd, tab, (bf16 *)st->window, W, win_idx, idx_stride,
                        dbg ? dbg->kv_codes : nullptr, dbg ? dbg->kv_scale : nullptr,
                        (float)(1.0 / std::sqrt((double)dI * std::max(Hi, 1))), wI};
    STEP(csa::launch_x_finish(xa, s), "x finish");
  }
  // a decode row's selection in one kernel (the fused indexer + top-k, or its cluster form for long
  // rows under a mask) is a programmatic dependent that reads proj qr's output only after its
  // dependency wait: proj qr lets it start early
  const int K_sel = r.ratio > 0 ? g.index_topk : 0;
  const bool fused_sel =
      r.ratio > 0 && r.is_index_source && !(dbg && dbg->scores) && !r.is_candidate_source &&
      (csa::index_fused_supported(qI, (const bf16 *)sh->index_k, T, start_pos, Hi, dI, sh->compress_len, r.ratio,
                                  K_sel) ||
       csa::index_gather_topk_supported(qI, (const bf16 *)sh->index_k, B, T, start_pos, Hi, dI, sh->compress_len,
                                        r.ratio, r.uses_candidates ? sh->candidates : nullptr, sh->cand_width,
                                        g.cand_block, K_sel, ctx->num_sms));
  // q path: q = wq_b qr (+ the indexer query q^I = W_IQ qr); RoPE on each head's tail
  {
    csa::LinearProblem pq[2] = {lin(qr, g.q_rank, g.q_rank, w->wq_b, H * hd, q, H * hd, 1),
                                lin(qr, g.q_rank, g.q_rank, w->idx_wq_b, Hi * dI, qI, Hi * dI, 1)};
    pq[0].early_dependents = pq[1].early_dependents = fused_sel ? 1 : 0;
    pq[0].pdl = pq[1].pdl = 1;  // (x finish lets it start early)
    STEP(csa::launch_linear(pq, idx_src ? 2 : 1, ctx->ws, ctx->gemm_ws_bytes(), ctx->num_sms, ctx->status, s), "proj qr");
  }
  // the sparse attention's arguments: the selection's buffers are known before the index stages fill
  // them; rows_a = the window ring at decode, the chunk's own kv rows at prefill
  const int rows_a_len = decode ? W : T;
  const int K = r.ratio > 0 ? g.index_topk : 0;
  csa::AttnArgs a{q, B, T, H, hd,
                  decode ? (const bf16 *)st->window : kv, decode ? (int64_t)W * hd : (int64_t)T * hd, rows_a_len,
                  r.ratio > 0 ? (const bf16 *)sh->compress_kv : nullptr,
                  r.ratio > 0 ? (int64_t)sh->compress_stride * hd : 0, r.ratio > 0 ? sh->compress_len : 0,
                  win_idx, W, r.ratio > 0 ? sh->topk_idxs : nullptr, K, w->sink, (float)(1.0 / std::sqrt((double)hd)),
                  o, ctx->o_rot, rd, start_pos, tab, ctx->status};
  // RoPE on q: inside the tensor-core attention kernel (on its own copy of q), unless the caller wants
  // the turned q itself in its debug buffer or the attention runs on the CUDA-core path
  a.rope_q = (dbg && dbg->q) ? 0 : 1;
  if (a.rope_q && !csa::sparse_attn_tc_supported(a)) a.rope_q = 0;
  if (!a.rope_q)
    STEP(csa::launch_rope(q, (int64_t)NT * H, hd, rd, pos_q, tab, ctx->tab_rows, 0, ctx->status, s), "rope q");
  // the compressed selection
  if (r.ratio > 0) {
    if (r.is_index_source) {
      float *S = dbg && dbg->scores ? dbg->scores : ctx->scores;
      const uint8_t *cand = r.uses_candidates ? sh->candidates : nullptr;
      // short decode rows: scores and selection in one kernel, the scores kept on chip (unless the
      // caller wants them in its debug buffer)
      if (!(dbg && dbg->scores) && !r.is_candidate_source &&
          csa::index_fused_supported(qI, (const bf16 *)sh->index_k, T, start_pos, Hi, dI, sh->compress_len, r.ratio,
                                     K)) {
        STEP(csa::launch_index_topk_fused(qI, wI, (const bf16 *)sh->index_k, B, start_pos, Hi, sh->compress_stride,
                                          sh->compress_len, r.ratio, cand, sh->cand_width, g.cand_block, K,
                                          rows_a_len, sh->topk_idxs, ctx->status, s),
             "index scores + topk");
      } else if (!(dbg && dbg->scores) && !r.is_candidate_source &&
                 csa::index_gather_topk_supported(qI, (const bf16 *)sh->index_k, B, T, start_pos, Hi, dI,
                                                  sh->compress_len, r.ratio, cand, sh->cand_width, g.cand_block, K,
                                                  ctx->num_sms)) {
        // long rows under a mask: gathered scores and the selection in one cluster launch
        STEP(csa::launch_index_gather_topk(qI, wI, (const bf16 *)sh->index_k, B, start_pos, Hi, sh->compress_stride,
                                           sh->compress_len, r.ratio, cand, sh->cand_width, g.cand_block, K,
                                           rows_a_len, sh->topk_idxs, ctx->status, ctx->num_sms, s),
             "index scores + topk");
      } else {
        // (the rows whose selection takes every valid position are not scored, unless the scores are
        // wanted: in the debug buffer, or for the candidate blocks below)
        const int skip_k = (dbg && dbg->scores) || r.is_candidate_source || cand ? 0 : K;
        STEP(csa::launch_index_scores(qI, wI, (const bf16 *)sh->index_k, B, T, start_pos, Hi, dI,
                                      sh->compress_stride, sh->compress_len, r.ratio, cand, sh->cand_width,
                                      g.cand_block, S, s, ctx->status, skip_k),
             "index scores");
        STEP(csa::launch_index_topk(S, B, T, start_pos, sh->compress_stride, sh->compress_len, r.ratio, cand,
                                    sh->cand_width, g.cand_block, K, rows_a_len, sh->topk_idxs, s),
             "index topk");
        // the candidate source publishes the block mask of its own scores for later index sources
        if (r.is_candidate_source)
          STEP(csa::launch_cand_blocks(S, B, T, start_pos, sh->compress_stride, sh->compress_len, r.ratio,
                                       g.cand_block, g.cand_topk_blocks, sh->candidates, sh->cand_width, s),
               "candidate blocks");
      }
      sh->has_topk = 1;
    }
    if (dbg && dbg->idx)
      COPY(cudaMemcpy2DAsync(dbg->idx + W, sizeof(int32_t) * (W + K), sh->topk_idxs, sizeof(int32_t) * K,
                             sizeof(int32_t) * K, NT, cudaMemcpyDeviceToDevice, s),
           "debug idx");
  }
  // the window selection in the debug buffer is strided; pass the stride through idx_a's row length
  if (idx_stride != W) {
    // compact copy of the window columns for the kernel
    COPY(cudaMemcpy2DAsync(ctx->idx_win, sizeof(int32_t) * W, win_idx, sizeof(int32_t) * idx_stride,
                           sizeof(int32_t) * W, NT, cudaMemcpyDeviceToDevice, s),
         "window idx");
    a.idx_a = ctx->idx_win;
  }
  int attn_kernels = 0;
  STAGE(csa::launch_sparse_attn(a, ctx->ws, ctx->ws_bytes, ctx->num_sms, s, &attn_kernels), "sparse_attn",
        attn_kernels);
  // grouped output: og[:, g] = o_rot[:, g*gw:(g+1)*gw] wo_a[g]^T, then out = og wo_b^T
  {
    csa::LinearProblem pa = lin(ctx->o_rot, gw, H * hd, w->wo_a, g.o_rank, og, G * g.o_rank, G);
    if (w->wo_a_fp8) {  // the codes and tile scales in place of the bf16 weights
      pa.W = nullptr;
      pa.W8 = w->wo_a_fp8;
      pa.w8_scale = w->wo_a_scale;
      pa.ldw = gw;
    }
    // wo_a and wo_b: programmatic dependents of the kernels before them (their weights start to stream
    // while those finish), each letting the next launch early
    pa.pdl = pa.early_dependents = 1;
    STEP(csa::launch_linear(&pa, 1, ctx->ws, ctx->gemm_ws_bytes(), ctx->num_sms, ctx->status, s), "wo_a");
    csa::LinearProblem pb = lin(og, G * g.o_rank, G * g.o_rank, w->wo_b, g.dim, out, g.dim, 1);
    pb.pdl = pb.early_dependents = 1;
    int wo_b_kernels = 0;  // (a prefill chunk's wo_b may split its last wave: three launches)
    STAGE(csa::launch_linear(&pb, 1, ctx->ws, ctx->gemm_ws_bytes(), ctx->num_sms, ctx->status, s, &wo_b_kernels),
          "wo_b", wo_b_kernels);
  }
#undef STEP
#undef COPY
#undef STAGE
  return CSA_OK;
}

int attn_v41_forward_host(csa_ctx *ctx, const csa_layer_weights *w, csa_layer_state *st, const csa_bf16 *x_host, int B,
                          int T, int start_pos, csa_shared *sh, csa_bf16 *out_host, csa_stream stream) {
  if (!ctx || !x_host || !out_host) return fail(CSA_ERR_ARG, "attn_v41_forward_host: NULL argument");
  int rc = check_forward(ctx, w, st, x_host, B, T, start_pos, sh, out_host);
  if (rc) return rc;
  const size_t bytes = sizeof(csa_bf16) * (size_t)B * T * ctx->cfg.dim;
  cudaStream_t s = (cudaStream_t)stream;
  CSA_CUDA(cudaMemcpyAsync(ctx->x_stage, x_host, bytes, cudaMemcpyHostToDevice, s), "attn_v41_forward_host: H2D");
  rc = attn_v41_forward(ctx, w, st, (const csa_bf16 *)ctx->x_stage, B, T, start_pos, sh, (csa_bf16 *)ctx->out_stage,
                        nullptr, stream);
  if (rc) return rc;
  CSA_CUDA(cudaMemcpyAsync(out_host, ctx->out_stage, bytes, cudaMemcpyDeviceToHost, s), "attn_v41_forward_host: D2H");
  return CSA_OK;
}

}  // extern "C"
