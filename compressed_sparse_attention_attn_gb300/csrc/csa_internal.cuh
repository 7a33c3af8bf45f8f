// csa_internal.cuh -- declarations shared by the library's translation units (not installed).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <atomic>
#include <cstdint>
#include <cstddef>
#include <mutex>

#include "../../include/csa.h"

namespace csa {

using bf16 = __nv_bfloat16;

// Bits of the device status word (csa_status).
constexpr int kStatusBadIndex = 1;
constexpr int kStatusTimeout = 2;

// Position of row r: pos[r / rows_per_pos] from an array, or start + (r / rows_per_pos) % T.
struct PosSpec {
  const int32_t *arr;
  int start;
  int T;
  int rows_per_pos;
  __device__ __forceinline__ int at(int64_t r) const {
    int64_t tok = r / rows_per_pos;
    return arr ? arr[tok] : start + (int)(tok % T);
  }
};

// The dynamic shared-memory limit of a kernel is a per-device attribute: each launcher keeps one of
// these (static) and raises the attribute of the current device when a launch needs more than it
// has, never lowering it, so that host threads launching the same kernel with different needs do
// not undo one another.  The per-device value last set is cached for the common case.
constexpr int kAttrDevices = 64;
struct SmemAttr {
  std::atomic<int> set[kAttrDevices] = {};
  std::mutex mu;
  cudaError_t ensure(const void *func, int need) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool tracked = dev >= 0 && dev < kAttrDevices;
    if (tracked && set[dev].load(std::memory_order_acquire) >= need) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu);
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, func);
    if (e != cudaSuccess) return e;
    int have = fa.maxDynamicSharedSizeBytes;
    if (have < need) {
      e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, need);
      if (e != cudaSuccess) return e;
      have = need;
    }
    if (tracked) set[dev].store(have, std::memory_order_release);
    return cudaSuccess;
  }
};

// ---- launchers (each returns a cudaError_t of the launch) ---------------------------------------

cudaError_t launch_rmsnorm(const bf16 *x, int M, int N, const float *w, float eps, bf16 *y, cudaStream_t s);
cudaError_t launch_rope(bf16 *x, int64_t rows, int row_len, int rd, PosSpec pos, const float *tab, int tab_rows,
                        int inverse, int *status, cudaStream_t s);
cudaError_t launch_act_quant(bf16 *x, int64_t n, uint8_t *codes, int8_t *scale_exp, cudaStream_t s);
cudaError_t launch_kv_finish(const bf16 *kv_in, bf16 *kv_out, int B, int T, int start_pos, int hd, int rd,
                             const float *tab, bf16 *ring, int W, int32_t *win_idx, int idx_stride, uint8_t *codes,
                             int8_t *scales, cudaStream_t s);
cudaError_t launch_scale_bf16_to_f32(const bf16 *x, int64_t n, float scale, float *y, cudaStream_t s);

// One product y[M][g*N + n] = sum_k x[m][g*K + k] W[g*N + n][k] for g < groups (f32 accumulation,
// bf16 out); x row stride ldx, W row stride ldw, y row stride ldy (elements).
struct LinearProblem {
  const bf16 *x;
  int M, K, ldx;
  const bf16 *W;
  int N, ldw;
  bf16 *y;
  int ldy, groups;
  float *part = nullptr;  // split-K mode: f32 partials [S][M][ldp], this problem's columns at part
  int ldp = 0;
  // fp8 weights (W unused): e4m3 codes uint8 [groups*N][ldw bytes] and one f32 scale per 128 x 128
  // tile, w8_scale [ceil(groups*N/128)][ceil(K/128)]; the product uses w = bf16(e4m3 * scale)
  const uint8_t *W8 = nullptr;
  const float *w8_scale = nullptr;
  // 1: the kernel launched right after this product is a programmatic dependent that reads the
  // product's output only after its dependency wait, so the tensor-core launch lets it start as soon
  // as this grid's CTAs have started (set on every problem of the launch)
  int early_dependents = 0;
  // 1: launched as a programmatic dependent of the kernel before it (decode-sized launches): the
  // weights of each CTA's first stages are copied before the dependency wait, the activations after
  int pdl = 0;
};
// Products sharing M run in one tensor-core launch (up to 4 at a time).  ws/ws_bytes: Stream-K
// arrival counters and partials (the counters must be zero between launches).  kernels (may be NULL):
// receives the kernels launched.
cudaError_t launch_linear(const LinearProblem *probs, int n, float *ws, size_t ws_bytes, int num_sms, int *status,
                          cudaStream_t s, int *kernels = nullptr);
constexpr size_t kGemmCounterBytes = 65536 * sizeof(int);
// Failure-detection test hook of the current device: while ns != 0 the projection kernels first
// wait, up to ns nanoseconds, on a barrier phase that nothing completes, then take their timeout path.
cudaError_t set_gemm_stall(unsigned long long ns);
// Split-K without fixup: products sharing M and K; CTA (tile, s) writes its f32 partial sum over
// its K range to part[s][m][col] (every problem's part/ldp set).  The consumer sums the S slices.
cudaError_t launch_gemm_tc_split(const LinearProblem *probs, int nprob, int S, int *status, cudaStream_t s);
// The Stream-K / waves / paired launch of up to four problems sharing the activations (the paired
// kernel, chosen for many token tiles, may write a problem's f32 result to `part` as one split slice).
// kernels (may be NULL): receives the kernels launched; only a caller that counts them lets a paired
// launch of one problem split its last partial wave by k-range (two more launches: the split tiles
// and their sum).
cudaError_t launch_gemm_tc(const LinearProblem *probs, int nprob, float *ws, size_t ws_bytes, int num_sms,
                           int *status, cudaStream_t s, int *kernels = nullptr);
// The largest split count S <= max_S dividing the problems' k-slices with tiles * S <= max_ctas (>= 1).
int gemm_tc_split_count(const LinearProblem *probs, int nprob, int max_ctas, int max_S);
bool gemm_tc_supported(const LinearProblem &q);

// The window rows and the query latent from split-K partials of [wq_a | wkv | weights_proj] x:
// per token, the sum of the S slices rounded to bf16 (linear_bf16), then qr = RMSNorm * q_norm,
// kv = RMSNorm * kv_norm -> RoPE -> fp8 -> ring + window selection (as csa_kv_finish), and
// w^I = bf16 * wscale.  Hi may be 0.
struct XFinishArgs {
  const float *part;
  int S, ldp, q_rank, hd, Hi;
  const float *q_norm, *kv_norm;
  float eps;
  bf16 *qr, *kv;
  int B, T, start_pos, rd;
  const float *tab;
  bf16 *ring;
  int W;
  int32_t *win_idx;
  int idx_stride;
  uint8_t *codes;
  int8_t *scales;
  float wscale;
  float *wI;
};
cudaError_t launch_x_finish(const XFinishArgs &a, cudaStream_t s);

// Tensor-core kernel when dI == 128, Hi is a multiple of 16 (<= 256) and qI, KI are 16-byte
// aligned; else the CUDA-core kernel.  status (may be NULL): the device status word for timeouts.
// skip_k > 0 (no candidate mask): the rows of queries with at most skip_k valid positions may be left
// unwritten -- a top-k of K = skip_k over the same limits takes all of them without reading a score.
cudaError_t launch_index_scores(const bf16 *qI, const float *wI, const bf16 *KI, int B, int T, int start_pos, int Hi,
                                int dI, int Lstride, int compress_len, int ratio, const uint8_t *cand, int cand_width,
                                int cand_block, float *S, cudaStream_t s, int *status = nullptr, int skip_k = 0);
cudaError_t launch_index_topk(const float *S, int B, int T, int start_pos, int Lstride, int compress_len, int ratio,
                              const uint8_t *cand, int cand_width, int cand_block, int K, int offset, int32_t *out,
                              cudaStream_t s);
// Long decode rows under a candidate mask: the gathered scores and the top-k in one launch, one
// thread-block cluster per query that selects together (the scores stay on chip).
bool index_gather_topk_supported(const bf16 *qI, const bf16 *KI, int B, int T, int start_pos, int Hi, int dI,
                                 int compress_len, int ratio, const uint8_t *cand, int cand_width, int cand_block,
                                 int K, int num_sms);
cudaError_t launch_index_gather_topk(const bf16 *qI, const float *wI, const bf16 *KI, int B, int start_pos, int Hi,
                                     int Lstride, int compress_len, int ratio, const uint8_t *cand, int cand_width,
                                     int cand_block, int K, int offset, int32_t *out, int *status, int num_sms,
                                     cudaStream_t s);
// The candidate source's block mask from its own scores: per query the top K blocks of cand_block
// positions by their largest valid score, mask uint8 [B*T][cand_width] (1 = candidate).
cudaError_t launch_cand_blocks(const float *S, int B, int T, int start_pos, int Lstride, int compress_len, int ratio,
                               int cand_block, int K, uint8_t *mask, int cand_width, cudaStream_t s);
// Scores and top-k in one kernel for decode rows (T == 1) with at most 512 valid positions (the
// scores stay on chip); same conditions on the operands as the tensor-core scores, K <= 512.
bool index_fused_supported(const bf16 *qI, const bf16 *KI, int T, int start_pos, int Hi, int dI, int compress_len,
                           int ratio, int K);
cudaError_t launch_index_topk_fused(const bf16 *qI, const float *wI, const bf16 *KI, int B, int start_pos, int Hi,
                                    int Lstride, int compress_len, int ratio, const uint8_t *cand, int cand_width,
                                    int cand_block, int K, int offset, int32_t *out, int *status, cudaStream_t s);

struct AttnArgs {
  const bf16 *q;
  int B, T, H, hd;
  const bf16 *rows_a;
  int64_t a_seq_stride;
  int a_len;
  const bf16 *rows_b;
  int64_t b_seq_stride;
  int b_len;
  const int32_t *idx_a;
  int na;
  const int32_t *idx_b;
  int nb;
  const float *sink;
  float scale;
  bf16 *o, *o_rot;
  int rd, start_pos;
  const float *tab;
  int *status;
  // 1: q has not been rotated yet; the kernel turns the last rd features of each head by the
  // query's position (RoPE, tab) on its own copy before the scores.  0: q is used as given.
  int rope_q = 0;
};
// Tensor-core kernel where the shapes allow (head_dim 512, heads in groups of 64), else the SIMT one.
// ws: the tensor-core path's per-split shares (after the GEMM counters).  *kernels (if given): the
// number of kernels launched.
cudaError_t launch_sparse_attn(const AttnArgs &a, float *ws, size_t ws_bytes, int num_sms, cudaStream_t s,
                               int *kernels = nullptr);
// Whether the tensor-core kernel takes these arguments (it alone applies rope_q, for rd <= 64).
bool sparse_attn_tc_supported(const AttnArgs &a);

// The compressor of a kv-source layer (k_compress.cu): products of x [B*T][dim] with wkv (f32 at
// ratio > 1, bf16 at ratio 1) and wgate, the partial group st_kv / st_score [B][ratio][hd], the
// closed groups' latent rows Z and index keys KI (with wk) at rows j of [B][Lstride][.]; y_dbg (may be
// NULL) receives the normed rows before RoPE and fp8.  Prefill (start_pos 0) or one decode token.
struct CompressArgs {
  const bf16 *x;
  int B, T, start_pos, ratio, dim, hd, rd, dI;
  const void *wkv;
  const float *wgate, *norm;
  const bf16 *wk;
  const float *k_norm;
  float *st_kv, *st_score;
  bf16 *Z, *KI, *y_dbg;
  int64_t Lstride;
  const float *tab;
  float eps;
};
bool compress_supported(const CompressArgs &a);
// ws: f32 partial sums (the splits are chosen to fit ws_bytes)
cudaError_t launch_compress(const CompressArgs &a, float *ws, size_t ws_bytes, int num_sms, cudaStream_t s);
cudaError_t launch_fill_f32(float *p, int64_t n, float v, cudaStream_t s);

// Record the calling thread's last error (attn_v41_last_error) and return `code`.
int set_error(int code, const char *fmt, ...);

// Host-side tables (double precision, rounded to f32).
void build_rope_table(int rd, int max_seq, double theta, int orig_seq, double factor, double beta_fast,
                      double beta_slow, float *tab);

}  // namespace csa
