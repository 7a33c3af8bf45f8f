/*
 * csa.h -- C ABI of the GB300 (sm_103a) compressed sparse attention layer core of DeepSeek-V4.1.
 *
 * One layer forward, attn_v41_forward, plus one entry point per step of the path.  Everything is
 * enqueued on the caller's CUDA stream; nothing synchronises the host unless a function says so.
 * All tensors are row-major and contiguous unless a stride argument says otherwise; bf16 tensors
 * are passed as their 16-bit patterns (csa_bf16).  Pointers are DEVICE pointers unless the name
 * ends in _host.  The caller owns every tensor passed in; the library owns only the workspaces of a
 * csa_ctx (allocated by csa_create, freed by csa_destroy).
 *
 * Sources the operations follow (page title, then section):
 *   [attn_v41]  "metrale_model_arch::attn_v41" rustdoc page and attn_v41.rs: AttnV41Cfg, LayerRole,
 *               AttnV41LayerWeights, AttnV41LayerState, SharedV41, AttnV41Run, "Invariants".
 *   [ref-attn]  "deepseek_v41_ref::attn" rustdoc page: the precision contract, act_quant_inplace,
 *               pow2_ceil, apply_rotary, freqs_cis, sparse_attn, window_topk_idxs, the ring fixture.
 *   [atlas]     "DeepSeek V4.1 - Compressed sparse attention" atlas page: "All 25 steps",
 *               Attention.forward excerpt, config.json.
 *   [join]      "Join rows" atlas page.
 *
 * Errors: every int-returning function returns CSA_OK (0) or a negative CSA_ERR_* code; the text of
 * the last error of the calling thread is attn_v41_last_error().  Arguments are validated on the
 * host before anything is enqueued: on an error nothing is launched.  CSA_ERR_CUDA reports a launch
 * or runtime failure seen by the host (asynchronous faults surface at the caller's next sync).
 *
 * Threads: the entry points may be called from several host threads at once.  A csa_ctx, though,
 * serves one stream at a time: its workspaces are shared by every call made with it, so calls on
 * one context whose work could overlap on the GPU must be ordered by the caller.  A csa_ctx belongs
 * to the device current at csa_create; the calls that launch work with it, or wait for it, return
 * CSA_ERR_ARG when another device is current.
 */
#ifndef CSA_H_
#define CSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define CSA_API __attribute__((visibility("default")))
#else
#define CSA_API
#endif

typedef uint16_t csa_bf16; /* bit pattern of a bfloat16 */
typedef void *csa_stream;  /* a cudaStream_t; NULL = the legacy default stream */

enum {
  CSA_OK = 0,
  CSA_ERR_ARG = -1,            /* null pointer, bad dimension, bad role */
  CSA_ERR_SHAPE = -2,          /* T > max_tokens, start_pos + T > max_seq, batch > max_batch, decode with T > 1 */
  CSA_ERR_NO_KV_SOURCE = -3,   /* ratio > 0 and no published latent cache ([attn_v41] "Invariants") */
  CSA_ERR_NO_SELECTION = -4,   /* a ratio > 0 layer that reuses the selection, and none is published */
  CSA_ERR_TOO_WIDE = -5,       /* selection wider than window + index_topk or 2048 ([attn_v41] "Invariants") */
  CSA_ERR_UNSUPPORTED = -6,    /* a role or shape this library does not take */
  CSA_ERR_CUDA = -7,           /* a CUDA call failed */
  CSA_ERR_DEVICE_TIMEOUT = -8, /* a bounded device-side wait ran out (kernel returned early, output invalid) */
  CSA_ERR_NOMEM = -9           /* workspace allocation failed in csa_create */
};

/* Model-wide attention geometry ([attn_v41] AttnV41Cfg; [atlas] config.json).  gw = n_heads *
 * head_dim / groups.  max_tokens bounds T per call, max_batch bounds B, max_seq bounds positions and
 * sizes the RoPE tables.  The ratio-0 table uses rope_theta; ratio > 0 uses compress_rope_theta with
 * YaRN (orig_seq, rope_factor, beta_fast, beta_slow) once max_seq > orig_seq. */
typedef struct csa_cfg {
  int dim, n_heads, head_dim, rope_dim, q_rank, o_rank, groups, window;
  float eps;
  int index_heads, index_hd, index_topk, cand_block, cand_topk_blocks;
  int max_seq, max_tokens, max_batch;
  float rope_theta, compress_rope_theta, rope_factor;
  int orig_seq;
  float beta_fast, beta_slow;
} csa_cfg;

/* A layer's compress ratio and the shared slots it writes or reads ([attn_v41] LayerRole).
 * ratio 0: window only.  ratio > 0 with is_index_source: computes and publishes its own selection
 * (a Reindex layer when it is not the kv source); ratio > 0 without it: reuses the published one.
 * uses_candidates: the index source applies the published candidate block mask. */
typedef struct csa_role {
  int ratio;
  int is_kv_source, is_index_source, is_candidate_source, uses_candidates;
} csa_role;

/* One layer's resident weights ([attn_v41] AttnV41LayerWeights).  Projections are bf16 [out, in]:
 * wq_a [q_rank, dim], wq_b [n_heads*head_dim, q_rank], wkv [head_dim, dim],
 * wo_a [groups*o_rank, gw], wo_b [dim, groups*o_rank], idx_wq_b [index_heads*index_hd, q_rank],
 * idx_wproj [index_heads, dim].  sink [n_heads], q_norm [q_rank], kv_norm [head_dim] are f32.
 * idx_* may be NULL unless role.is_index_source.  A candidate source (an index source with
 * role.is_candidate_source) also writes shared->candidates from its own scores, as
 * csa_candidate_blocks with K = cfg.cand_topk_blocks, for the index sources after it.
 * The grouped wo_a may instead stay in fp8 ([atlas] Attention excerpt: the checkpoint's converter
 * dequantises it to bf16, and an fp8 grouped product would halve its memory): wo_a_fp8 uint8
 * [groups*o_rank, gw] holds e4m3 codes and wo_a_scale f32 [groups*o_rank/128 rounded up][gw/128
 * rounded up] one scale per 128 x 128 tile; the layer then computes with w = bf16(e4m3 * scale), the
 * converter's bf16 weight, and wo_a may be NULL.  Both NULL: wo_a (bf16) is used. */
typedef struct csa_layer_weights {
  csa_role role;
  const float *sink, *q_norm, *kv_norm;
  const csa_bf16 *wq_a, *wq_b, *wkv, *wo_a, *wo_b, *idx_wq_b, *idx_wproj;
  const uint8_t *wo_a_fp8;
  const float *wo_a_scale;
  /* kv sources only ([attn_v41] CompressorWeightsGpu, IndexerWeightsGpu): comp_wkv [head_dim, dim],
   * f32 at ratio > 1 and bf16 at ratio 1; comp_wgate f32 [head_dim, dim] at ratio > 1 (NULL at
   * ratio 1); comp_norm f32 [head_dim].  idx_wk bf16 [index_hd, head_dim] and idx_k_norm f32
   * [index_hd] produce the index keys (NULL: the kv source publishes no index keys). */
  const void *comp_wkv;
  const float *comp_wgate, *comp_norm;
  const csa_bf16 *idx_wk;
  const float *idx_k_norm;
} csa_layer_weights;

/* One layer's per-sequence state ([attn_v41] AttnV41LayerState): the window ring bf16
 * [max_batch][window][head_dim]; slot of position p is p mod window.  A kv source also holds the
 * compressor's partial group, comp_kv and comp_score f32 [max_batch][comp_ratio][head_dim] (scores
 * -inf for empty slots), and the caches it publishes: latent bf16 [max_batch][cache_rows][head_dim]
 * and index_keys bf16 [max_batch][cache_rows][index_hd] (cache_rows >= max_seq / ratio).  Other
 * layers leave these NULL / 0. */
typedef struct csa_layer_state {
  csa_bf16 *window;
  float *comp_kv, *comp_score;
  int comp_ratio;
  csa_bf16 *latent, *index_keys;
  int cache_rows;
} csa_layer_state;

/* What source layers publish ([attn_v41] SharedV41), device buffers:
 *   compress_kv  bf16 [B][compress_stride][head_dim]   latent cache Z (kv source's)
 *   index_k      bf16 [B][compress_stride][index_hd]   index keys K^I
 *   compress_len rows of each sequence that are written (valid positions j < compress_len)
 *   topk_idxs    int32 [B*T][topk]: the selection, offset past the window rows, -1 = absent; an
 *                index-source layer writes it (has_topk becomes 1), a reuse layer reads it
 *   candidates   uint8 [B*T][cand_width], nonzero = block j / cand_block allowed (may be NULL
 *                unless the layer uses candidates); the candidate source writes it */
typedef struct csa_shared {
  const csa_bf16 *compress_kv;
  const csa_bf16 *index_k;
  int compress_len, compress_stride;
  int32_t *topk_idxs;
  int topk, has_topk;
  uint8_t *candidates;
  int cand_width;
} csa_shared;

/* Optional intermediates of one forward ([attn_v41] AttnV41Run); every member may be NULL.
 *   q        bf16 [B*T][n_heads][head_dim]  q after RoPE
 *   kv       bf16 [B*T][head_dim]           new kv rows after RoPE and the fp8 round trip
 *   kv_codes uint8 [B*T][head_dim]          their e4m3 codes
 *   kv_scale int8 [B*T][head_dim/32]        exponents k of the block scales 2^k
 *   idx      int32 [B*T][window + topk]     the joined selection (window slots, then compressed+|W|)
 *   scores   f32 [B*T][compress_stride]     indexer scores (valid positions only are written)
 *   o        bf16 [B*T][n_heads][head_dim]  sparse_attn output before the inverse rotation
 *   og       bf16 [B*T][groups*o_rank]      grouped projection
 *   qr       bf16 [B*T][q_rank]; qI bf16 [B*T][index_heads*index_hd]; wI f32 [B*T][index_heads] */
typedef struct csa_debug {
  csa_bf16 *q, *kv;
  uint8_t *kv_codes;
  int8_t *kv_scale;
  int32_t *idx;
  float *scores;
  csa_bf16 *o, *og, *qr, *qI;
  float *wI;
} csa_debug;

typedef struct csa_ctx csa_ctx;

/* ---------------------------------------------------------------------------------------------
 * Context and layer
 * -------------------------------------------------------------------------------------------*/

/* Create a context on the current CUDA device: validates cfg, allocates the workspaces for
 * max_batch * max_tokens positions, builds the two RoPE tables on the host ([ref-attn] freqs_cis)
 * and uploads them.  Synchronous.  *out receives the context. */
CSA_API int csa_create(const csa_cfg *cfg, csa_ctx **out);

/* Free a context and its workspaces (after synchronising the device).  NULL is a no-op. */
CSA_API int csa_destroy(csa_ctx *ctx);

/* Zero the window ring of `batch` sequences ([attn_v41] AttnV41LayerState::new), on `stream`; on a
 * kv source's state also empty the compressor's partial group (kv 0, scores -inf: "the score state
 * starts at -inf"). */
CSA_API int csa_state_init(csa_ctx *ctx, csa_layer_state *state, int batch, csa_stream stream);

/* One layer forward ([atlas] Attention.forward; [attn_v41] AttnV41::forward) for `batch` sequences
 * of T tokens at start_pos: prefill when start_pos == 0 (T >= 1), decode when start_pos > 0 (T == 1).
 * x bf16 [batch][T][dim] in, out bf16 [batch][T][dim] out.  Updates state->window; an index-source
 * layer writes shared->topk_idxs and sets shared->has_topk.  shared may be NULL for ratio 0.
 * dbg may be NULL.  Enqueued on `stream`, no host synchronisation (graph-capturable). */
CSA_API int attn_v41_forward(csa_ctx *ctx, const csa_layer_weights *w, csa_layer_state *state, const csa_bf16 *x, int batch,
                     int T, int start_pos, csa_shared *shared, csa_bf16 *out, const csa_debug *dbg, csa_stream stream);

/* attn_v41_forward with x_host / out_host in HOST memory (pinned for overlap, pageable accepted):
 * copies x to a context staging buffer, runs the layer, copies out back, all on `stream`.  Returns
 * once the work is enqueued; out_host is valid after the stream is synchronised. */
CSA_API int attn_v41_forward_host(csa_ctx *ctx, const csa_layer_weights *w, csa_layer_state *state, const csa_bf16 *x_host,
                          int batch, int T, int start_pos, csa_shared *shared, csa_bf16 *out_host, csa_stream stream);

/* The compressor of a kv-source layer ([attn_v41] module description: the compressor pooling;
 * CompressorWeightsGpu; AttnV41LayerState; SharedV41), for `batch` sequences of T tokens at
 * start_pos (prefill at 0, or one decode token): k_p = x_p comp_wkv^T and s_p = x_p comp_wgate^T in
 * f32 (at ratio 1, k_p = linear_bf16(x_p, comp_wkv) and no score) fill slot p mod ratio of the
 * state's partial group; every group j the call closes (positions j*ratio .. j*ratio + ratio - 1) is
 * pooled per feature with the softmax of its scores, z = sum_i e^{s_i} k_i / sum_i e^{s_i}, normed,
 * y = bf16(RMSNorm(z) * comp_norm); with idx_wk its index key bf16(RMSNorm(linear_bf16(y, idx_wk)) *
 * idx_k_norm) goes to row j of state->index_keys, and y with RoPE on its last rope_dim at position
 * j * ratio and the fp8 round trip to row j of state->latent.  The pooling is a reading (the pages
 * name the step but print no formula).  shared (may be NULL) then publishes the caches:
 * compress_kv = latent, index_k = index_keys (when written), compress_stride = cache_rows,
 * compress_len = max(compress_len, (start_pos + T) / ratio).  x bf16 [batch][T][dim] (16-byte
 * aligned); w->role.ratio in 1..16, head_dim <= 1024 a multiple of 64, index_hd <= 256; y_dbg (may
 * be NULL) bf16 [batch][cache_rows][head_dim] receives y.  attn_v41_forward runs this first on a kv
 * source.  The context's workspace holds the f32 partial products. */
CSA_API int csa_compress(csa_ctx *ctx, const csa_layer_weights *w, csa_layer_state *state, const csa_bf16 *x,
                         int batch, int T, int start_pos, csa_shared *shared, csa_bf16 *y_dbg, csa_stream stream);

/* Text of the calling thread's last error ("" if none). */
CSA_API const char *attn_v41_last_error(void);

/* Copy the context's RoPE table for a ratio class (0: ratio-0 layers; 1: ratio > 0) to host memory
 * tab_host f32 [max_seq][rope_dim/2][2] of (cos, sin).  Synchronous. */
CSA_API int csa_rope_table_get(const csa_ctx *ctx, int ratio_class, float *tab_host);

/* Synchronise the device and return the context's device status word as an error code:
 * CSA_OK, CSA_ERR_ARG (a kernel met an out-of-range index and skipped it) or CSA_ERR_DEVICE_TIMEOUT
 * (a bounded device-side wait ran out; the outputs since the last clear are invalid).  The word is
 * sticky: every kernel ORs its findings in until a call with clear != 0 resets it (after a timeout
 * that also re-zeroes the projections' Stream-K arrival counters, so the next call starts clean). */
CSA_API int csa_status(csa_ctx *ctx, int clear);

/* Test hook of failure detection, for checking how a device-side timeout is reported without any
 * fault: while ns != 0, every projection kernel launched on the current device (csa_linear,
 * csa_linear_noalloc, the layer's projections; every context) first waits on a barrier phase that
 * nothing completes, and gives up after ns nanoseconds (each wait of the kernels is bounded: 2 s by
 * default).  The kernel then takes its timeout path -- it lets the copies it has in flight land,
 * frees its tensor memory, returns, and sets CSA_ERR_DEVICE_TIMEOUT in the status word (csa_status,
 * csa_linear_noalloc_status); its output is invalid.  ns = 0 turns the hook off.  Synchronous. */
CSA_API int csa_debug_stall(unsigned long long ns);

/* Bytes of device workspace the context holds. */
CSA_API size_t csa_workspace_bytes(const csa_ctx *ctx);

/* Tracing.  While enabled, attn_v41_forward records a CUDA event pair on its stream around each of
 * its stages (at most 64 in all); on a stream being captured into a CUDA graph the pairs become
 * event-record nodes, so each replay of the graph re-times its stages.  enable 1: each forward
 * replaces the list with its own stages; enable 2: forwards append theirs to the list, which
 * restarts empty at this call (one list for several layers, or for a captured step); 0: off.
 * csa_trace_read waits for the listed events and writes, for the first `max` stages, a static stage
 * name and the elapsed milliseconds.  Returns the number of listed stages (>= 0) or an error code. */
CSA_API int csa_trace_enable(csa_ctx *ctx, int enable);
CSA_API int csa_trace_read(csa_ctx *ctx, int max, const char **names, float *ms);

/* Number of kernels the last attn_v41_forward enqueued. */
CSA_API int csa_last_launches(const csa_ctx *ctx);

/* ---------------------------------------------------------------------------------------------
 * Steps of the path (device pointers, enqueued on `stream`)
 * -------------------------------------------------------------------------------------------*/

/* linear_bf16 ([ref-attn] "Precision"): y[m][n] = bf16(sum_k x[m][k] W[n][k]), f32 accumulation.
 * x [M][K] with row stride ldx, W [N][K] row stride ldw, y [M][N] row stride ldy (elements).
 * groups > 1 runs `groups` independent products in one call ([atlas] "Grouped output", the
 * block-diagonal wo_a): product g reads x columns [g*K, (g+1)*K), W rows [g*N, (g+1)*N) and writes
 * y columns [g*N, (g+1)*N).  ctx provides the split-K workspace (a call on one context at a time
 * per stream: the workspace also holds the f32 partial sums when a product of 2048 or more rows
 * splits its last wave of tiles by k-range, which enqueues two more kernels). */
CSA_API int csa_linear(csa_ctx *ctx, const csa_bf16 *x, int M, int K, int ldx, const csa_bf16 *W, int N, int ldw, csa_bf16 *y,
               int ldy, int groups, csa_stream stream);

/* linear_bf16 with fp8 weights ([atlas] Attention excerpt: the grouped wo_a is dequantised to bf16
 * by the checkpoint's converter; an fp8 grouped product halves its memory): y[m][n] = bf16(sum_k
 * x[m][k] w[n][k]) with w[n][k] = bf16(e4m3(W8[n][k]) * scale[n/128][k/128]), f32 accumulation --
 * the result of csa_linear on the dequantised bf16 weights, reading half the weight bytes.
 * W8 uint8 [groups*N][ldw8 bytes] e4m3 codes (16-byte aligned, ldw8 a multiple of 16, K a multiple
 * of 16, of 64 when groups > 1); scale f32 [ceil(groups*N/128)][ceil(K/128)]; x, y and groups as
 * in csa_linear (product g reads x columns [g*K, (g+1)*K) and W8 rows [g*N, (g+1)*N)). */
CSA_API int csa_linear_fp8w(csa_ctx *ctx, const csa_bf16 *x, int M, int K, int ldx, const uint8_t *W8,
                            const float *scale, int N, int ldw8, csa_bf16 *y, int ldy, int groups, csa_stream stream);

/* RMSNorm ([ref-attn] "Precision"): y = bf16(x / sqrt(mean(x^2) + eps) * w) per row; x, y [M][N]
 * (may alias), w f32 [N]. */
CSA_API int csa_rmsnorm(const csa_bf16 *x, int M, int N, const float *w, float eps, csa_bf16 *y, csa_stream stream);

/* apply_rotary ([ref-attn]): rotate, in place, the last rd elements of each row_len-wide row of x
 * [rows][row_len]; pairs (2i, 2i+1) are complex, multiplied by tab[pos][i] = (cos, sin) (conjugate
 * when inverse) with each product and sum rounded to f32, written bf16.  Row r uses position
 * pos[r / rows_per_pos] (device int32); tab f32 [tab_rows][rd/2][2]. */
CSA_API int csa_rope(csa_bf16 *x, int64_t rows, int row_len, int rd, const int32_t *pos, int rows_per_pos, const float *tab,
             int tab_rows, int inverse, csa_stream stream);

/* act_quant_inplace ([ref-attn], FP8_BLOCK = 32): per block of 32 of x [n] (n a multiple of 32),
 * s = pow2_ceil(max(amax, 1e-4) / 448), codes = e4m3_rne(clamp(x / s, +-448)), x = bf16(code * s).
 * codes uint8 [n] and scale_exp int8 [n/32] (exponent of s) may be NULL. */
CSA_API int csa_act_quant(csa_bf16 *x, int64_t n, uint8_t *codes, int8_t *scale_exp, csa_stream stream);

/* The window keys and values after the norm ([atlas] "Window keys and values": RoPE of the last
 * rd, then W <- FP8(W)) with the ring update and the window selection ([ref-attn] WindowCache,
 * window_topk_idxs), in one pass.  kv_in bf16 [B*T][hd] (the normed rows), kv_out bf16 [B*T][hd]
 * (may alias kv_in), ring bf16 [B][W][hd], win_idx int32 [B*T][idx_stride] (first W columns),
 * codes uint8 [B*T][hd] and scales int8 [B*T][hd/32] may be NULL.  Prefill (start_pos == 0): the
 * last min(T, W) rows enter the ring, row t selects {t-W+1..t} (-1 below 0).  Decode (T == 1): slot
 * start_pos mod W is written, then the whole ring is selected oldest first (-1 for never-written). */
CSA_API int csa_kv_finish(const csa_bf16 *kv_in, csa_bf16 *kv_out, int B, int T, int start_pos, int hd, int rd,
                  const float *tab, int tab_rows, csa_bf16 *ring, int W, int32_t *win_idx, int idx_stride,
                  uint8_t *codes, int8_t *scales, csa_stream stream);

/* Indexer scores ([atlas] "Indexer, re-scored"): S[t][j] = sum_h wI[t][h] ReLU(qI[t][h] . KI[b][j])
 * for the valid j of query t (j < floor((start_pos + t%T + 1) / ratio), j < compress_len, candidate
 * block j / cand_block allowed when cand != NULL); other entries of S are not written.
 * qI bf16 [B*T][Hi][dI], wI f32 [B*T][Hi], KI bf16 [B][Lstride][dI], S f32 [B*T][Lstride],
 * cand uint8 [B*T][cand_width] or NULL. */
CSA_API int csa_index_scores(const csa_bf16 *qI, const float *wI, const csa_bf16 *KI, int B, int T, int start_pos, int Hi,
                     int dI, int Lstride, int compress_len, int ratio, const uint8_t *cand, int cand_width,
                     int cand_block, float *S, csa_stream stream);

/* The candidate source's block mask ([attn_v41] module description: the candidate-source layer
 * publishes a block-level candidate mask that later index sources apply; SharedV41 candidates;
 * [atlas] config.json candidate_block_size, candidate_topk_blocks): per query t, block c (positions
 * c*cand_block .. c*cand_block + cand_block - 1) scores the largest of its valid scores S[t][j]
 * (j < floor((start_pos + t%T + 1) / ratio), j < compress_len), a block without a valid position
 * is no candidate, and the K blocks of highest score (equal scores to the lower block, -0 == +0) get
 * mask[t][c] = 1, every other column 0.  The block score is a reading (the pages print none).
 * S f32 [B*T][Lstride] (this source's own scores, unmasked), mask uint8 [B*T][cand_width] with
 * cand_width * cand_block >= min(compress_len, Lstride); K <= 2048, cand_width <= 25600. */
CSA_API int csa_candidate_blocks(const float *S, int B, int T, int start_pos, int Lstride, int compress_len, int ratio,
                                 int cand_block, int K, uint8_t *mask, int cand_width, csa_stream stream);

/* Index top-k ([atlas] I_t = top_K over the valid scores; [attn_v41] selection offset past the
 * window rows, -1 = absent): per query, the K valid positions of highest score, equal scores to the
 * lower index, -0 == +0; written in that order as j + offset, then -1 when fewer are valid.
 * S f32 [B*T][Lstride] (only valid entries are read), out int32 [B*T][K]. */
CSA_API int csa_index_topk(const float *S, int B, int T, int start_pos, int Lstride, int compress_len, int ratio,
                   const uint8_t *cand, int cand_width, int cand_block, int K, int offset, int32_t *out,
                   csa_stream stream);

/* sparse_attn with the sink ([ref-attn] sparse_attn; [atlas] "Sparse attention"; [join]): per
 * query t and head h over Y = [rows_a; rows_b] of its sequence and J_t = [idx_a[t] (na columns);
 * idx_b[t] (nb columns)] with -1 skipped: S_i = scale * q.Y[J_i], O = sum_i exp(S_i) Y[J_i] /
 * (exp(sink_h) + sum_i exp(S_i)), in f32, bf16 out.  q bf16 [B*T][H][hd]; rows_a bf16, sequence b
 * at rows_a + b*a_seq_stride (elements), a_len rows; rows_b likewise (may be NULL with b_len 0);
 * idx_a int32 [B*T][na], idx_b int32 [B*T][nb] or NULL; sink f32 [H].  o bf16 [B*T][H][hd] (may be
 * NULL) receives O; o_rot (may be NULL) receives O with the inverse rotation of its last rd
 * ([atlas] "Grouped output": R_t^-1 on the last rd) at position start_pos + t%T from tab.
 * An index outside [-1, a_len + b_len) is a caller error: the kernel skips such an entry and
 * records it in the context's device status word (read with csa_status). */
CSA_API int csa_sparse_attn(csa_ctx *ctx, const csa_bf16 *q, int B, int T, int H, int hd, const csa_bf16 *rows_a,
                    int64_t a_seq_stride, int a_len, const csa_bf16 *rows_b, int64_t b_seq_stride, int b_len,
                    const int32_t *idx_a, int na, const int32_t *idx_b, int nb, const float *sink, float scale,
                    csa_bf16 *o, csa_bf16 *o_rot, int rd, int start_pos, const float *tab, int tab_rows,
                    csa_stream stream);

/* Allocation-free projection.  The pages have no counterpart: this is an addition for callers that
 * cannot allocate device memory -- a host runtime that owns a fixed device-memory budget and forbids
 * allocations outside it, or code that has no csa_ctx (csa_create allocates the context's
 * workspaces).  It computes exactly what csa_linear computes, y = x W^T with f32 accumulation and a
 * bf16 result (same arguments, same grouping), with the same tensor-core kernel, and allocates
 * nothing: no cudaMalloc, no cudaFree, no context.  Its scratch (Stream-K arrival counters, f32
 * partials, a status word) is one static device array of 5,505,280 bytes (5.25 MiB) inside the
 * library, which every GPU that loads the library holds until the process exits.
 * Limits: M <= 32 tokens; ceil(N/128) * groups <= 65536; x and W 16-byte aligned, ldx and ldw
 * multiples of 8, K a multiple of 8 (of 64 when groups > 1).  Beyond them it returns CSA_ERR_SHAPE or
 * CSA_ERR_ARG and launches nothing.
 * The first call on a device looks the array's device address up (cudaGetSymbolAddress, once per
 * device and CUDA context, with that device current); make that first call before any stream
 * capture.  After a device reset the next call looks the address up again.
 * Every call shares the one array and it keeps the last call's contents: each call clears the
 * counters it needs on `stream` before its launch, but calls whose work overlaps on the GPU (on
 * different streams or from different threads) race on the array and must not be issued.
 * A bounded device-side wait that runs out is not reported by the return code (the call returns
 * once the work is enqueued): it sets the array's status word, which csa_linear_noalloc_status
 * reads. */
CSA_API int csa_linear_noalloc(const csa_bf16 *x, int M, int K, int ldx, const csa_bf16 *W, int N, int ldw,
                               csa_bf16 *y, int ldy, int groups, csa_stream stream);

/* The status word of csa_linear_noalloc on the current device: synchronises the device, then returns
 * CSA_OK, or CSA_ERR_DEVICE_TIMEOUT when a bounded wait of some call since the last clear ran out (the
 * outputs of those calls are invalid).  The word is sticky; clear != 0 resets it.  Allocates
 * nothing.  CSA_OK when no call has run on this device. */
CSA_API int csa_linear_noalloc_status(int clear);

#ifdef __cplusplus
}
#endif

#endif /* CSA_H_ */
