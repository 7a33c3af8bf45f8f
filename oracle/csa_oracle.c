/*
 * csa_oracle.c -- CPU oracle for the DeepSeek-V4.1 compressed sparse attention layer core.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct CPU statement of what
 * the GPU library computes.  Only the test suite, the package smoke check and the benchmark's CPU
 * baseline leg load it; the product never does, and it shares no source, header or table with the
 * CUDA path.  Every function restates a definition from the pages it cites:
 *
 *   [ref-attn]   "deepseek_v41_ref::attn" rustdoc page: the precision contract, the ring fixture and
 *                the helpers act_quant_inplace, pow2_ceil, apply_rotary, freqs_cis, sparse_attn and
 *                window_topk_idxs.
 *   [atlas]      "DeepSeek V4.1 - Compressed sparse attention" (Re-indexing layer, decode p=1000)
 *                atlas page: the formula chain "All 25 steps", the parameter table, the
 *                Attention.forward excerpt of model.py and config.json.
 *   [join]       "Join rows" atlas page: Y = [W; Z], compressed indices offset by |W|.
 *   [attn_v41]   "metrale_model_arch::attn_v41" rustdoc page and attn_v41.rs source: roles, the
 *                shared selection (offset past the window rows, -1 = absent), the candidate mask and
 *                the refusal rules.
 *
 * Arithmetic: where the pages fix a precision (bf16 tensors, f32 scores and tables, f32 RoPE
 * products) the result is rounded to it at the same point; everything in between is carried in
 * double, i.e. the exact value up to one final rounding.  Compile with -ffp-contract=off so that no
 * product/sum pair is fused.
 *
 * Parity pins: every function here is checked by tests/test_oracle_*.py against facts the pages or
 * mathematics fix (the 12-into-8 ring fixture, the e4m3 format table, closed forms of the softmax
 * with sink, brute force on tiny inputs, the published parameter counts).  The YaRN variant of the
 * RoPE table follows the published method, as the pages give its constants but not its formula: its
 * frequency classes by rotation count and the blend weight of every pair inside the ramp are checked
 * against ramp ends found by searching the rotation counts.
 *
 * Parity unpinned: orc_compress, the kv source's compressor.  The pages give its weights, state and
 * caches but not its pooling formula, so the reading it follows (softmax-gated pooling of each closed
 * group, RMSNorm, RoPE at the group's first position, the fp8 round trip) is checked only against
 * what mathematics fixes (products, closed forms of the pooling, composition of pinned steps,
 * complete-group publication, chunking invariance), not against the real model.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_ARG -1
#define ORC_ERR_INDEX -2

/* ------------------------------------------------------------------------------------------------
 * Numeric primitives
 * ----------------------------------------------------------------------------------------------*/

static float f32_from_bits(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}
static uint32_t bits_from_f32(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

/* bf16 is the top half of an IEEE binary32. */
float orc_bf16_to_f32(uint16_t b) { return f32_from_bits((uint32_t)b << 16); }

/* binary32 -> bf16, round to nearest, ties to even on the dropped 16 bits; NaN stays a quiet NaN. */
uint16_t orc_f32_to_bf16(float f) {
  uint32_t u = bits_from_f32(f);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

static double bfd(uint16_t b) { return (double)orc_bf16_to_f32(b); }

/* [ref-attn] pow2_ceil: 2^ceil(log2 v) for a positive normal binary32, read off the IEEE fields:
 * v itself when its 23 mantissa bits are zero, else the power of two one binade up. */
float orc_pow2_ceil(float v) {
  uint32_t u = bits_from_f32(v);
  if ((u & 0x007fffffu) == 0) return v;
  uint32_t e = (u >> 23) & 0xffu;
  return f32_from_bits((e + 1u) << 23);
}

/* E4M3 ("fn" variant, OCP 8-bit floating point format): sign, 4 exponent bits with bias 7,
 * 3 mantissa bits, no infinities, S.1111.111 is NaN, so the largest finite magnitude is
 * 1.75 * 2^8 = 448.  Normal numbers (8+m) * 2^(E-10) for E = 1..15, subnormals m * 2^-9.
 * Encoding rounds to nearest, ties to even, and saturates at +-448 (the "clamped" in [ref-attn]
 * act_quant_inplace). */
uint8_t orc_e4m3_encode(float v) {
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (!(a < 448.0)) return (uint8_t)(sign | 0x7e);
  if (a < ldexp(1.0, -6)) {
    /* subnormal binade: quantum 2^-9; q == 8 lands exactly on the smallest normal, code 0x08 */
    double q = nearbyint(a * 512.0);
    return (uint8_t)(sign | (uint8_t)q);
  }
  int e2;
  frexp(a, &e2);   /* a = f * 2^e2 with f in [0.5, 1) */
  int E = e2 - 1;  /* floor(log2 a), in [-6, 8] */
  double q = nearbyint(ldexp(a, 3 - E)); /* significand scaled to [8, 16] */
  if (q == 16.0) {
    q = 8.0;
    E += 1;
  }
  if (E > 8 || (E == 8 && q > 14.0)) return (uint8_t)(sign | 0x7e);
  return (uint8_t)(sign | (uint8_t)(((E + 7) << 3) | ((int)q - 8)));
}

float orc_e4m3_decode(uint8_t c) {
  int s = c >> 7, E = (c >> 3) & 15, m = c & 7;
  if (E == 15 && m == 7) return NAN;
  double a = (E == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), E - 10);
  return (float)(s ? -a : a);
}

/* ------------------------------------------------------------------------------------------------
 * Steps of the layer
 * ----------------------------------------------------------------------------------------------*/

/* [ref-attn] "Precision": every projection is linear_bf16, f32 accumulation and a bf16 result.
 * y[m][n] = bf16( sum_k x[m][k] * W[n][k] ), W is [out, in] row-major.  The sum is exact in double
 * (products of two bf16 are exact) up to its final rounding, which is the f32 -> bf16 one. */
void orc_linear_bf16(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, const uint16_t *W, int64_t N,
                     int64_t ldw, uint16_t *y, int64_t ldy) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      const uint16_t *xr = x + m * ldx;
      const uint16_t *wr = W + n * ldw;
      for (int64_t k = 0; k < K; ++k) acc += bfd(xr[k]) * bfd(wr[k]);
      y[m * ldy + n] = orc_f32_to_bf16((float)acc);
    }
  }
}

/* [ref-attn] "Precision": RMSNorm computes in f32 and returns bf16.  y = x / sqrt(mean(x^2) + eps) * w,
 * w an f32 vector (q_norm / kv_norm in the attn_v41 layer weights). */
void orc_rmsnorm(const uint16_t *x, int64_t M, int64_t N, const float *w, float eps, uint16_t *y) {
  for (int64_t m = 0; m < M; ++m) {
    double ss = 0.0;
    for (int64_t n = 0; n < N; ++n) ss += bfd(x[m * N + n]) * bfd(x[m * N + n]);
    double r = 1.0 / sqrt(ss / (double)N + (double)eps);
    for (int64_t n = 0; n < N; ++n)
      y[m * N + n] = orc_f32_to_bf16((float)(bfd(x[m * N + n]) * r * (double)w[n]));
  }
}

/* [ref-attn] freqs_cis: the RoPE table [max_seq][rd/2] of (cos, sin), f32.  Pair i rotates at
 * frequency theta^(-2i/rd); position p turns it by the angle p * f_i.  The angle and its cosine and
 * sine are taken in double and rounded once to f32.
 *
 * Ratio > 0 layers use compress_rope_theta with YaRN ([atlas] Attention.__init__ excerpt:
 * original_seq_len and rope_factor, beta_fast, beta_slow).  The pages give the constants only; this
 * follows the published YaRN frequency interpolation (Peng et al., 2023, "NTK-by-parts"): for the
 * pair whose wavelength completes n rotations over the original length L, the index is
 * d(n) = rd * ln(L / (2 pi n)) / (2 ln theta); pairs below floor(d(beta_fast)) keep f_i, pairs above
 * ceil(d(beta_slow)) use f_i / factor, and a linear ramp over the pair index blends the two in
 * between.  Applied only when max_seq exceeds the original length, as the excerpt passes
 * original_seq_len through to the table.  Pinned by the tests: the frequency classes, and each pair's
 * blend weight against ramp ends found by searching the rotation counts. */
int orc_rope_table(int rd, int64_t max_seq, double theta, int64_t orig_seq, double factor, double beta_fast,
                   double beta_slow, float *tab) {
  if (rd <= 0 || (rd & 1) || max_seq <= 0 || !tab) return ORC_ERR_ARG;
  int half = rd / 2;
  double *f = (double *)malloc(sizeof(double) * (size_t)half);
  if (!f) return ORC_ERR_ARG;
  for (int i = 0; i < half; ++i) f[i] = pow(theta, -2.0 * (double)i / (double)rd);
  if (orig_seq > 0 && max_seq > orig_seq) {
    const double two_pi = 6.283185307179586476925286766559;
    double d_fast = (double)rd * log((double)orig_seq / (two_pi * beta_fast)) / (2.0 * log(theta));
    double d_slow = (double)rd * log((double)orig_seq / (two_pi * beta_slow)) / (2.0 * log(theta));
    double lo = floor(d_fast), hi = ceil(d_slow);
    if (lo < 0.0) lo = 0.0;
    if (hi > (double)(rd - 1)) hi = (double)(rd - 1);
    if (hi == lo) hi += 0.001;
    for (int i = 0; i < half; ++i) {
      double ramp = ((double)i - lo) / (hi - lo);
      if (ramp < 0.0) ramp = 0.0;
      if (ramp > 1.0) ramp = 1.0;
      f[i] = f[i] / factor * ramp + f[i] * (1.0 - ramp);
    }
  }
  for (int64_t p = 0; p < max_seq; ++p)
    for (int i = 0; i < half; ++i) {
      double ang = (double)p * f[i];
      tab[(p * half + i) * 2 + 0] = (float)cos(ang);
      tab[(p * half + i) * 2 + 1] = (float)sin(ang);
    }
  free(f);
  return ORC_OK;
}

/* [ref-attn] apply_rotary: rotate the last rd elements of each row_len-wide row; adjacent elements
 * (2i, 2i+1) are one complex number a + ib, multiplied by (c + is) = freqs_cis[pos][i] in f32
 * (the conjugate c - is when inverse), written back as bf16.  Each product and each sum is rounded
 * to f32 on its own: re = fl(fl(a c) - fl(b s)), im = fl(fl(a s) + fl(b c)).
 * Row r uses position pos[r / rows_per_pos] (rows_per_pos = n_heads for q and o, 1 for kv). */
int orc_apply_rotary(uint16_t *x, int64_t rows, int row_len, int rd, const int32_t *pos, int rows_per_pos,
                     const float *tab, int64_t tab_rows, int inverse) {
  if (rd > row_len || (rd & 1) || rows_per_pos <= 0) return ORC_ERR_ARG;
  int half = rd / 2;
  for (int64_t r = 0; r < rows; ++r) {
    int64_t p = pos[r / rows_per_pos];
    if (p < 0 || p >= tab_rows) return ORC_ERR_INDEX;
    uint16_t *t = x + r * row_len + (row_len - rd);
    for (int i = 0; i < half; ++i) {
      float a = orc_bf16_to_f32(t[2 * i]), b = orc_bf16_to_f32(t[2 * i + 1]);
      float c = tab[(p * half + i) * 2 + 0], s = tab[(p * half + i) * 2 + 1];
      if (inverse) s = -s;
      float ac = a * c, bs = b * s, as = a * s, bc = b * c;
      float re = ac - bs, im = as + bc;
      t[2 * i] = orc_f32_to_bf16(re);
      t[2 * i + 1] = orc_f32_to_bf16(im);
    }
  }
  return ORC_OK;
}

/* [ref-attn] act_quant_inplace, FP8_BLOCK = 32: per block, scale s = pow2_ceil(max(amax, 1e-4) / 448)
 * (f32 division), codes c = e4m3(clamp(v / s, -448, 448)) rounded to nearest even, value v' = bf16(c * s).
 * The result is bf16-exact (an e4m3 value times a power of two).  codes[i] receives c and
 * scale_exp[block] the exponent k of s = 2^k (either may be NULL).  n must be a multiple of 32. */
int orc_act_quant(uint16_t *x, int64_t n, uint8_t *codes, int8_t *scale_exp) {
  if (n % 32) return ORC_ERR_ARG;
  for (int64_t b = 0; b < n / 32; ++b) {
    uint16_t *blk = x + b * 32;
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) {
      float a = fabsf(orc_bf16_to_f32(blk[i]));
      if (a > amax) amax = a;
    }
    float floor_amax = amax > 1e-4f ? amax : 1e-4f;
    float s = orc_pow2_ceil(floor_amax / 448.0f);
    for (int i = 0; i < 32; ++i) {
      float v = orc_bf16_to_f32(blk[i]) / s;
      if (v > 448.0f) v = 448.0f;
      if (v < -448.0f) v = -448.0f;
      uint8_t c = orc_e4m3_encode(v);
      if (codes) codes[b * 32 + i] = c;
      blk[i] = orc_f32_to_bf16(orc_e4m3_decode(c) * s);
    }
    if (scale_exp) scale_exp[b] = (int8_t)((int)((bits_from_f32(s) >> 23) & 0xffu) - 127);
  }
  return ORC_OK;
}

/* [ref-attn] window_topk_idxs, prefill form (start_pos == 0): query t sees the causal window of its
 * own chunk, J^w_t = {max(0, t-W+1), ..., t} ([atlas] "Sparse attention" J^w); W columns in ascending
 * position, a column whose position would be negative holds -1.  Values index the chunk's rows. */
void orc_window_idx_prefill(int64_t T, int W, int32_t *idx) {
  for (int64_t t = 0; t < T; ++t)
    for (int k = 0; k < W; ++k) {
      int64_t p = t - W + 1 + k;
      idx[t * W + k] = p >= 0 ? (int32_t)p : -1;
    }
}

/* [ref-attn] window_topk_idxs, decode form (one query at position p, after the ring write of p):
 * the whole ring oldest first.  Slot of position p' is p' mod W, so the k-th oldest live position
 * p-W+1+k sits in slot (p+1+k) mod W; a slot whose position would be negative was never written: -1. */
void orc_window_idx_decode(int64_t p, int W, int32_t *idx) {
  for (int k = 0; k < W; ++k) {
    int64_t pk = p - W + 1 + k;
    idx[k] = pk >= 0 ? (int32_t)((p + 1 + k) % W) : -1;
  }
}

/* [ref-attn] WindowCache and the ring fixture: row of position p lives in slot p mod W.  A call
 * writes its T rows in order, so of a chunk longer than the ring only the last W land. */
void orc_ring_write(uint16_t *ring, int W, int hd, const uint16_t *rows, int64_t T, int64_t start_pos) {
  int64_t first = T > W ? T - W : 0;
  for (int64_t t = first; t < T; ++t) memcpy(ring + ((start_pos + t) % W) * hd, rows + t * hd, sizeof(uint16_t) * (size_t)hd);
}

/* Validity of compressed position j for a query at absolute position pos ([atlas] "Indexer"
 * I_t = top_512(S^I_{t,j} : j < floor((t+1)/ratio), M^c_{t,j})): causal limit, the published cache
 * length ([attn_v41] SharedV41.compress_len), and the candidate block mask when the layer uses it
 * ([attn_v41] LayerRole.uses_candidates; M^c_{t,j} = candidates[t][j / cand_block]). */
static int comp_valid(int64_t j, int64_t pos, int ratio, int64_t compress_len, const uint8_t *cand_row,
                      int cand_block) {
  if (ratio <= 0) return 0;
  if (j >= (pos + 1) / ratio) return 0;
  if (j >= compress_len) return 0;
  if (cand_row && !cand_row[j / cand_block]) return 0;
  return 1;
}

/* [atlas] "Indexer, re-scored": S^I[t][j] = sum_h w^I[t][h] * ReLU(Q^I[t][h] . K^I[j]) for the
 * valid j of query t; invalid j are written as -inf (they take no part in the selection).
 * qI [n_tok][Hi][dI] bf16, wI [n_tok][Hi] f32, KI [Lc][dI] bf16 (one sequence), pos [n_tok]. */
void orc_index_scores(const uint16_t *qI, const float *wI, const uint16_t *KI, int64_t n_tok, int Hi, int dI,
                      int64_t Lc, const int32_t *pos, int ratio, int64_t compress_len, const uint8_t *cand,
                      int cand_width, int cand_block, float *S) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t t = 0; t < n_tok; ++t) {
    for (int64_t j = 0; j < Lc; ++j) {
      const uint8_t *cr = cand ? cand + t * cand_width : NULL;
      if (!comp_valid(j, pos[t], ratio, compress_len, cr, cand_block)) {
        S[t * Lc + j] = -INFINITY;
        continue;
      }
      double acc = 0.0;
      for (int h = 0; h < Hi; ++h) {
        double dot = 0.0;
        for (int d = 0; d < dI; ++d) dot += bfd(qI[(t * Hi + h) * dI + d]) * bfd(KI[j * dI + d]);
        if (dot > 0.0) acc += (double)wI[t * Hi + h] * dot;
      }
      S[t * Lc + j] = (float)acc;
    }
  }
}

typedef struct {
  float s;
  int64_t j;
} orc_cand;

/* Order for the selection: higher score first, equal scores by lower index.  -0 and +0 compare
 * equal (IEEE), a NaN score ranks below every number. */
static int cand_cmp(const void *pa, const void *pb) {
  const orc_cand *a = (const orc_cand *)pa, *b = (const orc_cand *)pb;
  int an = isnan(a->s), bn = isnan(b->s);
  if (an != bn) return an ? 1 : -1;
  if (!an) {
    if (a->s > b->s) return -1;
    if (a->s < b->s) return 1;
  }
  return (a->j < b->j) ? -1 : (a->j > b->j);
}

/* [atlas] I_t = top_512 of the valid scores; [attn_v41] the selection is [queries][topk], offset
 * past the window rows, -1 = absent.  Equal scores go to the lower index (a fixed tie rule in place
 * of the pages' torch CPU tie order).  Fewer valid positions than K: all of them, then -1.
 * Output in selection order (score descending, index ascending), each value j + offset. */
void orc_index_topk(const float *S, int64_t n_tok, int64_t Lc, int K, const int32_t *pos, int ratio,
                    int64_t compress_len, const uint8_t *cand, int cand_width, int cand_block, int32_t offset,
                    int32_t *out) {
#pragma omp parallel for schedule(dynamic)
  for (int64_t t = 0; t < n_tok; ++t) {
    const uint8_t *cr = cand ? cand + t * cand_width : NULL;
    orc_cand *c = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)(Lc > 0 ? Lc : 1));
    int64_t n = 0;
    for (int64_t j = 0; j < Lc; ++j)
      if (comp_valid(j, pos[t], ratio, compress_len, cr, cand_block)) {
        c[n].s = S[t * Lc + j];
        c[n].j = j;
        ++n;
      }
    qsort(c, (size_t)n, sizeof(orc_cand), cand_cmp);
    for (int k = 0; k < K; ++k) out[t * K + k] = k < n ? (int32_t)(c[k].j + offset) : -1;
    free(c);
  }
}

/* [ref-attn] sparse_attn / [atlas] "Sparse attention": for query t and head h over the gathered
 * rows G_t = Y[J_t] of Y = [rows_a; rows_b] ([join]), with -1 entries skipped:
 *   S_i = (q_{t,h} . G_i) * scale,  A_i = exp(S_i) / (exp(sink_h) + sum_j exp(S_j)),  O = sum_i A_i G_i,
 * the sink counted in the denominator only.  Carried in double (max-shifted), output bf16.
 * q [n_tok][H][hd], idx [n_tok][n_idx]; returns ORC_ERR_INDEX for an entry outside [-1, rows). */
int orc_sparse_attn(const uint16_t *q, int64_t n_tok, int H, int hd, const uint16_t *rows_a, int64_t rows_a_len,
                    const uint16_t *rows_b, int64_t rows_b_len, const int32_t *idx, int n_idx, const float *sink,
                    double scale, uint16_t *o) {
  int64_t n_rows = rows_a_len + rows_b_len;
  for (int64_t t = 0; t < n_tok; ++t)
    for (int i = 0; i < n_idx; ++i) {
      int32_t v = idx[t * n_idx + i];
      if (v < -1 || v >= n_rows) return ORC_ERR_INDEX;
    }
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t t = 0; t < n_tok; ++t)
    for (int h = 0; h < H; ++h) {
      const int32_t *it = idx + t * n_idx;
      const uint16_t *qh = q + (t * H + h) * hd;
      double *sc = (double *)malloc(sizeof(double) * (size_t)(n_idx > 0 ? n_idx : 1));
      double *acc = (double *)calloc((size_t)hd, sizeof(double));
      double m = (double)sink[h];
      for (int i = 0; i < n_idx; ++i) {
        if (it[i] < 0) continue;
        const uint16_t *g = it[i] < rows_a_len ? rows_a + (int64_t)it[i] * hd : rows_b + ((int64_t)it[i] - rows_a_len) * hd;
        double d = 0.0;
        for (int k = 0; k < hd; ++k) d += bfd(qh[k]) * bfd(g[k]);
        sc[i] = d * scale;
        if (sc[i] > m) m = sc[i];
      }
      double den = exp((double)sink[h] - m);
      for (int i = 0; i < n_idx; ++i) {
        if (it[i] < 0) continue;
        const uint16_t *g = it[i] < rows_a_len ? rows_a + (int64_t)it[i] * hd : rows_b + ((int64_t)it[i] - rows_a_len) * hd;
        double e = exp(sc[i] - m);
        den += e;
        for (int k = 0; k < hd; ++k) acc[k] += e * bfd(g[k]);
      }
      for (int k = 0; k < hd; ++k) o[(t * H + h) * hd + k] = orc_f32_to_bf16((float)(acc[k] / den));
      free(sc);
      free(acc);
    }
  return ORC_OK;
}

/* ------------------------------------------------------------------------------------------------
 * The layer forward ([atlas] Attention.forward excerpt and "All 25 steps")
 * ----------------------------------------------------------------------------------------------*/

typedef struct orc_cfg {
  int dim, n_heads, head_dim, rope_dim, q_rank, o_rank, groups, window;
  float eps;
  int index_heads, index_hd, index_topk, cand_block;
} orc_cfg;

typedef struct orc_role {
  int ratio, is_index_source, uses_candidates;
} orc_role;

typedef struct orc_weights {
  const float *sink, *q_norm, *kv_norm;
  const uint16_t *wq_a, *wq_b, *wkv, *wo_a, *wo_b, *idx_wq_b, *idx_wproj;
} orc_weights;

/* Shared state published by source layers ([attn_v41] SharedV41), one block per sequence. */
typedef struct orc_shared {
  const uint16_t *compress_kv; /* [B][Lstride][hd] */
  const uint16_t *index_k;     /* [B][Lstride][dI] */
  int64_t compress_len, Lstride;
  int32_t *topk_idxs; /* [B*T][index_topk]: written by an index source, read by the other ratio > 0 layers */
  const uint8_t *candidates; /* [B*T][cand_width] or NULL */
  int cand_width;
} orc_shared;

/* Optional intermediates ([attn_v41] AttnV41Run), each NULL or a full [B*T ...] buffer. */
typedef struct orc_debug {
  uint16_t *q;         /* [B*T][H][hd]  q after RoPE */
  uint16_t *kv;        /* [B*T][hd]     kv row after RoPE and the fp8 round trip */
  uint8_t *kv_codes;   /* [B*T][hd]     e4m3 codes */
  int8_t *kv_scale;    /* [B*T][hd/32]  scale exponents */
  int32_t *idx;        /* [B*T][n_idx]  the joined selection J (window then compressed + rows_a_len) */
  float *scores;       /* [B*T][Lstride] indexer scores (index sources) */
  uint16_t *o;         /* [B*T][H][hd]  sparse_attn output before the inverse rotation */
  uint16_t *og;        /* [B*T][G*o_rank] grouped projection */
  uint16_t *qr;        /* [B*T][q_rank] */
  uint16_t *qI;        /* [B*T][Hi*dI] */
  float *wI;           /* [B*T][Hi] */
} orc_debug;

/* The number of joined selection columns: the window, plus index_topk when ratio > 0. */
int orc_n_idx(const orc_cfg *c, const orc_role *r) { return c->window + (r->ratio > 0 ? c->index_topk : 0); }

/* One layer forward for B sequences of T tokens at start_pos (prefill: start_pos == 0; decode:
 * start_pos > 0 and T == 1).  x [B][T][dim] bf16; ring [B][W][hd] bf16 (updated); out [B][T][dim].
 * tok_mask (NULL = all) restricts which rows of out (and of the debug outputs) are produced, for
 * sampled checks at full size; the ring is always updated in full.  Refusals follow [attn_v41]
 * "Invariants": a ratio > 0 layer without a published latent cache, or a reuse layer without a
 * published selection, returns ORC_ERR_ARG. */
int orc_attn_forward(const orc_cfg *c, const orc_role *role, const orc_weights *w, uint16_t *ring,
                     const uint16_t *x, int B, int64_t T, int64_t start_pos, orc_shared *sh, const float *rope_tab,
                     int64_t rope_rows, const uint8_t *tok_mask, uint16_t *out, orc_debug *dbg) {
  const int H = c->n_heads, hd = c->head_dim, rd = c->rope_dim, W = c->window;
  const int G = c->groups, gw = H * hd / G, Hi = c->index_heads, dI = c->index_hd, K = c->index_topk;
  const int ratio = role->ratio;
  if (B <= 0 || T <= 0 || start_pos < 0) return ORC_ERR_ARG;
  if (start_pos > 0 && T != 1) return ORC_ERR_ARG;
  if (start_pos + T > rope_rows) return ORC_ERR_ARG;
  if (ratio > 0 && (!sh || !sh->compress_kv)) return ORC_ERR_ARG;
  if (ratio > 0 && role->is_index_source && !sh->index_k) return ORC_ERR_ARG;
  if (ratio > 0 && !sh->topk_idxs) return ORC_ERR_ARG;
  const int n_idx = orc_n_idx(c, role);
  const int64_t NT = (int64_t)B * T;
  const int decode = start_pos > 0;

  /* which kv rows each sequence needs: the window of every produced token, the ring's last W */
  uint8_t *need_kv = (uint8_t *)calloc((size_t)NT, 1);
  uint8_t *need_tok = (uint8_t *)calloc((size_t)NT, 1);
  for (int64_t r = 0; r < NT; ++r) need_tok[r] = tok_mask ? tok_mask[r] : 1;
  for (int b = 0; b < B; ++b)
    for (int64_t t = 0; t < T; ++t) {
      int64_t r = (int64_t)b * T + t;
      if (t >= T - W) need_kv[r] = 1;
      if (need_tok[r]) {
        need_kv[r] = 1;
        if (!decode)
          for (int64_t u = (t - W + 1 > 0 ? t - W + 1 : 0); u <= t; ++u) need_kv[(int64_t)b * T + u] = 1;
      }
    }

  int32_t *pos = (int32_t *)malloc(sizeof(int32_t) * (size_t)NT);
  for (int64_t r = 0; r < NT; ++r) pos[r] = (int32_t)(start_pos + r % T);

  /* kv path: wkv -> kv_norm -> RoPE on the last rd -> fp8 round trip ([atlas] "Window keys and values") */
  uint16_t *kv = (uint16_t *)calloc((size_t)(NT * hd), sizeof(uint16_t));
  uint16_t *tmp = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(hd > c->q_rank ? hd : c->q_rank));
  for (int64_t r = 0; r < NT; ++r) {
    if (!need_kv[r]) continue;
    orc_linear_bf16(x + r * c->dim, 1, c->dim, c->dim, w->wkv, hd, c->dim, tmp, hd);
    orc_rmsnorm(tmp, 1, hd, w->kv_norm, c->eps, kv + r * hd);
    orc_apply_rotary(kv + r * hd, 1, hd, rd, pos + r, 1, rope_tab, rope_rows, 0);
    orc_act_quant(kv + r * hd, hd, dbg && dbg->kv_codes ? dbg->kv_codes + r * hd : NULL,
                  dbg && dbg->kv_scale ? dbg->kv_scale + r * (hd / 32) : NULL);
    if (dbg && dbg->kv) memcpy(dbg->kv + r * hd, kv + r * hd, sizeof(uint16_t) * (size_t)hd);
  }

  /* q path: wq_a -> q_norm -> wq_b -> RoPE on the last rd of every head ([atlas] "Query compression",
   * "Query heads") */
  uint16_t *qr = (uint16_t *)calloc((size_t)(NT * c->q_rank), sizeof(uint16_t));
  uint16_t *q = (uint16_t *)calloc((size_t)(NT * H * hd), sizeof(uint16_t));
  for (int64_t r = 0; r < NT; ++r) {
    if (!need_tok[r]) continue;
    orc_linear_bf16(x + r * c->dim, 1, c->dim, c->dim, w->wq_a, c->q_rank, c->dim, tmp, c->q_rank);
    orc_rmsnorm(tmp, 1, c->q_rank, w->q_norm, c->eps, qr + r * c->q_rank);
    orc_linear_bf16(qr + r * c->q_rank, 1, c->q_rank, c->q_rank, w->wq_b, (int64_t)H * hd, c->q_rank, q + r * H * hd,
                    (int64_t)H * hd);
    orc_apply_rotary(q + r * H * hd, H, hd, rd, pos + r, H, rope_tab, rope_rows, 0);
    if (dbg && dbg->q) memcpy(dbg->q + r * H * hd, q + r * H * hd, sizeof(uint16_t) * (size_t)(H * hd));
    if (dbg && dbg->qr) memcpy(dbg->qr + r * c->q_rank, qr + r * c->q_rank, sizeof(uint16_t) * (size_t)c->q_rank);
  }

  int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)(NT * n_idx));
  uint16_t *o = (uint16_t *)calloc((size_t)(NT * H * hd), sizeof(uint16_t));
  int rc = ORC_OK;
  for (int b = 0; b < B && rc == ORC_OK; ++b) {
    int64_t r0 = (int64_t)b * T;
    uint16_t *ring_b = ring + (int64_t)b * W * hd;
    /* ring update, then the window selection ([ref-attn] the fixture's order: write, then read) */
    orc_ring_write(ring_b, W, hd, kv + r0 * hd, T, start_pos);
    const uint16_t *rows_a = decode ? ring_b : kv + r0 * hd;
    int64_t rows_a_len = decode ? W : T;
    for (int64_t t = 0; t < T; ++t) {
      int32_t *it = idx + (r0 + t) * n_idx;
      if (decode)
        orc_window_idx_decode(start_pos, W, it);
      else
        for (int k = 0; k < W; ++k) {
          int64_t p = t - W + 1 + k;
          it[k] = p >= 0 ? (int32_t)p : -1;
        }
    }
    const uint16_t *rows_b = NULL;
    int64_t rows_b_len = 0;
    if (ratio > 0) {
      rows_b = sh->compress_kv + (int64_t)b * sh->Lstride * hd;
      rows_b_len = sh->compress_len;
      int32_t *sel = sh->topk_idxs + r0 * K;
      if (role->is_index_source) {
        /* [atlas] "Indexer, re-scored": q^I = c^Q W_IQ, w^I = x W_IW / sqrt(dI * Hi) */
        uint16_t *qI = (uint16_t *)calloc((size_t)(T * Hi * dI), sizeof(uint16_t));
        float *wI = (float *)calloc((size_t)(T * Hi), sizeof(float));
        uint16_t *wraw = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)Hi);
        double wscale = 1.0 / sqrt((double)dI * (double)Hi);
        for (int64_t t = 0; t < T; ++t) {
          if (!need_tok[r0 + t]) continue;
          orc_linear_bf16(qr + (r0 + t) * c->q_rank, 1, c->q_rank, c->q_rank, w->idx_wq_b, (int64_t)Hi * dI, c->q_rank,
                          qI + t * Hi * dI, (int64_t)Hi * dI);
          orc_linear_bf16(x + (r0 + t) * c->dim, 1, c->dim, c->dim, w->idx_wproj, Hi, c->dim, wraw, Hi);
          for (int h = 0; h < Hi; ++h) wI[t * Hi + h] = (float)(bfd(wraw[h]) * wscale);
          if (dbg && dbg->qI) memcpy(dbg->qI + (r0 + t) * Hi * dI, qI + t * Hi * dI, sizeof(uint16_t) * (size_t)(Hi * dI));
          if (dbg && dbg->wI) memcpy(dbg->wI + (r0 + t) * Hi, wI + t * Hi, sizeof(float) * (size_t)Hi);
        }
        float *S = (float *)malloc(sizeof(float) * (size_t)sh->Lstride);
        const uint8_t *cand = role->uses_candidates ? sh->candidates : NULL;
        if (role->uses_candidates && !cand) rc = ORC_ERR_ARG;
        for (int64_t t = 0; t < T && rc == ORC_OK; ++t) {
          if (!need_tok[r0 + t]) continue;
          const uint8_t *cr = cand ? cand + (r0 + t) * sh->cand_width : NULL;
          orc_index_scores(qI + t * Hi * dI, wI + t * Hi, sh->index_k + (int64_t)b * sh->Lstride * dI, 1, Hi, dI,
                           sh->Lstride, pos + r0 + t, ratio, sh->compress_len, cr, sh->cand_width, c->cand_block, S);
          orc_index_topk(S, 1, sh->Lstride, K, pos + r0 + t, ratio, sh->compress_len, cr, sh->cand_width,
                         c->cand_block, (int32_t)rows_a_len, sel + t * K);
          if (dbg && dbg->scores) memcpy(dbg->scores + (r0 + t) * sh->Lstride, S, sizeof(float) * (size_t)sh->Lstride);
        }
        free(S);
        free(wraw);
        free(wI);
        free(qI);
      }
      /* [join] J = [J^w; I + |W|]: the published selection is already offset past the window rows */
      for (int64_t t = 0; t < T; ++t) memcpy(idx + (r0 + t) * n_idx + W, sel + t * K, sizeof(int32_t) * (size_t)K);
    }
    if (rc != ORC_OK) break;
    /* sparse attention for the produced tokens of this sequence */
    for (int64_t t = 0; t < T; ++t) {
      int64_t r = r0 + t;
      if (!need_tok[r]) continue;
      int e = orc_sparse_attn(q + r * H * hd, 1, H, hd, rows_a, rows_a_len, rows_b, rows_b_len, idx + r * n_idx, n_idx,
                              w->sink, 1.0 / sqrt((double)hd), o + r * H * hd);
      if (e != ORC_OK) {
        rc = e;
        break;
      }
    }
  }
  if (dbg && dbg->idx)
    for (int64_t r = 0; r < NT; ++r)
      if (need_tok[r]) memcpy(dbg->idx + r * n_idx, idx + r * n_idx, sizeof(int32_t) * (size_t)n_idx);

  /* [atlas] "Grouped output": O-bar = R_t^-1 O on the last rd, o^g_r = [O-bar_h]_{h in r} W_OA,r,
   * Delta = o^g W_OB.  Group g is heads [g*H/G, (g+1)*H/G), contiguous (the view in the excerpt). */
  if (rc == ORC_OK) {
    uint16_t *og = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)((int64_t)G * c->o_rank));
    for (int64_t r = 0; r < NT; ++r) {
      if (!need_tok[r]) continue;
      if (dbg && dbg->o) memcpy(dbg->o + r * H * hd, o + r * H * hd, sizeof(uint16_t) * (size_t)(H * hd));
      orc_apply_rotary(o + r * H * hd, H, hd, rd, pos + r, H, rope_tab, rope_rows, 1);
      for (int g = 0; g < G; ++g)
        orc_linear_bf16(o + r * H * hd + (int64_t)g * gw, 1, gw, gw, w->wo_a + (int64_t)g * c->o_rank * gw, c->o_rank, gw,
                        og + (int64_t)g * c->o_rank, c->o_rank);
      if (dbg && dbg->og) memcpy(dbg->og + r * G * c->o_rank, og, sizeof(uint16_t) * (size_t)(G * c->o_rank));
      orc_linear_bf16(og, 1, (int64_t)G * c->o_rank, (int64_t)G * c->o_rank, w->wo_b, c->dim, (int64_t)G * c->o_rank,
                      out + r * c->dim, c->dim);
    }
    free(og);
  }
  free(o);
  free(idx);
  free(q);
  free(qr);
  free(tmp);
  free(kv);
  free(pos);
  free(need_tok);
  free(need_kv);
  return rc;
}

/* The candidate source's block mask ([attn_v41] module description: the candidate-source layer
 * publishes a block-level candidate mask that later index sources apply; SharedV41 candidates
 * [queries][cand_width]; [atlas] config.json candidate_block_size, candidate_topk_blocks; the
 * candidate-block selection runs as a top-k, like the index selection).  The pages give no block
 * score; the reading taken here: block c of query t scores the largest of its valid positions'
 * indexer scores S[t][j] (j in [c*cb, (c+1)*cb), j < floor((pos+1)/ratio), j < compress_len); a block
 * with no valid position is not a candidate; the top cand_topk blocks by score (ties to the lower
 * block; -0 == +0) are marked 1, the rest 0.  S [n_tok][Lstride] f32 (this source's own, unmasked),
 * mask [n_tok][cand_width] uint8. */
void orc_candidate_blocks(const float *S, int64_t n_tok, int64_t Lstride, const int32_t *pos, int ratio,
                          int64_t compress_len, int cand_block, int cand_topk, int cand_width, uint8_t *mask) {
  orc_cand *c = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)(cand_width > 0 ? cand_width : 1));
  for (int64_t t = 0; t < n_tok; ++t) {
    int64_t limit = ((int64_t)pos[t] + 1) / ratio;
    if (limit > compress_len) limit = compress_len;
    int n = 0;
    for (int b = 0; b < cand_width; ++b) {
      float best = 0.0f;
      int any = 0;
      for (int64_t j = (int64_t)b * cand_block; j < (int64_t)(b + 1) * cand_block && j < limit; ++j) {
        float v = S[t * Lstride + j];
        if (!any || v > best) best = v;
        any = 1;
      }
      if (any) {
        c[n].s = best == 0.0f ? 0.0f : best; /* -0 -> +0 */
        c[n].j = b;
        ++n;
      }
    }
    qsort(c, (size_t)n, sizeof(orc_cand), cand_cmp);
    uint8_t *m = mask + t * cand_width;
    for (int b = 0; b < cand_width; ++b) m[b] = 0;
    for (int k = 0; k < n && k < cand_topk; ++k) m[c[k].j] = 1;
  }
  free(c);
}

/* ------------------------------------------------------------------------------------------------
 * Compressor of a kv-source layer
 * ----------------------------------------------------------------------------------------------*/

/* Weights of the compressor ([attn_v41] CompressorWeightsGpu): at ratio > 1 kv and gate are f32
 * [hd][dim]; at ratio 1 kv is bf16 [hd][dim] and there is no gate; norm is f32 [hd].  The index
 * keys of a kv source that is also an index source come from wk bf16 [dI][hd] and k_norm f32 [dI]
 * ([attn_v41] IndexerWeightsGpu); wk may be NULL (no index keys published). */
typedef struct orc_comp_weights {
  const float *wkv_f32;    /* ratio > 1 */
  const float *wgate;      /* ratio > 1 */
  const uint16_t *wkv_bf16; /* ratio 1 */
  const float *norm;
  const uint16_t *wk;
  const float *k_norm;
} orc_comp_weights;

/* The compressor ([attn_v41] module description "the compressor pooling"; AttnV41LayerState: the
 * partial group of f32 kv and score [ratio][hd], the score starting at -inf, the bf16 latent cache
 * [max_seq/ratio][hd] and index-key cache [max_seq/ratio][dI]; SharedV41: compress_len, the number
 * of groups written, only grows).  The pages give these shapes but not the pooling formula, so its
 * parity against the real model is unpinned; the reading taken here, token by token in position
 * order p = start_pos + t of each sequence:
 *   k_p = x_p Wkv^T and s_p = x_p Wgate^T, each an f32 [hd] (sums exact in double, one rounding to
 *     f32); at ratio 1 k_p = linear_bf16(x_p, Wkv) and there is no score;
 *   they fill slot p mod ratio of the partial group;
 *   when p closes group j = p / ratio ((p + 1) mod ratio == 0): per feature d, the group's rows are
 *     pooled with softmax weights of their scores, z[d] = sum_i e^{s_i[d]} k_i[d] / sum_i e^{s_i[d]}
 *     (at ratio 1, z = k_p), rounded to f32; y = RMSNorm(z) * norm (f32 arithmetic, bf16 result, as
 *     every RMSNorm of the precision contract); the index key is RMSNorm(linear_bf16(y, wk)) * k_norm;
 *     the latent row is y with RoPE on its last rd at the group's first position j * ratio, then the
 *     fp8 round trip of the window rows ([ref-attn] act_quant_inplace); row j of both caches is
 *     written, compress_len becomes at least j + 1, and the partial group restarts empty (scores
 *     -inf, kv 0), so rows of an unfinished group are never published.
 * st_kv, st_score: [B][ratio][hd]; Z [B][Lstride][hd], KI [B][Lstride][dI] (KI ignored without wk);
 * y_dbg (NULL or [B][Lstride][hd]): the normed rows before RoPE and fp8. */
int orc_compress(const orc_cfg *c, int ratio, const orc_comp_weights *w, float *st_kv, float *st_score,
                 const uint16_t *x, int B, int64_t T, int64_t start_pos, const float *rope_tab, int64_t rope_rows,
                 uint16_t *Z, uint16_t *KI, int64_t Lstride, int64_t *compress_len, uint16_t *y_dbg) {
  const int hd = c->head_dim, rd = c->rope_dim, dim = c->dim, dI = c->index_hd;
  if (ratio <= 0 || B <= 0 || T <= 0 || start_pos < 0 || !w || !w->norm) return ORC_ERR_ARG;
  if (ratio > 1 && (!w->wkv_f32 || !w->wgate)) return ORC_ERR_ARG;
  if (ratio == 1 && !w->wkv_bf16) return ORC_ERR_ARG;
  if ((start_pos + T) / ratio > Lstride) return ORC_ERR_ARG;
  double *z = (double *)malloc(sizeof(double) * (size_t)hd);
  float *zf = (float *)malloc(sizeof(float) * (size_t)hd);
  uint16_t *kb = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)hd);
  uint16_t *y = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)hd);
  uint16_t *kraw = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(dI > 0 ? dI : 1));
  for (int b = 0; b < B; ++b) {
    float *skv = st_kv + (int64_t)b * ratio * hd, *ssc = st_score + (int64_t)b * ratio * hd;
    for (int64_t t = 0; t < T; ++t) {
      const int64_t p = start_pos + t;
      const uint16_t *xr = x + ((int64_t)b * T + t) * dim;
      const int slot = (int)(p % ratio);
      if (ratio > 1) {
        for (int d = 0; d < hd; ++d) {
          double a = 0.0, g = 0.0;
          for (int k = 0; k < dim; ++k) {
            a += bfd(xr[k]) * (double)w->wkv_f32[(int64_t)d * dim + k];
            g += bfd(xr[k]) * (double)w->wgate[(int64_t)d * dim + k];
          }
          skv[slot * hd + d] = (float)a;
          ssc[slot * hd + d] = (float)g;
        }
      } else {
        orc_linear_bf16(xr, 1, dim, dim, w->wkv_bf16, hd, dim, kb, hd);
        for (int d = 0; d < hd; ++d) skv[d] = orc_bf16_to_f32(kb[d]);
      }
      if ((p + 1) % ratio) continue;
      const int64_t j = p / ratio;
      /* pooling of the closed group */
      for (int d = 0; d < hd; ++d) {
        if (ratio == 1) {
          z[d] = skv[d];
          continue;
        }
        double m = -INFINITY;
        for (int i = 0; i < ratio; ++i)
          if ((double)ssc[i * hd + d] > m) m = (double)ssc[i * hd + d];
        double num = 0.0, den = 0.0;
        for (int i = 0; i < ratio; ++i) {
          double e = exp((double)ssc[i * hd + d] - m);
          num += e * (double)skv[i * hd + d];
          den += e;
        }
        z[d] = num / den;
      }
      /* RMSNorm of the f32 pooled row */
      double ss = 0.0;
      for (int d = 0; d < hd; ++d) {
        zf[d] = (float)z[d];
        ss += (double)zf[d] * (double)zf[d];
      }
      double rs = 1.0 / sqrt(ss / (double)hd + (double)c->eps);
      for (int d = 0; d < hd; ++d) y[d] = orc_f32_to_bf16((float)((double)zf[d] * rs * (double)w->norm[d]));
      if (y_dbg) memcpy(y_dbg + ((int64_t)b * Lstride + j) * hd, y, sizeof(uint16_t) * (size_t)hd);
      /* index key */
      if (w->wk && KI) {
        orc_linear_bf16(y, 1, hd, hd, w->wk, dI, hd, kraw, dI);
        orc_rmsnorm(kraw, 1, dI, w->k_norm, c->eps, KI + ((int64_t)b * Lstride + j) * dI);
      }
      /* latent row: RoPE at the group's first position, then the fp8 round trip */
      uint16_t *zr = Z + ((int64_t)b * Lstride + j) * hd;
      memcpy(zr, y, sizeof(uint16_t) * (size_t)hd);
      int32_t gp = (int32_t)(j * ratio);
      if (gp >= rope_rows) {
        free(z), free(zf), free(kb), free(y), free(kraw);
        return ORC_ERR_INDEX;
      }
      orc_apply_rotary(zr, 1, hd, rd, &gp, 1, rope_tab, rope_rows, 0);
      orc_act_quant(zr, hd, NULL, NULL);
      if (j + 1 > *compress_len) *compress_len = j + 1;
      /* the partial group restarts empty */
      for (int i = 0; i < ratio * hd; ++i) {
        skv[i] = 0.0f;
        ssc[i] = -INFINITY;
      }
    }
  }
  free(z), free(zf), free(kb), free(y), free(kraw);
  return ORC_OK;
}

/* A kv source's partial group before its first token: kv 0, scores -inf ([attn_v41]
 * AttnV41LayerState::new, "the score state starts at -inf"). */
void orc_compress_state_init(float *st_kv, float *st_score, int64_t n) {
  for (int64_t i = 0; i < n; ++i) {
    st_kv[i] = 0.0f;
    st_score[i] = -INFINITY;
  }
}

/* Element counts of the weights orc_attn_forward reads, in the order of the [atlas] parameter
 * table: query compression (wq_a + q_norm), query heads (wq_b), window keys and values
 * (wkv + kv_norm), indexer (idx_wq_b + idx_wproj), sparse attention (sink), grouped output
 * (wo_a + wo_b).  counts[6] = the total. */
void orc_param_counts(const orc_cfg *c, int with_indexer, int64_t *counts) {
  int64_t H = c->n_heads, hd = c->head_dim, G = c->groups, gw = H * hd / G;
  counts[0] = (int64_t)c->q_rank * c->dim + c->q_rank;
  counts[1] = H * hd * c->q_rank;
  counts[2] = hd * c->dim + hd;
  counts[3] = with_indexer ? (int64_t)c->index_heads * c->index_hd * c->q_rank + (int64_t)c->index_heads * c->dim : 0;
  counts[4] = H;
  counts[5] = G * c->o_rank * gw + (int64_t)c->dim * G * c->o_rank;
  counts[6] = counts[0] + counts[1] + counts[2] + counts[3] + counts[4] + counts[5];
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ------------------------------------------------------------------------------------------------
 * Array forms of the primitives, for the test suite
 * ----------------------------------------------------------------------------------------------*/

void orc_f32_to_bf16_n(const float *x, uint16_t *y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = orc_f32_to_bf16(x[i]);
}
void orc_pow2_ceil_n(const float *x, float *y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = orc_pow2_ceil(x[i]);
}
void orc_e4m3_encode_n(const float *x, uint8_t *y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = orc_e4m3_encode(x[i]);
}
void orc_e4m3_decode_n(const uint8_t *x, float *y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = orc_e4m3_decode(x[i]);
}
