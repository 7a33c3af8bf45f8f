// k_attn_tc.cu -- sparse attention with the per-head sink on the 5th-generation tensor cores
// ("deepseek_v41_ref::attn" sparse_attn; "DeepSeek V4.1 - Compressed sparse attention", "Sparse
// attention" and "Grouped output"; "Join rows").
//
// One CTA per (query, group of HG heads).  All 64 heads of a query share one K = V row per selected
// position, so the CTA gathers the query's selected rows once per 128-row tile into shared memory
// (Y = [rows_a; rows_b] and J = [idx_a; idx_b] are never materialised: the two index lists are
// compacted to the valid entries and each entry names its source) and uses the tile twice:
//   S^T[r][h] = sum_d G[r][d] q[h][d]      (M = 128 rows, N = HG, K = 512; G and q K-major)
//   O^T[d][h] += sum_r G[r][d] P[h][r]     (M = 4 x 128 features, N = HG, K = 128 rows; the same G
//                                           tile read as an MN-major operand, P K-major)
// with the accumulators in TMEM.  The softmax runs on the scores in f32: a running maximum that
// starts at the head's sink (so the sink enters the denominator only, exp(sink - m)), raised only when
// a tile's maximum exceeds it by more than 2^8 (then O and the sum are rescaled), P rounded to bf16
// for the second product.  The epilogue divides by the sum, writes O as bf16 and, for the last
// rope_dim features, the inverse rotation of the bf16 value at the query's position.
//
// Warps 0-3: softmax and epilogue (TMEM lane quadrant = warp); warps 4-7: row gather (cp.async, one
// thread per tile row, into the 128-byte swizzled layout) and the compaction of the index lists;
// warp 8: TMEM allocation and MMA issue.  Every mbarrier wait is time-bounded.
#include "csa_internal.cuh"
#include "tc_ptx.cuh"

namespace csa {

namespace attn {

constexpr int HD = 512;              // head_dim this kernel serves
constexpr int KB = HD / 64;          // 64-feature K-blocks
constexpr int TILE = 128;            // rows per tile
constexpr int kThreads = 288;
constexpr int kMaxList = 2048;       // selection width bound (the API refuses wider)
constexpr uint32_t kSrcB = 0x80000000u;

struct Params {
  const bf16 *q;
  int T, H;
  const bf16 *rows_a;
  int64_t a_seq_rows;  // rows per sequence in rows_a
  int a_len;
  const bf16 *rows_b;
  int64_t b_seq_rows;
  int b_len;
  const int32_t *idx_a;
  int na;
  const int32_t *idx_b;
  int nb;
  const float *sink;
  float scale_log2;  // softmax scale * log2(e)
  bf16 *o, *o_rot;
  int rd, start_pos;
  const float *tab;
  int *status;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

template <int HG>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[HG]) {
#pragma unroll
  for (int c = 0; c < HG; c += 16) {
    uint32_t r[16];
    tc::tmem_ld16(taddr + (uint32_t)c, r);
    tc::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) v[c + i] = __uint_as_float(r[i]);
  }
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

template <int HG>
__global__ void __launch_bounds__(kThreads, 1) k_sparse_attn_tc(const __grid_constant__ Params P) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  uint8_t *sG = smem;                              // [KB][128 rows][128 B]
  uint8_t *sQ = sG + KB * TILE * 128;              // [KB][HG rows][128 B]
  uint8_t *sP = sQ + KB * HG * 128;                // [2][HG rows][128 B]
  uint32_t *list = reinterpret_cast<uint32_t *>(sP + 2 * HG * 128);  // [kMaxList] compacted rows
  float *red_max = reinterpret_cast<float *>(list + kMaxList);       // [4][HG]
  float *red_sum = red_max + 4 * HG;                                 // [4][HG]
  float *m_sm = red_sum + 4 * HG, *l_sm = m_sm + HG, *alpha_sm = l_sm + HG;  // [HG] each
  uint64_t *bars = reinterpret_cast<uint64_t *>(alpha_sm + HG + (HG & 1));
  uint64_t *g_full = bars + 0, *s_full = bars + 1, *p_full = bars + 2, *o_full = bars + 3, *sm_bar = bars + 4,
           *drain = bars + 5;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 6);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *s_nvalid = const_cast<int *>(abort_flag) + 1;
  int *s_cnt = s_nvalid + 1;  // [4] loader warp counts
  int *s_rescale = s_cnt + 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = blockIdx.y;  // query b*T + t
  const int hg = blockIdx.x;
  const int b = (int)(row / P.T), t = (int)(row % P.T);
  constexpr uint32_t kCols = (5 * HG <= 32) ? 32 : (5 * HG <= 64) ? 64 : (5 * HG <= 128) ? 128 : (5 * HG <= 256) ? 256 : 512;

  if (threadIdx.x == 0) {
    tc::mbar_init(g_full, 128);
    tc::mbar_init(s_full, 1);
    tc::mbar_init(p_full, 128);
    tc::mbar_init(o_full, 1);
    tc::mbar_init(sm_bar, 128);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    *s_nvalid = 0;
    *s_rescale = 0;
    tc::fence_barrier_init();
  }
  if (warp == 8) tc::tmem_alloc(tmem_slot, kCols);
  __syncthreads();

  // ---- compaction of the joined selection (loader warps): valid entries, in order, with their source
  const int n_all = P.na + P.nb;
  const int n_rows = P.a_len + P.b_len;
  if (warp >= 4 && warp < 8) {
    const int j = threadIdx.x - 128, lw = warp - 4;
    int base = 0;
    for (int e0 = 0; e0 < n_all; e0 += TILE) {
      const int e = e0 + j;
      int v = -1;
      if (e < P.na)
        v = P.idx_a[row * P.na + e];
      else if (e < n_all)
        v = P.idx_b[row * P.nb + (e - P.na)];
      const bool bad = e < n_all && (v < -1 || v >= n_rows);
      if (bad) atomicOr(P.status, kStatusBadIndex);
      const bool ok = e < n_all && v >= 0 && v < n_rows;
      const unsigned bal = __ballot_sync(0xffffffffu, ok);
      if (lane == 0) s_cnt[lw] = __popc(bal);
      tc::named_bar(2, 128);
      int before = base;
      for (int w = 0; w < lw; ++w) before += s_cnt[w];
      before += __popc(bal & ((1u << lane) - 1u));
      if (ok) {
        const uint32_t enc = v < P.a_len ? (uint32_t)(b * P.a_seq_rows + v)
                                         : (kSrcB | (uint32_t)(b * P.b_seq_rows + (v - P.a_len)));
        list[before] = enc;
      }
      int tot = 0;
      for (int w = 0; w < 4; ++w) tot += s_cnt[w];
      base += tot;
      tc::named_bar(2, 128);
    }
    if (j == 0) *s_nvalid = base;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nvalid = *s_nvalid;
  const int ntiles = (nvalid + TILE - 1) / TILE;
  const uint32_t tS = tmem, tO = tmem + HG;  // S^T: HG columns; O^T chunk c: HG columns at tO + c*HG

  if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------------ gather
    const int j = threadIdx.x - 128;  // tile row this thread loads
    const uint32_t g_base = tc::smem_u32(sG), q_base = tc::smem_u32(sQ);
    // q of this head group: HG rows x 512, K-major swizzled
    for (int c = j; c < HG * 64; c += 128) {
      const int h = c / 64, ch = c % 64, kb = ch / 8, cc = ch % 8;
      const bf16 *src = P.q + (row * P.H + hg * HG + h) * HD + ch * 8;
      cp_async16(q_base + kb * HG * 128 + h * 128 + ((cc ^ (h & 7)) << 4), src, true);
    }
    for (int k = 0; k < ntiles; ++k) {
      if (k > 0 && !tc::mbar_wait(o_full, (uint32_t)((k - 1) & 1), abort_flag)) break;
      const int e = k * TILE + j;
      const bool valid = e < nvalid;
      const bf16 *src = P.rows_a;
      if (valid) {
        const uint32_t enc = list[e];
        src = (enc & kSrcB) ? P.rows_b + (int64_t)(enc & ~kSrcB) * HD : P.rows_a + (int64_t)enc * HD;
      }
#pragma unroll 8
      for (int ch = 0; ch < 64; ++ch) {
        const int kb = ch / 8, cc = ch % 8;
        cp_async16(g_base + kb * TILE * 128 + j * 128 + ((cc ^ (j & 7)) << 4), src + (valid ? ch * 8 : 0), valid);
      }
      cp_async_wait_all();
      fence_proxy_async();
      tc::mbar_arrive(g_full);
    }
    cp_async_wait_all();  // no copy may be in flight when the CTA exits (q when nothing is selected)
  } else if (warp == 8) {
    // ------------------------------------------------------------------ MMA issue
    if (lane == 0 && ntiles > 0) {
      const uint32_t id1 = tc::idesc_bf16_f32(TILE, HG);
      const uint32_t id2 = tc::idesc_bf16_f32(TILE, HG, /*a_mn_major=*/true, /*b_mn_major=*/false);
      const uint32_t g_base = tc::smem_u32(sG), q_base = tc::smem_u32(sQ), p_base = tc::smem_u32(sP);
      for (int k = 0; k < ntiles; ++k) {
        if (!tc::mbar_wait(g_full, (uint32_t)(k & 1), abort_flag)) break;
        tc::tc_fence_after();
        // S^T = G q^T
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
          const uint64_t ad = tc::sdesc_sw128(g_base + kb * TILE * 128, 16, 1024);
          const uint64_t bd = tc::sdesc_sw128(q_base + kb * HG * 128, 16, 1024);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) tc::mma_bf16(tS, ad + 2ull * k4, bd + 2ull * k4, id1, (kb | k4) ? 1u : 0u);
        }
        tc::mma_commit(s_full);
        if (!tc::mbar_wait(p_full, (uint32_t)(k & 1), abort_flag)) break;
        tc::tc_fence_after();
        // O^T += G^T P^T, feature chunk c = K-blocks 2c, 2c+1 of the tile
#pragma unroll
        for (int c = 0; c < KB / 2; ++c) {
#pragma unroll
          for (int i = 0; i < TILE / 16; ++i) {
            const uint64_t ad = tc::sdesc_sw128(g_base + (2 * c) * TILE * 128 + i * 2048, TILE * 128, 1024);
            const uint64_t bd = tc::sdesc_sw128(p_base + (i / 4) * HG * 128 + (i % 4) * 32, 16, 1024);
            tc::mma_bf16(tO + (uint32_t)(c * HG), ad, bd, id2, (k > 0 || i > 0) ? 1u : 0u);
          }
        }
        tc::mma_commit(o_full);
      }
      tc::mma_commit(drain);
      const uint64_t t0 = tc::global_ns();
      while (!tc::mbar_try_wait(drain, 0) && tc::global_ns() - t0 < tc::kWaitLimitNs) {
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax + epilogue (warps 0-3)
    const int r = warp * 32 + lane;  // tile row (for S^T) and feature within a chunk (for O^T)
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    // running maximum (log2 domain) and sum per head, one copy each in shared memory, written by
    // thread h only; they start at the sink: m = sink, l = exp2(sink - m) = 1
    if (r < HG) {
      m_sm[r] = P.sink[hg * HG + r] * 1.4426950408889634f;
      l_sm[r] = 1.0f;
    }
    uint32_t sm_uses = 0;
    auto sm_sync = [&]() -> bool {
      tc::mbar_arrive(sm_bar);
      return tc::mbar_wait(sm_bar, (sm_uses++) & 1u, abort_flag);
    };
    bool ok = sm_sync();
    for (int k = 0; k < ntiles && ok; ++k) {
      if (!tc::mbar_wait(s_full, (uint32_t)(k & 1), abort_flag)) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      float s[HG];
      tmem_ld_cols<HG>(tS + lane_off, s);
      const bool valid = k * TILE + r < nvalid;
#pragma unroll
      for (int h = 0; h < HG; ++h) s[h] = valid ? s[h] * P.scale_log2 : -INFINITY;
      // tile maximum per head
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        float v = s[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) red_max[warp * HG + h] = v;
      }
      if (!(ok = sm_sync())) break;
      if (r < HG) {
        const float tmax = fmaxf(fmaxf(red_max[r], red_max[HG + r]), fmaxf(red_max[2 * HG + r], red_max[3 * HG + r]));
        float a = 1.0f;
        if (tmax > m_sm[r] + 8.0f) {  // keep exp2(s - m) below 2^8; rescale what has accumulated
          a = exp2f(m_sm[r] - tmax);
          m_sm[r] = tmax;
          l_sm[r] *= a;
          if (k > 0) *s_rescale = 1;
        }
        alpha_sm[r] = a;
      }
      if (!(ok = sm_sync())) break;
      if (*s_rescale) {
        // O^T columns h scale by alpha[h]; the previous tile's product has completed (its commit
        // released this tile's rows before the scores could be computed)
#pragma unroll 1
        for (int c = 0; c < KB / 2; ++c) {
#pragma unroll
          for (int c0 = 0; c0 < HG; c0 += 16) {
            uint32_t v[16];
            const uint32_t ta = tO + (uint32_t)(c * HG + c0) + lane_off;
            tc::tmem_ld16(ta, v);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha_sm[c0 + i]);
            tmem_st16(ta, v);
          }
        }
        tmem_st_wait();
      }
      // probabilities, their per-head sums, and P (bf16, K-major [HG][128 rows], swizzled)
      uint8_t *prow = sP + (r / 64) * HG * 128;
      const int rc = (r % 64) / 8, ro = (r % 8) * 2;
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        const float p = exp2f(s[h] - m_sm[h]);
        *reinterpret_cast<bf16 *>(prow + h * 128 + ((rc ^ (h & 7)) << 4) + ro) = __float2bfloat16_rn(p);
        float v = p;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red_sum[warp * HG + h] = v;
      }
      fence_proxy_async();
      tc::tc_fence_before();
      tc::mbar_arrive(p_full);
      if (!(ok = sm_sync())) break;
      if (r < HG) {
        l_sm[r] += (red_sum[r] + red_sum[HG + r]) + (red_sum[2 * HG + r] + red_sum[3 * HG + r]);
        if (r == 0) *s_rescale = 0;
      }
    }
    if (ok) ok = sm_sync();  // the last sums are visible to every thread
    // epilogue: O = O^T / l, bf16; inverse rotation of the last rd features at the query's position
    if (ok && ntiles > 0 && !tc::mbar_wait(o_full, (uint32_t)((ntiles - 1) & 1), abort_flag)) ok = false;
    ok = __all_sync(0xffffffffu, ok);  // the shuffles below need the whole warp
    if (ok) {
      tc::tc_fence_after();
      const int p_pos = P.start_pos + t;
      const int tail = HD - P.rd;
#pragma unroll 1
      for (int c = 0; c < KB / 2; ++c) {
        float v[HG];
        if (ntiles > 0) {
          tmem_ld_cols<HG>(tO + (uint32_t)(c * HG) + lane_off, v);
        } else {
#pragma unroll
          for (int h = 0; h < HG; ++h) v[h] = 0.f;
        }
        const int d = c * 128 + r;
        float2 cs = make_float2(1.f, 0.f);
        const bool rot = P.o_rot && d >= tail;
        if (rot) cs = reinterpret_cast<const float2 *>(P.tab)[(int64_t)p_pos * (P.rd >> 1) + ((d - tail) >> 1)];
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          const bf16 ob = __float2bfloat16_rn(v[h] / l_sm[h]);
          const int64_t off = (row * P.H + hg * HG + h) * (int64_t)HD + d;
          if (P.o) P.o[off] = ob;
          if (P.o_rot) {
            const float x = __bfloat162float(ob);
            const float partner = __shfl_xor_sync(0xffffffffu, x, 1);
            bf16 out = ob;
            if (rot) {
              const float sn = -cs.y;
              const float x0 = (d & 1) ? partner : x, x1 = (d & 1) ? x : partner;
              const float re = __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, sn));
              const float im = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, cs.x));
              out = __float2bfloat16_rn((d & 1) ? im : re);
            }
            P.o_rot[off] = out;
          }
        }
      }
    }
  }
  __syncthreads();
  if (warp == 8) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(P.status, kStatusTimeout);
}

template <int HG>
size_t smem_bytes() {
  return 1024 + (size_t)KB * TILE * 128 + (size_t)KB * HG * 128 + 2 * HG * 128 + kMaxList * 4 + 12 * HG * 4 + 6 * 8 + 64;
}

template <int HG>
cudaError_t launch_hg(const Params &p, int nq, cudaStream_t s) {
  static bool attr = false;
  const size_t smem = smem_bytes<HG>();
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_sparse_attn_tc<HG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(p.H / HG, nq);
  k_sparse_attn_tc<HG><<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace attn

bool sparse_attn_tc_supported(const AttnArgs &a) {
  return a.hd == attn::HD && a.H % 16 == 0 && a.na + a.nb <= attn::kMaxList && a.a_seq_stride % attn::HD == 0 &&
         (a.rows_b == nullptr || a.b_seq_stride % attn::HD == 0) && (a.o_rot == nullptr || a.rd % 2 == 0);
}

cudaError_t launch_sparse_attn_tc(const AttnArgs &a, int num_sms, cudaStream_t s) {
  using namespace attn;
  Params p;
  p.q = a.q;
  p.T = a.T;
  p.H = a.H;
  p.rows_a = a.rows_a;
  p.a_seq_rows = a.a_seq_stride / HD;
  p.a_len = a.a_len;
  p.rows_b = a.rows_b ? a.rows_b : a.rows_a;
  p.b_seq_rows = a.rows_b ? a.b_seq_stride / HD : 0;
  p.b_len = a.rows_b ? a.b_len : 0;
  p.idx_a = a.idx_a;
  p.na = a.na;
  p.idx_b = a.idx_b;
  p.nb = a.idx_b ? a.nb : 0;
  p.sink = a.sink;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.o = a.o;
  p.o_rot = a.o_rot;
  p.rd = a.rd;
  p.start_pos = a.start_pos;
  p.tab = a.tab;
  p.status = a.status;
  const int nq = a.B * a.T;
  if (nq <= 0) return cudaSuccess;
  // heads per CTA: enough CTAs to cover the SMs at least once
  if ((int64_t)nq * (a.H / 64) >= 2 * num_sms && a.H % 64 == 0) return launch_hg<64>(p, nq, s);
  if ((int64_t)nq * (a.H / 32) >= num_sms && a.H % 32 == 0) return launch_hg<32>(p, nq, s);
  return launch_hg<16>(p, nq, s);
}

}  // namespace csa
