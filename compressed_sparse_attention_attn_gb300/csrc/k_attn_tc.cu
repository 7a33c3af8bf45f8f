// k_attn_tc.cu -- sparse attention with the per-head sink on the 5th-generation tensor cores
// ("deepseek_v41_ref::attn" sparse_attn; "DeepSeek V4.1 - Compressed sparse attention", "Sparse
// attention" and "Grouped output"; "Join rows").
//
// One CTA per (query, group of HG heads).  All heads of a query share one K = V row per selected
// position.  Y = [rows_a; rows_b] and J = [idx_a; idx_b] are never materialised: the valid entries
// of both index lists are compacted per source, and the four loader warps copy the selected rows
// (cp.async, 16 lanes per 256-byte row segment, so each warp instruction reads two whole segments)
// into a ring of eight 16 KiB K-block slots in the 128-byte swizzled layout (slot kb holds features
// [64 kb, 64 kb + 64) of a 128-row tile; loader warp w owns slots 2w and 2w + 1).
//
//   pass 1  S^T_k[r][h] = sum_d G_k[r][d] q[h][d]   for every tile k (M = 128 rows, N = HG, K = 512),
//           each tile's scores in their own TMEM columns;
//   softmax over all tiles at once: m_h = max(sink_h, max S), p = exp(S - m) (0 for padding rows),
//           l_h = exp(sink_h - m_h) + sum p (the sink in the denominator only), P_k bf16 in shared
//           memory, K-major [HG][128];
//   pass 2  O^T[d][h] += sum_r G_k[r][d] P_k[h][r]  (M = 4 x 128 features, N = HG, K = 128 rows; the
//           slots read as MN-major operands), the last tile of pass 1 reused in place, the others
//           gathered again (their loads overlap the softmax);
//   epilogue O = O^T / l as bf16, and the inverse rotation of the last rope_dim features of the
//           bf16 value at the query's position.
//
// Warps 0-3: softmax and epilogue (TMEM lane quadrant = warp); warps 4-7: compaction of the index
// lists, then the row copies (warp 4 lane 0 also loads q by TMA); warp 8: TMEM allocation and MMA
// issue.  Every mbarrier wait is time-bounded.
#include "csa_internal.cuh"
#include "tc_ptx.cuh"

namespace csa {

// 2-D bf16 tensor map with 128-byte swizzle (defined with the GEMM's TMA helpers).
bool tma_map_2d_bf16(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner,
                     uint32_t box_outer);

namespace attn {

constexpr int HD = 512;              // head_dim this kernel serves
constexpr int KB = HD / 64;          // 64-feature K-blocks = ring slots
constexpr int TILE = 128;            // rows per tile
constexpr int kThreads = 288;
constexpr int kMaxTiles = 6;         // selections up to 768 rows
constexpr int kMaxEntries = kMaxTiles * TILE;
constexpr int kSlotBytes = TILE * 128;

struct Params {
  CUtensorMap tm_q;  // q [NT*H][512], box {64, HG}
  const bf16 *rows_a, *rows_b;
  int T, H;
  int64_t a_seq_rows, b_seq_rows;
  int a_len, b_len;
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
__device__ __forceinline__ void tma_load_2d_nohint(uint32_t dst, const CUtensorMap *tm, uint64_t *bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"((uint64_t)tm), "r"(tc::smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
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

template <int HG>
struct Smem {
  static constexpr size_t slots = 0;                                      // KB x 16 KiB
  static constexpr size_t q = slots + (size_t)KB * kSlotBytes;              // KB x HG x 128
  static constexpr size_t p = q + (size_t)KB * HG * 128;                    // kMaxTiles x 2 x HG x 128
  static constexpr size_t list = p + (size_t)kMaxTiles * 2 * HG * 128;      // int32 [2][kMaxEntries] (A, B)
  static constexpr size_t valid = list + (size_t)2 * kMaxEntries * 4;      // uint8 [kMaxEntries]
  static constexpr size_t red = valid + (size_t)kMaxEntries;              // float [2][4][HG]
  static constexpr size_t stat = red + (size_t)2 * 4 * HG * 4;            // float m[HG], l[HG]
  static constexpr size_t bars = (stat + (size_t)2 * HG * 4 + 7) / 8 * 8;  // u64 [2*KB + 6]
  static constexpr size_t misc = bars + (size_t)(2 * KB + 6) * 8;         // tmem slot, flags, counts
  static constexpr size_t total = misc + 128;
};

template <int HG>
__global__ void __launch_bounds__(kThreads, 1) k_sparse_attn_tc(const __grid_constant__ Params P) {
  using L = Smem<HG>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  const uint32_t s_slots = tc::smem_u32(smem + L::slots), s_q = tc::smem_u32(smem + L::q),
                 s_p = tc::smem_u32(smem + L::p);
  uint8_t *sP = smem + L::p;
  int32_t *listA = reinterpret_cast<int32_t *>(smem + L::list), *listB = listA + kMaxEntries;
  uint8_t *valid = smem + L::valid;
  float *red_max = reinterpret_cast<float *>(smem + L::red), *red_sum = red_max + 4 * HG;
  float *m_sm = reinterpret_cast<float *>(smem + L::stat), *l_sm = m_sm + HG;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bars);
  uint64_t *slot_full = bars, *slot_empty = bars + KB, *q_full = bars + 2 * KB, *s_done = q_full + 1,
           *p_full = q_full + 2, *o_done = q_full + 3, *sm_bar = q_full + 4, *drain = q_full + 5;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *s_cnt = const_cast<int *>(abort_flag) + 1;  // [2 buffers][2 sources][4 loader warps]
  int *s_nA = s_cnt + 16, *s_nB = s_nA + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = blockIdx.y;  // query b*T + t
  const int hg = blockIdx.x;
  const int b = (int)(row / P.T), t = (int)(row % P.T);
  constexpr uint32_t kCols = ((kMaxTiles + 4) * HG <= 128) ? 128 : ((kMaxTiles + 4) * HG <= 256) ? 256 : 512;

  if (threadIdx.x == 0) {
    for (int i = 0; i < KB; ++i) {
      tc::mbar_init(&slot_full[i], 32);  // the lanes of the loader warp that owns the slot
      tc::mbar_init(&slot_empty[i], 1);
    }
    tc::mbar_init(q_full, 1);
    tc::mbar_init(s_done, 1);
    tc::mbar_init(p_full, 128);
    tc::mbar_init(o_done, 1);
    tc::mbar_init(sm_bar, 128);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 8) tc::tmem_alloc(tmem_slot, kCols);
  __syncthreads();

  // ---- compaction (warps 4-7): the valid entries of [idx_a; idx_b] in order, split by source (rows
  //      of rows_a in listA, of rows_b in listB); one block-wide count per 128 entries
  const int n_all = P.na + P.nb;
  const int n_rows = P.a_len + P.b_len;
  if (warp >= 4 && warp < 8) {
    const int j = threadIdx.x - 128, lw = warp - 4;
    constexpr int kPer = kMaxEntries / 128;
    int v[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {  // every index of this query, loaded up front
      const int e = i * 128 + j;
      v[i] = e < P.na ? P.idx_a[row * P.na + e] : (e < n_all ? P.idx_b[row * P.nb + (e - P.na)] : -1);
    }
    int baseA = 0, baseB = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = i * 128 + j;
      if (e < n_all && (v[i] < -1 || v[i] >= n_rows)) atomicOr(P.status, kStatusBadIndex);
      const bool ok = e < n_all && v[i] >= 0 && v[i] < n_rows;
      const bool inA = ok && v[i] < P.a_len, inB = ok && v[i] >= P.a_len;
      const unsigned balA = __ballot_sync(0xffffffffu, inA), balB = __ballot_sync(0xffffffffu, inB);
      int *cnt = s_cnt + (i & 1) * 8;
      if (lane == 0) {
        cnt[lw] = __popc(balA);
        cnt[4 + lw] = __popc(balB);
      }
      tc::named_bar(2, 128);
      int bA = baseA, bB = baseB;
      for (int w = 0; w < lw; ++w) {
        bA += cnt[w];
        bB += cnt[4 + w];
      }
      const unsigned below = (1u << lane) - 1u;
      if (inA) {
        const int at = bA + __popc(balA & below);
        if (at < kMaxEntries) listA[at] = (int32_t)(b * P.a_seq_rows + v[i]);
      }
      if (inB) {
        const int at = bB + __popc(balB & below);
        if (at < kMaxEntries) listB[at] = (int32_t)(b * P.b_seq_rows + (v[i] - P.a_len));
      }
      baseA += cnt[0] + cnt[1] + cnt[2] + cnt[3];
      baseB += cnt[4] + cnt[5] + cnt[6] + cnt[7];
    }
    const int nA = min(baseA, kMaxEntries), nB = min(baseB, kMaxEntries - nA);
    const int padded = min((nA + nB + TILE - 1) / TILE * TILE, kMaxEntries);
    for (int e = j; e < padded; e += 128) valid[e] = e < nA + nB;
    if (j == 0) {
      *s_nA = nA;
      *s_nB = nB;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nA = *s_nA, nB = *s_nB;
  const int ntiles = min((nA + nB + TILE - 1) / TILE, kMaxTiles);
  const uint32_t tS = tmem, tO = tmem + (uint32_t)(kMaxTiles * HG);  // S_k at tS + k*HG; O^T chunk c at tO + c*HG

  if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------------ loaders
    const int w = warp - 4;
    if (w == 0 && lane == 0 && ntiles > 0) {
      tc::prefetch_tmap(&P.tm_q);
      tc::mbar_expect_tx(q_full, KB * HG * 128);
#pragma unroll 1
      for (int kb = 0; kb < KB; ++kb)
        tma_load_2d_nohint(s_q + kb * HG * 128, &P.tm_q, q_full, kb * 64, (int)(row * P.H + hg * HG));
    }
    // fills in order: pass 1 tiles 0..n-1, then pass 2 tiles n-2..0 (tile n-1 stays from pass 1).
    // This warp writes features [128 w, 128 w + 128) = slots 2w, 2w+1 of every row of the tile:
    // lanes 0-15 one row, lanes 16-31 the next, 16 bytes each.
    const int half = lane >> 4, sub = lane & 15;
    const int kb = 2 * w + (sub >> 3), cc = sub & 7;
    const uint32_t slot_base = s_slots + kb * kSlotBytes;
    int fill = 0;
    bool ok = true;
    const int nfills = ntiles > 0 ? 2 * ntiles - 1 : 0;
    for (int fi = 0; fi < nfills && ok; ++fi) {
      const int k = fi < ntiles ? fi : 2 * ntiles - 2 - fi;
      const uint32_t par = (uint32_t)(fill & 1) ^ 1u;
      if (!(ok = tc::mbar_wait(&slot_empty[2 * w], par, abort_flag) &&
                 tc::mbar_wait(&slot_empty[2 * w + 1], par, abort_flag)))
        break;
#pragma unroll 4
      for (int i = 0; i < TILE / 2; ++i) {
        const int r = 2 * i + half, e = k * TILE + r;
        const bool vr = e < nA + nB;
        const bf16 *src = P.rows_a;
        if (vr) src = e < nA ? P.rows_a + (int64_t)listA[e] * HD : P.rows_b + (int64_t)listB[e - nA] * HD;
        cp_async16(slot_base + r * 128 + ((cc ^ (r & 7)) << 4), src + (vr ? 128 * w + 8 * sub : 0), vr);
      }
      cp_async_wait_all();
      fence_proxy_async();
      tc::mbar_arrive(&slot_full[2 * w]);
      tc::mbar_arrive(&slot_full[2 * w + 1]);
      ++fill;
    }
    cp_async_wait_all();
    if (w == 0 && lane == 0 && ntiles > 0) {  // the q copies have landed before the CTA can exit
      const uint64_t t0 = tc::global_ns();
      while (!tc::mbar_try_wait(q_full, 0) && tc::global_ns() - t0 < tc::kWaitLimitNs) {
      }
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------------ MMA issue
    if (lane == 0 && ntiles > 0) {
      const uint32_t id1 = tc::idesc_bf16_f32(TILE, HG);
      const uint32_t id2 = tc::idesc_bf16_f32(TILE, HG, /*a_mn_major=*/true, /*b_mn_major=*/false);
      bool ok = tc::mbar_wait(q_full, 0, abort_flag);
      int fill = 0;
      // pass 1: scores of every tile
      for (int k = 0; k < ntiles && ok; ++k) {
        for (int kb = 0; kb < KB; ++kb) {
          if (!(ok = tc::mbar_wait(&slot_full[kb], (uint32_t)(fill & 1), abort_flag))) break;
          tc::tc_fence_after();
          const uint64_t ad = tc::sdesc_sw128(s_slots + kb * kSlotBytes, 16, 1024);
          const uint64_t bd = tc::sdesc_sw128(s_q + kb * HG * 128, 16, 1024);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            tc::mma_bf16(tS + (uint32_t)(k * HG), ad + 2ull * k4, bd + 2ull * k4, id1, (kb | k4) ? 1u : 0u);
          if (k + 1 < ntiles) tc::mma_commit(&slot_empty[kb]);  // the last tile stays for pass 2
        }
        ++fill;
      }
      if (ok) tc::mma_commit(s_done);
      if (ok) ok = tc::mbar_wait(p_full, 0, abort_flag);
      // pass 2: O^T += G^T P^T, the last tile first (still in the slots), then the refills
      for (int pi = 0; pi < ntiles && ok; ++pi) {
        const int k = ntiles - 1 - pi;
        const bool resident = pi == 0;
#pragma unroll 1
        for (int c = 0; c < KB / 2 && ok; ++c) {
          if (!resident) {
            if (!(ok = tc::mbar_wait(&slot_full[2 * c], (uint32_t)(fill & 1), abort_flag))) break;
            if (!(ok = tc::mbar_wait(&slot_full[2 * c + 1], (uint32_t)(fill & 1), abort_flag))) break;
            tc::tc_fence_after();
          }
#pragma unroll
          for (int i = 0; i < TILE / 16; ++i) {
            const uint64_t ad = tc::sdesc_sw128(s_slots + (2 * c) * kSlotBytes + i * 2048, kSlotBytes, 1024);
            const uint64_t bd =
                tc::sdesc_sw128(s_p + k * 2 * HG * 128 + (i / 4) * HG * 128 + (i % 4) * 32, 16, 1024);
            tc::mma_bf16(tO + (uint32_t)(c * HG), ad, bd, id2, (pi > 0 || i > 0) ? 1u : 0u);
          }
          tc::mma_commit(&slot_empty[2 * c]);
          tc::mma_commit(&slot_empty[2 * c + 1]);
        }
        if (!resident) ++fill;
      }
      if (ok) tc::mma_commit(o_done);
      tc::mma_commit(drain);
      const uint64_t t0 = tc::global_ns();
      while (!tc::mbar_try_wait(drain, 0) && tc::global_ns() - t0 < tc::kWaitLimitNs) {
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------------ softmax + epilogue (warps 0-3)
    const int r = warp * 32 + lane;  // tile row (S^T) and feature within a chunk (O^T)
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    uint32_t sm_uses = 0;
    auto sm_sync = [&]() -> bool {
      tc::mbar_arrive(sm_bar);
      return tc::mbar_wait(sm_bar, (sm_uses++) & 1u, abort_flag);
    };
    bool ok = true;
    if (ntiles > 0) {
      ok = tc::mbar_wait(s_done, 0, abort_flag);
      if (ok) tc::tc_fence_after();
      float m[HG], l[HG];
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
      }
      // maximum over every row of every tile
      for (int k = 0; k < ntiles && ok; ++k) {
        float s[HG];
        tmem_ld_cols<HG>(tS + (uint32_t)(k * HG) + lane_off, s);
        if (valid[k * TILE + r]) {
#pragma unroll
          for (int h = 0; h < HG; ++h) m[h] = fmaxf(m[h], s[h] * P.scale_log2);
        }
      }
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        float x = m[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
        if (lane == 0) red_max[warp * HG + h] = x;
      }
      if (ok) ok = sm_sync();
      if (r < HG) {
        const float sink2 = P.sink[hg * HG + r] * 1.4426950408889634f;
        m_sm[r] = fmaxf(fmaxf(fmaxf(red_max[r], red_max[HG + r]), fmaxf(red_max[2 * HG + r], red_max[3 * HG + r])),
                        sink2);
      }
      if (ok) ok = sm_sync();
#pragma unroll
      for (int h = 0; h < HG; ++h) m[h] = m_sm[h];
      // probabilities (bf16, K-major [HG][128 rows] per tile, swizzled) and their sums
      const int rc = (r % 64) / 8, ro = (r % 8) * 2;
      for (int k = 0; k < ntiles && ok; ++k) {
        float s[HG];
        tmem_ld_cols<HG>(tS + (uint32_t)(k * HG) + lane_off, s);
        const bool vr = valid[k * TILE + r] != 0;
        uint8_t *prow = sP + k * 2 * HG * 128 + (r / 64) * HG * 128;
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          const float p = vr ? exp2f(s[h] * P.scale_log2 - m[h]) : 0.f;
          l[h] += p;
          *reinterpret_cast<bf16 *>(prow + h * 128 + ((rc ^ (h & 7)) << 4) + ro) = __float2bfloat16_rn(p);
        }
      }
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        float x = l[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (lane == 0) red_sum[warp * HG + h] = x;
      }
      fence_proxy_async();
      tc::tc_fence_before();
      tc::mbar_arrive(p_full);
      if (ok) ok = sm_sync();
      if (r < HG) {
        const float sink2 = P.sink[hg * HG + r] * 1.4426950408889634f;
        l_sm[r] =
            exp2f(sink2 - m_sm[r]) + ((red_sum[r] + red_sum[HG + r]) + (red_sum[2 * HG + r] + red_sum[3 * HG + r]));
      }
      if (ok) ok = sm_sync();
      if (ok) ok = tc::mbar_wait(o_done, 0, abort_flag);
    } else {
      if (r < HG) l_sm[r] = 1.f;
      ok = sm_sync();
    }
    ok = __all_sync(0xffffffffu, ok);  // the shuffles below need the whole warp
    // epilogue: O = O^T / l, bf16; inverse rotation of the last rd features at the query's position
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
cudaError_t launch_hg(const Params &p, int nq, cudaStream_t s) {
  static bool attr = false;
  const size_t smem = 1024 + Smem<HG>::total;
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
  // every selection must fit kMaxTiles tiles of rows
  return a.hd == attn::HD && a.H % 16 == 0 && a.na + a.nb <= attn::kMaxEntries && a.a_seq_stride % attn::HD == 0 &&
         (a.rows_b == nullptr || a.b_seq_stride % attn::HD == 0) && (a.o_rot == nullptr || a.rd % 2 == 0) &&
         ((uintptr_t)a.q & 15) == 0 && ((uintptr_t)a.rows_a & 15) == 0 && ((uintptr_t)a.rows_b & 15) == 0;
}

cudaError_t launch_sparse_attn_tc(const AttnArgs &a, int num_sms, cudaStream_t s) {
  using namespace attn;
  const int nq = a.B * a.T;
  if (nq <= 0) return cudaSuccess;
  Params p;
  memset(&p, 0, sizeof(p));
  // heads per CTA: 32 once that still gives about one CTA per SM, else 16
  const int HG = ((int64_t)nq * (a.H / 32) >= num_sms && a.H % 32 == 0) ? 32 : 16;
  if (!tma_map_2d_bf16(&p.tm_q, a.q, HD, (uint64_t)nq * a.H, HD, 64, (uint32_t)HG)) return cudaErrorInvalidValue;
  p.rows_a = a.rows_a;
  p.rows_b = a.rows_b ? a.rows_b : a.rows_a;
  p.b_seq_rows = a.rows_b ? a.b_seq_stride / HD : 0;
  p.b_len = a.rows_b ? a.b_len : 0;
  p.T = a.T;
  p.H = a.H;
  p.a_seq_rows = a.a_seq_stride / HD;
  p.a_len = a.a_len;
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
  return HG == 32 ? launch_hg<32>(p, nq, s) : launch_hg<16>(p, nq, s);
}

}  // namespace csa
