// k_attn_queries_tc.cu -- the sparse attention of many queries (a prefill chunk) on a persistent grid
// ("deepseek_v41_ref::attn" sparse_attn; "DeepSeek V4.1 - Compressed sparse attention", "Sparse
// attention" and "Grouped output").
//
// Each (query, 64-head group) unit is computed exactly as k_sparse_attn_tc computes a unit that one
// CTA holds whole: the 128-entry tiles of J = [idx_a; idx_b], S^T = G q^T per tile, the running
// maximum raised only past 2^8, p = exp2(S - m) rounded to bf16, O^T += G^T P^T, and the result
// O e^{m-M} / (l e^{m-M} + e^{sink-M}) with the inverse rotation of its last rope_dim features.  What
// differs is the schedule: one CTA an SM takes units c, c + G, c + 2G, ... and the work between two
// units overlaps the tile pipeline instead of running with the SM otherwise idle:
//   * warp 9 forms the next unit's index lists (two list buffers) and loads and turns its q as soon as
//     the last scores MMA of the unit before has read q;
//   * warps 0-7 start copying the next unit's first tile as soon as the last P.V chunks have freed
//     its K-blocks, and write the finished unit's result (staged a warp at a time through the P
//     buffer, 16-byte stores) while that tile's scores are formed;
//   * warp 8 issues the MMAs of consecutive units without a break (TMEM allocated once).
// Every mbarrier wait is time-bounded.
#include "attn_common.cuh"

namespace csa {
namespace attn {

constexpr int kQThreads = 320;  // warps 0-7 copies, softmax and results; 8 MMA; 9 lists and q

struct QSmem {
  static constexpr size_t g = 0;                                            // KB x 16 KiB: one tile
  static constexpr size_t q = g + (size_t)KB * kBlockBytes;                 // KB x 64 x 128
  static constexpr size_t p = q + (size_t)KB * HG * 128;                    // P [2][64][128]; result staging
  static constexpr size_t src = p + (size_t)2 * HG * 128;                   // const bf16 * [2][kMaxTiles][TILE]
  static constexpr size_t red = src + (size_t)2 * kMaxTiles * TILE * 8;     // float [2][4][HG]
  static constexpr size_t stat = red + (size_t)2 * 4 * HG * 4;              // float m, l, alpha, f [HG]
  static constexpr size_t wcnt = stat + (size_t)4 * HG * 4;                 // int [2][kMaxTiles][4]
  static constexpr size_t bars = wcnt + (size_t)2 * kMaxTiles * 4 * 4;      // u64 [20]
  static constexpr size_t misc = bars + (size_t)20 * 8;                     // TMEM slot, abort, s_need[2]
  static constexpr size_t total = misc + 64;
};
static_assert(QSmem::total + 1024 <= 232448, "one CTA's shared memory");
static_assert(2 * HG * 128 == 8 * 32 * 32 * 2, "the P buffer holds the eight warps' 32 x 32 staging blocks");

// The index lists of one unit, by one warp: each entry's row address (nullptr for an invalid entry,
// -1) and per tile the valid entries of each quarter (32 entries).  An index outside -1 .. rows-1
// raises the bad-index status.  Every index is loaded before the first is used.
__device__ __forceinline__ void index_lists_warp(const Params &P, int64_t row, int b, int lane, const bf16 **src,
                                                 int *wcnt) {
  const int n_all = P.na + P.nb, n_rows = P.a_len + P.b_len;
  int v[kMaxTiles * 4];
#pragma unroll
  for (int k = 0; k < kMaxTiles * 4; ++k) {
    const int e = 32 * k + lane;
    v[k] = -1;
    if (k < 4 * P.ntiles)
      v[k] = e < P.na ? P.idx_a[row * P.na + e] : (e < n_all ? P.idx_b[row * P.nb + (e - P.na)] : -1);
  }
#pragma unroll
  for (int k = 0; k < kMaxTiles * 4; ++k) {
    if (k < 4 * P.ntiles) {
      const int e = 32 * k + lane;
      if (e < n_all && (v[k] < -1 || v[k] >= n_rows)) atomicOr(P.status, kStatusBadIndex);
      const bool ok = e < n_all && v[k] >= 0 && v[k] < n_rows;
      const bf16 *p = nullptr;
      if (ok)
        p = v[k] < P.a_len ? P.rows_a + (b * P.a_seq_rows + v[k]) * HD
                           : P.rows_b + (b * P.b_seq_rows + (v[k] - P.a_len)) * HD;
      src[e] = p;
      const unsigned bal = __ballot_sync(0xffffffffu, ok);
      if (lane == 0) wcnt[k] = __popc(bal);
    }
  }
}

// RoPE on q's last rd features in shared memory, by one warp (the same arithmetic as rope_q_apply)
__device__ __forceinline__ void rope_q_warp(const Params &P, uint8_t *sq, int t, int lane) {
  const int q_tail = HD - P.rd, q_nch = P.rd / 8;
  const float2 *tp = reinterpret_cast<const float2 *>(P.tab) + (int64_t)(P.start_pos + t) * (P.rd >> 1);
  for (int u = lane; u < HG * q_nch; u += 32) {
    const int f0 = q_tail + 8 * (u % q_nch);
    const float4 c01 = *reinterpret_cast<const float4 *>(tp + (f0 - q_tail) / 2);
    const float4 c23 = *reinterpret_cast<const float4 *>(tp + (f0 - q_tail) / 2 + 2);
    const float cs[8] = {c01.x, c01.y, c01.z, c01.w, c23.x, c23.y, c23.z, c23.w};
    rope_q_chunk(sq, u / q_nch, f0, cs);
  }
  fence_proxy_async();  // the turned q is read by the MMA (async proxy)
}

// every lane waits (each acquires what the barrier publishes); the warp goes on only if all succeeded
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
  const bool ok = tc::mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

__global__ void __launch_bounds__(kQThreads, 1) k_sparse_attn_queries_tc(const __grid_constant__ Params P, int units) {
  using L = QSmem;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  const uint32_t s_g = tc::smem_u32(smem + L::g), s_q = tc::smem_u32(smem + L::q), s_p = tc::smem_u32(smem + L::p);
  uint8_t *sP = smem + L::p;
  const bf16 **src_all = reinterpret_cast<const bf16 **>(smem + L::src);  // [2][kMaxTiles * TILE]
  float *red_max = reinterpret_cast<float *>(smem + L::red), *red_sum = red_max + 4 * HG;
  float *m_sm = reinterpret_cast<float *>(smem + L::stat), *l_sm = m_sm + HG, *alpha_sm = l_sm + HG,
        *f_sm = alpha_sm + HG;
  int *wcnt_all = reinterpret_cast<int *>(smem + L::wcnt);  // [2][kMaxTiles * 4]
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bars);
  uint64_t *g_full = bars, *s_full = bars + 4, *p_full = bars + 5, *pv_done = bars + 6, *sm_bar = bars + 10,
           *drain = bars + 11, *q_full = bars + 12, *q_ready = bars + 13, *q_free = bars + 14,
           *list_full = bars + 15, *list_free = bars + 17;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *s_need = const_cast<int *>(abort_flag) + 1;  // [2]: by tile parity, some score above its head's maximum

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int groups = P.H / HG;
  const int nmy = (int)blockIdx.x < units ? (units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  auto unit_row = [&](int j) { return ((int64_t)blockIdx.x + (int64_t)j * gridDim.x) / groups; };
  auto unit_hg = [&](int j) { return (int)(((int64_t)blockIdx.x + (int64_t)j * gridDim.x) % groups); };
  auto tile_live = [](const int *wc, int i) { return (wc[4 * i] | wc[4 * i + 1] | wc[4 * i + 2] | wc[4 * i + 3]) != 0; };
  constexpr uint32_t kCols = 512;  // S: 64 columns, O^T: 4 x 64
  constexpr uint32_t kQBytes = KB * HG * 128;

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) tc::mbar_init(&g_full[i], 64);  // the lanes of the pair's two copy warps
    tc::mbar_init(s_full, 1);
    tc::mbar_init(p_full, 256);
    for (int c = 0; c < 4; ++c) tc::mbar_init(&pv_done[c], 1);
    tc::mbar_init(sm_bar, 256);
    tc::mbar_init(drain, 1);
    tc::mbar_init(q_full, 1);
    tc::mbar_init(q_ready, 32);  // the lanes of warp 9
    tc::mbar_init(q_free, 1);
    for (int bb = 0; bb < 2; ++bb) {
      tc::mbar_init(&list_full[bb], 32);
      tc::mbar_init(&list_free[bb], 257);  // warps 0-7 and the MMA thread
    }
    *abort_flag = 0;
    s_need[0] = s_need[1] = 0;
    tc::fence_barrier_init();
  }
  if (warp == 8) tc::tmem_alloc(tmem_slot, kCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + HG;  // O^T chunk c at tO + c*HG
  // the first unit's q (written two launches earlier) is copied while the kernel before still runs
  if (warp == 9 && lane == 0 && nmy > 0) {
    tc::prefetch_tmap(&P.tm_q);
    tc::mbar_expect_tx(q_full, kQBytes);
#pragma unroll 1
    for (int kb = 0; kb < KB; ++kb)
      tma_load_2d_nohint(s_q + kb * HG * 128, &P.tm_q, q_full, kb * 64, (int)(unit_row(0) * P.H + unit_hg(0) * HG));
  }
  // a programmatic dependent of the selection kernel: the index lists it writes are read after this
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == 9) {
    // ------------------------------------------------------------------ lists and q, a unit ahead
    bool ok = true;
    int q_issued = nmy > 0 ? 1 : 0, q_landed = 0;  // q copies issued, and seen landed
    for (int j = 0; j < nmy && ok; ++j) {
      const int64_t row = unit_row(j);
      const int bj = j & 1;
      // the list buffer's previous unit (j - 2) is no longer read
      if (!(ok = warp_wait(&list_free[bj], (uint32_t)((j >> 1) & 1) ^ 1u, abort_flag))) break;
      index_lists_warp(P, row, (int)(row / P.T), lane, src_all + bj * kMaxTiles * TILE, wcnt_all + bj * kMaxTiles * 4);
      tc::mbar_arrive(&list_full[bj]);
      if (j > 0) {  // q of unit j once the last scores MMA of unit j - 1 has read the buffer
        if (!(ok = warp_wait(q_free, (uint32_t)((j - 1) & 1), abort_flag))) break;
        if (lane == 0) {
          tc::mbar_expect_tx(q_full, kQBytes);
#pragma unroll 1
          for (int kb = 0; kb < KB; ++kb)
            tma_load_2d_nohint(s_q + kb * HG * 128, &P.tm_q, q_full, kb * 64, (int)(row * P.H + unit_hg(j) * HG));
        }
        ++q_issued;
      }
      if (!(ok = warp_wait(q_full, (uint32_t)(j & 1), abort_flag))) break;
      ++q_landed;
      if (P.rope_q) rope_q_warp(P, smem + L::q, (int)(row % P.T), lane);
      tc::mbar_arrive(q_ready);
    }
    if (q_issued > q_landed && lane == 0) {  // stopped early: the copy in flight lands before the CTA ends
      const uint64_t t0 = tc::global_ns();
      while (!tc::mbar_try_wait(q_full, (uint32_t)((q_issued - 1) & 1)) && tc::global_ns() - t0 < tc::kWaitLimitNs) {
      }
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t id1 = tc::idesc_bf16_f32(TILE, HG);
      const uint32_t id2 = tc::idesc_bf16_f32(TILE, HG, /*a_mn_major=*/true, /*b_mn_major=*/false);
      bool ok = true;
      int G = 0;  // tiles issued so far (all units): the barriers' phases
      for (int j = 0; j < nmy && ok; ++j) {
        const int bj = j & 1;
        if (!(ok = tc::mbar_wait(&list_full[bj], (uint32_t)((j >> 1) & 1), abort_flag))) break;
        const int *wc = wcnt_all + bj * kMaxTiles * 4;
        unsigned live = 0;
        for (int i = 0; i < P.ntiles; ++i)
          if (tile_live(wc, i)) live |= 1u << i;
        tc::mbar_arrive(&list_free[bj]);
        // q has landed (and, with RoPE, been turned)
        if (!(ok = tc::mbar_wait(q_ready, (uint32_t)(j & 1), abort_flag))) break;
        tc::tc_fence_after();
        int n = 0;
        for (int i = 0; i < P.ntiles && ok; ++i) {
          if (!((live >> i) & 1u)) continue;
          const uint32_t par = (uint32_t)(G & 1);
          // S^T = G q^T, each K-block pair as soon as its two copy warps are done
          for (int w = 0; w < 4 && ok; ++w) {
            if (!(ok = tc::mbar_wait(&g_full[w], par, abort_flag))) break;
            tc::tc_fence_after();
#pragma unroll
            for (int kb = 2 * w; kb < 2 * w + 2; ++kb) {
              const uint64_t ad = tc::sdesc_sw128(s_g + kb * kBlockBytes, 16, 1024);
              const uint64_t bd = tc::sdesc_sw128(s_q + kb * HG * 128, 16, 1024);
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4) tc::mma_bf16(tS, ad + 2ull * k4, bd + 2ull * k4, id1, (kb | k4) ? 1u : 0u);
            }
          }
          if (!ok) break;
          tc::mma_commit(s_full);
          if ((live >> (i + 1)) == 0u) tc::mma_commit(q_free);  // the unit's last scores MMA: q may be replaced
          if (!(ok = tc::mbar_wait(p_full, par, abort_flag))) break;
          tc::tc_fence_after();
          // O^T += G^T P^T, feature chunk c = K-blocks 2c, 2c+1; each chunk's completion frees them
#pragma unroll
          for (int c = 0; c < KB / 2; ++c) {
#pragma unroll
            for (int ii = 0; ii < TILE / 16; ++ii) {
              const uint64_t ad = tc::sdesc_sw128(s_g + (2 * c) * kBlockBytes + ii * 2048, kBlockBytes, 1024);
              const uint64_t bd = tc::sdesc_sw128(s_p + (ii / 4) * HG * 128 + (ii % 4) * 32, 16, 1024);
              tc::mma_bf16(tO + (uint32_t)(c * HG), ad, bd, id2, (n > 0 || ii > 0) ? 1u : 0u);
            }
            tc::mma_commit(&pv_done[c]);
          }
          ++n;
          ++G;
        }
        if (ok && live == 0u) tc::mma_commit(q_free);  // a unit without rows still hands q back
      }
      if (nmy > 0) {  // nothing may still write TMEM, read shared memory or arrive when the CTA ends
        tc::mma_commit(drain);
        const uint64_t t0 = tc::global_ns();
        while (!tc::mbar_try_wait(drain, 0) && tc::global_ns() - t0 < tc::kWaitLimitNs) {
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ warps 0-7: copies, softmax, results
    // warp w: TMEM lane quadrant w % 4 (tile rows, and features of an O^T chunk), heads hh .. hh+31,
    // and K-block (w + 4) % 8 of every tile's rows
    const int quad = warp & 3, hh = (warp >> 2) * 32;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int kbw = (warp + 4) & 7, pw = kbw >> 1, rq = lane >> 3, cc = lane & 7;
    uint32_t sm_uses = 0;
    auto sm_sync = [&]() -> bool {
      tc::mbar_arrive(sm_bar);
      return tc::mbar_wait(sm_bar, (sm_uses++) & 1u, abort_flag);
    };
    auto issue_tile = [&](const bf16 *const *srcs) {
      const uint32_t blk = s_g + kbw * kBlockBytes;
#pragma unroll 1
      for (int i0 = 0; i0 < TILE / 4; i0 += 8) {
        const bf16 *ps[8];  // eight row addresses read before the copies that use them are issued
#pragma unroll
        for (int u = 0; u < 8; ++u) ps[u] = srcs[4 * (i0 + u) + rq];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int rr = 4 * (i0 + u) + rq;
          cp_async16(blk + rr * 128 + ((cc ^ (rr & 7)) << 4), ps[u] ? ps[u] + 64 * kbw + 8 * cc : P.rows_a,
                     ps[u] != nullptr);
        }
      }
    };
    if (tid < HG) m_sm[tid] = -INFINITY;
    float lsum[32];  // this thread's sums of p over its rows, per head (reduced over the CTA per unit)
#pragma unroll
    for (int h = 0; h < 32; ++h) lsum[h] = 0.f;
    int G = 0;  // tiles completed so far (all units): the barriers' phases
    // A unit's result in two steps.  finish_sums, right after its last softmax (overlapping its last
    // P.V): the sums over the CTA, the factor f with the sink, the inverse rotation's angles of this
    // lane's last-chunk features; m back to -inf and the sums to 0 for the next unit.  finish_write,
    // once the next unit's first rows are published to the MMA (so its scores are formed meanwhile):
    // O * f a 128-feature chunk at a time, staged per warp in the P buffer (its last reader, the
    // unit's last P.V, has completed) and written with 16-byte stores.
    int64_t pr_row = -1;
    int pr_hg = 0, pr_live = 0;
    bool pending = false;
    const int tail = HD - P.rd;
    const int d3 = 3 * 128 + quad * 32 + (lane & 3) * 8;  // this lane's first feature of the last chunk
    float4 rc01 = make_float4(0.f, 0.f, 0.f, 0.f), rc23 = rc01;
    auto finish_sums = [&](int64_t row, int hg, int live) -> bool {
      red_sum[quad * HG + hh + lane] = warp_reduce_32<false>(lsum, lane);
#pragma unroll
      for (int h = 0; h < 32; ++h) lsum[h] = 0.f;
      if (P.o_rot && d3 >= tail) {
        const float2 *tp = reinterpret_cast<const float2 *>(P.tab) + (int64_t)(P.start_pos + row % P.T) * (P.rd >> 1);
        rc01 = *reinterpret_cast<const float4 *>(tp + ((d3 - tail) >> 1));
        rc23 = *reinterpret_cast<const float4 *>(tp + ((d3 - tail) >> 1) + 2);
      }
      if (!sm_sync()) return false;
      if (tid < HG) {
        const float l = (red_sum[tid] + red_sum[HG + tid]) + (red_sum[2 * HG + tid] + red_sum[3 * HG + tid]);
        const float s2 = P.sink[hg * HG + tid] * 1.4426950408889634f;
        const float M = fmaxf(m_sm[tid], s2);
        const float em = live > 0 ? exp2f(m_sm[tid] - M) : 0.f;
        f_sm[tid] = em / (l * em + exp2f(s2 - M));
        m_sm[tid] = -INFINITY;
      }
      if (!sm_sync()) return false;
      pr_row = row;
      pr_hg = hg;
      pr_live = live;
      pending = true;
      return true;
    };
    auto finish_write = [&]() -> bool {
      pending = false;
      if (G > 0 && !tc::mbar_wait(&pv_done[3], (uint32_t)((G - 1) & 1), abort_flag)) return false;
      tc::tc_fence_after();
      const float2 *tp = P.o_rot ? reinterpret_cast<const float2 *>(P.tab) + (int64_t)(P.start_pos + pr_row % P.T) * (P.rd >> 1)
                                 : nullptr;
      bf16 *stg = reinterpret_cast<bf16 *>(sP + warp * 2048);  // [32 heads][32 features]
      const int64_t obase = (pr_row * P.H + pr_hg * HG + hh) * (int64_t)HD;
#pragma unroll 1
      for (int c = 0; c < KB / 2; ++c) {
        float v[32];
        if (pr_live > 0) {
          tmem_ld_32cols(tO + (uint32_t)(c * HG + hh) + lane_off, v);
        } else {
#pragma unroll
          for (int h = 0; h < 32; ++h) v[h] = 0.f;
        }
#pragma unroll
        for (int h0 = 0; h0 < 32; h0 += 16) {
          float fv[16];
          lds16(fv, f_sm + hh + h0);
#pragma unroll
          for (int k = 0; k < 16; ++k) stg[(h0 + k) * 32 + lane] = __float2bfloat16_rn(v[h0 + k] * fv[k]);
        }
        __syncwarp();
        // lane l writes features d0 .. d0+7 (d0 the same for all four of its vectors) of heads
        // l/4, l/4 + 8, l/4 + 16, l/4 + 24
        const int d0 = c * 128 + quad * 32 + (lane & 3) * 8;
        const bool turn = P.o_rot && d0 >= tail;
        float2 cs[4] = {make_float2(rc01.x, rc01.y), make_float2(rc01.z, rc01.w), make_float2(rc23.x, rc23.y),
                        make_float2(rc23.z, rc23.w)};
        if (turn && c < 3) {  // (features below the last chunk turn only when rope_dim > 128)
          const float4 c01 = *reinterpret_cast<const float4 *>(tp + ((d0 - tail) >> 1));
          const float4 c23 = *reinterpret_cast<const float4 *>(tp + ((d0 - tail) >> 1) + 2);
          cs[0] = make_float2(c01.x, c01.y);
          cs[1] = make_float2(c01.z, c01.w);
          cs[2] = make_float2(c23.x, c23.y);
          cs[3] = make_float2(c23.z, c23.w);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int h = (lane >> 2) + 8 * k;
          const uint4 ob = *reinterpret_cast<const uint4 *>(stg + h * 32 + (lane & 3) * 8);
          const int64_t off = obase + (int64_t)h * HD + d0;
          if (P.o) *reinterpret_cast<uint4 *>(P.o + off) = ob;
          if (P.o_rot) {
            uint4 orr = ob;
            if (turn) {
              const bf16 *xb = reinterpret_cast<const bf16 *>(&ob);
              bf16 *yb = reinterpret_cast<bf16 *>(&orr);
#pragma unroll
              for (int qq = 0; qq < 4; ++qq) {
                float re, im;
                unrotate(__bfloat162float(xb[2 * qq]), __bfloat162float(xb[2 * qq + 1]), cs[qq], re, im);
                yb[2 * qq] = __float2bfloat16_rn(re);
                yb[2 * qq + 1] = __float2bfloat16_rn(im);
              }
            }
            *reinterpret_cast<uint4 *>(P.o_rot + off) = orr;
          }
        }
        __syncwarp();
      }
      tc::tc_fence_before();
      return true;
    };
    bool ok = true;
    for (int j = 0; j < nmy && ok; ++j) {
      const int bj = j & 1;
      if (!(ok = tc::mbar_wait(&list_full[bj], (uint32_t)((j >> 1) & 1), abort_flag))) break;
      const bf16 *const *srcj = src_all + bj * kMaxTiles * TILE;
      const int *wc = wcnt_all + bj * kMaxTiles * 4;
      int n = 0;
      for (int i = 0; i < P.ntiles && ok; ++i) {
        if (!tile_live(wc, i)) continue;
        // this warp's K-block of the tile before (this unit's or the last unit's) has been read by its
        // P.V chunk: refill it
        if (G > 0 && !(ok = tc::mbar_wait(&pv_done[pw], (uint32_t)((G - 1) & 1), abort_flag))) break;
        issue_tile(srcj + i * TILE);
        cp_async_wait_all();
        fence_proxy_async();
        tc::mbar_arrive(&g_full[pw]);
        // the unit before is written while this unit's first scores are formed
        if (pending && !(ok = finish_write())) break;
        {  // the next tile's segments of this warp's K-block on their way to L2 while this one is used
          int nx = i + 1;
          while (nx < P.ntiles && !tile_live(wc, nx)) ++nx;
          if (nx < P.ntiles) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const bf16 *prr = srcj[nx * TILE + lane + 32 * k];
              if (prr) asm volatile("prefetch.global.L2 [%0];" ::"l"(prr + 64 * kbw));
            }
          }
        }
        if (!(ok = tc::mbar_wait(s_full, (uint32_t)(G & 1), abort_flag))) break;
        tc::tc_fence_after();
        float s[32];
        tmem_ld_32cols(tS + (uint32_t)hh + lane_off, s);
        const bool vr = srcj[i * TILE + r] != nullptr;
#pragma unroll
        for (int h = 0; h < 32; ++h) s[h] = vr ? s[h] * P.scale_log2 : -INFINITY;
        // the running maximum of a head moves only when a score exceeds it by more than 2^8; the
        // maxima over the tile are formed only when some score does (always on a unit's first tile)
        bool full = true;
        if (n > 0) {
          bool need = false;
#pragma unroll
          for (int h0 = 0; h0 < 32; h0 += 16) {
            float mv[16];
            lds16(mv, m_sm + hh + h0);
#pragma unroll
            for (int k = 0; k < 16; ++k) need |= s[h0 + k] > mv[k] + 8.0f;
          }
          if (need) s_need[G & 1] = 1;
          if (!(ok = sm_sync())) break;
          full = s_need[G & 1] != 0;
          if (tid == 0) s_need[(G + 1) & 1] = 0;  // the flag of the tile before, read by all by now
        }
        if (full) {
          red_max[quad * HG + hh + lane] = warp_reduce_32<true>(s, lane);
          if (!(ok = sm_sync())) break;
          if (n == 0 && tid == 0) s_need[(G + 1) & 1] = 0;
          if (tid < HG) {
            const float tmax =
                fmaxf(fmaxf(red_max[tid], red_max[HG + tid]), fmaxf(red_max[2 * HG + tid], red_max[3 * HG + tid]));
            float a = 1.0f;
            if (tmax > m_sm[tid] + 8.0f) {  // rescale what has accumulated
              a = exp2f(m_sm[tid] - tmax);
              m_sm[tid] = tmax;
            }
            alpha_sm[tid] = a;
          }
          if (!(ok = sm_sync())) break;
          if (n > 0) {
            // the tile before's product has completed: its commit released this tile's rows
#pragma unroll 1
            for (int c = 0; c < KB / 2; ++c) {
#pragma unroll
              for (int c0 = 0; c0 < 32; c0 += 16) {
                uint32_t v[16];
                const uint32_t ta = tO + (uint32_t)(c * HG + hh + c0) + lane_off;
                float av[16];
                lds16(av, alpha_sm + hh + c0);
                tc::tmem_ld16(ta, v);
                tc::tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 16; ++q) v[q] = __float_as_uint(__uint_as_float(v[q]) * av[q]);
                tmem_st16(ta, v);
              }
            }
            tmem_st_wait();
#pragma unroll
            for (int h0 = 0; h0 < 32; h0 += 16) {
              float av[16];
              lds16(av, alpha_sm + hh + h0);
#pragma unroll
              for (int k = 0; k < 16; ++k) lsum[h0 + k] *= av[k];
            }
          }
        }
        uint8_t *prow = sP + (r / 64) * HG * 128;
        const int rc = (r % 64) / 8, ro = (r % 8) * 2;
#pragma unroll
        for (int h0 = 0; h0 < 32; h0 += 16) {
          float mv[16];  // the maxima read before the stores below (which the compiler cannot tell apart)
          lds16(mv, m_sm + hh + h0);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int h = hh + h0 + k;
            s[h0 + k] = exp2f(s[h0 + k] - mv[k]);  // 0 for masked rows
            lsum[h0 + k] += s[h0 + k];
            *reinterpret_cast<bf16 *>(prow + h * 128 + ((rc ^ (h & 7)) << 4) + ro) = __float2bfloat16_rn(s[h0 + k]);
          }
        }
        fence_proxy_async();
        tc::tc_fence_before();
        tc::mbar_arrive(p_full);
        ++n;
        ++G;
      }
      if (!ok) break;
      // this unit's lists are no longer read
      tc::mbar_arrive(&list_free[bj]);
      // a unit without rows: the unit before is written here
      if (pending && !(ok = finish_write())) break;
      if (!(ok = finish_sums(unit_row(j), unit_hg(j), n))) break;
    }
    if (ok && pending) ok = finish_write();  // the last unit's result
    cp_async_wait_all();
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kCols);
  }
  if (tid == 0 && *abort_flag) atomicOr(P.status, kStatusTimeout);
}

cudaError_t launch_sparse_attn_queries_tc(const Params &p, int units, int num_sms, cudaStream_t s) {
  static SmemAttr attr;
  const size_t smem = 1024 + QSmem::total;
  cudaError_t e = attr.ensure((const void *)k_sparse_attn_queries_tc, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)std::min(units, num_sms));
  cfg.blockDim = dim3(kQThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_sparse_attn_queries_tc, p, units);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace attn
}  // namespace csa
