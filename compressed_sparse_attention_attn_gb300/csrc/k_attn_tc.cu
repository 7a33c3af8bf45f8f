// k_attn_tc.cu -- sparse attention with the per-head sink on the 5th-generation tensor cores
// ("deepseek_v41_ref::attn" sparse_attn; "DeepSeek V4.1 - Compressed sparse attention", "Sparse
// attention" and "Grouped output"; "Join rows").
//
// All heads of a query share one K = V row per selected position, so a CTA works on one query, a
// group of 64 heads, and a range of 128-entry tiles of the query's index list J = [idx_a; idx_b]:
// tile k covers entries 128k .. 128k+127 as they stand (an invalid entry, -1, is a masked row that
// fetches nothing; a tile with no valid entry is skipped).  Y = [rows_a; rows_b] is never
// materialised: eight warps copy each tile's rows straight from the two sources (cp.async, a warp
// per 64-feature K-block, 8 lanes per 128-byte row segment) into the 128-byte swizzled layout.  Per
// tile, with the accumulators in TMEM:
//   S^T[r][h] = sum_d G[r][d] q[h][d]       (M = 128 rows, N = 64 heads, K = 512; G and q K-major)
//   softmax step: a running maximum per head, raised only when a score exceeds it by more than 2^8
//   (the accumulated output and sums are then rescaled), p = exp(S - m) rounded to bf16 in shared
//   memory (K-major [64][128]); eight warps share it (a TMEM lane quadrant and 32 heads each).  After
//   the first tile every thread checks its scores against the running maxima and the tile's maxima
//   (butterfly reductions that leave each lane one head) are formed only when one exceeds them; each
//   thread keeps its own f32 sums of p per head, reduced over the CTA once after the last tile
//   O^T[d][h] += sum_r G[r][d] P[h][r]      (M = 4 x 128 features, N = 64, K = 128 rows; the same tile
//                                            read as an MN-major operand)
// When a query's tiles are split over several CTAs (decode: few queries; the split minimises tiles
// per CTA x waves of CTAs), each CTA writes (m, l) and its share O / l, and a second, wide kernel (a
// programmatic dependent) merges the shares in CTA order with the sink, which enters the
// denominator only:
//   O = sum_c e^{m_c - M} O_c / (e^{sink - M} + sum_c e^{m_c - M} l_c).
// A query held by one CTA (prefill: many queries) is finished in place.  The result (or share) is
// staged in shared memory and written with 16-byte stores as bf16, the result together with the
// inverse rotation of its last rope_dim features at the query's position.
//
// Warps 0-7: softmax, the row copies and the result or share; warps 4-7 also run the index pass.
// Each owns one 64-feature K-block of the tile, which it refills for the next tile as soon as the
// P.V chunk reading it has completed (the next tile's rows are prefetched into L2 once the current
// one has landed); warp 8: TMEM allocation and MMA issue; all nine warps write the result or share.
// Every mbarrier wait is time-bounded.
#include "attn_common.cuh"

namespace csa {

// 2-D bf16 tensor map with 128-byte swizzle (defined with the GEMM's TMA helpers).
bool tma_map_2d_bf16(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner,
                     uint32_t box_outer);

namespace attn {

constexpr int kThreads = 288;

struct Smem {
  static constexpr size_t g = 0;                                         // KB x 16 KiB: one tile; output staging
  static constexpr size_t q = g + (size_t)KB * kBlockBytes;              // KB x 64 x 128
  static constexpr size_t p = q + (size_t)KB * HG * 128;                 // 2 x 64 x 128
  static constexpr size_t src = p + (size_t)2 * HG * 128;                // const bf16 * [kMaxTiles][TILE]
  static constexpr size_t valid = src + (size_t)kMaxTiles * TILE * 8;    // uint8 [kMaxTiles][TILE]
  static constexpr size_t red = valid + (size_t)kMaxTiles * TILE;        // float [2][4][HG]
  static constexpr size_t stat = red + (size_t)2 * 4 * HG * 4;           // float m, l, alpha, f [HG]
  static constexpr size_t wcnt = stat + (size_t)4 * HG * 4;              // int [kMaxTiles][4]
  static constexpr size_t bars = wcnt + (size_t)kMaxTiles * 4 * 4;       // u64 [16]
  static constexpr size_t misc = bars + (size_t)16 * 8;
  static constexpr size_t rot = misc + 64;                               // float2 [kRotPairs]
  static constexpr size_t total = rot + (size_t)kRotPairs * 8;
};

__global__ void __launch_bounds__(kThreads, 1) k_sparse_attn_tc(const __grid_constant__ Params P) {
  using L = Smem;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  const uint32_t s_g = tc::smem_u32(smem + L::g), s_q = tc::smem_u32(smem + L::q), s_p = tc::smem_u32(smem + L::p);
  uint8_t *sP = smem + L::p;
  const bf16 **src_list = reinterpret_cast<const bf16 **>(smem + L::src);
  uint8_t *valid = smem + L::valid;
  float *red_max = reinterpret_cast<float *>(smem + L::red), *red_sum = red_max + 4 * HG;
  float *m_sm = reinterpret_cast<float *>(smem + L::stat), *l_sm = m_sm + HG, *alpha_sm = l_sm + HG,
        *f_sm = alpha_sm + HG;
  int *wcnt = reinterpret_cast<int *>(smem + L::wcnt);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bars);
  uint64_t *g_full = bars, *q_full = bars + 4, *s_full = bars + 5, *p_full = bars + 6, *pv_done = bars + 7,
           *sm_bar = bars + 11, *drain = bars + 12, *q_ready = bars + 13;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *s_need = const_cast<int *>(abort_flag) + 1;  // [2]: by tile parity, some score above its head's maximum

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t row = blockIdx.x;  // query b*T + t
  const int split = blockIdx.y;
  const int hg = blockIdx.z;  // head group of 64
  const int b = (int)(row / P.T), t = (int)(row % P.T);
  const int k0 = split * P.tpc, nk = max(0, min(k0 + P.tpc, P.ntiles) - k0);
  constexpr uint32_t kCols = 512;  // S: 64 columns, O^T: 4 x 64

  // ---- phase 1: barriers, q, TMEM, and the index pass with the first tile's copies in flight
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) tc::mbar_init(&g_full[i], 64);  // the lanes of the pair's two loader warps
    tc::mbar_init(q_full, 1);
    tc::mbar_init(s_full, 1);
    tc::mbar_init(p_full, 256);
    for (int c = 0; c < 4; ++c) tc::mbar_init(&pv_done[c], 1);
    tc::mbar_init(sm_bar, 256);
    tc::mbar_init(q_ready, 256);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    s_need[0] = s_need[1] = 0;
    tc::fence_barrier_init();
    // q of this query's head group, independent of the selection
    tc::prefetch_tmap(&P.tm_q);
    tc::mbar_expect_tx(q_full, KB * HG * 128);
#pragma unroll 1
    for (int kb = 0; kb < KB; ++kb)
      tma_load_2d_nohint(s_q + kb * HG * 128, &P.tm_q, q_full, kb * 64, (int)(row * P.H + hg * HG));
  }
  if (warp == 8) tc::tmem_alloc(tmem_slot, kCols);

  // loader geometry: each of warps 0-7 copies one K-block (a 128-byte segment of every row), four
  // rows per instruction, 8 lanes per row; warps 4-7 take K-blocks 0-3 (they run the index pass and
  // the first S^T chunks wait for those), warps 0-3 K-blocks 4-7.  K-block pair c (features 128c ..
  // 128c+127) is one P.V chunk and one g_full barrier.
  const int kbw = (warp + 4) & 7, pw = kbw >> 1, rq = lane >> 3, cc = lane & 7;
  auto issue_tile = [&](int i) {
    const uint32_t blk = s_g + kbw * kBlockBytes;
    const bf16 *const *srcs = src_list + i * TILE;
#pragma unroll 1
    for (int i0 = 0; i0 < TILE / 4; i0 += 8) {
      const bf16 *ps[8];  // eight row addresses read before the copies that use them are issued
#pragma unroll
      for (int u = 0; u < 8; ++u) ps[u] = srcs[4 * (i0 + u) + rq];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int r = 4 * (i0 + u) + rq;
        cp_async16(blk + r * 128 + ((cc ^ (r & 7)) << 4), ps[u] ? ps[u] + 64 * kbw + 8 * cc : P.rows_a,
                   ps[u] != nullptr);
      }
    }
  };
  auto tile_ok = [&](int i) { return (wcnt[4 * i] | wcnt[4 * i + 1] | wcnt[4 * i + 2] | wcnt[4 * i + 3]) != 0; };
  // A CTA whose first tile is a whole tile of the first list (the window: its indices and rows were
  // written two or more launches earlier) forms that tile's list and starts its copies before the
  // dependency wait.
  const bool early = k0 == 0 && nk > 0 && P.na >= TILE;
  if (early) {
    if (warp >= 4 && warp < 8) index_pass(P, row, b, 0, 1, tid - 128, warp - 4, lane, src_list, valid, wcnt);
    if (warp < 8) {
      tc::named_bar(1, 256);
      if (tile_ok(0)) issue_tile(0);
    }
  }
  // Launched as a programmatic dependent of the selection kernel before it: everything above (and
  // q, written two launches earlier) overlaps that kernel; the index lists it writes are read only
  // after this wait.  The kernel after (the merge, or wo_a: programmatic dependents reading this
  // kernel's output after their own waits) may start at once.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int t1 = early ? 1 : 0;  // the first tile the pass after the wait forms
  if (warp >= 4 && warp < 8 && nk > t1)
    index_pass(P, row, b, k0 + t1, nk - t1, tid - 128, warp - 4, lane, src_list + t1 * TILE, valid + t1 * TILE,
               wcnt + 4 * t1);
  if (warp < 8) {  // the first live tile's copies (unless already started), once the lists are filled
    tc::named_bar(1, 256);
    if (!(early && tile_ok(0)))
      for (int i = t1; i < nk; ++i)
        if (tile_ok(i)) {
          issue_tile(i);
          break;
        }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  int nmine = 0;
  for (int i = 0; i < nk; ++i) nmine += tile_ok(i) ? 1 : 0;
  const uint32_t tS = tmem, tO = tmem + HG;  // O^T chunk c at tO + c*HG
  const bool single = P.nsplit == 1;

  // ---- phase 2: the tile pipeline
  if (warp == 8) {
    // ------------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t id1 = tc::idesc_bf16_f32(TILE, HG);
      const uint32_t id2 = tc::idesc_bf16_f32(TILE, HG, /*a_mn_major=*/true, /*b_mn_major=*/false);
      // q has landed (and, with RoPE, been turned): this also keeps the CTA alive until the copy is in
      bool ok = tc::mbar_wait(q_ready, 0, abort_flag);
      int n = 0;
      bool issued = false;
      for (int i = 0; i < nk && ok; ++i) {
        if (!tile_ok(i)) continue;
        const uint32_t par = (uint32_t)(n & 1);
        // S^T = G q^T, each K-block pair as soon as its two loader warps are done
        for (int w = 0; w < 4 && ok; ++w) {
          if (!(ok = tc::mbar_wait(&g_full[w], par, abort_flag))) break;
          tc::tc_fence_after();
          issued = true;
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
        if (!(ok = tc::mbar_wait(p_full, par, abort_flag))) break;
        tc::tc_fence_after();
        // O^T += G^T P^T, feature chunk c = K-blocks 2c, 2c+1; each chunk's completion frees those
        // K-blocks for their loader warps
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
      }
      if (issued) {  // nothing may still write TMEM or read shared memory when the CTA moves on
        tc::mma_commit(drain);
        const uint64_t t0 = tc::global_ns();
        while (!tc::mbar_try_wait(drain, 0) && tc::global_ns() - t0 < tc::kWaitLimitNs) {
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ warps 0-7: softmax + staging
    // warp w: TMEM lane quadrant w % 4 (tile rows, and features of an O^T chunk), heads hh .. hh+31;
    // every one of these warps also copies its K-block of each tile's rows
    const int quad = warp & 3, hh = (warp >> 2) * 32;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    uint32_t sm_uses = 0;
    auto sm_sync = [&]() -> bool {
      tc::mbar_arrive(sm_bar);
      return tc::mbar_wait(sm_bar, (sm_uses++) & 1u, abort_flag);
    };
    if (tid < HG) m_sm[tid] = -INFINITY;
    // this thread's sums of p over its rows, per head (reduced over the CTA at the end)
    float lsum[32];
#pragma unroll
    for (int h = 0; h < 32; ++h) lsum[h] = 0.f;
    // RoPE on q's last rd features (the angles read while q is still in flight)
    float4 qcs[2][2];
    if (P.rope_q) rope_q_angles(P, t, tid, qcs);
    // the angles of the result's inverse rotation, read while q is in flight (used after the tiles)
    if (single && P.o_rot && (P.rd >> 1) <= kRotPairs && tid < (P.rd >> 1))
      reinterpret_cast<float2 *>(smem + L::rot)[tid] =
          reinterpret_cast<const float2 *>(P.tab)[(int64_t)(P.start_pos + t) * (P.rd >> 1) + tid];
    bool ok = tc::mbar_wait(q_full, 0, abort_flag);
    if (ok && P.rope_q) rope_q_apply(P, smem + L::q, tid, qcs);
    tc::mbar_arrive(q_ready);
    if (ok) ok = sm_sync();
    int n = 0;
    for (int i = 0; i < nk && ok; ++i) {
      if (!tile_ok(i)) continue;
      {
        if (n > 0) {  // this warp's K-block of the previous tile has been read by its P.V chunk
          if (!(ok = tc::mbar_wait(&pv_done[pw], (uint32_t)((n - 1) & 1), abort_flag))) break;
          issue_tile(i);
        }
        cp_async_wait_all();
        fence_proxy_async();
        tc::mbar_arrive(&g_full[pw]);
        // the next tile's segments of this warp's K-block on their way to L2 while this one is used
        int nx = i + 1;
        while (nx < nk && !tile_ok(nx)) ++nx;
        if (nx < nk) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const bf16 *pr = src_list[nx * TILE + lane + 32 * k];
            if (pr) asm volatile("prefetch.global.L2 [%0];" ::"l"(pr + 64 * kbw));
          }
        }
      }
      if (!(ok = tc::mbar_wait(s_full, (uint32_t)(n & 1), abort_flag))) break;
      tc::tc_fence_after();
      float s[32];
      tmem_ld_32cols(tS + (uint32_t)hh + lane_off, s);
      const bool vr = valid[i * TILE + r] != 0;
#pragma unroll
      for (int h = 0; h < 32; ++h) s[h] = vr ? s[h] * P.scale_log2 : -INFINITY;
      // The running maximum of a head moves only when a score exceeds it by more than 2^8 (that keeps
      // exp2(s - m) below 2^8): every thread checks its scores against it and the maxima over the
      // tile are formed only when one of them does.
      bool full = true;  // the first tile always
      if (n > 0) {
        bool need = false;
#pragma unroll
        for (int h0 = 0; h0 < 32; h0 += 16) {
          float mv[16];
          lds16(mv, m_sm + hh + h0);
#pragma unroll
          for (int k = 0; k < 16; ++k) need |= s[h0 + k] > mv[k] + 8.0f;
        }
        if (need) s_need[n & 1] = 1;
        if (!(ok = sm_sync())) break;
        full = s_need[n & 1] != 0;
        if (tid == 0) s_need[(n + 1) & 1] = 0;  // the previous tile's flag, read by all by now
      }
      if (full) {
        red_max[quad * HG + hh + lane] = warp_reduce_32<true>(s, lane);
        if (!(ok = sm_sync())) break;
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
          // the previous tile's product has completed: its commit released this tile's rows
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
    }
    cp_async_wait_all();
    // l per head: this thread's sums over the warp, then over the four lane quadrants
    red_sum[quad * HG + hh + lane] = warp_reduce_32<false>(lsum, lane);
    if (ok) ok = sm_sync();
    if (ok && tid < HG)
      l_sm[tid] = (red_sum[tid] + red_sum[HG + tid]) + (red_sum[2 * HG + tid] + red_sum[3 * HG + tid]);
    if (ok && nmine > 0) ok = tc::mbar_wait(&pv_done[3], (uint32_t)((nmine - 1) & 1), abort_flag);
    if (ok && tid < HG) {
      if (single) {  // finish in place: the sink joins the denominator
        const float s2 = P.sink[hg * HG + tid] * 1.4426950408889634f;
        const float M = fmaxf(m_sm[tid], s2);
        const float em = nmine > 0 ? exp2f(m_sm[tid] - M) : 0.f;
        f_sm[tid] = em / (l_sm[tid] * em + exp2f(s2 - M));
      } else {
        f_sm[tid] = nmine > 0 ? 1.0f / l_sm[tid] : 0.f;
        float *ml = P.part_ml + ((row * P.nsplit + split) * P.H + hg * HG + tid) * 2;
        ml[0] = m_sm[tid];
        ml[1] = l_sm[tid];
      }
    }
    if (ok) ok = sm_sync();
    if (ok && nmine > 0) {
      // stage O * f as bf16 [64 heads][512] in the (now idle) tile buffer
      tc::tc_fence_after();
      bf16 *stage = reinterpret_cast<bf16 *>(smem + L::g);
#pragma unroll 1
      for (int c = 0; c < KB / 2; ++c) {
        float v[32];
        tmem_ld_32cols(tO + (uint32_t)(c * HG + hh) + lane_off, v);
#pragma unroll
        for (int h0 = 0; h0 < 32; h0 += 16) {
          float fv[16];  // the factors read before the stores below
          lds16(fv, f_sm + hh + h0);
#pragma unroll
          for (int k = 0; k < 16; ++k)
            stage[(hh + h0 + k) * HD + c * 128 + r] = __float2bfloat16_rn(v[h0 + k] * fv[k]);
        }
      }
    }
  }
  __syncthreads();

  // ---- phase 3: the result, or this CTA's share of it, by all nine warps (16-byte vectors: head h,
  // features d0 .. d0+7)
  const bf16 *stage = reinterpret_cast<const bf16 *>(smem + L::g);
  if (single) {
    const float2 *tp = !P.o_rot ? nullptr
                       : (P.rd >> 1) <= kRotPairs
                           ? reinterpret_cast<const float2 *>(smem + L::rot)
                           : reinterpret_cast<const float2 *>(P.tab) + (int64_t)(P.start_pos + t) * (P.rd >> 1);
    for (int it = tid; it < kVecs; it += kThreads) {
      const int h = it >> 6, d0 = (it & 63) * 8;
      uint4 ob = make_uint4(0u, 0u, 0u, 0u);
      if (nmine > 0) ob = *reinterpret_cast<const uint4 *>(stage + h * HD + d0);
      store_out(P.o, P.o_rot, (row * P.H + hg * HG + h) * (int64_t)HD + d0, d0, HD - P.rd, tp, ob);
    }
  } else if (nmine > 0) {
    bf16 *mine = P.part_o + ((row * P.nsplit + split) * P.H + hg * HG) * (int64_t)HD;
    for (int it = tid; it < kVecs; it += kThreads) {
      const int h = it >> 6, d0 = (it & 63) * 8;
      *reinterpret_cast<uint4 *>(mine + h * HD + d0) = *reinterpret_cast<const uint4 *>(stage + h * HD + d0);
    }
  }
  __syncthreads();
  if (warp == 8) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kCols);
  }
  if (tid == 0 && *abort_flag) atomicOr(P.status, kStatusTimeout);
}

// Merge of the split shares: block (query, 8 heads), one warp per head, two 16-byte vectors per
// thread.  The weights e^{m_c - M} l_c / den put each share O_c / l_c back on the common scale, with
// the sink in den; every thread forms its head's weights itself (no barrier).  The (m, l) of every
// share are read first, and only the shares of CTAs that found something (l > 0; the others never
// wrote theirs) after them.
constexpr int kCombHeads = 8;
constexpr int kCombThreads = 256;
struct CombineParams {
  const bf16 *part_o;
  const float *part_ml;
  int nsplit, H, T;
  const float *sink;
  bf16 *o, *o_rot;
  int rd, start_pos;
  const float *tab;
};

__global__ void __launch_bounds__(kCombThreads) k_attn_combine(const __grid_constant__ CombineParams C) {
  const int64_t row = blockIdx.x;
  const int h0 = blockIdx.y * kCombHeads, tid = threadIdx.x;
  const int t = (int)(row % C.T);
  constexpr int kPer = kCombHeads * (HD / 8) / kCombThreads;  // consecutive vectors per thread
  static_assert((HD / 8) % kPer == 0, "a thread's vectors belong to one head");
  const int h = h0 + (tid * kPer) / (HD / 8);
  const int dv = ((tid * kPer) % (HD / 8)) * 8;  // this thread's first feature
  // what does not depend on the attention kernel, before the wait: the sink term and the angles
  const float s2 = C.sink[h] * 1.4426950408889634f;
  const int tail = HD - C.rd;
  const float2 *tp = C.o_rot ? reinterpret_cast<const float2 *>(C.tab) + (int64_t)(C.start_pos + t) * (C.rd >> 1)
                             : nullptr;
  float4 cs[kPer][2];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int d0 = dv + 8 * k;
    if (tp && d0 >= tail) {
      cs[k][0] = *reinterpret_cast<const float4 *>(tp + ((d0 - tail) >> 1));
      cs[k][1] = *reinterpret_cast<const float4 *>(tp + ((d0 - tail) >> 1) + 2);
    }
  }
  // (a programmatic dependent of the attention kernel: the shares are read after this wait; wo_a,
  // a programmatic dependent of this kernel, may start at once)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float2 ml[kMaxTiles];
#pragma unroll
  for (int c = 0; c < kMaxTiles; ++c) {
    ml[c] = make_float2(-INFINITY, 0.f);
    if (c < C.nsplit) ml[c] = __ldcg(reinterpret_cast<const float2 *>(C.part_ml + ((row * C.nsplit + c) * C.H + h) * 2));
  }
  uint4 u[kPer][kMaxTiles];
#pragma unroll
  for (int c = 0; c < kMaxTiles; ++c)
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      u[k][c] = make_uint4(0u, 0u, 0u, 0u);
      if (ml[c].y > 0.f)
        u[k][c] = __ldcg(reinterpret_cast<const uint4 *>(C.part_o + ((row * C.nsplit + c) * C.H + h) * (int64_t)HD + dv + 8 * k));
    }
  // this head's weights e^{m_c - M} l_c / den
  float M = s2;
#pragma unroll
  for (int c = 0; c < kMaxTiles; ++c)
    if (ml[c].y > 0.f) M = fmaxf(M, ml[c].x);
  float den = exp2f(s2 - M), w[kMaxTiles];
#pragma unroll
  for (int c = 0; c < kMaxTiles; ++c) {
    w[c] = ml[c].y > 0.f ? ml[c].y * exp2f(ml[c].x - M) : 0.f;
    den += w[c];
  }
  const float inv = 1.0f / den;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int d0 = dv + 8 * k;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < kMaxTiles; ++c) {
      if (w[c] == 0.f) continue;
      const float wv = w[c] * inv;
      const __nv_bfloat162 *pv = reinterpret_cast<const __nv_bfloat162 *>(&u[k][c]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] = fmaf(wv, __low2float(pv[q]), acc[2 * q]);
        acc[2 * q + 1] = fmaf(wv, __high2float(pv[q]), acc[2 * q + 1]);
      }
    }
    uint4 ob;
    __nv_bfloat162 *po = reinterpret_cast<__nv_bfloat162 *>(&ob);
#pragma unroll
    for (int q = 0; q < 4; ++q) po[q] = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
    const int64_t off = (row * C.H + h) * (int64_t)HD + d0;
    if (C.o) *reinterpret_cast<uint4 *>(C.o + off) = ob;
    if (C.o_rot) {
      uint4 orr = ob;
      if (d0 >= tail) {
        const float2 c2[4] = {make_float2(cs[k][0].x, cs[k][0].y), make_float2(cs[k][0].z, cs[k][0].w),
                              make_float2(cs[k][1].x, cs[k][1].y), make_float2(cs[k][1].z, cs[k][1].w)};
        const bf16 *xb = reinterpret_cast<const bf16 *>(&ob);
        bf16 *yb = reinterpret_cast<bf16 *>(&orr);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float re, im;
          unrotate(__bfloat162float(xb[2 * q]), __bfloat162float(xb[2 * q + 1]), c2[q], re, im);
          yb[2 * q] = __float2bfloat16_rn(re);
          yb[2 * q + 1] = __float2bfloat16_rn(im);
        }
      }
      *reinterpret_cast<uint4 *>(C.o_rot + off) = orr;
    }
  }
}

}  // namespace attn

bool sparse_attn_tc_supported(const AttnArgs &a) {
  return a.hd == attn::HD && a.H % attn::HG == 0 && a.H / attn::HG <= attn::kMaxHeadGroups &&
         a.na + a.nb <= attn::kMaxTiles * attn::TILE && a.a_seq_stride % attn::HD == 0 &&
         (a.rows_b == nullptr || a.b_seq_stride % attn::HD == 0) &&
         (a.o_rot == nullptr || (a.rd % 8 == 0 && ((uintptr_t)a.tab & 15) == 0)) && ((uintptr_t)a.q & 15) == 0 &&
         ((uintptr_t)a.rows_a & 15) == 0 && ((uintptr_t)a.rows_b & 15) == 0 && ((uintptr_t)a.o & 15) == 0 &&
         ((uintptr_t)a.o_rot & 15) == 0 &&
         (a.rope_q == 0 || (a.rd % 8 == 0 && a.rd <= 64 && ((uintptr_t)a.tab & 15) == 0));  // two units a thread
}

cudaError_t launch_sparse_attn_tc(const AttnArgs &a, float *ws, size_t ws_bytes, int num_sms, cudaStream_t s,
                                  int *kernels) {
  *kernels = 0;
  using namespace attn;
  const int nq = a.B * a.T;
  if (nq <= 0) return cudaSuccess;
  Params p;
  memset(&p, 0, sizeof(p));
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
  p.rope_q = a.rope_q;
  p.ntiles = std::max(1, (a.na + p.nb + TILE - 1) / TILE);
  // tiles per CTA: the choice with the least (tiles a CTA runs) x (waves of CTAs), where CTAs past
  // the first wave that all hold the list's last tile count half a wave (that tile is the selection's
  // tail, padding whenever fewer than K positions are valid, so its CTAs mostly end after their index
  // pass); ties go to fewer CTAs.  The shares must fit the workspace (after the GEMM's counters).
  const int groups = a.H / HG;
  const size_t avail = ws_bytes > kGemmCounterBytes ? ws_bytes - kGemmCounterBytes : 0;
  int tpc = p.ntiles;
  int64_t best = INT64_MAX;
  for (int c = 1; c <= p.ntiles; ++c) {
    const int ns = (p.ntiles + c - 1) / c;
    const size_t need = (size_t)nq * ns * a.H * (HD * sizeof(bf16) + 2 * sizeof(float));
    if (ns > 1 && need > avail) continue;
    const int64_t units = (int64_t)nq * groups, ctas = units * ns;
    int64_t cost2;  // twice the cost
    if (ctas <= num_sms)
      cost2 = 2 * (int64_t)c;
    else if (ctas - num_sms <= units && (ns - 1) * c < p.ntiles)
      cost2 = 3 * (int64_t)c;  // only CTAs of the last split spill over
    else
      cost2 = 2 * (int64_t)c * ((ctas + num_sms - 1) / num_sms);
    if (cost2 <= best) {
      best = cost2;
      tpc = c;
    }
  }
  p.tpc = tpc;
  p.nsplit = (p.ntiles + tpc - 1) / tpc;
  // many units held whole (a prefill chunk): a persistent CTA an SM takes a sequence of them, the work
  // between two units overlapping the tile pipeline
  if (p.nsplit == 1 && (int64_t)nq * groups >= 2 * (int64_t)num_sms) {
    *kernels = 1;
    return launch_sparse_attn_queries_tc(p, nq * groups, num_sms, s);
  }
  uint8_t *base = reinterpret_cast<uint8_t *>(ws) + kGemmCounterBytes;
  p.part_o = reinterpret_cast<bf16 *>(base);
  p.part_ml = reinterpret_cast<float *>(base + (size_t)nq * p.nsplit * a.H * HD * sizeof(bf16));
  static SmemAttr attr;
  const size_t smem = 1024 + Smem::total;
  {
    cudaError_t e = attr.ensure((const void *)k_sparse_attn_tc, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // a programmatic dependent launch: the CTAs start (barriers, TMEM, q's copy) while the kernel before
  // them on the stream still runs, and wait for it before they read the selection
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(nq, p.nsplit, groups);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_sparse_attn_tc, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  *kernels = 1;
  if (p.nsplit == 1 || e != cudaSuccess) return e;
  CombineParams c;
  c.part_o = p.part_o;
  c.part_ml = p.part_ml;
  c.nsplit = p.nsplit;
  c.H = a.H;
  c.T = a.T;
  c.sink = a.sink;
  c.o = a.o;
  c.o_rot = a.o_rot;
  c.rd = a.rd;
  c.start_pos = a.start_pos;
  c.tab = a.tab;
  // launched as a programmatic dependent, so its launch overlaps the attention kernel's tail
  cudaLaunchConfig_t cc;
  memset(&cc, 0, sizeof(cc));
  cc.gridDim = dim3(nq, a.H / kCombHeads);
  cc.blockDim = dim3(kCombThreads);
  cc.stream = s;
  cc.attrs = at;
  cc.numAttrs = 1;
  e = cudaLaunchKernelEx(&cc, k_attn_combine, c);
  *kernels = 2;
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace csa
