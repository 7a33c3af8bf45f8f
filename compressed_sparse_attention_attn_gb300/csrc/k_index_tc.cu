// k_index_tc.cu -- the indexer's scores on the 5th-generation tensor cores ("DeepSeek V4.1 -
// Compressed sparse attention", "Indexer, re-scored": S^I[t][j] = sum_h w^I[t][h] ReLU(Q^I[t][h] . K^I[j])).
//
// The compressed keys of a sequence are contiguous rows, so a CTA takes a 128-key tile of one
// sequence and a group of up to QG of its queries, loads both by TMA (128-byte swizzled, two
// 64-element K-blocks of dI = 128) and computes every query head's dot products in one MMA chain:
//   D[j][(t, h)] = sum_d K^I[j][d] Q^I[t][h][d]      (M = 128 keys, N = QG * Hi, K = 128; TMEM)
// The four warps then read their 32 keys' rows of D and form sum_h w^I[t][h] ReLU(D) in f32 for
// each query, writing the valid positions only (j below the causal limit floor((p+1)/ratio) and the
// published length, and inside an allowed candidate block).  A decode query whose candidate mask
// spans more than 1024 keys goes to a gathered variant that reads the kept blocks' keys only.  Every
// mbarrier wait is time-bounded.
#include "csa_internal.cuh"
#include "tc_ptx.cuh"
#include "topk_core.cuh"

#include <algorithm>
#include <cstring>

namespace csa {

bool tma_map_2d_bf16(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner,
                     uint32_t box_outer);

namespace idx {

constexpr int DI = 128;
constexpr int TILE = 128;
constexpr int kThreads = 128;
constexpr int kMaxN = 256;  // MMA N: query group x heads

struct Params {
  CUtensorMap tm_k;  // K^I [B*Lstride][128], box {64, 128}
  CUtensorMap tm_q;  // Q^I [B*T*Hi][128], box {64, QG*Hi}
  const float *wI;   // [B*T][Hi]
  int T, Hi, QG, Lstride, compress_len, ratio, start_pos;
  const uint8_t *cand;
  int cand_width, cand_block;
  float *S;  // [B*T][Lstride]
  int *status;
};

__global__ void __launch_bounds__(kThreads) k_index_scores_tc(const __grid_constant__ Params P) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  const int N = P.QG * P.Hi;
  const uint32_t k_blk = TILE * 128, q_blk = (uint32_t)N * 128;
  uint8_t *sk = smem, *sq = smem + 2 * k_blk;
  float *w_s = reinterpret_cast<float *>(sq + 2 * q_blk);  // [QG][Hi]
  uint64_t *bars = reinterpret_cast<uint64_t *>(w_s + kMaxN);
  uint64_t *full = bars, *done = bars + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int j0 = blockIdx.x * TILE, t0 = blockIdx.y * P.QG, b = blockIdx.z;
  const int nqg = min(P.QG, P.T - t0);
  // the group's last query has the largest causal limit
  const int lim_max = min((P.start_pos + t0 + nqg) / P.ratio, P.compress_len);
  if (j0 >= lim_max) return;
  const uint32_t ncols = N <= 32 ? 32 : N <= 64 ? 64 : N <= 128 ? 128 : 256;

  if (tid == 0) {
    tc::mbar_init(full, 1);
    tc::mbar_init(done, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
    tc::prefetch_tmap(&P.tm_k);
    tc::prefetch_tmap(&P.tm_q);
  }
  if (warp == 0) tc::tmem_alloc(tmem_slot, ncols);
  if (tid == 0) {
    tc::mbar_expect_tx(full, 2 * (k_blk + q_blk));
    const uint64_t pol = tc::policy_evict_first();
    for (int kb = 0; kb < 2; ++kb) {
      tc::tma_load_2d(sk + kb * k_blk, &P.tm_k, full, kb * 64, b * P.Lstride + j0, pol);
      tc::tma_load_2d(sq + kb * q_blk, &P.tm_q, full, kb * 64, (b * P.T + t0) * P.Hi, pol);
    }
  }
  for (int e = tid; e < N; e += kThreads) {
    const int tq = e / P.Hi;
    w_s[e] = tq < nqg ? P.wI[(int64_t)(b * P.T + t0) * P.Hi + e] : 0.f;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (tid == 0) {
    if (tc::mbar_wait(full, 0, abort_flag)) {
      tc::tc_fence_after();
      const uint32_t id = tc::idesc_bf16_f32(TILE, N);
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
        const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sk + kb * k_blk), 16, 1024);
        const uint64_t bd = tc::sdesc_sw128(tc::smem_u32(sq + kb * q_blk), 16, 1024);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) tc::mma_bf16(tmem, ad + 2ull * k4, bd + 2ull * k4, id, (kb | k4) ? 1u : 0u);
      }
      tc::mma_commit(done);
    } else {
      // the copies may still land: wait for them (bounded) before the CTA can exit
      const uint64_t t0w = tc::global_ns();
      while (!tc::mbar_try_wait(full, 0) && tc::global_ns() - t0w < tc::kWaitLimitNs) {
      }
    }
  }
  if (tc::mbar_wait(done, 0, abort_flag)) {
    tc::tc_fence_after();
    const int r = tid;  // key within the tile = TMEM lane
    const int j = j0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    for (int tq = 0; tq < nqg; ++tq) {
      const int t = t0 + tq;
      const int64_t row = (int64_t)b * P.T + t;
      const int limit = min((P.start_pos + t + 1) / P.ratio, P.compress_len);
      float acc = 0.f;
      for (int h0 = 0; h0 < P.Hi; h0 += 16) {
        uint32_t v[16];
        tc::tmem_ld16(lane_base + (uint32_t)(tq * P.Hi + h0), v);
        tc::tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 16; ++k) acc = fmaf(w_s[tq * P.Hi + h0 + k], fmaxf(__uint_as_float(v[k]), 0.f), acc);
      }
      const bool ok = j < limit && (P.cand == nullptr || P.cand[row * P.cand_width + j / P.cand_block] != 0);
      if (ok) P.S[row * P.Lstride + j] = acc;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, ncols);
  }
  if (tid == 0 && *abort_flag && P.status) atomicOr(P.status, kStatusTimeout);
}

// An empty instruction that takes the 16 registers as inputs and outputs: placed after a
// tcgen05.wait::ld, it keeps every use of the loaded values below the wait.
__device__ __forceinline__ void tie_regs16(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}

// ---- many query groups (prefill): persistent CTAs, Q^I resident, the key tiles streamed -------------
// With more query groups than SMs, a CTA takes whole groups in turn (largest causal range first, the
// groups dealt to the CTAs in a back-and-forth order so that every CTA gets about the same number of
// key tiles) and runs each group's key tiles through a pipeline: warp 8 copies Q^I (two buffers, the
// next group's while the current one is in use) and the key tiles (a ring of three) by TMA, warp 9
// issues each tile's MMA chain into one of two TMEM accumulators, and warps 0-7 (two per TMEM lane
// quadrant, each half of the group's queries) form the head-weighted ReLU sums of a finished tile
// while the next one is multiplied.
constexpr int kRowsThreads = 576;  // warps 0-15: sums; warp 16: TMA; warp 17: TMEM and MMA
constexpr int kRowsEpi = 512;      // the epilogue threads
constexpr int kRowsKSlots = 3;

struct RowsParams {
  CUtensorMap tm_k;  // K^I [B*Lstride][128], box {64, 128}
  CUtensorMap tm_q;  // Q^I [B*T*Hi][128], box {64, QG*Hi}
  const float *wI;   // [B*T][Hi]
  int T, Hi, QG, Lstride, compress_len, ratio, start_pos;
  int gps, ngroups;  // query groups a sequence, B * gps
  int nwork;         // groups run: the first nwork in order of decreasing key range (the others'
                     // selections take every valid position, so their scores are not needed)
  const uint8_t *cand;
  int cand_width, cand_block;
  float *S;  // [B*T][Lstride]
  int *status;
};

// The r-th group in order of decreasing key range: the sequences' last groups first.
__device__ __forceinline__ void rows_group(const RowsParams &P, int r, int &b, int &t0, int &nqg, int &ntiles) {
  const int B = P.ngroups / P.gps;
  b = r % B;
  const int gq = P.gps - 1 - r / B;
  t0 = gq * P.QG;
  nqg = min(P.QG, P.T - t0);
  const int lim = min((P.start_pos + t0 + nqg) / P.ratio, P.compress_len);
  ntiles = lim > 0 ? (lim + TILE - 1) / TILE : 0;
}
// The k-th group of CTA c among G: rounds of G ranks, every other round dealt in reverse.
__device__ __forceinline__ int rows_rank(int k, int c, int G) { return k * G + ((k & 1) ? G - 1 - c : c); }

__global__ void __launch_bounds__(kRowsThreads, 1) k_index_scores_rows_tc(const __grid_constant__ RowsParams P) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  const int N = P.QG * P.Hi;
  constexpr uint32_t k_blk = TILE * 128, k_slot = 2 * k_blk;
  const uint32_t q_blk = (uint32_t)N * 128, q_buf = 2 * q_blk;
  uint8_t *sk = smem, *sq = smem + kRowsKSlots * k_slot;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sq + 2 * q_buf);
  uint64_t *k_full = bars, *k_empty = bars + kRowsKSlots, *q_full = bars + 2 * kRowsKSlots, *q_empty = q_full + 2,
           *acc_full = q_full + 4, *acc_empty = q_full + 6, *drain = q_full + 8, *wbar = q_full + 9;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 16);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  float *w_s = reinterpret_cast<float *>(bars + 18);  // [QG * Hi]: the current group's head weights, then
                                                      // [QG <= 16] int: its queries' causal limits

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const uint32_t acc_cols = N <= 32 ? 32 : N <= 64 ? 64 : N <= 128 ? 128 : 256;

  if (tid == 0) {
    for (int s = 0; s < kRowsKSlots; ++s) {
      tc::mbar_init(&k_full[s], 1);
      tc::mbar_init(&k_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&q_full[i], 1);
      tc::mbar_init(&q_empty[i], 1);
      tc::mbar_init(&acc_full[i], 1);
      tc::mbar_init(&acc_empty[i], kRowsEpi);
    }
    tc::mbar_init(drain, 1);
    tc::mbar_init(wbar, kRowsEpi);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 17) tc::tmem_alloc(tmem_slot, 2 * acc_cols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 16) {
    // ---------------------------------------------------------------- TMA: Q^I per group, key tiles
    if (lane == 0) {
      tc::prefetch_tmap(&P.tm_k);
      tc::prefetch_tmap(&P.tm_q);
      const uint64_t pol_k = tc::policy_evict_last(), pol_q = tc::policy_evict_first();
      int qi = 0, ki = 0;
      bool ok = true;
      for (int k = 0; ok && k * G < P.nwork; ++k) {
        const int r = rows_rank(k, c, G);
        if (r >= P.nwork) continue;
        int b, t0, nqg, nt;
        rows_group(P, r, b, t0, nqg, nt);
        if (nt == 0) continue;
        const int qb = qi & 1;
        if (qi >= 2 && !(ok = tc::mbar_wait(&q_empty[qb], (uint32_t)((qi / 2 - 1) & 1), abort_flag))) break;
        tc::mbar_expect_tx(&q_full[qb], 2 * q_blk);
        for (int kb = 0; kb < 2; ++kb)
          tc::tma_load_2d(sq + qb * q_buf + kb * q_blk, &P.tm_q, &q_full[qb], kb * 64, (b * P.T + t0) * P.Hi, pol_q);
        ++qi;
        for (int kt = 0; kt < nt; ++kt, ++ki) {
          const int s = ki % kRowsKSlots;
          if (ki >= kRowsKSlots &&
              !(ok = tc::mbar_wait(&k_empty[s], (uint32_t)((ki / kRowsKSlots - 1) & 1), abort_flag)))
            break;
          tc::mbar_expect_tx(&k_full[s], k_slot);
          for (int kb = 0; kb < 2; ++kb)
            tc::tma_load_2d(sk + s * k_slot + kb * k_blk, &P.tm_k, &k_full[s], kb * 64, b * P.Lstride + kt * TILE,
                            pol_k);
        }
      }
      {  // every copy has landed before the CTA can exit (bounded, whatever the flag; at once normally)
        for (int s = 0; s < kRowsKSlots && s < ki; ++s) {
          const int last = ki - 1 - ((ki - 1 - s) % kRowsKSlots);  // the last copy into slot s
          const uint64_t t0w = tc::global_ns();
          while (!tc::mbar_try_wait(&k_full[last % kRowsKSlots], (uint32_t)((last / kRowsKSlots) & 1)) &&
                 tc::global_ns() - t0w < tc::kWaitLimitNs) {
          }
        }
        for (int i = (qi >= 2 ? qi - 2 : 0); i < qi; ++i) {
          const uint64_t t0w = tc::global_ns();
          while (!tc::mbar_try_wait(&q_full[i & 1], (uint32_t)((i / 2) & 1)) && tc::global_ns() - t0w < tc::kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 17) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      const uint32_t id = tc::idesc_bf16_f32(TILE, N);
      int qi = 0, ki = 0, ai = 0;
      bool ok = true, issued = false;
      for (int k = 0; ok && k * G < P.nwork; ++k) {
        const int r = rows_rank(k, c, G);
        if (r >= P.nwork) continue;
        int b, t0, nqg, nt;
        rows_group(P, r, b, t0, nqg, nt);
        if (nt == 0) continue;
        const int qb = qi & 1;
        if (!(ok = tc::mbar_wait(&q_full[qb], (uint32_t)((qi / 2) & 1), abort_flag))) break;
        for (int kt = 0; kt < nt; ++kt, ++ki, ++ai) {
          const int s = ki % kRowsKSlots, a = ai & 1;
          if (!(ok = tc::mbar_wait(&k_full[s], (uint32_t)((ki / kRowsKSlots) & 1), abort_flag))) break;
          if (ai >= 2 && !(ok = tc::mbar_wait(&acc_empty[a], (uint32_t)((ai / 2 - 1) & 1), abort_flag))) break;
          tc::tc_fence_after();
          issued = true;
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) {
            const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sk + s * k_slot + kb * k_blk), 16, 1024);
            const uint64_t bd = tc::sdesc_sw128(tc::smem_u32(sq + qb * q_buf + kb * q_blk), 16, 1024);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
              tc::mma_bf16(tmem + (uint32_t)a * acc_cols, ad + 2ull * k4, bd + 2ull * k4, id, (kb | k4) ? 1u : 0u);
          }
          tc::mma_commit(&k_empty[s]);
          tc::mma_commit(&acc_full[a]);
        }
        if (!ok) break;
        tc::mma_commit(&q_empty[qb]);
        ++qi;
      }
      if (issued) {  // nothing may still write TMEM when the CTA frees it
        tc::mma_commit(drain);
        const uint64_t t0w = tc::global_ns();
        while (!tc::mbar_try_wait(drain, 0) && tc::global_ns() - t0w < tc::kWaitLimitNs) {
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- warps 0-15: the weighted sums
    // warp w: TMEM lane quadrant w % 4 (32 keys of the tile) and a quarter of the group's queries; the
    // group's head weights and causal limits staged in shared memory once per group.  The sums run
    // on pairs of heads (packed f32x2 multiply-adds) in four independent chains.
    const int quad = warp & 3, part = warp >> 2;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int bpq = P.Hi / 16;  // 16-column blocks a query
    int *lim_s = reinterpret_cast<int *>(w_s + kMaxN);
    int ai = 0;
    uint32_t syncs = 0;
    auto ep_sync = [&]() -> bool {  // the epilogue threads, a bounded wait
      tc::mbar_arrive(wbar);
      return tc::mbar_wait(wbar, (syncs++) & 1u, abort_flag);
    };
    bool ok = true;
    for (int k = 0; ok && k * G < P.nwork; ++k) {
      const int r = rows_rank(k, c, G);
      if (r >= P.nwork) continue;
      int b, t0, nqg, nt;
      rows_group(P, r, b, t0, nqg, nt);
      if (nt == 0) continue;
      if (!(ok = ep_sync())) break;  // every epilogue warp is done with the previous group's values
      if (tid < N) w_s[tid] = tid / P.Hi < nqg ? P.wI[(int64_t)(b * P.T + t0) * P.Hi + tid] : 0.f;
      if (tid < nqg) lim_s[tid] = min((P.start_pos + t0 + tid + 1) / P.ratio, P.compress_len);
      if (!(ok = ep_sync())) break;
      const int qw = (nqg + 3) / 4, qa = min(nqg, part * qw), qe = min(nqg, qa + qw);
      const int blk0 = qa * bpq, blk1 = qe * bpq;  // this warp's blocks, in query order
      const int64_t row0 = (int64_t)b * P.T + t0;
      for (int kt = 0; kt < nt; ++kt, ++ai) {
        const int a = ai & 1;
        if (!(ok = tc::mbar_wait(&acc_full[a], (uint32_t)((ai / 2) & 1), abort_flag))) break;
        tc::tc_fence_after();
        const uint32_t tb = tmem + (uint32_t)a * acc_cols + lane_off;
        const int j = kt * TILE + quad * 32 + lane;
        uint64_t acc2[4] = {0, 0, 0, 0};  // pairs of f32 partial sums (0.0f is all zero bits)
        int tq = qa, hb = 0;              // query, and block within it, of the next block
        if (blk1 <= blk0) {               // no queries for this warp
          tc::tc_fence_before();
          tc::mbar_arrive(&acc_empty[a]);
        }
        for (int k0 = blk0; k0 < blk1; k0 += 2) {
          // up to two 16-column blocks in flight, then one wait
          uint32_t v[2][16];
          const int nb = min(2, blk1 - k0);
#pragma unroll
          for (int u = 0; u < 2; ++u)
            if (u < nb) tc::tmem_ld16(tb + (uint32_t)((k0 + u) * 16), v[u]);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
          for (int u = 0; u < 2; ++u)
            if (u < nb) tie_regs16(v[u]);  // no use of a loaded register moves above the wait
          if (k0 + nb >= blk1) {  // every load of this accumulator has completed: the MMA may reuse it
            tc::tc_fence_before();
            tc::mbar_arrive(&acc_empty[a]);
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            if (u >= nb) break;
            const ulonglong2 *w2 = reinterpret_cast<const ulonglong2 *>(w_s + tq * P.Hi + hb * 16);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const ulonglong2 w = w2[q4];  // heads 4 q4 .. 4 q4 + 3 as two f32 pairs
              uint64_t r0, r1;
              asm("mov.b64 %0, {%1, %2};"
                  : "=l"(r0)
                  : "f"(fmaxf(__uint_as_float(v[u][4 * q4]), 0.f)), "f"(fmaxf(__uint_as_float(v[u][4 * q4 + 1]), 0.f)));
              asm("mov.b64 %0, {%1, %2};"
                  : "=l"(r1)
                  : "f"(fmaxf(__uint_as_float(v[u][4 * q4 + 2]), 0.f)), "f"(fmaxf(__uint_as_float(v[u][4 * q4 + 3]), 0.f)));
              asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[(2 * q4) & 3]) : "l"(w.x), "l"(r0));
              asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[(2 * q4 + 1) & 3]) : "l"(w.y), "l"(r1));
            }
            if (++hb == bpq) {  // query tq is complete
              float sp[8];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                asm("mov.b64 {%0, %1}, %2;" : "=f"(sp[2 * e]), "=f"(sp[2 * e + 1]) : "l"(acc2[e]));
              const float acc = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
              const int64_t row = row0 + tq;
              if (j < lim_s[tq] && (P.cand == nullptr || P.cand[row * P.cand_width + j / P.cand_block] != 0))
                P.S[row * P.Lstride + j] = acc;
#pragma unroll
              for (int e = 0; e < 4; ++e) acc2[e] = 0;
              hb = 0;
              ++tq;
            }
          }
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 17) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 2 * acc_cols);
  }
  if (tid == 0 && *abort_flag && P.status) atomicOr(P.status, kStatusTimeout);
}


// ---- candidate-gathered variant (one query per CTA group, T == 1) --------------------------------
// With a candidate block mask, only the kept blocks' keys can be selected, so only those are read:
// each CTA scans the query's mask row into the ordered list of kept 64-key units (a block of
// cand_block keys is cand_block / 64 units), and takes the unit pairs c, c + P, c + 2P, ... of it.
// A pair is two TMA boxes of 64 keys stacked into one 128-row operand (the 128-byte swizzle repeats
// every 8 rows, so two 64-row boxes form the layout of one 128-row box); pairs are double-buffered
// against the MMA and the epilogue, each buffer with its own TMEM accumulator.
constexpr int kGatherBufs = 3;

struct GatherParams {
  CUtensorMap tm_k;  // K^I [B*Lstride][128], box {64, 64}
  CUtensorMap tm_q;  // Q^I [B*Hi][128], box {64, Hi}
  const float *wI;   // [B][Hi]
  int Hi, Lstride, compress_len, ratio, start_pos, P, max_units;
  const uint8_t *cand;
  int cand_width, cand_block;
  float *S;  // [B][Lstride]
  int *status;
};

__global__ void __launch_bounds__(kThreads) k_index_scores_gather_tc(const __grid_constant__ GatherParams P) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  const int N = P.Hi;
  constexpr uint32_t k_buf = TILE * 128 * 2;  // a pair: two 64-column halves of 128 keys
  const uint32_t q_half = (uint32_t)N * 128;
  uint8_t *sk = smem, *sq = smem + kGatherBufs * k_buf;
  float *w_s = reinterpret_cast<float *>(sq + 2 * q_half);        // [Hi]
  int *units = reinterpret_cast<int *>(w_s + kMaxN);              // [max_units] kept 64-key units
  uint64_t *bars = reinterpret_cast<uint64_t *>(units + ((P.max_units + 1) & ~1));
  uint64_t *full = bars, *done = bars + kGatherBufs, *qbar = bars + 2 * kGatherBufs;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(qbar + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *s_nunits = const_cast<int *>(abort_flag) + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, b = blockIdx.y;
  const int limit = min((P.start_pos + 1) / P.ratio, P.compress_len);
  const int per_block = P.cand_block / 64;
  const uint32_t ncols = N * kGatherBufs <= 32 ? 32 : N * kGatherBufs <= 64 ? 64 : N * kGatherBufs <= 128 ? 128
                         : N * kGatherBufs <= 256 ? 256 : 512;

  if (tid == 0) {
    for (int i = 0; i < 2 * kGatherBufs + 1; ++i) tc::mbar_init(&bars[i], 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
    tc::prefetch_tmap(&P.tm_k);
    tc::prefetch_tmap(&P.tm_q);
    tc::mbar_expect_tx(qbar, 2 * q_half);
    const uint64_t pol = tc::policy_evict_first();
    for (int kb = 0; kb < 2; ++kb) tc::tma_load_2d(sq + kb * q_half, &P.tm_q, qbar, kb * 64, b * N, pol);
  }
  for (int e = tid; e < N; e += kThreads) w_s[e] = P.wI[(int64_t)b * N + e];
  if (warp == 1) {
    // the kept units in ascending key order
    const uint8_t *cr = P.cand + (int64_t)b * P.cand_width;
    const int nblk = min((limit + P.cand_block - 1) / P.cand_block, P.cand_width);
    int n = 0;
    for (int b0 = 0; b0 < nblk; b0 += 8 * 32) {
      uint32_t kv[8];  // eight rounds of mask bytes in flight at once
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int blk = b0 + k * 32 + lane;
        kv[k] = blk < nblk ? cr[blk] : 0u;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int blk = b0 + k * 32 + lane;
        const bool keep = kv[k] != 0u;
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
        if (keep) {
          const int base = n + __popc(bal & ((1u << lane) - 1u)) * per_block;
          for (int s = 0; s < per_block; ++s)
            if (base + s < P.max_units) units[base + s] = blk * per_block + s;
        }
        n += __popc(bal) * per_block;
      }
    }
    // units past the causal limit hold no valid key
    if (lane == 0) {
      while (n > 0 && n <= P.max_units && units[n - 1] * 64 >= limit) --n;
      *s_nunits = min(n, P.max_units);
    }
  }
  if (warp == 0) tc::tmem_alloc(tmem_slot, ncols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nunits = *s_nunits;
  const int npairs_all = (nunits + 1) / 2;
  const int mine = c < npairs_all ? (npairs_all - c + P.P - 1) / P.P : 0;
  auto issue = [&](int i) {  // pair i of this CTA into buffer i % kGatherBufs
    const int pi = c + i * P.P;
    const int u0 = units[2 * pi], two = 2 * pi + 1 < nunits;
    uint64_t *bar = &full[i % kGatherBufs];
    uint8_t *dst = sk + (i % kGatherBufs) * k_buf;
    const uint64_t pol = tc::policy_evict_first();
    tc::mbar_expect_tx(bar, (two ? 2u : 1u) * 2u * 64u * 128u);
    for (int kb = 0; kb < 2; ++kb) {
      tc::tma_load_2d(dst + kb * (k_buf / 2), &P.tm_k, bar, kb * 64, b * P.Lstride + u0 * 64, pol);
      if (two)
        tc::tma_load_2d(dst + kb * (k_buf / 2) + 64 * 128, &P.tm_k, bar, kb * 64,
                        b * P.Lstride + units[2 * pi + 1] * 64, pol);
    }
  };
  int issued = 0, landed = 0;  // (thread 0) pairs whose copies were issued / seen complete
  bool q_landed = false;
  if (tid == 0)
    for (; issued < min(mine, kGatherBufs); ++issued) issue(issued);
  bool ok = true;
  if (tid == 0 && mine > 0) ok = q_landed = tc::mbar_wait(qbar, 0, abort_flag);
  const uint32_t id = tc::idesc_bf16_f32(TILE, N);
  const float *Srow_w = w_s;
  float *Srow = P.S + (int64_t)b * P.Lstride;
  for (int i = 0; i < mine; ++i) {
    const int buf = i % kGatherBufs;
    const uint32_t par = (uint32_t)(i / kGatherBufs) & 1u;
    if (tid == 0 && ok) {
      ok = tc::mbar_wait(&full[buf], par, abort_flag);
      if (ok) {
        ++landed;
        tc::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * N);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sk + buf * k_buf + kb * (k_buf / 2)), 16, 1024);
          const uint64_t bd = tc::sdesc_sw128(tc::smem_u32(sq + kb * q_half), 16, 1024);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) tc::mma_bf16(d, ad + 2ull * k4, bd + 2ull * k4, id, (kb | k4) ? 1u : 0u);
        }
        tc::mma_commit(&done[buf]);
      }
    }
    const bool got = tc::mbar_wait(&done[buf], par, abort_flag);
    tc::tc_fence_after();
    // the buffer is free once the MMA has read it: refill it with pair i + kGatherBufs
    if (got && tid == 0 && i + kGatherBufs < mine) issue(issued++);
    const int pi = c + i * P.P;
    const int r = tid;
    const int slot = 2 * pi + (r >> 6);
    const int j = slot < nunits ? units[slot] * 64 + (r & 63) : limit;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(buf * N);
    float acc = 0.f;
    for (int h0 = 0; h0 < N; h0 += 16) {
      uint32_t v[16];
      tc::tmem_ld16_wait(lane_base + (uint32_t)h0, v);
#pragma unroll
      for (int k = 0; k < 16; ++k) acc = fmaf(Srow_w[h0 + k], fmaxf(__uint_as_float(v[k]), 0.f), acc);
    }
    if (got && j < limit) Srow[j] = acc;
    // every thread has read accumulator buf before the MMA of pair i + kGatherBufs overwrites it;
    // a wait that gave up anywhere ends the loop for every thread alike
    tc::tc_fence_before();
    const int failed = __syncthreads_or(!got);
    tc::tc_fence_after();
    if (failed) break;
  }
  if (tid == 0) {
    // copies that may still be in flight (none unless a wait gave up): let them land, bounded,
    // before the CTA exits
    const uint64_t t0w = tc::global_ns();
    auto drain = [&](uint64_t *bar, uint32_t par) {
      while (!tc::mbar_try_wait(bar, par) && tc::global_ns() - t0w < tc::kWaitLimitNs) {
      }
    };
    if (!q_landed) drain(qbar, 0);
    for (int i = landed; i < issued; ++i) drain(&full[i % kGatherBufs], (uint32_t)(i / kGatherBufs) & 1u);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, ncols);
  }
  if (tid == 0 && *abort_flag && P.status) atomicOr(P.status, kStatusTimeout);
}


// ---- gathered scores + top-k across a cluster (long decode rows) ---------------------------------
// The gathered variant's work for one query split over a thread-block cluster of P CTAs: CTA c takes
// the contiguous run of kept unit pairs [c np / P, (c+1) np / P), so the CTAs' ranges are in
// ascending position.  Within a CTA the work is a pipeline: warp 4 copies the pairs' keys by TMA into
// a ring of NB 32 KiB slots as far ahead as the ring allows, warp 5 issues each pair's MMA chain into
// one of two TMEM accumulators as soon as its keys have landed (the slot is free again when the chain
// completes), and warps 0-3 turn each accumulator into scores while the next pair's chain runs.  Each
// CTA keeps its keys' scores in shared memory as 32-bit order keys with a validity bit (the position
// of entry i follows from the unit list), and the cluster then selects together: the counts and, per
// radix pass, the 256-bin histograms are read from every CTA through distributed shared memory,
// every CTA takes the same digit, and each writes its taken positions in ascending order at the
// offset of the CTAs before it.  The scores never go to global memory and the top-k needs no launch
// of its own.
constexpr int kGtThreads = 192;   // warps 0-3: scores; warp 4: key copies; warp 5: TMEM and MMA
constexpr int kGtMaxBufs = 6;     // key slots
constexpr int kGtMaxKeys = 8192;  // keys a CTA holds (its pairs x 128)
constexpr uint32_t kGtSlot = TILE * 128 * 2;  // a pair: two 64-column halves of 128 keys

struct GatherTopkParams {
  CUtensorMap tm_k;  // K^I [B*Lstride][128], box {64, 64}
  CUtensorMap tm_q;  // Q^I [B*Hi][128], box {64, Hi}
  const float *wI;   // [B][Hi]
  int Hi, Lstride, compress_len, ratio, start_pos, P, max_units;
  int nbufs, cap_keys;  // key slots; keys a CTA can hold (a multiple of 128)
  const uint8_t *cand;
  int cand_width, cand_block, K, offset;
  int32_t *out;  // [B][K]
  int *status;
};

__global__ void __launch_bounds__(kGtThreads) k_index_gather_topk_tc(const __grid_constant__ GatherTopkParams P) {
  // Launched as a programmatic dependent of the projection that writes Q^I: the unit list, the head
  // weights and the key copies (all written before that launch began) start at once, Q^I is read only
  // after the dependency wait, and the attention after this kernel (which reads q before its own
  // wait) may launch only after it.
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  const int N = P.Hi, NB = P.nbufs;
  const uint32_t q_half = (uint32_t)N * 128;
  uint8_t *sk = smem, *sq = smem + NB * kGtSlot;
  float *w_s = reinterpret_cast<float *>(sq + 2 * q_half);      // [Hi]
  uint32_t *keys = reinterpret_cast<uint32_t *>(w_s + kMaxN);   // [cap_keys] order keys
  uint32_t *vmask = keys + P.cap_keys;                          // [cap_keys / 32] validity bits
  unsigned *hists = vmask + P.cap_keys / 32;                    // [2][256] per pass
  // [12]: count, taken, count of positive scores, -, then the least, the largest and the least
  // positive value (u64)
  unsigned *xchg = hists + 512;
  unsigned long long *xval = reinterpret_cast<unsigned long long *>(xchg + 4);
  int *units = reinterpret_cast<int *>(xchg + 12);              // [max_units]
  uint64_t *bars = reinterpret_cast<uint64_t *>(units + ((P.max_units + 1) & ~1));
  uint64_t *full = bars, *sfree = bars + NB, *done = bars + 2 * NB, *accfree = done + 2, *qbar = accfree + 2,
           *drain = qbar + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *s_nunits = const_cast<int *>(abort_flag) + 1;
  __shared__ TopkShared sh;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = tc::cluster_ctarank();
  const int b = blockIdx.y;
  const int limit = min((P.start_pos + 1) / P.ratio, P.compress_len);
  const int per_block = P.cand_block / 64;
  const uint32_t ncols = 2 * N <= 32 ? 32 : 2 * N <= 64 ? 64 : 2 * N <= 128 ? 128 : 2 * N <= 256 ? 256 : 512;

  if (tid == 0) {
    for (int i = 0; i < NB; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&sfree[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&done[i], 1);
      tc::mbar_init(&accfree[i], 128);  // the scoring threads
    }
    tc::mbar_init(qbar, 1);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    topk_shared_init(sh, P.K);
    tc::fence_barrier_init();
    tc::prefetch_tmap(&P.tm_k);
    tc::prefetch_tmap(&P.tm_q);
  }
  for (int e = tid; e < N; e += kGtThreads) w_s[e] = P.wI[(int64_t)b * N + e];
  if (warp == 1) {
    // the kept units in ascending key order
    const uint8_t *cr = P.cand + (int64_t)b * P.cand_width;
    const int nblk = min((limit + P.cand_block - 1) / P.cand_block, P.cand_width);
    int n = 0;
    for (int b0 = 0; b0 < nblk; b0 += 8 * 32) {
      uint32_t kv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int blk = b0 + k * 32 + lane;
        kv[k] = blk < nblk ? cr[blk] : 0u;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int blk = b0 + k * 32 + lane;
        const bool keep = kv[k] != 0u;
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
        if (keep) {
          const int base = n + __popc(bal & ((1u << lane) - 1u)) * per_block;
          for (int s2 = 0; s2 < per_block; ++s2)
            if (base + s2 < P.max_units) units[base + s2] = blk * per_block + s2;
        }
        n += __popc(bal) * per_block;
      }
    }
    if (lane == 0) {
      while (n > 0 && n <= P.max_units && units[n - 1] * 64 >= limit) --n;
      *s_nunits = min(n, P.max_units);
    }
  }
  if (warp == 5) tc::tmem_alloc(tmem_slot, ncols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nunits = *s_nunits;
  const int npairs_all = (nunits + 1) / 2;
  const int pa = (int)(((int64_t)rank * npairs_all) / P.P), pb = (int)(((int64_t)(rank + 1) * npairs_all) / P.P);
  const int mine = min(pb - pa, P.cap_keys / TILE);  // (the host sizes P so that every range fits)
  bool ok = true;
  unsigned my_valid = 0;
  if (warp == 4) {
    // ------------------------------------------------------------------ key copies
    if (lane == 0) {
      const uint64_t pol = tc::policy_evict_first();
      int issued = 0;
      for (int i = 0; i < mine && ok; ++i) {
        const int buf = i % NB;
        if (i >= NB && !(ok = tc::mbar_wait(&sfree[buf], (uint32_t)((i / NB) - 1) & 1u, abort_flag))) break;
        const int pi = pa + i;
        const int u0 = units[2 * pi], two = 2 * pi + 1 < nunits;
        uint8_t *dst = sk + buf * kGtSlot;
        tc::mbar_expect_tx(&full[buf], (two ? 2u : 1u) * 2u * 64u * 128u);
        for (int kb = 0; kb < 2; ++kb) {
          tc::tma_load_2d(dst + kb * (kGtSlot / 2), &P.tm_k, &full[buf], kb * 64, b * P.Lstride + u0 * 64, pol);
          if (two)
            tc::tma_load_2d(dst + kb * (kGtSlot / 2) + 64 * 128, &P.tm_k, &full[buf], kb * 64,
                            b * P.Lstride + units[2 * pi + 1] * 64, pol);
        }
        ++issued;
      }
      // copies that may still be in flight (none unless a wait gave up): let them land, bounded
      const uint64_t t0 = tc::global_ns();
      for (int i = max(0, issued - NB); i < issued; ++i)
        while (!tc::mbar_try_wait(&full[i % NB], (uint32_t)(i / NB) & 1u) && tc::global_ns() - t0 < tc::kWaitLimitNs) {
        }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t id = tc::idesc_bf16_f32(TILE, N);
      bool issued = false;
      asm volatile("griddepcontrol.wait;" ::: "memory");
      asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
      if (mine > 0) {
        tc::mbar_expect_tx(qbar, 2 * q_half);
        const uint64_t pol = tc::policy_evict_first();
        for (int kb = 0; kb < 2; ++kb) tc::tma_load_2d(sq + kb * q_half, &P.tm_q, qbar, kb * 64, b * N, pol);
        ok = tc::mbar_wait(qbar, 0, abort_flag);
      }
      for (int i = 0; i < mine && ok; ++i) {
        const int buf = i % NB, acc = i & 1;
        if (!(ok = tc::mbar_wait(&full[buf], (uint32_t)(i / NB) & 1u, abort_flag))) break;
        if (i >= 2 && !(ok = tc::mbar_wait(&accfree[acc], (uint32_t)((i >> 1) - 1) & 1u, abort_flag))) break;
        tc::tc_fence_after();
        issued = true;
        const uint32_t d = tmem + (uint32_t)(acc * N);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sk + buf * kGtSlot + kb * (kGtSlot / 2)), 16, 1024);
          const uint64_t bd = tc::sdesc_sw128(tc::smem_u32(sq + kb * q_half), 16, 1024);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) tc::mma_bf16(d, ad + 2ull * k4, bd + 2ull * k4, id, (kb | k4) ? 1u : 0u);
        }
        tc::mma_commit(&done[acc]);
        tc::mma_commit(&sfree[buf]);
      }
      if (mine > 0 && !ok) {  // q may still be in flight after a wait gave up: let it land, bounded
        const uint64_t t0 = tc::global_ns();
        while (!tc::mbar_try_wait(qbar, 0) && tc::global_ns() - t0 < tc::kWaitLimitNs) {
        }
      }
      if (issued) {  // nothing may still write TMEM or read shared memory when the CTA moves on
        tc::mma_commit(drain);
        const uint64_t t0 = tc::global_ns();
        while (!tc::mbar_try_wait(drain, 0) && tc::global_ns() - t0 < tc::kWaitLimitNs) {
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ scores (warps 0-3)
    for (int i = 0; i < mine && ok; ++i) {
      const int acc = i & 1;
      if (!(ok = tc::mbar_wait(&done[acc], (uint32_t)(i >> 1) & 1u, abort_flag))) break;
      tc::tc_fence_after();
      const int slot = 2 * (pa + i) + (tid >> 6);
      const int j = slot < nunits ? units[slot] * 64 + (tid & 63) : limit;
      const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(acc * N);
      float sacc = 0.f;
      for (int h0 = 0; h0 < N; h0 += 16) {
        uint32_t v[16];
        tc::tmem_ld16_wait(lane_base + (uint32_t)h0, v);
#pragma unroll
        for (int k = 0; k < 16; ++k) sacc = fmaf(w_s[h0 + k], fmaxf(__uint_as_float(v[k]), 0.f), sacc);
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&accfree[acc]);
      const bool valid = j < limit;
      keys[i * TILE + tid] = order_key(sacc);
      const unsigned bal = __ballot_sync(0xffffffffu, valid);
      if (lane == 0) vmask[i * 4 + warp] = bal;
      my_valid += valid ? 1u : 0u;
    }
  }
  // (every thread past the dependency wait before the selection is written: the kernels before may
  // read the previous selection)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int failed = __syncthreads_or(!ok);
  // ---- the selection, across the cluster ---------------------------------------------------------
  // entry i (key pair i / 128 of this CTA's range, row i % 128) as the top-k's 64-bit value (0: not a
  // valid position), built once into the key slots, all copies and products having completed
  const int n_iter = failed ? 0 : mine * TILE;
  unsigned long long *vals = reinterpret_cast<unsigned long long *>(sk);  // (cap_keys x 8 <= 2 slots)
  for (int i = tid; i < n_iter; i += kGtThreads) {
    unsigned long long v = 0ull;
    if ((vmask[i >> 5] >> (i & 31)) & 1u) {
      const int row = i % TILE;
      const int j = units[2 * (pa + i / TILE) + (row >> 6)] * 64 + (row & 63);
      v = ((unsigned long long)keys[i] << 32) | (unsigned long long)(~(uint32_t)j);
    }
    vals[i] = v;
  }
  __syncthreads();
  // thread t owns the contiguous entries [c0, c1) (ascending position) for the output
  const int chunk = (n_iter + kGtThreads - 1) / kGtThreads;
  const int c0 = min(n_iter, tid * chunk), c1 = min(n_iter, c0 + chunk);
  unsigned wv = failed ? 0u : my_valid;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wv += __shfl_xor_sync(0xffffffffu, wv, o);
  // the range the selection lies in: the least and the largest valid value, and the least value of
  // a positive score (its top bit set) with their count -- when at least K scores are positive the
  // K largest all are, and only the positive range needs resolving
  unsigned long long vmin = ~0ull, vmax = 0ull, vpos = ~0ull;
  unsigned npos = 0;
  for (int i = tid; i < n_iter; i += kGtThreads) {
    const unsigned long long v = vals[i];
    if (v) {
      vmin = min(vmin, v);
      vmax = max(vmax, v);
      if (v >> 63) {
        vpos = min(vpos, v);
        ++npos;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    vmin = min(vmin, __shfl_xor_sync(0xffffffffu, vmin, o));
    vmax = max(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
    vpos = min(vpos, __shfl_xor_sync(0xffffffffu, vpos, o));
    npos += __shfl_xor_sync(0xffffffffu, npos, o);
  }
  if (tid == 0) {
    xval[0] = ~0ull;
    xval[1] = 0ull;
    xval[2] = ~0ull;
    xchg[2] = 0;
  }
  __syncthreads();
  if (lane == 0) {
    atomicAdd(&sh.count, wv);
    atomicMin(&xval[0], vmin);
    atomicMax(&xval[1], vmax);
    atomicMin(&xval[2], vpos);
    atomicAdd(&xchg[2], npos);
  }
  __syncthreads();
  if (tid == 0) xchg[0] = sh.count;
  tc::cluster_sync();  // every CTA's counts and value ranges are published
  // lane c of every warp reads CTA c's figures (all remote loads in flight together), then the warp
  // reduces them
  unsigned total = 0, total_pos = 0;
  unsigned long long gmin = ~0ull, gmax = 0ull, gpos = ~0ull;
  if (lane < P.P) {
    const uint32_t c = (uint32_t)lane;
    total = tc::ld_cluster_u32(tc::cluster_map(tc::smem_u32(&xchg[0]), c));
    total_pos = tc::ld_cluster_u32(tc::cluster_map(tc::smem_u32(&xchg[2]), c));
    gmin = tc::ld_cluster_u64(tc::cluster_map(tc::smem_u32(&xval[0]), c));
    gmax = tc::ld_cluster_u64(tc::cluster_map(tc::smem_u32(&xval[1]), c));
    gpos = tc::ld_cluster_u64(tc::cluster_map(tc::smem_u32(&xval[2]), c));
  }
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) {  // (P <= 8 lanes hold figures)
    total += __shfl_xor_sync(0xffffffffu, total, o);
    total_pos += __shfl_xor_sync(0xffffffffu, total_pos, o);
    gmin = min(gmin, __shfl_xor_sync(0xffffffffu, gmin, o));
    gmax = max(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
    gpos = min(gpos, __shfl_xor_sync(0xffffffffu, gpos, o));
  }
  total = __shfl_sync(0xffffffffu, total, 0);
  total_pos = __shfl_sync(0xffffffffu, total_pos, 0);
  gmin = __shfl_sync(0xffffffffu, gmin, 0);
  gmax = __shfl_sync(0xffffffffu, gmax, 0);
  gpos = __shfl_sync(0xffffffffu, gpos, 0);
  if (total_pos >= (unsigned)P.K) gmin = gpos;
  const bool all = total <= (unsigned)P.K;
  int fs = 0;
  unsigned long long thr = 0ull;
  if (!all) {
    // the K largest share the bits above the first one where the least value of their range and the
    // largest differ: each pass resolves the next (up to) 8 bits below the resolved ones, bit-aligned
    const unsigned long long diff = gmin ^ gmax;
    int lo = diff ? 64 - __clzll((long long)diff) : 0;  // bits >= lo are resolved
    if (tid == 0) sh.prefix = lo >= 64 ? 0ull : (gmax & (~0ull << lo));
    int pass = 0;
    for (; lo > 0; ++pass) {
      const int w = min(8, lo), shift = lo - w;
      unsigned *hist = hists + (pass & 1) * 256;
      for (int i = tid; i < 256; i += kGtThreads) hist[i] = 0;
      __syncthreads();
      const unsigned long long prefix = sh.prefix;
      const unsigned long long hi_mask = lo >= 64 ? 0ull : (~0ull << lo);
      const unsigned dmask = (1u << w) - 1u;
      for (int i = tid; i < n_iter; i += kGtThreads) {
        const unsigned long long v = vals[i];
        if (v && (v & hi_mask) == (prefix & hi_mask)) atomicAdd(&hist[(unsigned)(v >> shift) & dmask], 1u);
      }
      tc::cluster_sync();  // every CTA's histogram of this pass is complete
      for (int i = tid; i < 256; i += kGtThreads) {
        unsigned hv[8];  // every CTA's bin, the remote loads in flight together
#pragma unroll
        for (int c = 0; c < 8; ++c)
          hv[c] = c < P.P ? tc::ld_cluster_u32(tc::cluster_map(tc::smem_u32(&hist[i]), (uint32_t)c)) : 0u;
        unsigned t = 0;
#pragma unroll
        for (int c = 0; c < 8; ++c) t += hv[c];
        sh.hist[i] = t;
      }
      __syncthreads();
      if (warp == 0) radix_pick(sh, sh.hist, shift);
      __syncthreads();
      if (sh.done) break;  // the same in every CTA: each summed the same histograms
      lo = shift;
    }
    fs = sh.shift;
    thr = sh.prefix >> fs;
  }
  // taken positions: this CTA's in ascending order (one block-wide scan of the chunks' counts), after
  // those of the CTAs before it
  unsigned cnt = 0;
  for (int i = c0; i < c1; ++i) {
    const unsigned long long v = vals[i];
    cnt += (v != 0ull && (all || (v >> fs) >= thr)) ? 1u : 0u;
  }
  unsigned incl = cnt;
#pragma unroll
  for (int o2 = 1; o2 < 32; o2 <<= 1) {
    const unsigned n2 = __shfl_up_sync(0xffffffffu, incl, o2);
    if (lane >= o2) incl += n2;
  }
  if (lane == 31) sh.wsum[warp] = incl;
  __syncthreads();
  unsigned excl = incl - cnt;
  for (int w2 = 0; w2 < warp; ++w2) excl += sh.wsum[w2];
  if (tid == 0) {
    unsigned ct = 0;
    for (int w2 = 0; w2 < kGtThreads / 32; ++w2) ct += sh.wsum[w2];
    xchg[1] = ct;
  }
  tc::cluster_sync();  // every CTA's taken count is published
  unsigned before = 0, taken_all = 0;
  {
    const unsigned t = lane < P.P ? tc::ld_cluster_u32(tc::cluster_map(tc::smem_u32(&xchg[1]), (uint32_t)lane)) : 0u;
    before = lane < (int)rank ? t : 0u;
    taken_all = t;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) {
      before += __shfl_xor_sync(0xffffffffu, before, o);
      taken_all += __shfl_xor_sync(0xffffffffu, taken_all, o);
    }
    before = __shfl_sync(0xffffffffu, before, 0);
    taken_all = __shfl_sync(0xffffffffu, taken_all, 0);
  }
  int32_t *o = P.out + (int64_t)b * P.K;
  unsigned slot = before + excl;
  for (int i = c0; i < c1; ++i) {
    const unsigned long long v = vals[i];
    if (v != 0ull && (all || (v >> fs) >= thr)) {
      if (slot < (unsigned)P.K) o[slot] = (int32_t)(~(uint32_t)(v & 0xffffffffull)) + P.offset;
      ++slot;
    }
  }
  if (rank == (uint32_t)P.P - 1)
    for (int k = (int)taken_all + tid; k < P.K; k += kGtThreads) o[k] = -1;
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, ncols);
  }
  if (tid == 0 && *abort_flag && P.status) atomicOr(P.status, kStatusTimeout);
  tc::cluster_sync();  // no CTA leaves while another may still read its shared memory
}

// ---- fused scores + top-k for short decode rows --------------------------------------------------
// A decode query (T == 1) with at most kFusedTiles * 128 valid positions: one CTA loads its key tiles
// and Q^I by TMA (one barrier a tile, the copies issued by several lanes), runs one MMA chain per
// tile into its own TMEM columns as soon as the tile has landed, and the epilogue turns each valid
// key's score straight into the top-k's 64-bit value in shared memory, tile by tile behind the
// chains; the selection and ordering then run in the same CTA (the scores never go to global memory,
// and the top-k needs no launch of its own).  The scores' arithmetic is the dense kernel's, so the
// selection is the same.
constexpr int kFusedTiles = 4;
constexpr int kFusedThreads = 512;

struct FusedParams {
  CUtensorMap tm_k;  // K^I [B*Lstride][128], box {64, 128}
  CUtensorMap tm_q;  // Q^I [B*Hi][128], box {64, Hi}
  const float *wI;   // [B][Hi]
  int Hi, Lstride, compress_len, ratio, start_pos;
  const uint8_t *cand;
  int cand_width, cand_block, K, offset;
  int32_t *out;      // [B][K]
  int *status;
};

__global__ void __launch_bounds__(kFusedThreads, 1) k_index_topk_fused_tc(const __grid_constant__ FusedParams P) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  __shared__ TopkShared sh;
  const int N = P.Hi;
  constexpr uint32_t k_blk = TILE * 128;  // one 64-column half of a 128-key tile
  const uint32_t q_blk = (uint32_t)N * 128;
  uint8_t *sk = smem, *sq = smem + kFusedTiles * 2 * k_blk;
  float *w_s = reinterpret_cast<float *>(sq + 2 * q_blk);                        // [Hi]
  unsigned long long *vals = reinterpret_cast<unsigned long long *>(w_s + kMaxN);  // [512] by position
  uint64_t *bars = reinterpret_cast<uint64_t *>(vals + kFusedTiles * TILE);
  uint64_t *full = bars, *done = bars + kFusedTiles, *qbar = bars + 2 * kFusedTiles;  // full, done: a tile each
  uint64_t *drain = qbar + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x;
  const int limit = max(0, min((P.start_pos + 1) / P.ratio, P.compress_len));
  const int ntiles = min(kFusedTiles, (limit + TILE - 1) / TILE);
  const uint32_t ncols = N * kFusedTiles <= 32 ? 32 : N * kFusedTiles <= 64 ? 64 : N * kFusedTiles <= 128 ? 128
                         : N * kFusedTiles <= 256 ? 256 : 512;
  if (tid == 0) {
    for (int i = 0; i < 2 * kFusedTiles + 2; ++i) tc::mbar_init(&bars[i], 1);
    *abort_flag = 0;
    topk_shared_init(sh, P.K);
    tc::fence_barrier_init();
  }
  __syncthreads();
  // the copies: lane 0 of warp 1 takes q, lane i + 1 tile i.  Launched as a programmatic dependent of
  // the projection that writes Q^I: the key tiles, w^I and the mask (all written before that launch
  // began) are read at once, Q^I only after the dependency wait.
  if (warp == 1 && lane <= ntiles && ntiles > 0) {
    const uint64_t pol = tc::policy_evict_first();
    if (lane == 0) {
      tc::prefetch_tmap(&P.tm_q);
      asm volatile("griddepcontrol.wait;" ::: "memory");
      // the attention after this kernel may start its set-up now: it reads q (written by the
      // projection just waited for) before its own wait, and the selection only after it
      asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
      tc::mbar_expect_tx(qbar, 2 * q_blk);
      for (int kb = 0; kb < 2; ++kb) tc::tma_load_2d(sq + kb * q_blk, &P.tm_q, qbar, kb * 64, b * N, pol);
    } else {
      const int i = lane - 1;
      tc::prefetch_tmap(&P.tm_k);
      tc::mbar_expect_tx(&full[i], 2 * k_blk);
      for (int kb = 0; kb < 2; ++kb)
        tc::tma_load_2d(sk + (2 * i + kb) * k_blk, &P.tm_k, &full[i], kb * 64, b * P.Lstride + i * TILE, pol);
    }
  }
  for (int e = tid; e < N; e += kFusedThreads) w_s[e] = P.wI[(int64_t)b * N + e];
  // the epilogue threads' candidate-mask bytes, read while the keys are in flight
  const uint8_t *cr = P.cand ? P.cand + (int64_t)b * P.cand_width : nullptr;
  uint8_t keep[kFusedTiles];
#pragma unroll
  for (int i = 0; i < kFusedTiles; ++i) {
    const int j = i * TILE + tid;
    keep[i] = (warp < 4 && i < ntiles && j < limit) ? (cr ? cr[j / P.cand_block] : (uint8_t)1) : (uint8_t)0;
  }
  if (warp == 0) tc::tmem_alloc(tmem_slot, ncols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 2 && lane == 0 && ntiles > 0) {
    bool issued = false;
    // one MMA chain per tile as it lands
    bool ok = tc::mbar_wait(qbar, 0, abort_flag);
    const uint32_t id = tc::idesc_bf16_f32(TILE, N);
    for (int i = 0; i < ntiles && ok; ++i) {
      if (!(ok = tc::mbar_wait(&full[i], 0, abort_flag))) break;
      tc::tc_fence_after();
      issued = true;
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
        const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sk + (2 * i + kb) * k_blk), 16, 1024);
        const uint64_t bd = tc::sdesc_sw128(tc::smem_u32(sq + kb * q_blk), 16, 1024);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          tc::mma_bf16(tmem + (uint32_t)(i * N), ad + 2ull * k4, bd + 2ull * k4, id, (kb | k4) ? 1u : 0u);
      }
      tc::mma_commit(&done[i]);
    }
    if (!ok) {
      // copies that may still land: wait for them (bounded) before the CTA can exit
      const uint64_t t0w = tc::global_ns();
      while (!tc::mbar_try_wait(qbar, 0) && tc::global_ns() - t0w < tc::kWaitLimitNs) {
      }
      for (int i = 0; i < ntiles; ++i)
        while (!tc::mbar_try_wait(&full[i], 0) && tc::global_ns() - t0w < tc::kWaitLimitNs) {
        }
    }
    if (issued) {  // nothing may still write TMEM when the CTA frees it
      tc::mma_commit(drain);
      const uint64_t t0 = tc::global_ns();
      while (!tc::mbar_try_wait(drain, 0) && tc::global_ns() - t0 < tc::kWaitLimitNs) {
      }
    }
  }
  // scores of the valid keys as 64-bit values at their positions, 0 for an invalid one (warps 0-3:
  // TMEM lane = key within a tile), tile by tile as each chain completes
  bool got = true;
  if (warp < 4) {
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    for (int i = 0; i < ntiles; ++i) {
      got = got && tc::mbar_wait(&done[i], 0, abort_flag);
      tc::tc_fence_after();
      const int j = i * TILE + tid;
      float acc = 0.f;
      if (got)
        for (int h0 = 0; h0 < N; h0 += 16) {
          uint32_t v[16];
          tc::tmem_ld16_wait(lane_base + (uint32_t)(i * N + h0), v);
#pragma unroll
          for (int k = 0; k < 16; ++k) acc = fmaf(w_s[h0 + k], fmaxf(__uint_as_float(v[k]), 0.f), acc);
        }
      const bool ok = got && keep[i] != 0;
      vals[j] = ok ? topk_value(acc, j) : 0ull;
      const unsigned bal = __ballot_sync(0xffffffffu, ok);
      if (lane == 0 && bal) atomicAdd(&sh.count, (unsigned)__popc(bal));
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) sh.count = 0;  // a wait gave up: no score is trusted, nothing selected
  __syncthreads();
  auto at = [&](int i, bool &ok) -> unsigned long long {
    const unsigned long long v = vals[i];
    ok = v != 0ull;
    return v;
  };
  const unsigned nvalid = sh.count;
  // (every thread past the dependency wait before the selection is written: the kernels before may
  // read the previous selection)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  topk_select(sh, nvalid, nvalid ? ntiles * TILE : 0, at, P.K, P.offset, P.out + (int64_t)b * P.K);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, ncols);
  }
  if (tid == 0 && *abort_flag && P.status) atomicOr(P.status, kStatusTimeout);
}

}  // namespace idx

bool index_scores_tc_supported(const bf16 *qI, const bf16 *KI, int Hi, int dI) {
  return dI == idx::DI && Hi % 16 == 0 && Hi <= idx::kMaxN && ((uintptr_t)qI & 15) == 0 && ((uintptr_t)KI & 15) == 0;
}

// One query per sequence with a candidate mask: CTA group of P per query over its kept 64-key units.
static cudaError_t launch_index_scores_gather_tc(const bf16 *qI, const float *wI, const bf16 *KI, int B, int start_pos,
                                                 int Hi, int Lstride, int compress_len, int ratio, const uint8_t *cand,
                                                 int cand_width, int cand_block, float *S, int *status,
                                                 cudaStream_t s) {
  using namespace idx;
  GatherParams p;
  memset(&p, 0, sizeof(p));
  const int limit = std::min((start_pos + 1) / ratio, compress_len);
  if (limit <= 0 || B <= 0) return cudaSuccess;
  const int per_block = cand_block / 64;
  const int nblk = std::min((limit + cand_block - 1) / cand_block, cand_width);
  p.max_units = nblk * per_block;
  if (p.max_units <= 0) return cudaSuccess;
  if (!tma_map_2d_bf16(&p.tm_k, KI, DI, (uint64_t)B * Lstride, DI, 64, 64)) return cudaErrorInvalidValue;
  if (!tma_map_2d_bf16(&p.tm_q, qI, DI, (uint64_t)B * Hi, DI, 64, (uint32_t)Hi)) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int max_pairs = (p.max_units + 1) / 2;
  // CTAs per query: as many as fill the SMs in one wave (two CTAs fit on an SM), rounded down so
  // that no CTA waits for a second wave
  p.P = std::max(1, std::min(max_pairs, 2 * sms / B));
  p.wI = wI;
  p.Hi = Hi;
  p.Lstride = Lstride;
  p.compress_len = compress_len;
  p.ratio = ratio;
  p.start_pos = start_pos;
  p.cand = cand;
  p.cand_width = cand_width;
  p.cand_block = cand_block;
  p.S = S;
  p.status = status;
  const size_t smem = 1024 + (size_t)kGatherBufs * TILE * 128 * 2 + 2 * (size_t)Hi * 128 + kMaxN * 4 +
                      4 * (size_t)((p.max_units + 1) & ~1) + (2 * kGatherBufs + 1) * 8 + 16;
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  static SmemAttr attr;
  e = attr.ensure((const void *)k_index_scores_gather_tc, (int)smem);
  if (e != cudaSuccess) return e;
  k_index_scores_gather_tc<<<dim3(p.P, B), kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

// Many query groups: persistent CTAs (one an SM), each running whole groups' key tiles.
static cudaError_t launch_index_scores_rows_tc(const bf16 *qI, const float *wI, const bf16 *KI, int B, int T,
                                               int start_pos, int Hi, int QG, int Lstride, int compress_len, int ratio,
                                               const uint8_t *cand, int cand_width, int cand_block, float *S,
                                               int *status, int grid, int skip_k, int skip_len, cudaStream_t s) {
  using namespace idx;
  RowsParams p;
  memset(&p, 0, sizeof(p));
  p.QG = QG;
  if (!tma_map_2d_bf16(&p.tm_k, KI, DI, (uint64_t)B * Lstride, DI, 64, TILE)) return cudaErrorInvalidValue;
  if (!tma_map_2d_bf16(&p.tm_q, qI, DI, (uint64_t)B * T * Hi, DI, 64, (uint32_t)(QG * Hi)))
    return cudaErrorInvalidValue;
  p.wI = wI;
  p.T = T;
  p.Hi = Hi;
  p.Lstride = Lstride;
  p.compress_len = compress_len;
  p.ratio = ratio;
  p.start_pos = start_pos;
  p.gps = (T + QG - 1) / QG;
  p.ngroups = B * p.gps;
  p.nwork = p.ngroups;
  if (skip_k > 0 && !cand) {
    // the leading groups whose every query has at most skip_k valid positions (by the selection's own
    // limit, skip_len being its compress_len) are not run: those selections take every position
    int gq_min = 0;
    while (gq_min < p.gps) {
      const int t_last = std::min(T, (gq_min + 1) * QG) - 1;
      if (std::min((start_pos + t_last + 1) / ratio, skip_len) > skip_k) break;
      ++gq_min;
    }
    p.nwork = B * (p.gps - gq_min);
    if (p.nwork == 0) return cudaSuccess;
  }
  p.cand = cand;
  p.cand_width = cand_width;
  p.cand_block = cand_block;
  p.S = S;
  p.status = status;
  const size_t smem = 1024 + (size_t)kRowsKSlots * 2 * TILE * 128 + 2 * 2 * (size_t)QG * Hi * 128 + 18 * 8 + kMaxN * 4 + 16 * 4;
  static SmemAttr attr;
  {
    cudaError_t e = attr.ensure((const void *)k_index_scores_rows_tc,
                                (int)(1024 + kRowsKSlots * 2 * TILE * 128 + 4 * kMaxN * 128 + 18 * 8 + kMaxN * 4 + 16 * 4));
    if (e != cudaSuccess) return e;
  }
  k_index_scores_rows_tc<<<std::min(grid, p.nwork), kRowsThreads, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_index_scores_tc(const bf16 *qI, const float *wI, const bf16 *KI, int B, int T, int start_pos,
                                   int Hi, int Lstride, int compress_len, int ratio, const uint8_t *cand,
                                   int cand_width, int cand_block, float *S, int *status, cudaStream_t s, int skip_k) {
  using namespace idx;
  Params p;
  memset(&p, 0, sizeof(p));
  p.QG = std::max(1, std::min(T, kMaxN / Hi));
  if (!tma_map_2d_bf16(&p.tm_k, KI, DI, (uint64_t)B * Lstride, DI, 64, TILE)) return cudaErrorInvalidValue;
  if (!tma_map_2d_bf16(&p.tm_q, qI, DI, (uint64_t)B * T * Hi, DI, 64, (uint32_t)(p.QG * Hi)))
    return cudaErrorInvalidValue;
  p.wI = wI;
  p.T = T;
  p.Hi = Hi;
  p.Lstride = Lstride;
  p.compress_len = std::min(compress_len, Lstride);
  p.ratio = ratio;
  p.start_pos = start_pos;
  p.cand = cand;
  p.cand_width = cand_width;
  p.cand_block = cand_block;
  p.S = S;
  p.status = status;
  const size_t smem = 1024 + 2 * (size_t)TILE * 128 + 2 * (size_t)p.QG * Hi * 128 + kMaxN * 4 + 64;
  static SmemAttr attr;
  {
    cudaError_t e = attr.ensure((const void *)k_index_scores_tc,
                                (int)(1024 + 2 * TILE * 128 + 2 * kMaxN * 128 + kMaxN * 4 + 64));
    if (e != cudaSuccess) return e;
  }
  const int tiles = (p.compress_len + TILE - 1) / TILE;
  if (tiles <= 0) return cudaSuccess;
  // gathering pays once the candidate keys of a query span more than a few tiles: its key copies wait
  // for the mask scan, while the dense kernel's start at once
  if (cand && T == 1 && cand_block % 64 == 0 && Hi * kGatherBufs <= 512 &&
      (int64_t)std::min((std::min((start_pos + 1) / ratio, compress_len) + cand_block - 1) / cand_block, cand_width) *
              cand_block > 1024)
    return launch_index_scores_gather_tc(qI, wI, KI, B, start_pos, Hi, Lstride, p.compress_len, ratio, cand,
                                         cand_width, cand_block, S, status, s);
  // more query groups than SMs: persistent CTAs keep each group's Q^I resident over its key tiles
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      T > 1 && (int64_t)B * ((T + p.QG - 1) / p.QG) >= nsm && ((uintptr_t)wI & 15) == 0)
    return launch_index_scores_rows_tc(qI, wI, KI, B, T, start_pos, Hi, p.QG, Lstride, p.compress_len, ratio, cand,
                                       cand_width, cand_block, S, status, nsm, skip_k, compress_len, s);
  dim3 grid(tiles, (T + p.QG - 1) / p.QG, B);
  k_index_scores_tc<<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

// CTAs per query of the cluster-fused gathered scores + top-k, or 0 when the launch does not take it:
// a decode query with a candidate mask in 64-key units whose span exceeds 1024 keys (where the
// gathered kernel pays), P <= 8 CTAs (a portable cluster) that each hold at most kGtMaxKeys keys even
// if the mask kept every block, and otherwise as many as fill two CTAs an SM in one wave.
static int gather_topk_ctas(const bf16 *qI, const bf16 *KI, int B, int T, int start_pos, int Hi, int dI,
                            int compress_len, int ratio, const uint8_t *cand, int cand_width, int cand_block, int K,
                            int num_sms) {
  using namespace idx;
  if (!cand || T != 1 || ratio <= 0 || cand_block % 64 || K > kTopkMaxK || B <= 0) return 0;
  if (!index_scores_tc_supported(qI, KI, Hi, dI) || 2 * Hi > 512) return 0;
  const int limit = std::min((start_pos + 1) / ratio, compress_len);
  const int nblk = std::min((limit + cand_block - 1) / cand_block, cand_width);
  if ((int64_t)nblk * cand_block <= 1024) return 0;
  const int max_pairs = (nblk * (cand_block / 64) + 1) / 2;
  const int need = (max_pairs + kGtMaxKeys / TILE - 1) / (kGtMaxKeys / TILE);
  if (need > 8) return 0;
  return std::max(need, std::min(8, std::min(max_pairs, std::max(1, 2 * num_sms / B))));
}

bool index_gather_topk_supported(const bf16 *qI, const bf16 *KI, int B, int T, int start_pos, int Hi, int dI,
                                 int compress_len, int ratio, const uint8_t *cand, int cand_width, int cand_block,
                                 int K, int num_sms) {
  return gather_topk_ctas(qI, KI, B, T, start_pos, Hi, dI, compress_len, ratio, cand, cand_width, cand_block, K,
                          num_sms) > 0;
}

cudaError_t launch_index_gather_topk(const bf16 *qI, const float *wI, const bf16 *KI, int B, int start_pos, int Hi,
                                     int Lstride, int compress_len, int ratio, const uint8_t *cand, int cand_width,
                                     int cand_block, int K, int offset, int32_t *out, int *status, int num_sms,
                                     cudaStream_t s) {
  using namespace idx;
  const int Pc = gather_topk_ctas(qI, KI, B, 1, start_pos, Hi, DI, compress_len, ratio, cand, cand_width, cand_block, K,
                                  num_sms);
  if (Pc <= 0) return cudaErrorInvalidValue;
  GatherTopkParams p;
  memset(&p, 0, sizeof(p));
  const int limit = std::min((start_pos + 1) / ratio, compress_len);
  const int nblk = std::min((limit + cand_block - 1) / cand_block, cand_width);
  p.max_units = nblk * (cand_block / 64);
  if (!tma_map_2d_bf16(&p.tm_k, KI, DI, (uint64_t)B * Lstride, DI, 64, 64)) return cudaErrorInvalidValue;
  if (!tma_map_2d_bf16(&p.tm_q, qI, DI, (uint64_t)B * Hi, DI, 64, (uint32_t)Hi)) return cudaErrorInvalidValue;
  p.wI = wI;
  p.Hi = Hi;
  p.Lstride = Lstride;
  p.compress_len = std::min(compress_len, Lstride);
  p.ratio = ratio;
  p.start_pos = start_pos;
  p.P = Pc;
  p.cand = cand;
  p.cand_width = cand_width;
  p.cand_block = cand_block;
  p.K = K;
  p.offset = offset;
  p.out = out;
  p.status = status;
  // keys a CTA holds (its share of the unit pairs if the mask kept every block), then as many key
  // slots as the shared memory left takes
  const int max_pairs = (p.max_units + 1) / 2;
  p.cap_keys = ((max_pairs + Pc - 1) / Pc) * TILE;
  const size_t fixed = 1024 + 2 * (size_t)Hi * 128 + kMaxN * 4 + (size_t)p.cap_keys * 4 + (size_t)p.cap_keys / 8 +
                       524 * 4 + 4 * (size_t)((p.max_units + 1) & ~1) + (2 * kGtMaxBufs + 6) * 8 + 16;
  // two CTAs an SM when the grid needs them, else one with a deeper ring
  const size_t budget = (size_t)B * Pc > (size_t)num_sms ? 112 * 1024 : 225 * 1024;
  p.nbufs = fixed < budget ? (int)std::min<size_t>(kGtMaxBufs, (budget - fixed) / kGtSlot) : 0;
  if (p.nbufs < 2) return cudaErrorInvalidValue;
  const size_t smem = fixed + (size_t)p.nbufs * kGtSlot;
  static SmemAttr attr;
  cudaError_t e = attr.ensure((const void *)k_index_gather_topk_tc, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(Pc, B);
  cfg.blockDim = dim3(kGtThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = Pc;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  // a programmatic dependent of the projection before it (see the kernel)
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, k_index_gather_topk_tc, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

bool index_fused_supported(const bf16 *qI, const bf16 *KI, int T, int start_pos, int Hi, int dI, int compress_len,
                           int ratio, int K) {
  if (T != 1 || ratio <= 0 || K > kTopkMaxK || !index_scores_tc_supported(qI, KI, Hi, dI)) return false;
  if (Hi * idx::kFusedTiles > 512) return false;
  return std::min((start_pos + 1) / ratio, compress_len) <= idx::kFusedTiles * idx::TILE;
}

cudaError_t launch_index_topk_fused(const bf16 *qI, const float *wI, const bf16 *KI, int B, int start_pos, int Hi,
                                    int Lstride, int compress_len, int ratio, const uint8_t *cand, int cand_width,
                                    int cand_block, int K, int offset, int32_t *out, int *status, cudaStream_t s) {
  using namespace idx;
  if (B <= 0) return cudaSuccess;
  FusedParams p;
  memset(&p, 0, sizeof(p));
  if (!tma_map_2d_bf16(&p.tm_k, KI, DI, (uint64_t)B * Lstride, DI, 64, TILE)) return cudaErrorInvalidValue;
  if (!tma_map_2d_bf16(&p.tm_q, qI, DI, (uint64_t)B * Hi, DI, 64, (uint32_t)Hi)) return cudaErrorInvalidValue;
  p.wI = wI;
  p.Hi = Hi;
  p.Lstride = Lstride;
  p.compress_len = std::min(compress_len, Lstride);
  p.ratio = ratio;
  p.start_pos = start_pos;
  p.cand = cand;
  p.cand_width = cand_width;
  p.cand_block = cand_block;
  p.K = K;
  p.offset = offset;
  p.out = out;
  p.status = status;
  const size_t smem = 1024 + (size_t)kFusedTiles * 2 * TILE * 128 + 2 * (size_t)Hi * 128 + kMaxN * 4 +
                      (size_t)kFusedTiles * TILE * 8 + (2 * kFusedTiles + 2) * 8 + 16;
  static SmemAttr attr;
  {
    cudaError_t e = attr.ensure((const void *)k_index_topk_fused_tc,
                                (int)(1024 + kFusedTiles * 2 * TILE * 128 + 2 * kMaxN * 128 + kMaxN * 4 +
                                      kFusedTiles * TILE * 8 + (2 * kFusedTiles + 2) * 8 + 16));
    if (e != cudaSuccess) return e;
  }
  // a programmatic dependent launch: the CTAs start (barriers, TMEM, the key tiles' copies) while the
  // projection before them on the stream finishes, and wait for it before they read Q^I
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(B);
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_index_topk_fused_tc, p);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace csa
