// k_index_tc.cu -- the indexer's scores on the 5th-generation tensor cores ("DeepSeek V4.1 -
// Compressed sparse attention", "Indexer, re-scored": S^I[t][j] = sum_h w^I[t][h] ReLU(Q^I[t][h] . K^I[j])).
//
// The compressed keys of a sequence are contiguous rows, so a CTA takes a 128-key tile of one
// sequence and a group of up to QG of its queries, loads both by TMA (128-byte swizzled, two
// 64-element K-blocks of dI = 128) and computes every query head's dot products in one MMA chain:
//   D[j][(t, h)] = sum_d K^I[j][d] Q^I[t][h][d]      (M = 128 keys, N = QG * Hi, K = 128; TMEM)
// The four warps then read their 32 keys' rows of D and form sum_h w^I[t][h] ReLU(D) in f32 for
// each query, writing the valid positions only (j below the causal limit floor((p+1)/ratio) and the
// published length, and inside an allowed candidate block).  Every mbarrier wait is time-bounded.
#include "csa_internal.cuh"
#include "tc_ptx.cuh"

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

}  // namespace idx

bool index_scores_tc_supported(const bf16 *qI, const bf16 *KI, int Hi, int dI) {
  return dI == idx::DI && Hi % 16 == 0 && Hi <= idx::kMaxN && ((uintptr_t)qI & 15) == 0 && ((uintptr_t)KI & 15) == 0;
}

cudaError_t launch_index_scores_tc(const bf16 *qI, const float *wI, const bf16 *KI, int B, int T, int start_pos,
                                   int Hi, int Lstride, int compress_len, int ratio, const uint8_t *cand,
                                   int cand_width, int cand_block, float *S, int *status, cudaStream_t s) {
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
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_index_scores_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(1024 + 2 * TILE * 128 + 2 * kMaxN * 128 + kMaxN * 4 + 64));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int tiles = (p.compress_len + TILE - 1) / TILE;
  if (tiles <= 0) return cudaSuccess;
  dim3 grid(tiles, (T + p.QG - 1) / p.QG, B);
  k_index_scores_tc<<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace csa
