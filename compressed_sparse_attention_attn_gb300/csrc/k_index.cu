// k_index.cu -- the indexer's scores and the index top-k ("DeepSeek V4.1 - Compressed sparse
// attention", "Indexer, re-scored": S^I[t][j] = sum_h w^I[t][h] ReLU(Q^I[t][h] . K^I[j]),
// I_t = top_K over valid j; "metrale_model_arch::attn_v41": selection offset past the window rows,
// -1 = absent).
#include "csa_internal.cuh"
#include "topk_core.cuh"

namespace csa {

// Valid compressed position j for query position p: causal limit floor((p+1)/ratio), the published
// length, and the candidate block mask when given.
__device__ __forceinline__ bool comp_valid(int j, int limit, const uint8_t *cand_row, int cand_block) {
  return j < limit && (cand_row == nullptr || cand_row[j / cand_block] != 0);
}

// ---------------------------------------------------------------------------------------------
// Scores: one CTA per (query, 128 positions); one thread per position.  Q^I of the query sits in
// shared memory as f32; each thread keeps its key row's dI values in registers (dI == 128).
// ---------------------------------------------------------------------------------------------
template <int DI>
__global__ void __launch_bounds__(128) k_index_scores(const bf16 *__restrict__ qI, const float *__restrict__ wI,
                                                      const bf16 *__restrict__ KI, int T, int start_pos, int Hi,
                                                      int Lstride, int compress_len, int ratio,
                                                      const uint8_t *__restrict__ cand, int cand_width,
                                                      int cand_block, float *__restrict__ S) {
  extern __shared__ float qs[];  // [Hi][DI] then w [Hi]
  const int64_t row = blockIdx.y;
  const int b = (int)(row / T), t = (int)(row % T);
  const int p = start_pos + t;
  const int limit = min((p + 1) / ratio, compress_len);
  const int j0 = blockIdx.x * 128;
  if (j0 >= limit) return;
  for (int e = threadIdx.x; e < Hi * DI; e += blockDim.x) qs[e] = __bfloat162float(qI[row * Hi * DI + e]);
  for (int e = threadIdx.x; e < Hi; e += blockDim.x) qs[Hi * DI + e] = wI[row * Hi + e];
  __syncthreads();
  const int j = j0 + threadIdx.x;
  const uint8_t *cr = cand ? cand + row * cand_width : nullptr;
  if (!comp_valid(j, limit, cr, cand_block)) return;
  float k[DI];
  const uint4 *kp = reinterpret_cast<const uint4 *>(KI + ((int64_t)b * Lstride + j) * DI);
#pragma unroll
  for (int v = 0; v < DI / 8; ++v) {
    uint4 u = kp[v];
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      k[v * 8 + 2 * e] = __low2float(h[e]);
      k[v * 8 + 2 * e + 1] = __high2float(h[e]);
    }
  }
  float acc = 0.f;
  for (int h = 0; h < Hi; ++h) {
    const float *q = qs + h * DI;
    float d = 0.f;
#pragma unroll
    for (int e = 0; e < DI; ++e) d = fmaf(q[e], k[e], d);
    acc = fmaf(qs[Hi * DI + h], fmaxf(d, 0.f), acc);
  }
  S[row * Lstride + j] = acc;
}

bool index_scores_tc_supported(const bf16 *qI, const bf16 *KI, int Hi, int dI);
cudaError_t launch_index_scores_tc(const bf16 *qI, const float *wI, const bf16 *KI, int B, int T, int start_pos,
                                   int Hi, int Lstride, int compress_len, int ratio, const uint8_t *cand,
                                   int cand_width, int cand_block, float *S, int *status, cudaStream_t s, int skip_k);

cudaError_t launch_index_scores(const bf16 *qI, const float *wI, const bf16 *KI, int B, int T, int start_pos, int Hi,
                                int dI, int Lstride, int compress_len, int ratio, const uint8_t *cand, int cand_width,
                                int cand_block, float *S, cudaStream_t s, int *status, int skip_k) {
  if (B * T <= 0 || Lstride <= 0) return cudaSuccess;
  if (index_scores_tc_supported(qI, KI, Hi, dI))
    return launch_index_scores_tc(qI, wI, KI, B, T, start_pos, Hi, Lstride, compress_len, ratio, cand, cand_width,
                                  cand_block, S, status, s, skip_k);
  const size_t smem = sizeof(float) * (size_t)Hi * (dI + 1);
  dim3 grid((Lstride + 127) / 128, B * T);
  switch (dI) {
    case 128: {
      static SmemAttr attr;
      const cudaError_t e = attr.ensure((const void *)k_index_scores<128>, (int)smem);
      if (e != cudaSuccess) return e;
      k_index_scores<128><<<grid, 128, smem, s>>>(qI, wI, KI, T, start_pos, Hi, Lstride, compress_len, ratio, cand,
                                                  cand_width, cand_block, S);
      break;
    }
    case 64:
      k_index_scores<64><<<grid, 128, smem, s>>>(qI, wI, KI, T, start_pos, Hi, Lstride, compress_len, ratio, cand,
                                                 cand_width, cand_block, S);
      break;
    case 32:
      k_index_scores<32><<<grid, 128, smem, s>>>(qI, wI, KI, T, start_pos, Hi, Lstride, compress_len, ratio, cand,
                                                 cand_width, cand_block, S);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
// Top-k: one CTA per query (512 threads, four CTAs an SM, for rows of at most 2048 positions; 1024
// otherwise).  A first pass gathers the valid positions' 64-bit values into shared memory in
// ascending position (with a candidate mask: the kept blocks listed first, only their positions
// visited, each round compacted in order); the selection and its position-ordered output are
// topk_core.cuh's.  (A query with more valid positions than shared memory holds runs the same
// passes over its scores in global memory.)
// ---------------------------------------------------------------------------------------------
constexpr int kTopkCap = 12288;  // valid positions of one query held in shared memory (96 KiB at most)
// dynamic shared memory: `cap` values and the kept-block list
constexpr size_t topk_smem(int cap, int nt) { return (size_t)cap * 8 + (size_t)2 * nt * 4; }

// NT threads: 1024 for long rows, 512 (four CTAs an SM) for rows of at most 2048 positions
template <int NT>
__global__ void __launch_bounds__(NT, 2048 / NT) k_index_topk(const float *__restrict__ S, int T, int start_pos,
                                                             int Lstride, int compress_len, int ratio,
                                                             const uint8_t *__restrict__ cand, int cand_width,
                                                             int cand_block, int K, int offset, int32_t *__restrict__ out,
                                                             int cap_vals) {
  // the attention after this kernel may start its set-up now (it waits for this grid before it reads
  // the selection)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ unsigned long long tk_smem[];
  unsigned long long *vals = tk_smem;                      // [cap_vals] valid values, ascending position
  int *klist = reinterpret_cast<int *>(vals + cap_vals);   // [2 NT] kept blocks
  __shared__ TopkShared sh;
  const int64_t row = blockIdx.x;
  const int t = (int)(row % T);
  const int p = start_pos + t;
  const int limit = min((p + 1) / ratio, compress_len);
  const uint8_t *cr = cand ? cand + row * cand_width : nullptr;
  const float *Sr = S + row * Lstride;
  const int tid = threadIdx.x;
  // no mask and at most K valid positions: all are taken, and in ascending position they are
  // 0 .. limit-1, so the scores need not be read (the early queries of a prefill chunk)
  if (!cr && limit <= K) {
    for (int k = tid; k < K; k += NT) out[row * K + k] = k < limit ? k + offset : -1;
    return;
  }

  if (tid == 0) topk_shared_init(sh, K);
  __syncthreads();
  const int nblk = cr ? min((limit + cand_block - 1) / cand_block, cand_width) : 0;
  unsigned nvalid = 0;
  if (!cr) {
    // every position below the limit is valid: value j at slot j
    for (int j = tid; j < min(limit, cap_vals); j += NT) vals[j] = topk_value(Sr[j], j);
    nvalid = (unsigned)max(limit, 0);
  } else if (nblk <= 2 * NT) {
    // the kept blocks in order, then only their positions
    unsigned nk = 0;
    for (int b0 = 0; b0 < nblk; b0 += NT) {
      const int blk = b0 + tid;
      const bool keep = blk < nblk && cr[blk] != 0;
      const unsigned slot = ordered_slot(sh, keep, nk);
      if (keep) klist[slot] = blk;
    }
    __syncthreads();
    const int npos = (int)nk * cand_block;
    for (int i0 = 0; i0 < npos; i0 += NT) {
      const int i = i0 + tid;
      int j = 0;
      bool v = false;
      if (i < npos) {
        j = klist[i / cand_block] * cand_block + i % cand_block;
        v = j < limit;
      }
      const unsigned slot = ordered_slot(sh, v, nvalid);
      if (v && slot < (unsigned)cap_vals) vals[slot] = topk_value(Sr[j], j);
    }
  } else {
    for (int j0 = 0; j0 < limit; j0 += NT) {
      const int j = j0 + tid;
      const bool v = j < limit && comp_valid(j, limit, cr, cand_block);
      const unsigned slot = ordered_slot(sh, v, nvalid);
      if (v && slot < (unsigned)cap_vals) vals[slot] = topk_value(Sr[j], j);
    }
  }
  __syncthreads();
  if (nvalid <= (unsigned)cap_vals) {
    auto from_smem = [&](int i, bool &ok) -> unsigned long long {
      ok = true;
      return vals[i];
    };
    topk_select(sh, nvalid, (int)nvalid, from_smem, K, offset, out + row * K);
  } else {
    auto from_global = [&](int i, bool &ok) -> unsigned long long {  // position i, read from S
      ok = comp_valid(i, limit, cr, cand_block);
      return ok ? topk_value(Sr[i], i) : 0ull;
    };
    topk_select(sh, nvalid, limit, from_global, K, offset, out + row * K);
  }
}

// ---------------------------------------------------------------------------------------------
// Candidate blocks (the candidate source's mask, "metrale_model_arch::attn_v41": a block-level
// candidate mask published for later index sources; config.json candidate_block_size and
// candidate_topk_blocks): per query, block c scores the largest valid score S[t][j] inside it
// (blocks without a valid position are not candidates), the top cand_topk by that score (ties to the
// lower block, the index top-k's order keys) are marked 1, the others 0.  One CTA per query; the
// selection is topk_core.cuh's over the block values, written to shared memory, then scattered.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(512) k_cand_blocks(const float *__restrict__ S, int T, int start_pos, int Lstride,
                                                     int compress_len, int ratio, int cand_block, int K,
                                                     uint8_t *__restrict__ mask, int cand_width) {
  extern __shared__ unsigned long long cb_smem[];
  unsigned long long *vals = cb_smem;                           // [cand_width] block values (0: none)
  int32_t *sel = reinterpret_cast<int32_t *>(vals + cand_width);  // [K] chosen blocks
  __shared__ TopkShared sh;
  const int64_t row = blockIdx.x;
  const int p = start_pos + (int)(row % T);
  const int limit = min((p + 1) / ratio, compress_len);
  const float *Sr = S + row * Lstride;
  const int nb = min((limit + cand_block - 1) / cand_block, cand_width);
  if (threadIdx.x == 0) topk_shared_init(sh, K);
  __syncthreads();
  unsigned mine = 0;
  for (int c = threadIdx.x; c < cand_width; c += blockDim.x) {
    unsigned long long v = 0ull;
    if (c < nb) {
      const int j1 = min((c + 1) * cand_block, limit);
      float m = Sr[c * cand_block];
      for (int j = c * cand_block + 1; j < j1; ++j) m = fmaxf(m, Sr[j]);
      v = topk_value(m, c);
      ++mine;
    }
    vals[c] = v;
  }
  if (mine) atomicAdd(&sh.count, mine);
  __syncthreads();
  const unsigned nvalid = sh.count;
  auto at = [&](int i, bool &ok) -> unsigned long long {
    ok = vals[i] != 0ull;
    return vals[i];
  };
  topk_select(sh, nvalid, nb, at, K, 0, sel);
  __syncthreads();
  uint8_t *mr = mask + row * cand_width;
  for (int c = threadIdx.x; c < cand_width; c += blockDim.x) mr[c] = 0;
  __syncthreads();
  const int nsel = (int)min(nvalid, (unsigned)K);
  for (int k = threadIdx.x; k < nsel; k += blockDim.x) mr[sel[k]] = 1;
}

cudaError_t launch_cand_blocks(const float *S, int B, int T, int start_pos, int Lstride, int compress_len, int ratio,
                               int cand_block, int K, uint8_t *mask, int cand_width, cudaStream_t s) {
  if (B * T <= 0) return cudaSuccess;
  const size_t smem = (size_t)cand_width * 8 + (size_t)K * 4;
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  static SmemAttr attr;
  cudaError_t e = attr.ensure((const void *)k_cand_blocks, (int)smem);
  if (e != cudaSuccess) return e;
  k_cand_blocks<<<B * T, 512, smem, s>>>(S, T, start_pos, Lstride, compress_len, ratio, cand_block, K, mask,
                                         cand_width);
  return cudaGetLastError();
}

cudaError_t launch_index_topk(const float *S, int B, int T, int start_pos, int Lstride, int compress_len, int ratio,
                              const uint8_t *cand, int cand_width, int cand_block, int K, int offset, int32_t *out,
                              cudaStream_t s) {
  if (B * T <= 0) return cudaSuccess;
  if (K > kTopkMaxK) return cudaErrorInvalidValue;
  static SmemAttr attr512, attr1024;
  {
    cudaError_t e = attr1024.ensure((const void *)k_index_topk<1024>, (int)topk_smem(kTopkCap, 1024));
    if (e == cudaSuccess) e = attr512.ensure((const void *)k_index_topk<512>, (int)topk_smem(kTopkCap, 512));
    if (e != cudaSuccess) return e;
  }
  // room for the largest causal limit of the launch (the last query's), so that short ones keep
  // several CTAs per SM
  const int max_limit = std::max(0, std::min((start_pos + T) / std::max(ratio, 1), compress_len));
  const int cap = std::max(32, std::min(kTopkCap, max_limit));
  // short rows (every query's limit within 2048): 512 threads, four CTAs an SM, cheaper barriers
  if (max_limit <= 2048)
    k_index_topk<512><<<B * T, 512, topk_smem(cap, 512), s>>>(S, T, start_pos, Lstride, compress_len, ratio, cand,
                                                              cand_width, cand_block, K, offset, out, cap);
  else
    k_index_topk<1024><<<B * T, 1024, topk_smem(cap, 1024), s>>>(S, T, start_pos, Lstride, compress_len, ratio, cand,
                                                                 cand_width, cand_block, K, offset, out, cap);
  return cudaGetLastError();
}

}  // namespace csa
