// k_index.cu -- the indexer's scores and the index top-k ("DeepSeek V4.1 - Compressed sparse
// attention", "Indexer, re-scored": S^I[t][j] = sum_h w^I[t][h] ReLU(Q^I[t][h] . K^I[j]),
// I_t = top_K over valid j; "metrale_model_arch::attn_v41": selection offset past the window rows,
// -1 = absent).
#include "csa_internal.cuh"

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
                                   int cand_width, int cand_block, float *S, int *status, cudaStream_t s);

cudaError_t launch_index_scores(const bf16 *qI, const float *wI, const bf16 *KI, int B, int T, int start_pos, int Hi,
                                int dI, int Lstride, int compress_len, int ratio, const uint8_t *cand, int cand_width,
                                int cand_block, float *S, cudaStream_t s, int *status) {
  if (B * T <= 0 || Lstride <= 0) return cudaSuccess;
  if (index_scores_tc_supported(qI, KI, Hi, dI))
    return launch_index_scores_tc(qI, wI, KI, B, T, start_pos, Hi, Lstride, compress_len, ratio, cand, cand_width,
                                  cand_block, S, status, s);
  const size_t smem = sizeof(float) * (size_t)Hi * (dI + 1);
  dim3 grid((Lstride + 127) / 128, B * T);
  switch (dI) {
    case 128:
      cudaFuncSetAttribute(k_index_scores<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      k_index_scores<128><<<grid, 128, smem, s>>>(qI, wI, KI, T, start_pos, Hi, Lstride, compress_len, ratio, cand,
                                                  cand_width, cand_block, S);
      break;
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
// Top-k: one CTA per query.  Scores map to order-preserving 32-bit keys (-0 folded onto +0, NaN
// below every number) and each valid position j to the 64-bit value (key << 32) | ~j, so that the
// values are distinct and larger means selected first (higher score, then lower position).  A first
// pass compacts the valid values into shared memory; when they are at most K, all are taken.
// Otherwise a radix select on the 64-bit values (8 bits per pass, warp-aggregated histograms, over
// shared memory) finds the K-th largest, and the values at or above it are taken.  (A query with more
// valid positions than shared memory holds runs the same passes over its scores in global memory.)
// The chosen values are then sorted descending by a bitonic network whose stages within a warp run
// on shuffles and whose wider stages go through shared memory.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_key(float f) {
  if (f != f) return 0u;   // NaN: below every number
  if (f == 0.0f) f = 0.0f;  // -0 == +0
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kTopkMaxK = 2048;
constexpr int kTopkCap = 12288;  // valid positions of one query held in shared memory (96 KiB at most)
// dynamic shared memory for candidate buffers of `cap` values
constexpr size_t topk_smem(int cap, int nt) { return (size_t)(cap + kTopkMaxK + nt) * 8; }

// NT threads: 1024 for long rows, 512 (four CTAs an SM) for rows of at most 2048 positions
template <int NT>
__global__ void __launch_bounds__(NT, 2048 / NT) k_index_topk(const float *__restrict__ S, int T, int start_pos,
                                                             int Lstride, int compress_len, int ratio,
                                                             const uint8_t *__restrict__ cand, int cand_width,
                                                             int cand_block, int K, int offset, int32_t *__restrict__ out,
                                                             int cap_vals) {
  extern __shared__ unsigned long long tk_smem[];
  unsigned long long *vals = tk_smem;                 // [cap_vals] the valid values
  unsigned long long *chosen = vals + cap_vals;       // [kTopkMaxK] the selection
  unsigned long long *swap = chosen + kTopkMaxK;      // [NT] sort buffer
  __shared__ unsigned hist[256];
  __shared__ unsigned s_count, s_nchosen;
  __shared__ unsigned long long s_prefix;
  __shared__ unsigned s_remain, s_done;
  __shared__ int s_shift;
  const int64_t row = blockIdx.x;
  const int t = (int)(row % T);
  const int p = start_pos + t;
  const int limit = min((p + 1) / ratio, compress_len);
  const uint8_t *cr = cand ? cand + row * cand_width : nullptr;
  const float *Sr = S + row * Lstride;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const unsigned below = (1u << lane) - 1u;
  auto value_at = [&](int j) {
    return ((unsigned long long)order_key(Sr[j]) << 32) | (unsigned long long)(~(uint32_t)j);
  };
  // append v (where take) to buf[cap] through counter cnt: one atomic per warp
  auto append = [&](bool take, unsigned long long v, unsigned *cnt, unsigned long long *buf, unsigned cap) {
    const unsigned bal = __ballot_sync(0xffffffffu, take);
    unsigned base = 0;
    if (lane == 0 && bal) base = atomicAdd(cnt, (unsigned)__popc(bal));
    base = __shfl_sync(0xffffffffu, base, 0);
    const unsigned slot = base + __popc(bal & below);
    if (take && slot < cap) buf[slot] = v;
  };

  // pass 1: count the valid positions, compacting their values while they fit
  if (tid == 0) {
    s_count = 0;
    s_nchosen = 0;
    s_prefix = 0ull;
    s_remain = (unsigned)K;
    s_done = 0;
    s_shift = 0;
  }
  __syncthreads();
  for (int j0 = 0; j0 < limit; j0 += blockDim.x) {
    const int j = j0 + tid;
    const bool v = j < limit && comp_valid(j, limit, cr, cand_block);
    append(v, v ? value_at(j) : 0ull, &s_count, vals, (unsigned)cap_vals);
  }
  __syncthreads();
  const unsigned nvalid = s_count;
  const bool all = nvalid <= (unsigned)K;
  const bool in_smem = nvalid <= (unsigned)cap_vals;
  const int n_iter = in_smem ? (int)nvalid : limit;  // candidates: vals[0..nvalid) or positions 0..limit
  unsigned long long *sorted = vals;
  if (!all) {
    // radix select of the K-th largest value, 8 bits per pass from the top
    for (int shift = 56; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      const unsigned long long prefix = s_prefix;
      const unsigned long long hi_mask = shift == 56 ? 0ull : (~0ull << (shift + 8));
      for (int i0 = 0; i0 < n_iter; i0 += blockDim.x) {
        const int i = i0 + tid;
        int bin = 256 + lane;  // no bin: a value of every lane of its own
        if (i < n_iter) {
          bool ok = true;
          unsigned long long v = 0ull;
          if (in_smem) {
            v = vals[i];
          } else {
            ok = comp_valid(i, limit, cr, cand_block);
            if (ok) v = value_at(i);
          }
          if (ok && (v & hi_mask) == (prefix & hi_mask)) bin = (int)((v >> shift) & 255u);
        }
        const unsigned peers = __match_any_sync(0xffffffffu, bin);
        if (bin < 256 && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], (unsigned)__popc(peers));
      }
      __syncthreads();
      if (wid == 0) {
        // the digit holding the remain-th largest value: lane l scans digits 255-8l down to 248-8l
        unsigned c[8], tot = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          c[k] = hist[255 - 8 * lane - k];
          tot += c[k];
        }
        unsigned incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned n = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += n;
        }
        const unsigned excl = incl - tot, remain = s_remain;
        if (excl < remain && remain <= incl) {
          unsigned above = excl;
          int d = 255 - 8 * lane;
          unsigned cd = 0;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            d = 255 - 8 * lane - k;
            cd = c[k];
            if (above + cd >= remain) break;
            above += cd;
          }
          s_prefix = prefix | ((unsigned long long)d << shift);
          s_remain = remain - above;
          s_shift = shift;
          if (cd == remain - above) s_done = 1;  // every value with this prefix is taken
        }
      }
      __syncthreads();
      if (s_done) break;
    }
    // the selection: values above the prefix at the final digit, and every value equal to it there
    const int sh = s_shift;
    const unsigned long long thr = s_prefix >> sh;
    for (int i0 = 0; i0 < n_iter; i0 += blockDim.x) {
      const int i = i0 + tid;
      bool take = false;
      unsigned long long v = 0ull;
      if (i < n_iter) {
        bool ok = true;
        if (in_smem) {
          v = vals[i];
        } else {
          ok = comp_valid(i, limit, cr, cand_block);
          if (ok) v = value_at(i);
        }
        take = ok && (v >> sh) >= thr;
      }
      append(take, v, &s_nchosen, chosen, (unsigned)kTopkMaxK);
    }
    __syncthreads();
    sorted = chosen;
  }
  const int nsel = all ? (int)nvalid : K;
  int cap = 32;
  while (cap < nsel) cap <<= 1;
  int32_t *o = out + row * K;
  auto pos_of = [&](unsigned long long x) { return (int32_t)(~(uint32_t)(x & 0xffffffffull)) + offset; };
  if (cap <= NT) {
    // bitonic sort, descending: thread i holds element i; warps past the padded length only keep
    // the shared stages' barriers
    const bool holds = (tid & ~31) < cap;
    unsigned long long x = 0ull;  // padding sorts last
    if (tid < nsel) x = sorted[tid];
    int nb = 0;
    for (int size = 2; size <= cap; size <<= 1) {
      // stages of stride 32 and up go through shared memory, the rest are shuffles
      for (int stride = size >> 1; stride >= 32; stride >>= 1) {
        unsigned long long *bp = nb ? swap : chosen;  // alternate buffers: one barrier per stage
        if (tid < cap) bp[tid] = x;
        __syncthreads();
        if (tid < cap) {
          const unsigned long long y = bp[tid ^ stride];
          const bool keep_max = ((tid & size) == 0) == ((tid & stride) == 0);
          x = keep_max ? (x > y ? x : y) : (x < y ? x : y);
        }
        nb ^= 1;
      }
      if (holds) {
        for (int stride = min(size >> 1, 16); stride > 0; stride >>= 1) {
          const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, stride);
          const bool keep_max = ((tid & size) == 0) == ((tid & stride) == 0);
          x = keep_max ? (x > y ? x : y) : (x < y ? x : y);
        }
      }
    }
    for (int k = tid; k < K; k += blockDim.x) o[k] = (k == tid && k < nsel) ? pos_of(x) : -1;
  } else {
    unsigned long long *a = sorted;
    for (int i = nsel + tid; i < cap; i += blockDim.x) a[i] = 0ull;
    __syncthreads();
    for (int size = 2; size <= cap; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < cap; i += blockDim.x) {
          const int jx = i ^ stride;
          if (jx > i) {
            const bool desc = (i & size) == 0;
            const unsigned long long u = a[i], w = a[jx];
            if (desc ? (u < w) : (u > w)) {
              a[i] = w;
              a[jx] = u;
            }
          }
        }
        __syncthreads();
      }
    }
    for (int k = tid; k < K; k += blockDim.x) o[k] = k < nsel ? pos_of(a[k]) : -1;
  }
}

cudaError_t launch_index_topk(const float *S, int B, int T, int start_pos, int Lstride, int compress_len, int ratio,
                              const uint8_t *cand, int cand_width, int cand_block, int K, int offset, int32_t *out,
                              cudaStream_t s) {
  if (B * T <= 0) return cudaSuccess;
  if (K > kTopkMaxK) return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_index_topk<1024>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)topk_smem(kTopkCap, 1024));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_index_topk<512>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)topk_smem(kTopkCap, 512));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  // room for the largest causal limit of the launch (the last query's), so that short ones keep
  // two CTAs per SM; the sort buffers need at least as many values as the sort's padded length
  const int max_limit = std::min((start_pos + T) / std::max(ratio, 1), compress_len);
  const int cap = std::min(kTopkCap, std::max(max_limit, kTopkMaxK));
  // short rows (every query's limit within 2048, K within the 512-thread sort): 512 threads, four
  // CTAs an SM, cheaper block barriers
  if (max_limit <= 2048 && K <= 512)
    k_index_topk<512><<<B * T, 512, topk_smem(cap, 512), s>>>(S, T, start_pos, Lstride, compress_len, ratio, cand,
                                                              cand_width, cand_block, K, offset, out, cap);
  else
    k_index_topk<1024><<<B * T, 1024, topk_smem(cap, 1024), s>>>(S, T, start_pos, Lstride, compress_len, ratio, cand,
                                                                 cand_width, cand_block, K, offset, out, cap);
  return cudaGetLastError();
}

}  // namespace csa
