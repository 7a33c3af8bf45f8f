// topk_core.cuh -- the index top-k's selection and ordering, shared by the top-k kernel and the
// fused indexer + top-k ("DeepSeek V4.1 - Compressed sparse attention", "Indexer, re-scored": I_t =
// the top K valid positions by score, ties to the lower position).
//
// Scores map to order-preserving 32-bit keys (-0 folded onto +0, NaN below every number) and each
// valid position j to the 64-bit value (key << 32) | ~j, so that the values are distinct and larger
// means selected first.  Given the count of valid values (compacted into shared memory when they
// fit), topk_finish takes all of them when they are at most K; otherwise a radix select on the 64-bit
// values (8 bits per pass from the top) finds the K-th largest and the values at or above it are
// taken.  The histograms count with one shared atomic per value: measured at 4096 values a query,
// that is 2-5x faster a pass than aggregating equal digits across a warp first (__match_any_sync),
// even in the top digit where most values share one or two bins.  The chosen values are then sorted
// descending by a bitonic network whose stages within a warp run on shuffles and whose wider stages
// go through shared memory, and written as j + offset, -1 past the valid ones.  (Four values a
// thread, so that strides 1 and 2 stay in registers, measured 1.6x slower at 512 values: only four
// warps then hold values, and each stage's shuffle latency is exposed.)
#pragma once

#include <cstdint>

namespace csa {

__device__ __forceinline__ uint32_t order_key(float f) {
  if (f != f) return 0u;   // NaN: below every number
  if (f == 0.0f) f = 0.0f;  // -0 == +0
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kTopkMaxK = 2048;

// The block's shared scalars of one selection.
struct TopkShared {
  unsigned hist[256];
  unsigned count, nchosen, remain, done;
  unsigned long long prefix;
  int shift;
};

__device__ __forceinline__ void topk_shared_init(TopkShared &sh, int K) {
  sh.count = 0;
  sh.nchosen = 0;
  sh.prefix = 0ull;
  sh.remain = (unsigned)K;
  sh.done = 0;
  sh.shift = 0;
}

// Append v (where take) to buf[cap] through counter *cnt: one shared atomic per warp.
__device__ __forceinline__ void topk_append(bool take, unsigned long long v, unsigned *cnt, unsigned long long *buf,
                                            unsigned cap) {
  const int lane = threadIdx.x & 31;
  const unsigned bal = __ballot_sync(0xffffffffu, take);
  unsigned base = 0;
  if (lane == 0 && bal) base = atomicAdd(cnt, (unsigned)__popc(bal));
  base = __shfl_sync(0xffffffffu, base, 0);
  const unsigned slot = base + __popc(bal & ((1u << lane) - 1u));
  if (take && slot < cap) buf[slot] = v;
}

// After the first pass: nvalid valid values, compacted in vals[0, nvalid) when in_smem; otherwise
// candidate i < n_iter is value_at(i, ok) (ok false: not valid).  NT threads, all of which call this.
// chosen: [kTopkMaxK], swap: [NT] shared buffers; o: the query's K outputs.
template <int NT, class ValueAt>
__device__ __forceinline__ void topk_finish(TopkShared &sh, unsigned nvalid, bool in_smem, int n_iter,
                                            ValueAt value_at_i, int K, int offset, unsigned long long *vals,
                                            unsigned long long *chosen, unsigned long long *swap, int32_t *o) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  unsigned *hist = sh.hist;
  auto append = [&](bool take, unsigned long long v, unsigned *cnt, unsigned long long *buf, unsigned cap) {
    topk_append(take, v, cnt, buf, cap);
  };
  const bool all = nvalid <= (unsigned)K;
  unsigned long long *sorted = vals;
  if (!all) {
    // radix select of the K-th largest value, 8 bits per pass from the top
    for (int shift = 56; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      const unsigned long long prefix = sh.prefix;
      const unsigned long long hi_mask = shift == 56 ? 0ull : (~0ull << (shift + 8));
      for (int i0 = 0; i0 < n_iter; i0 += blockDim.x) {
        const int i = i0 + tid;
        int bin = 256;  // no bin
        if (i < n_iter) {
          bool ok = true;
          unsigned long long v = 0ull;
          if (in_smem) {
            v = vals[i];
          } else {
            v = value_at_i(i, ok);
          }
          if (ok && (v & hi_mask) == (prefix & hi_mask)) bin = (int)((v >> shift) & 255u);
        }
        if (bin < 256) atomicAdd(&hist[bin], 1u);
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
        const unsigned excl = incl - tot, remain = sh.remain;
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
          sh.prefix = prefix | ((unsigned long long)d << shift);
          sh.remain = remain - above;
          sh.shift = shift;
          if (cd == remain - above) sh.done = 1;  // every value with this prefix is taken
        }
      }
      __syncthreads();
      if (sh.done) break;
    }
    // the selection: values above the prefix at the final digit, and every value equal to it there
    const int fs = sh.shift;  // the final digit's shift
    const unsigned long long thr = sh.prefix >> fs;
    for (int i0 = 0; i0 < n_iter; i0 += blockDim.x) {
      const int i = i0 + tid;
      bool take = false;
      unsigned long long v = 0ull;
      if (i < n_iter) {
        bool ok = true;
        if (in_smem) {
          v = vals[i];
        } else {
          v = value_at_i(i, ok);
        }
        take = ok && (v >> fs) >= thr;
      }
      append(take, v, &sh.nchosen, chosen, (unsigned)kTopkMaxK);
    }
    __syncthreads();
    sorted = chosen;
  }
  const int nsel = all ? (int)nvalid : K;
  int cap = 32;
  while (cap < nsel) cap <<= 1;
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

}  // namespace csa
