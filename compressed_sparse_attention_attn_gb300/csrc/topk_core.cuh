// topk_core.cuh -- the index top-k's selection, shared by the top-k kernel and the fused indexer +
// top-k ("DeepSeek V4.1 - Compressed sparse attention", "Indexer, re-scored": I_t = the top K valid
// positions by score, ties to the lower position).
//
// Scores map to order-preserving 32-bit keys (-0 folded onto +0, NaN below every number) and each
// valid position j to the 64-bit value (key << 32) | ~j, so that the values are distinct, nonzero,
// and larger means selected first.  The candidates are visited in ascending position.  When at most
// K are valid all of them are taken; otherwise a radix select on the 64-bit values (8 bits per pass
// from the top; the histograms count with one shared atomic per value, which measured 2-5x faster a
// pass than aggregating equal digits across a warp first) finds the K-th largest, and the values at
// or above it are taken.  The selection is written in ascending position (a block-wide ordered
// compaction), as j + offset, then -1 up to K: the pages leave the order of the selected positions
// open (the attention that reads them does not depend on it), and position order needs no sort.
#pragma once

#include <cstdint>

namespace csa {

__device__ __forceinline__ uint32_t order_key(float f) {
  if (f != f) return 0u;   // NaN: below every number
  if (f == 0.0f) f = 0.0f;  // -0 == +0
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The 64-bit value of position j with score s (never 0: ~j has its top bit set for j < 2^31).
__device__ __forceinline__ unsigned long long topk_value(float s, int j) {
  return ((unsigned long long)order_key(s) << 32) | (unsigned long long)(~(uint32_t)j);
}

constexpr int kTopkMaxK = 2048;

// The block's shared scalars of one selection.
struct TopkShared {
  unsigned hist[256];
  unsigned wsum[32];  // per-warp counts of one round of an ordered compaction
  unsigned count, remain, done;
  unsigned long long prefix;
  int shift;
};

__device__ __forceinline__ void topk_shared_init(TopkShared &sh, int K) {
  sh.count = 0;
  sh.prefix = 0ull;
  sh.remain = (unsigned)K;
  sh.done = 0;
  sh.shift = 0;
}

// Block-wide ordered compaction, one round: the threads whose `take` is set get consecutive slots
// base, base + 1, ... in thread order; returns this thread's slot (meaningful where take) and adds
// the round's total to base (the same in every thread).  All blockDim.x (a multiple of 32, <= 1024)
// threads call it; it holds two block barriers.
__device__ __forceinline__ unsigned ordered_slot(TopkShared &sh, bool take, unsigned &base) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, take);
  if (lane == 0) sh.wsum[wid] = (unsigned)__popc(bal);
  __syncthreads();
  unsigned c = lane < nw ? sh.wsum[lane] : 0u, incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  const unsigned before = __shfl_sync(0xffffffffu, incl - c, wid);  // warps ahead of this one
  const unsigned total = __shfl_sync(0xffffffffu, incl, 31);
  const unsigned slot = base + before + (unsigned)__popc(bal & ((1u << lane) - 1u));
  base += total;
  __syncthreads();  // wsum is rewritten by the next round
  return slot;
}

// One radix step, run by warp 0: in the 256-bin histogram `hist` of the values that match the
// current prefix at digit `shift`, find the digit holding the remain-th largest value; update the
// prefix, remain and shift, and set done when every value with the new prefix is taken.
__device__ __forceinline__ void radix_pick(TopkShared &sh, const unsigned *hist, int shift) {
  const int lane = threadIdx.x & 31;
  unsigned c[8], tot = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    c[k] = hist[255 - 8 * lane - k];
    tot += c[k];
  }
  unsigned incl = tot;
#pragma unroll
  for (int o2 = 1; o2 < 32; o2 <<= 1) {
    const unsigned n = __shfl_up_sync(0xffffffffu, incl, o2);
    if (lane >= o2) incl += n;
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
    sh.prefix = sh.prefix | ((unsigned long long)d << shift);
    sh.remain = remain - above;
    sh.shift = shift;
    if (cd == remain - above) sh.done = 1;  // every value with this prefix is taken
  }
}

// The selection of one query.  value_at(i, ok) gives candidate i < n_iter in ascending position
// (ok false: not a valid position); nvalid counts the valid ones.  All blockDim.x threads call this;
// o receives the query's K outputs.
template <class ValueAt>
__device__ __forceinline__ void topk_select(TopkShared &sh, unsigned nvalid, int n_iter, ValueAt value_at, int K,
                                            int offset, int32_t *o) {
  const int tid = threadIdx.x, wid = tid >> 5;
  unsigned *hist = sh.hist;
  const bool all = nvalid <= (unsigned)K;
  int fs = 0;
  unsigned long long thr = 0ull;
  if (!all) {
    // radix select of the K-th largest value, 8 bits per pass from the top
    for (int shift = 56; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      const unsigned long long prefix = sh.prefix;
      const unsigned long long hi_mask = shift == 56 ? 0ull : (~0ull << (shift + 8));
      for (int i0 = 0; i0 < n_iter; i0 += blockDim.x) {
        const int i = i0 + tid;
        if (i < n_iter) {
          bool ok = true;
          const unsigned long long v = value_at(i, ok);
          if (ok && (v & hi_mask) == (prefix & hi_mask)) atomicAdd(&hist[(v >> shift) & 255u], 1u);
        }
      }
      __syncthreads();
      // the digit holding the remain-th largest value: lane l scans digits 255-8l down to 248-8l
      if (wid == 0) radix_pick(sh, hist, shift);
      __syncthreads();
      if (sh.done) break;
    }
    // taken: the values above the prefix at the final digit, and every value equal to it there
    fs = sh.shift;
    thr = sh.prefix >> fs;
  }
  // the taken positions in ascending order
  unsigned base = 0;
  for (int i0 = 0; i0 < n_iter; i0 += blockDim.x) {
    const int i = i0 + tid;
    bool take = false;
    unsigned long long v = 0ull;
    if (i < n_iter) {
      bool ok = true;
      v = value_at(i, ok);
      take = ok && (all || (v >> fs) >= thr);
    }
    const unsigned slot = ordered_slot(sh, take, base);
    if (take && slot < (unsigned)K) o[slot] = (int32_t)(~(uint32_t)(v & 0xffffffffull)) + offset;
  }
  for (int k = (int)base + tid; k < K; k += blockDim.x) o[k] = -1;
}

}  // namespace csa
