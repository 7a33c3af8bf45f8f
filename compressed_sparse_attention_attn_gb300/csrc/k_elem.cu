// k_elem.cu -- row-wise kernels of the layer core: RMSNorm, RoPE, the fp8 round trip, and the fused
// window-row finish (RoPE + fp8 + ring update + window selection).
//
// Each is bandwidth-trivial (a few KiB per token); they are written for exactness first: the RoPE
// complex product rounds each product and each sum to f32 separately (__fmul_rn / __fadd_rn, no
// contraction), the fp8 scale uses IEEE division (__fdiv_rn), and e4m3 conversion is the hardware
// round-to-nearest-even saturating convert.
#include <cuda_fp8.h>

#include <cstring>

#include "csa_internal.cuh"
#include "rowops.cuh"

namespace csa {


// ---------------------------------------------------------------------------------------------
// RMSNorm, "deepseek_v41_ref::attn" precision contract: f32 compute, bf16 result.
// One CTA per row; the sum of squares in f32 (warp shuffles, then shared memory).
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_rmsnorm(const bf16 *x, int N, const float *__restrict__ w,
                                                 float eps, bf16 *y) {
  const int64_t row = blockIdx.x;
  const bf16 *xr = x + row * N;
  bf16 *yr = y + row * N;
  float ss = 0.f;
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    float v = __bfloat162float(xr[i]);
    ss = fmaf(v, v, ss);
  }
  __shared__ float part[32];
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? part[threadIdx.x] : 0.f;
    v = warp_sum(v);
    if (threadIdx.x == 0) part[0] = v;
  }
  __syncthreads();
  const float r = 1.0f / sqrtf(part[0] / (float)N + eps);
  for (int i = threadIdx.x; i < N; i += blockDim.x) yr[i] = __float2bfloat16_rn(__bfloat162float(xr[i]) * r * w[i]);
}

cudaError_t launch_rmsnorm(const bf16 *x, int M, int N, const float *w, float eps, bf16 *y, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  k_rmsnorm<<<M, 256, 0, s>>>(x, N, w, eps, y);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
// RoPE, "deepseek_v41_ref::attn" apply_rotary: last rd elements of each row, adjacent pairs as
// complex numbers times (cos, sin) of the row's position (conjugate when inverse).
// ---------------------------------------------------------------------------------------------

// One warp per row; lane i takes pairs i, i+32, ...
__global__ void k_rope(bf16 *__restrict__ x, int64_t rows, int row_len, int rd, PosSpec pos,
                       const float *__restrict__ tab, int tab_rows, int inverse, int *status) {
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const int half = rd >> 1;
  const int p = pos.at(row);
  if (p < 0 || p >= tab_rows) {  // a position outside the table: leave the row, report it
    if (lane == 0 && status) atomicOr(status, kStatusBadIndex);
    return;
  }
  __nv_bfloat162 *t = reinterpret_cast<__nv_bfloat162 *>(x + row * row_len + (row_len - rd));
  const float2 *tp = reinterpret_cast<const float2 *>(tab) + (int64_t)p * half;
  for (int i = lane; i < half; i += 32) {
    float2 cs = tp[i];
    float sn = inverse ? -cs.y : cs.y;
    __nv_bfloat162 v = t[i];
    float re, im;
    rotate_pair(__low2float(v), __high2float(v), cs.x, sn, re, im);
    t[i] = __halves2bfloat162(__float2bfloat16_rn(re), __float2bfloat16_rn(im));
  }
}

cudaError_t launch_rope(bf16 *x, int64_t rows, int row_len, int rd, PosSpec pos, const float *tab, int tab_rows,
                        int inverse, int *status, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int warps = 8;
  k_rope<<<(unsigned)((rows + warps - 1) / warps), warps * 32, 0, s>>>(x, rows, row_len, rd, pos, tab, tab_rows,
                                                                       inverse, status);
  return cudaGetLastError();
}


// In-place act_quant over x [n]: one warp per block of 32.
__global__ void k_act_quant(bf16 *__restrict__ x, int64_t nblocks, uint8_t *__restrict__ codes,
                            int8_t *__restrict__ scale_exp) {
  const int64_t blk = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (blk >= nblocks) return;
  const int lane = threadIdx.x & 31;
  const int64_t i = blk * 32 + lane;
  uint8_t c;
  int se;
  float v = fp8_block_roundtrip(__bfloat162float(x[i]), c, se);
  x[i] = __float2bfloat16_rn(v);
  if (codes) codes[i] = c;
  if (scale_exp && lane == 0) scale_exp[blk] = (int8_t)se;
}

cudaError_t launch_act_quant(bf16 *x, int64_t n, uint8_t *codes, int8_t *scale_exp, cudaStream_t s) {
  const int64_t nb = n / 32;
  if (nb <= 0) return cudaSuccess;
  k_act_quant<<<(unsigned)((nb + 7) / 8), 256, 0, s>>>(x, nb, codes, scale_exp);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
// Window rows ("DeepSeek V4.1 - Compressed sparse attention", "Window keys and values": RoPE of the
// last rd, then FP8), plus the ring update and window selection ("deepseek_v41_ref::attn"
// WindowCache, window_topk_idxs).  One CTA of hd threads per token row; warp w owns fp8 block w.
// ---------------------------------------------------------------------------------------------
// Element i of window row `row` (b, t): v is the normed bf16 value.  Called by every thread of
// whole warps (the pair partner and the fp8 block come from lane shuffles).
__device__ __forceinline__ void kv_row_finish(float v, int64_t row, int b, int t, int i, int T, int start_pos,
                                              int hd, int rd, const float *__restrict__ tab, bf16 *kv_out,
                                              bf16 *__restrict__ ring, int W, int32_t *__restrict__ win_idx,
                                              int idx_stride, uint8_t *__restrict__ codes,
                                              int8_t *__restrict__ scales, int nthreads) {
  const int p = start_pos + t;
  const int tail = hd - rd;
  // RoPE: lanes (2k, 2k+1) hold one complex number; each lane produces its own component.
  const float partner = __shfl_xor_sync(0xffffffffu, v, 1);
  if (i >= tail) {
    const int pair = (i - tail) >> 1;
    const float2 cs = reinterpret_cast<const float2 *>(tab)[(int64_t)p * (rd >> 1) + pair];
    float re, im;
    if ((i & 1) == 0)
      rotate_pair(v, partner, cs.x, cs.y, re, im);
    else
      rotate_pair(partner, v, cs.x, cs.y, re, im);
    v = __bfloat162float(__float2bfloat16_rn((i & 1) ? im : re));
  }
  uint8_t c;
  int se;
  const float q = fp8_block_roundtrip(v, c, se);
  const bf16 qb = __float2bfloat16_rn(q);
  kv_out[row * hd + i] = qb;
  if (codes) codes[row * hd + i] = c;
  if (scales && (i & 31) == 0) scales[row * (hd / 32) + (i >> 5)] = (int8_t)se;
  // ring: position p lives in slot p mod W; of a chunk only the last W rows land
  if (t >= T - W) ring[((int64_t)b * W + (p % W)) * hd + i] = qb;
  // window selection
  if (win_idx) {
    int32_t *wi = win_idx + row * idx_stride;
    for (int k = i; k < W; k += nthreads) {
      const int pk = p - W + 1 + k;
      if (start_pos == 0)
        wi[k] = pk >= 0 ? pk : -1;  // the chunk's own rows
      else
        wi[k] = pk >= 0 ? (p + 1 + k) % W : -1;  // ring slots, oldest first
    }
  }
}

__global__ void k_kv_finish(const bf16 *kv_in, bf16 *kv_out, int T, int start_pos, int hd, int rd,
                            const float *__restrict__ tab, bf16 *__restrict__ ring, int W,
                            int32_t *__restrict__ win_idx, int idx_stride, uint8_t *__restrict__ codes,
                            int8_t *__restrict__ scales) {
  const int64_t row = blockIdx.x;  // b * T + t
  const int b = (int)(row / T), t = (int)(row % T);
  const int i = threadIdx.x;
  const float v = __bfloat162float(kv_in[row * hd + i]);
  kv_row_finish(v, row, b, t, i, T, start_pos, hd, rd, tab, kv_out, ring, W, win_idx, idx_stride, codes, scales,
                blockDim.x);
}

// ---------------------------------------------------------------------------------------------
// Split-K reduction of [wq_a | wkv | weights_proj] x fused with everything that consumes it:
// qr = RMSNorm(sum) * q_norm, the window row (RMSNorm * kv_norm, RoPE, fp8, ring, selection), and
// w^I = bf16(sum) * wscale.  One CTA per token, blockDim >= hd, a multiple of 32.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) k_x_finish(XFinishArgs a) {
  extern __shared__ float xs[];  // [ldp] the token's projections, rounded to bf16
  __shared__ float red[2][32];
  // a programmatic dependent of the split-K projection writing the slices: nothing is read or written
  // before that grid has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t row = blockIdx.x;
  const int b = (int)(row / a.T), t = (int)(row % a.T);
  const int M = a.B * a.T;
  const int n = a.q_rank + a.hd + a.Hi;
  float sq = 0.f, skv = 0.f;
  auto take = [&](int c, float v) {
    v = __bfloat162float(__float2bfloat16_rn(v));  // linear_bf16 rounds the projection to bf16
    xs[c] = v;
    if (c < a.q_rank)
      sq = fmaf(v, v, sq);
    else if (c < a.q_rank + a.hd)
      skv = fmaf(v, v, skv);
  };
  // the split partials of a column are summed in split order; up to 8 of them in flight at once
  constexpr int kB = 8;
  if ((n & 3) == 0 && (a.ldp & 3) == 0 && ((uintptr_t)a.part & 15) == 0) {
    for (int c4 = threadIdx.x; c4 < n / 4; c4 += blockDim.x) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s0 = 0; s0 < a.S; s0 += kB) {
        float4 v[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u)
          if (s0 + u < a.S)
            v[u] = __ldcg(reinterpret_cast<const float4 *>(a.part + ((int64_t)(s0 + u) * M + row) * a.ldp) + c4);
#pragma unroll
        for (int u = 0; u < kB; ++u)
          if (s0 + u < a.S) {
            acc.x += v[u].x;
            acc.y += v[u].y;
            acc.z += v[u].z;
            acc.w += v[u].w;
          }
      }
      take(4 * c4, acc.x);
      take(4 * c4 + 1, acc.y);
      take(4 * c4 + 2, acc.z);
      take(4 * c4 + 3, acc.w);
    }
  } else {
    for (int c = threadIdx.x; c < n; c += blockDim.x) {
      float acc = 0.f;
      for (int s0 = 0; s0 < a.S; s0 += kB) {
        float v[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u)
          if (s0 + u < a.S) v[u] = __ldcg(a.part + ((int64_t)(s0 + u) * M + row) * a.ldp + c);
#pragma unroll
        for (int u = 0; u < kB; ++u)
          if (s0 + u < a.S) acc += v[u];
      }
      take(c, acc);
    }
  }
  sq = warp_sum(sq);
  skv = warp_sum(skv);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (lane == 0) {
    red[0][wid] = sq;
    red[1][wid] = skv;
  }
  __syncthreads();
  if (wid == 0) {
    float x0 = lane < nw ? red[0][lane] : 0.f, x1 = lane < nw ? red[1][lane] : 0.f;
    x0 = warp_sum(x0);
    x1 = warp_sum(x1);
    if (lane == 0) {
      red[0][0] = x0;
      red[1][0] = x1;
    }
  }
  __syncthreads();
  const float rq = 1.0f / sqrtf(red[0][0] / (float)a.q_rank + a.eps);
  const float rkv = 1.0f / sqrtf(red[1][0] / (float)a.hd + a.eps);
  for (int c = threadIdx.x; c < a.q_rank; c += blockDim.x)
    a.qr[row * a.q_rank + c] = __float2bfloat16_rn(xs[c] * rq * a.q_norm[c]);
  for (int h = threadIdx.x; h < a.Hi; h += blockDim.x) a.wI[row * a.Hi + h] = xs[a.q_rank + a.hd + h] * a.wscale;
  if (threadIdx.x < a.hd) {
    const int i = threadIdx.x;
    const float v = __bfloat162float(__float2bfloat16_rn(xs[a.q_rank + i] * rkv * a.kv_norm[i]));
    kv_row_finish(v, row, b, t, i, a.T, a.start_pos, a.hd, a.rd, a.tab, a.kv, a.ring, a.W, a.win_idx, a.idx_stride,
                  a.codes, a.scales, a.hd);
  }
}

cudaError_t launch_x_finish(const XFinishArgs &a, cudaStream_t s) {
  const int M = a.B * a.T;
  if (M <= 0) return cudaSuccess;
  const int threads = a.hd > 256 ? a.hd : 256;
  const size_t smem = sizeof(float) * (size_t)(a.q_rank + a.hd + a.Hi);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_x_finish, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // launched as a programmatic dependent: its CTAs can be resident (beside the projection's) when the
  // projection ends
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(M);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_x_finish, a);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

cudaError_t launch_kv_finish(const bf16 *kv_in, bf16 *kv_out, int B, int T, int start_pos, int hd, int rd,
                             const float *tab, bf16 *ring, int W, int32_t *win_idx, int idx_stride, uint8_t *codes,
                             int8_t *scales, cudaStream_t s) {
  if (B * T <= 0) return cudaSuccess;
  k_kv_finish<<<B * T, hd, 0, s>>>(kv_in, kv_out, T, start_pos, hd, rd, tab, ring, W, win_idx, idx_stride, codes,
                                   scales);
  return cudaGetLastError();
}

__global__ void k_scale_bf16_to_f32(const bf16 *__restrict__ x, int64_t n, float scale, float *__restrict__ y) {
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) y[i] = __bfloat162float(x[i]) * scale;
}

cudaError_t launch_scale_bf16_to_f32(const bf16 *x, int64_t n, float scale, float *y, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  k_scale_bf16_to_f32<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(x, n, scale, y);
  return cudaGetLastError();
}

}  // namespace csa
