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
// The angle of window-row element i's RoPE pair at position p ((1, 0) outside the last rd elements).
__device__ __forceinline__ float2 kv_angle(const float *__restrict__ tab, int p, int rd, int hd, int i) {
  const int tail = hd - rd;
  return i >= tail ? reinterpret_cast<const float2 *>(tab)[(int64_t)p * (rd >> 1) + ((i - tail) >> 1)]
                   : make_float2(1.f, 0.f);
}

// Element i of window row `row` (b, t): v is the normed bf16 value.  Called by every thread of
// whole warps (the pair partner and the fp8 block come from lane shuffles).
__device__ __forceinline__ void kv_row_finish(float v, int64_t row, int b, int t, int i, int T, int start_pos,
                                              int hd, int rd, float2 cs, bf16 *kv_out,
                                              bf16 *__restrict__ ring, int W, int32_t *__restrict__ win_idx,
                                              int idx_stride, uint8_t *__restrict__ codes,
                                              int8_t *__restrict__ scales, int nthreads) {
  const int p = start_pos + t;
  const int tail = hd - rd;
  // RoPE: lanes (2k, 2k+1) hold one complex number; each lane produces its own component.
  const float partner = __shfl_xor_sync(0xffffffffu, v, 1);
  if (i >= tail) {  // cs: the angle of element i's pair at position p (read by the caller)
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
  kv_row_finish(v, row, b, t, i, T, start_pos, hd, rd, kv_angle(tab, start_pos + t, rd, hd, i), kv_out, ring, W,
                win_idx, idx_stride, codes, scales,
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
  const int64_t row = blockIdx.x;
  const int b = (int)(row / a.T), t = (int)(row % a.T);
  // the norm weights and the angle (inputs of no kernel before) read before the dependency wait
  constexpr int kQn = 3;
  float qn[kQn];
#pragma unroll
  for (int k = 0; k < kQn; ++k) {
    const int c = threadIdx.x + k * blockDim.x;
    qn[k] = c < a.q_rank ? __ldg(a.q_norm + c) : 0.f;
  }
  const bool kv_thread = threadIdx.x < a.hd;
  const float kvn = kv_thread ? __ldg(a.kv_norm + threadIdx.x) : 0.f;
  const float2 cs = kv_thread ? kv_angle(a.tab, a.start_pos + t, a.rd, a.hd, threadIdx.x) : make_float2(1.f, 0.f);
  // a programmatic dependent of the split-K projection writing the slices: nothing is read or written
  // before that grid has completed; the projection after it (also a programmatic dependent, reading
  // this kernel's output after its own wait) may start at once
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
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
#pragma unroll
  for (int k = 0; k < kQn; ++k) {
    const int c = threadIdx.x + k * blockDim.x;
    if (c < a.q_rank) a.qr[row * a.q_rank + c] = __float2bfloat16_rn(xs[c] * rq * qn[k]);
  }
  for (int c = threadIdx.x + kQn * blockDim.x; c < a.q_rank; c += blockDim.x)
    a.qr[row * a.q_rank + c] = __float2bfloat16_rn(xs[c] * rq * a.q_norm[c]);
  for (int h = threadIdx.x; h < a.Hi; h += blockDim.x) a.wI[row * a.Hi + h] = xs[a.q_rank + a.hd + h] * a.wscale;
  if (kv_thread) {
    const int i = threadIdx.x;
    const float v = __bfloat162float(__float2bfloat16_rn(xs[a.q_rank + i] * rkv * kvn));
    kv_row_finish(v, row, b, t, i, a.T, a.start_pos, a.hd, a.rd, cs, a.kv, a.ring, a.W, a.win_idx, a.idx_stride,
                  a.codes, a.scales, a.hd);
  }
}

// The same for many tokens (a prefill chunk): a warp per token, eight tokens a CTA.  Each lane sums
// the slices of its 16-byte groups of the token's columns into the warp's shared row (rounded to bf16,
// as above, and kept as bf16) with the sums of squares by warp shuffles; then qr and w^I from the
// row, and the window row in 32-element rounds (a round is one fp8 block, the RoPE pairs adjacent
// lanes).  The window norm weights (for the CTA) and each token's angles go to shared memory before
// the dependency wait.
constexpr int kXRowsWarps = 8;
__global__ void __launch_bounds__(kXRowsWarps * 32) k_x_finish_rows(XFinishArgs a) {
  extern __shared__ __align__(16) uint8_t xsm[];  // bf16 rows [kXRowsWarps][ldr], kv_norm [hd], angles [warps][rd/2]
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t row = (int64_t)blockIdx.x * kXRowsWarps + wid;
  const int M = a.B * a.T;
  const int b = (int)(row / a.T), t = (int)(row % a.T);
  const int n = a.q_rank + a.hd + a.Hi, ldr = (n + 7) & ~7, tail = a.hd - a.rd;
  bf16 *xs = reinterpret_cast<bf16 *>(xsm) + (size_t)wid * ldr;
  float *kvn = reinterpret_cast<float *>(xsm + (size_t)kXRowsWarps * ldr * 2);
  float2 *cs = reinterpret_cast<float2 *>(kvn + a.hd) + (size_t)wid * (a.rd >> 1);
  for (int i = threadIdx.x; i < a.hd; i += blockDim.x) kvn[i] = __ldg(a.kv_norm + i);
  if (row < M)
    for (int k = lane; k < (a.rd >> 1); k += 32)
      cs[k] = reinterpret_cast<const float2 *>(a.tab)[(int64_t)(a.start_pos + t) * (a.rd >> 1) + k];
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (row >= M) return;
  float sq = 0.f, skv = 0.f;
  for (int c4 = lane; c4 < n / 4; c4 += 32) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < a.S; ++s) {
      const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.part + ((int64_t)s * M + row) * a.ldp) + c4);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    // linear_bf16 rounds the projection to bf16
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(acc.x, acc.y), h1 = __floats2bfloat162_rn(acc.z, acc.w);
    *reinterpret_cast<__nv_bfloat162 *>(xs + 4 * c4) = h0;
    *reinterpret_cast<__nv_bfloat162 *>(xs + 4 * c4 + 2) = h1;
    const float r0 = __low2float(h0), r1 = __high2float(h0), r2 = __low2float(h1), r3 = __high2float(h1);
    const float s2 = fmaf(r0, r0, fmaf(r1, r1, fmaf(r2, r2, r3 * r3)));
    if (4 * c4 < a.q_rank)  // q_rank and hd are multiples of 4: a group lies in one part
      sq += s2;
    else if (4 * c4 < a.q_rank + a.hd)
      skv += s2;
  }
  sq = warp_sum(sq);
  skv = warp_sum(skv);
  __syncwarp();
  const float rq = 1.0f / sqrtf(sq / (float)a.q_rank + a.eps);
  const float rkv = 1.0f / sqrtf(skv / (float)a.hd + a.eps);
  for (int c4 = lane; c4 < a.q_rank / 4; c4 += 32) {
    const __nv_bfloat162 x0 = *reinterpret_cast<const __nv_bfloat162 *>(xs + 4 * c4);
    const __nv_bfloat162 x1 = *reinterpret_cast<const __nv_bfloat162 *>(xs + 4 * c4 + 2);
    const float4 w = __ldg(reinterpret_cast<const float4 *>(a.q_norm) + c4);
    const __nv_bfloat162 o0 = __floats2bfloat162_rn(__low2float(x0) * rq * w.x, __high2float(x0) * rq * w.y);
    const __nv_bfloat162 o1 = __floats2bfloat162_rn(__low2float(x1) * rq * w.z, __high2float(x1) * rq * w.w);
    *reinterpret_cast<__nv_bfloat162 *>(a.qr + row * a.q_rank + 4 * c4) = o0;
    *reinterpret_cast<__nv_bfloat162 *>(a.qr + row * a.q_rank + 4 * c4 + 2) = o1;
  }
  for (int h = lane; h < a.Hi; h += 32)
    a.wI[row * a.Hi + h] = __bfloat162float(xs[a.q_rank + a.hd + h]) * a.wscale;
  // the window row (hd = 512): lane l holds elements 16l .. 16l+15, so a RoPE pair lies in one lane
  // and an fp8 block of 32 in the lanes (2m, 2m+1); the same arithmetic as kv_row_finish
  const int p = a.start_pos + t, i0 = 16 * lane;
  float v[16];
  {
    const uint4 x0 = *reinterpret_cast<const uint4 *>(xs + a.q_rank + i0);
    const uint4 x1 = *reinterpret_cast<const uint4 *>(xs + a.q_rank + i0 + 8);
    const bf16 *xb0 = reinterpret_cast<const bf16 *>(&x0), *xb1 = reinterpret_cast<const bf16 *>(&x1);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[k] = __bfloat162float(__float2bfloat16_rn(__bfloat162float(xb0[k]) * rkv * kvn[i0 + k]));
      v[8 + k] = __bfloat162float(__float2bfloat16_rn(__bfloat162float(xb1[k]) * rkv * kvn[i0 + 8 + k]));
    }
  }
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int i = i0 + 2 * m;
    if (i >= tail) {
      const float2 c2 = cs[(i - tail) >> 1];
      float re, im;
      rotate_pair(v[2 * m], v[2 * m + 1], c2.x, c2.y, re, im);
      v[2 * m] = __bfloat162float(__float2bfloat16_rn(re));
      v[2 * m + 1] = __bfloat162float(__float2bfloat16_rn(im));
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(v[k]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  const float sc = pow2_ceil_f(__fdiv_rn(fmaxf(amax, 1e-4f), 448.0f));
  const uint32_t eb = (__float_as_uint(sc) >> 23) & 0xffu;
  const float inv = eb >= 254u ? 0.f : __uint_as_float((254u - eb) << 23);  // exact: sc is a power of two
  uint32_t qw[8], cw[4];
#pragma unroll
  for (int k = 0; k < 16; k += 2) {
    float qv[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float r = fminf(fmaxf(__fmul_rn(v[k + e], inv), -448.0f), 448.0f);
      const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(r, __NV_SATFINITE, __NV_E4M3);
      const __half_raw hr = __nv_cvt_fp8_to_halfraw(c, __NV_E4M3);
      qv[e] = __fmul_rn(__half2float(__half(hr)), sc);
      const int kk = k + e;
      if ((kk & 3) == 0) cw[kk >> 2] = 0u;
      cw[kk >> 2] |= (uint32_t)c << (8 * (kk & 3));
    }
    const __nv_bfloat162 qb = __floats2bfloat162_rn(qv[0], qv[1]);
    qw[k >> 1] = *reinterpret_cast<const uint32_t *>(&qb);
  }
  const uint4 q0 = make_uint4(qw[0], qw[1], qw[2], qw[3]), q1 = make_uint4(qw[4], qw[5], qw[6], qw[7]);
  uint4 *ko = reinterpret_cast<uint4 *>(a.kv + row * a.hd + i0);
  ko[0] = q0;
  ko[1] = q1;
  if (a.codes) *reinterpret_cast<uint4 *>(a.codes + row * a.hd + i0) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
  if (a.scales && (lane & 1) == 0)
    a.scales[row * (a.hd / 32) + (lane >> 1)] = (int8_t)((int)eb - 127);
  if (t >= a.T - a.W) {  // ring: position p lives in slot p mod W; of a chunk only the last W rows land
    uint4 *ro = reinterpret_cast<uint4 *>(a.ring + ((int64_t)b * a.W + (p % a.W)) * a.hd + i0);
    ro[0] = q0;
    ro[1] = q1;
  }
  if (a.win_idx) {
    int32_t *wi = a.win_idx + row * a.idx_stride;
    for (int k = lane; k < a.W; k += 32) {
      const int pk = p - a.W + 1 + k;
      if (a.start_pos == 0)
        wi[k] = pk >= 0 ? pk : -1;  // the chunk's own rows
      else
        wi[k] = pk >= 0 ? (p + 1 + k) % a.W : -1;  // ring slots, oldest first
    }
  }
}

cudaError_t launch_x_finish(const XFinishArgs &a, cudaStream_t s) {
  const int M = a.B * a.T;
  if (M <= 0) return cudaSuccess;
  const int n = a.q_rank + a.hd + a.Hi;
  const bool rows = M >= 512 && a.q_rank % 4 == 0 && a.hd == 512 && a.Hi % 4 == 0 && a.ldp % 4 == 0 &&
                    ((uintptr_t)a.part & 15) == 0 && ((uintptr_t)a.q_norm & 15) == 0 && ((uintptr_t)a.qr & 7) == 0 &&
                    ((uintptr_t)a.kv & 15) == 0 && ((uintptr_t)a.ring & 15) == 0 && ((uintptr_t)a.codes & 15) == 0;
  const int threads = rows ? kXRowsWarps * 32 : (a.hd > 256 ? a.hd : 256);
  const size_t smem = rows ? sizeof(bf16) * (size_t)kXRowsWarps * ((n + 7) & ~7) + sizeof(float) * (size_t)a.hd +
                                 sizeof(float2) * (size_t)kXRowsWarps * (a.rd >> 1)
                           : sizeof(float) * (size_t)n;
  const void *fn = rows ? (const void *)k_x_finish_rows : (const void *)k_x_finish;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // launched as a programmatic dependent: its CTAs can be resident (beside the projection's) when the
  // projection ends
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(rows ? (unsigned)((M + kXRowsWarps - 1) / kXRowsWarps) : (unsigned)M);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = rows ? cudaLaunchKernelEx(&cfg, k_x_finish_rows, a) : cudaLaunchKernelEx(&cfg, k_x_finish, a);
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
