// k_attn_simt.cu -- sparse attention with the per-head sink on CUDA cores ("deepseek_v41_ref::attn"
// sparse_attn; "DeepSeek V4.1 - Compressed sparse attention", "Sparse attention"; "Join rows").
// One warp per (query, head): the lane holds DPL = hd/32 consecutive features of q and of the
// running output; rows are gathered straight from the two sources through the joined index
// [idx_a; idx_b] (Y = [rows_a; rows_b] is never materialised).  The softmax is the running
// (max, sum) form started from the sink: m = sink, l = exp(sink - m) = 1, acc = 0, so the sink
// enters the denominator only.  The inverse rotation of the output's last rd features
// ("Grouped output": R_t^-1) is applied in the same pass.
#include "csa_internal.cuh"

namespace csa {

template <int DPL>
__device__ __forceinline__ void load_row(const bf16 *src, float (&v)[DPL]) {
  if constexpr (DPL % 8 == 0) {
    const uint4 *p = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int u = 0; u < DPL / 8; ++u) {
      uint4 w = p[u];
      const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&w);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[u * 8 + 2 * e] = __low2float(h[e]);
        v[u * 8 + 2 * e + 1] = __high2float(h[e]);
      }
    }
  } else {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(src);
#pragma unroll
    for (int e = 0; e < DPL / 2; ++e) {
      v[2 * e] = __low2float(h[e]);
      v[2 * e + 1] = __high2float(h[e]);
    }
  }
}

template <int DPL>
__global__ void __launch_bounds__(256) k_sparse_attn_simt(AttnArgs a) {
  const int H = a.H, hd = a.hd;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x * (blockDim.x >> 5) + warp;
  const int64_t row = blockIdx.y;  // b * T + t
  if (h >= H) return;
  const int b = (int)(row / a.T), t = (int)(row % a.T);
  float q[DPL];
  load_row<DPL>(a.q + (row * H + h) * hd + lane * DPL, q);
  const bf16 *ya = a.rows_a + b * a.a_seq_stride;
  const bf16 *yb = a.rows_b ? a.rows_b + b * a.b_seq_stride : nullptr;
  const int n_rows = a.a_len + a.b_len;
  const float sink = a.sink[h];
  float m = sink, l = 1.0f;
  float acc[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
  const int ntot = a.na + a.nb;
  for (int i = 0; i < ntot; ++i) {
    const int id = i < a.na ? a.idx_a[row * a.na + i] : a.idx_b[row * a.nb + (i - a.na)];
    if (id < 0 || id >= n_rows) {
      if ((id < -1 || id >= n_rows) && lane == 0 && h == 0) atomicOr(a.status, kStatusBadIndex);
      continue;
    }
    const bf16 *src = id < a.a_len ? ya + (int64_t)id * hd : yb + (int64_t)(id - a.a_len) * hd;
    float g[DPL];
    load_row<DPL>(src + lane * DPL, g);
    float d = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) d = fmaf(q[e], g[e], d);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    const float s = d * a.scale;
    const float mn = fmaxf(m, s);
    const float corr = __expf(m - mn);
    const float p = __expf(s - mn);
    l = l * corr + p;
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = fmaf(p, g[e], acc[e] * corr);
    m = mn;
  }
  const float inv = 1.0f / l;
  bf16 ob[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) ob[e] = __float2bfloat16_rn(acc[e] * inv);
  bf16 *od = a.o ? a.o + (row * H + h) * hd + lane * DPL : nullptr;
  if (od) {
#pragma unroll
    for (int e = 0; e < DPL; ++e) od[e] = ob[e];
  }
  if (a.o_rot) {
    bf16 *orr = a.o_rot + (row * H + h) * hd + lane * DPL;
    const int f0 = lane * DPL, tail = hd - a.rd;
    const int p = a.start_pos + t;
#pragma unroll
    for (int e = 0; e < DPL; e += 2) {
      const int f = f0 + e;
      if (f >= tail) {
        const float2 cs = reinterpret_cast<const float2 *>(a.tab)[(int64_t)p * (a.rd >> 1) + ((f - tail) >> 1)];
        const float x0 = __bfloat162float(ob[e]), x1 = __bfloat162float(ob[e + 1]);
        const float sn = -cs.y;
        const float re = __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, sn));
        const float im = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, cs.x));
        orr[e] = __float2bfloat16_rn(re);
        orr[e + 1] = __float2bfloat16_rn(im);
      } else {
        orr[e] = ob[e];
        orr[e + 1] = ob[e + 1];
      }
    }
  }
}

cudaError_t launch_sparse_attn_simt(const AttnArgs &a, cudaStream_t s) {
  const int n = a.B * a.T;
  if (n <= 0) return cudaSuccess;
  dim3 grid((a.H + 7) / 8, n);
  switch (a.hd / 32) {
    case 16: k_sparse_attn_simt<16><<<grid, 256, 0, s>>>(a); break;
    case 8: k_sparse_attn_simt<8><<<grid, 256, 0, s>>>(a); break;
    case 4: k_sparse_attn_simt<4><<<grid, 256, 0, s>>>(a); break;
    case 2: k_sparse_attn_simt<2><<<grid, 256, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace csa
