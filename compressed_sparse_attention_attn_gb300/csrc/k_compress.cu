// k_compress.cu -- the compressor of a kv-source layer ("metrale_model_arch::attn_v41": the module
// description's compressor pooling; CompressorWeightsGpu, IndexerWeightsGpu, AttnV41LayerState,
// SharedV41).  The pages fix the weights (f32 kv and gate [hd, dim] at ratio > 1, bf16 kv at ratio
// 1, f32 norm; bf16 wk [index_hd, hd] and f32 k_norm on a kv source that is also an index source),
// the state (a partial group of f32 kv and score [ratio, hd], scores starting at -inf), the caches
// and compress_len; the pooling itself is a reading (the oracle's orc_compress states it):
//   k_p = x_p Wkv^T, s_p = x_p Wgate^T (f32; at ratio 1 k_p = linear_bf16(x_p, Wkv), no score);
//   a closed group j (positions j*ratio .. j*ratio + ratio - 1) pools per feature with the softmax
//   of its scores, z = sum_i e^{s_i} k_i / sum_i e^{s_i}; y = RMSNorm(z) * norm (bf16);
//   index key = RMSNorm(linear_bf16(y, wk)) * k_norm; latent row = fp8 round trip of y with RoPE on
//   its last rd at position j * ratio; an unfinished group waits in the state.
// Two launches: the products as f32 partial sums over k-ranges (CUDA cores: the f32 weights stream
// once, every token of a tile reusing each weight from shared memory), then one CTA of hd threads
// per (sequence, group touched by the call) that sums the partials in split order and either pools
// and publishes a closed group or writes the open group's slots to the state.
#include "csa_internal.cuh"
#include "rowops.cuh"

namespace csa {
namespace comp {

constexpr int FT = 64;  // features per CTA
constexpr int TT = 32;  // tokens per CTA
constexpr int KC = 64;  // k per chunk
constexpr int kProjThreads = 256;
constexpr int kMaxRatio = 16;

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(bf16 v) { return __bfloat162float(v); }

// part[s][row][f] = sum over split s's k-range of x[row][k] W[f][k] (f32 FMA chain in k order); W
// rows f < hd are wkv's, f >= hd wgate's.  Thread (fl = tid % 64, tg = tid / 64): feature f0 + fl,
// tokens t0 + 8 tg .. + 7.
template <typename WT>
__global__ void __launch_bounds__(kProjThreads) k_comp_proj(const bf16 *__restrict__ x, int NT, int dim,
                                                            const WT *__restrict__ wkv, const WT *__restrict__ wgate,
                                                            int hd, int F, int chunks_per_split,
                                                            float *__restrict__ part) {
  __shared__ __align__(16) float Xs[KC][TT + 4];  // k-major: the 8 tokens of a thread are two float4
  __shared__ float Ws[FT][KC + 1];
  const int f0 = blockIdx.x * FT, t0 = blockIdx.y * TT, s = blockIdx.z;
  const int tid = threadIdx.x, fl = tid & 63, tg = tid >> 6;
  const int k_begin = s * chunks_per_split * KC, k_end = min(dim, k_begin + chunks_per_split * KC);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int k0 = k_begin; k0 < k_end; k0 += KC) {
    {  // x: token tid % 32, eight k from 8 (tid / 32)
      const int tok = tid & 31, kk = (tid >> 5) * 8, row = t0 + tok, k = k0 + kk;
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = 0.f;
      if (row < NT && k + 8 <= k_end) {
        const uint4 u = *reinterpret_cast<const uint4 *>(x + (int64_t)row * dim + k);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[2 * e] = __low2float(h[e]);
          v[2 * e + 1] = __high2float(h[e]);
        }
      } else if (row < NT) {
        for (int e = 0; e < 8; ++e)
          if (k + e < k_end) v[e] = __bfloat162float(x[(int64_t)row * dim + k + e]);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) Xs[kk + e][tok] = v[e];
    }
    {  // weights: feature tid / 4, sixteen k from 16 (tid % 4)
      const int fr = tid >> 2, kk = (tid & 3) * 16, f = f0 + fr;
      const WT *src = f < hd ? wkv + (int64_t)f * dim : wgate + (int64_t)(f - hd) * dim;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int k = k0 + kk + e;
        Ws[fr][kk + e] = (f < F && k < k_end) ? to_f(src[k]) : 0.f;
      }
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < KC; ++k) {
      const float w = Ws[fl][k];
      const float4 xa = *reinterpret_cast<const float4 *>(&Xs[k][tg * 8]);
      const float4 xb = *reinterpret_cast<const float4 *>(&Xs[k][tg * 8 + 4]);
      acc[0] = fmaf(w, xa.x, acc[0]);
      acc[1] = fmaf(w, xa.y, acc[1]);
      acc[2] = fmaf(w, xa.z, acc[2]);
      acc[3] = fmaf(w, xa.w, acc[3]);
      acc[4] = fmaf(w, xb.x, acc[4]);
      acc[5] = fmaf(w, xb.y, acc[5]);
      acc[6] = fmaf(w, xb.z, acc[6]);
      acc[7] = fmaf(w, xb.w, acc[7]);
    }
    __syncthreads();
  }
  const int f = f0 + fl;
  if (f < F) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = t0 + tg * 8 + i;
      if (row < NT) part[((int64_t)s * NT + row) * F + f] = acc[i];
    }
  }
}

struct PoolArgs {
  const float *part;
  int S, NT, F;
  float *st_kv, *st_score;  // [B][ratio][hd]
  int T, start_pos, ratio, hd, rd, dI, j0;
  const float *norm, *k_norm;
  const bf16 *wk;  // NULL: no index keys
  const float *tab;
  float eps;
  bf16 *Z, *KI, *y_dbg;  // [B][Lstride][hd], [B][Lstride][dI], [B][Lstride][hd] or NULL
  int64_t Lstride;
};

// Sum of v over the block (blockDim.x a multiple of 32, at most 1024); every thread gets it.
__device__ __forceinline__ float block_sum(float v, float *red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.f;
  return warp_sum(t);
}

// One CTA of hd threads per (group j0 + blockIdx.x, sequence blockIdx.y); thread d = feature d.
__global__ void __launch_bounds__(1024) k_comp_pool(const __grid_constant__ PoolArgs a) {
  __shared__ float red[32];
  __shared__ float ys[1024];
  __shared__ float kr[256];
  const int b = blockIdx.y, j = a.j0 + blockIdx.x, d = threadIdx.x;
  const int r = a.ratio, hd = a.hd;
  const int q0 = j * r, qend = a.start_pos + a.T;
  const bool closed = q0 + r <= qend;
  float kv[kMaxRatio], sc[kMaxRatio];
  float *skv = a.st_kv + (int64_t)b * r * hd, *ssc = a.st_score + (int64_t)b * r * hd;
#pragma unroll
  for (int i = 0; i < kMaxRatio; ++i) {
    if (i >= r) break;
    const int q = q0 + i;
    if (q < a.start_pos) {  // written by an earlier call
      kv[i] = skv[i * hd + d];
      sc[i] = r > 1 ? ssc[i * hd + d] : 0.f;
    } else if (q < qend) {  // this call's token: the split partial sums, in split order
      const int64_t row = (int64_t)b * a.T + (q - a.start_pos);
      float k = 0.f, g = 0.f;
      for (int s = 0; s < a.S; ++s) {
        const float *ps = a.part + ((int64_t)s * a.NT + row) * a.F;
        k += ps[d];
        if (r > 1) g += ps[hd + d];
      }
      if (r == 1) k = __bfloat162float(__float2bfloat16_rn(k));  // linear_bf16
      kv[i] = k;
      sc[i] = g;
    } else {  // not yet seen: an empty slot
      kv[i] = 0.f;
      sc[i] = -INFINITY;
    }
  }
  if (!closed) {  // the open group: this call's slots and the empty ones go to the state
    if (r > 1) {
#pragma unroll
      for (int i = 0; i < kMaxRatio; ++i)
        if (i < r && q0 + i >= a.start_pos) {
          skv[i * hd + d] = kv[i];
          ssc[i * hd + d] = sc[i];
        }
    }
    return;
  }
  // pooling
  float z = kv[0];
  if (r > 1) {
    float m = sc[0];
#pragma unroll
    for (int i = 1; i < kMaxRatio; ++i)
      if (i < r) m = fmaxf(m, sc[i]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxRatio; ++i)
      if (i < r) {
        const float e = expf(sc[i] - m);
        num = fmaf(e, kv[i], num);
        den += e;
      }
    z = num / den;
  }
  // y = RMSNorm(z) * norm, bf16
  const float ss = block_sum(z * z, red);
  const float rs = 1.0f / sqrtf(ss / (float)hd + a.eps);
  const float y = __bfloat162float(__float2bfloat16_rn(z * rs * a.norm[d]));
  const int64_t zrow = (int64_t)b * a.Lstride + j;
  if (a.y_dbg) a.y_dbg[zrow * hd + d] = __float2bfloat16_rn(y);
  // index key: RMSNorm(linear_bf16(y, wk)) * k_norm; warp w takes outputs w, w + nw, ...
  if (a.wk) {
    ys[d] = y;
    __syncthreads();
    const int lane = d & 31, wid = d >> 5, nw = hd >> 5;
    for (int o = wid; o < a.dI; o += nw) {
      const bf16 *wr = a.wk + (int64_t)o * hd;
      float acc = 0.f;
      for (int e = lane; e < hd; e += 32) acc = fmaf(ys[e], __bfloat162float(wr[e]), acc);
      acc = warp_sum(acc);
      if (lane == 0) kr[o] = __bfloat162float(__float2bfloat16_rn(acc));
    }
    __syncthreads();
    float kv2 = 0.f;
    for (int o = d; o < a.dI; o += hd) kv2 = fmaf(kr[o], kr[o], kv2);
    const float ss2 = block_sum(kv2, red);
    const float rs2 = 1.0f / sqrtf(ss2 / (float)a.dI + a.eps);
    for (int o = d; o < a.dI; o += hd) a.KI[zrow * a.dI + o] = __float2bfloat16_rn(kr[o] * rs2 * a.k_norm[o]);
  }
  // latent row: RoPE at the group's first position on the last rd, then the fp8 round trip
  float v = y;
  const float partner = __shfl_xor_sync(0xffffffffu, v, 1);
  const int tail = hd - a.rd;
  if (d >= tail) {
    const float2 cs = reinterpret_cast<const float2 *>(a.tab)[(int64_t)q0 * (a.rd >> 1) + ((d - tail) >> 1)];
    float re, im;
    if ((d & 1) == 0)
      rotate_pair(v, partner, cs.x, cs.y, re, im);
    else
      rotate_pair(partner, v, cs.x, cs.y, re, im);
    v = __bfloat162float(__float2bfloat16_rn((d & 1) ? im : re));
  }
  uint8_t c;
  int se;
  a.Z[zrow * hd + d] = __float2bfloat16_rn(fp8_block_roundtrip(v, c, se));
  // a closed group that ends the call leaves the partial group empty
  if (r > 1 && q0 + r == qend)
    for (int i = 0; i < r; ++i) {
      skv[i * hd + d] = 0.f;
      ssc[i * hd + d] = -INFINITY;
    }
}

__global__ void k_fill_f32(float *p, int64_t n, float v) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    p[i] = v;
}

}  // namespace comp

cudaError_t launch_fill_f32(float *p, int64_t n, float v, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  comp::k_fill_f32<<<(unsigned)std::min<int64_t>((n + 255) / 256, 4096), 256, 0, s>>>(p, n, v);
  return cudaGetLastError();
}

bool compress_supported(const CompressArgs &a) {
  return a.ratio >= 1 && a.ratio <= comp::kMaxRatio && a.hd % 64 == 0 && a.hd <= 1024 && a.rd <= a.hd &&
         a.rd % 2 == 0 && a.dim % 8 == 0 && ((uintptr_t)a.x & 15) == 0 && (a.wk == nullptr || a.dI <= 256) &&
         (a.start_pos == 0 || a.T == 1);
}

cudaError_t launch_compress(const CompressArgs &a, float *ws, size_t ws_bytes, int num_sms, cudaStream_t s) {
  using namespace comp;
  const int NT = a.B * a.T;
  if (NT <= 0) return cudaSuccess;
  const int F = a.ratio > 1 ? 2 * a.hd : a.hd;
  const int ftiles = (F + FT - 1) / FT, ttiles = (NT + TT - 1) / TT;
  const int nchunks = (a.dim + KC - 1) / KC;
  // k-splits: about two CTAs per SM, as many as the workspace holds
  int S = std::max(1, std::min(nchunks, (2 * num_sms + ftiles * ttiles - 1) / (ftiles * ttiles)));
  while (S > 1 && (size_t)S * NT * F * sizeof(float) > ws_bytes) --S;
  if ((size_t)S * NT * F * sizeof(float) > ws_bytes) return cudaErrorInvalidValue;
  const int per = (nchunks + S - 1) / S;
  S = (nchunks + per - 1) / per;
  dim3 g1(ftiles, ttiles, S);
  if (a.ratio > 1)
    k_comp_proj<float><<<g1, kProjThreads, 0, s>>>(a.x, NT, a.dim, (const float *)a.wkv, a.wgate, a.hd, F, per, ws);
  else
    k_comp_proj<bf16><<<g1, kProjThreads, 0, s>>>(a.x, NT, a.dim, (const bf16 *)a.wkv, nullptr, a.hd, F, per, ws);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  PoolArgs p;
  p.part = ws;
  p.S = S;
  p.NT = NT;
  p.F = F;
  p.st_kv = a.st_kv;
  p.st_score = a.st_score;
  p.T = a.T;
  p.start_pos = a.start_pos;
  p.ratio = a.ratio;
  p.hd = a.hd;
  p.rd = a.rd;
  p.dI = a.dI;
  p.j0 = a.start_pos / a.ratio;
  p.norm = a.norm;
  p.k_norm = a.k_norm;
  p.wk = a.wk;
  p.tab = a.tab;
  p.eps = a.eps;
  p.Z = a.Z;
  p.KI = a.KI;
  p.y_dbg = a.y_dbg;
  p.Lstride = a.Lstride;
  const int ngroups = (a.start_pos + a.T - 1) / a.ratio - p.j0 + 1;
  k_comp_pool<<<dim3(ngroups, a.B), a.hd, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace csa
