// rowops.cuh -- per-row building blocks shared by the row-wise kernels (k_elem.cu) and the
// compressor (k_compress.cu): warp reductions, the RoPE complex product with each product and sum
// rounded to f32 ("deepseek_v41_ref::attn" apply_rotary), and the fp8 round trip of one block of 32
// values ("deepseek_v41_ref::attn" act_quant_inplace, pow2_ceil).
#pragma once

#include <cuda_fp8.h>

#include "csa_internal.cuh"

namespace csa {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ void rotate_pair(float a, float b, float c, float s, float &re, float &im) {
  re = __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, s));
  im = __fadd_rn(__fmul_rn(a, s), __fmul_rn(b, c));
}

// fp8 round trip of one block of 32 held one value per lane of a full warp: scale s =
// pow2_ceil(max(amax, 1e-4) / 448) with IEEE division, code = e4m3 RNE of clamp(v / s, +-448)
// (saturating hardware convert), value = code * s.  Returns the new value; code / sexp receive the
// lane's e4m3 code and the block's scale exponent.
__device__ __forceinline__ float pow2_ceil_f(float v) {
  uint32_t u = __float_as_uint(v);
  if ((u & 0x007fffffu) == 0u) return v;
  return __uint_as_float(((u >> 23) + 1u) << 23);
}

__device__ __forceinline__ float fp8_block_roundtrip(float v, uint8_t &code, int &sexp) {
  float amax = warp_max(fabsf(v));
  float s = pow2_ceil_f(__fdiv_rn(fmaxf(amax, 1e-4f), 448.0f));
  // s is a power of two (2^-22 .. 2^120 for finite values), so v / s is v times the exact reciprocal
  // 2^-e: the same exact quotient, rounded once (to 0 when s is infinite)
  const uint32_t eb = (__float_as_uint(s) >> 23) & 0xffu;
  float r = __fmul_rn(v, eb >= 254u ? 0.f : __uint_as_float((254u - eb) << 23));
  r = fminf(fmaxf(r, -448.0f), 448.0f);
  __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(r, __NV_SATFINITE, __NV_E4M3);
  __half_raw hr = __nv_cvt_fp8_to_halfraw(c, __NV_E4M3);
  float dq = __half2float(__half(hr));
  code = (uint8_t)c;
  sexp = (int)((__float_as_uint(s) >> 23) & 0xffu) - 127;
  return __fmul_rn(dq, s);
}

}  // namespace csa
