// attn_common.cuh -- device helpers the two sparse-attention kernels share: cp.async row copies,
// the q tile's TMA load, TMEM loads and stores, butterfly reductions over a warp, and the output
// store with the inverse rotation ("DeepSeek V4.1 - Compressed sparse attention", "Sparse attention"
// and "Grouped output").
#pragma once

#include "csa_internal.cuh"
#include "tc_ptx.cuh"

namespace csa {
namespace attn {

constexpr int HD = 512;      // head_dim the tensor-core attention serves
constexpr int KB = HD / 64;  // 64-feature K-blocks
constexpr int TILE = 128;    // index-list entries per tile (the MMA's M)

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void tma_load_2d_nohint(uint32_t dst, const CUtensorMap *tm, uint64_t *bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"((uint64_t)tm), "r"(tc::smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive columns, then the wait (the registers are operands of the wait)
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  tc::tmem_ld32(taddr, r);
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
                 "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Reduce v[h] (h < 32) over the 32 lanes of the warp for max or sum; lane l ends with head l.
template <bool kMax>
__device__ __forceinline__ float warp_reduce_32(const float (&v)[32], int lane) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  float b[16], c[8], d[4], e[2];
  bool up = (lane & 16) != 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) b[j] = op(up ? v[j + 16] : v[j], __shfl_xor_sync(0xffffffffu, up ? v[j] : v[j + 16], 16));
  up = (lane & 8) != 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) c[j] = op(up ? b[j + 8] : b[j], __shfl_xor_sync(0xffffffffu, up ? b[j] : b[j + 8], 8));
  up = (lane & 4) != 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) d[j] = op(up ? c[j + 4] : c[j], __shfl_xor_sync(0xffffffffu, up ? c[j] : c[j + 4], 4));
  up = (lane & 2) != 0;
#pragma unroll
  for (int j = 0; j < 2; ++j) e[j] = op(up ? d[j + 2] : d[j], __shfl_xor_sync(0xffffffffu, up ? d[j] : d[j + 2], 2));
  up = (lane & 1) != 0;
  return op(up ? e[1] : e[0], __shfl_xor_sync(0xffffffffu, up ? e[0] : e[1], 1));
}

// 16 floats from shared memory (16-byte aligned) into registers
__device__ __forceinline__ void lds16(float (&d)[16], const float *src) {
#pragma unroll
  for (int k = 0; k < 16; k += 4) *reinterpret_cast<float4 *>(d + k) = *reinterpret_cast<const float4 *>(src + k);
}

// bf16 of the inverse rotation of the pair (x0, x1) (both already bf16 values) at table entry cs
__device__ __forceinline__ void unrotate(float x0, float x1, float2 cs, float &re, float &im) {
  const float sn = -cs.y;
  re = __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, sn));
  im = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, cs.x));
}

// Write the bf16 vector ob (features d0 .. d0+7 of one head, element offset off) to o, and its
// inverse rotation to o_rot: pairs at or past `tail` turn back by their angle at the query's
// position (tp: that position's row of the cos/sin table), the others are copied.
__device__ __forceinline__ void store_out(bf16 *o, bf16 *o_rot, int64_t off, int d0, int tail, const float2 *tp,
                                          uint4 ob) {
  if (o) *reinterpret_cast<uint4 *>(o + off) = ob;
  if (o_rot) {
    uint4 orr = ob;
    if (d0 >= tail) {
      const float4 c01 = *reinterpret_cast<const float4 *>(tp + ((d0 - tail) >> 1));
      const float4 c23 = *reinterpret_cast<const float4 *>(tp + ((d0 - tail) >> 1) + 2);
      const float2 cs[4] = {make_float2(c01.x, c01.y), make_float2(c01.z, c01.w), make_float2(c23.x, c23.y),
                            make_float2(c23.z, c23.w)};
      const bf16 *xb = reinterpret_cast<const bf16 *>(&ob);
      bf16 *yb = reinterpret_cast<bf16 *>(&orr);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float re, im;
        unrotate(__bfloat162float(xb[2 * q]), __bfloat162float(xb[2 * q + 1]), cs[q], re, im);
        yb[2 * q] = __float2bfloat16_rn(re);
        yb[2 * q + 1] = __float2bfloat16_rn(im);
      }
    }
    *reinterpret_cast<uint4 *>(o_rot + off) = orr;
  }
}

}  // namespace attn
}  // namespace csa
