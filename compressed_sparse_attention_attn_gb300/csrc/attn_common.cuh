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

// ---- the sparse-attention kernels' shared parameters -----------------------------------------------
constexpr int HG = 64;        // heads per CTA
constexpr int kMaxTiles = 6;  // index lists up to 768 entries
constexpr int kBlockBytes = TILE * 128;  // one K-block of a tile
constexpr int kMaxHeadGroups = 4;        // H <= 256
constexpr int kVecs = HG * (HD / 8);     // 16-byte vectors of one head group's output
constexpr int kRotPairs = 64;            // angles of the result's inverse rotation kept in shared memory

struct Params {
  CUtensorMap tm_q;  // q [NT*H][512], box {64, 64}
  const bf16 *rows_a, *rows_b;
  int T, H;
  int64_t a_seq_rows, b_seq_rows;
  int a_len, b_len;
  const int32_t *idx_a;
  int na;
  const int32_t *idx_b;
  int nb;
  const float *sink;
  float scale_log2;  // softmax scale * log2(e)
  bf16 *o, *o_rot;
  int rd, start_pos;
  const float *tab;
  int *status;
  int rope_q;       // turn q's last rd features by RoPE in shared memory before the scores
  int ntiles;       // tiles of the index list
  int tpc, nsplit;  // tiles per CTA, CTAs per query
  bf16 *part_o;     // [NT][nsplit][H][512]  O_c / l_c of each split
  float *part_ml;   // [NT][nsplit][H][2]    (m_c, l_c), log2 domain
};


// The index pass of one 128-entry slot j of a CTA's tiles k0 .. k0+nk-1 (a thread per slot, four
// warps): each entry's row address (nullptr for an invalid entry, -1), its validity, and per tile the
// count of valid entries of this thread's warp (warp iw of the four).  An index outside -1 .. rows-1
// raises the bad-index status.
__device__ __forceinline__ void index_pass(const Params &P, int64_t row, int b, int k0, int nk, int j, int iw, int lane,
                                           const bf16 **src_list, uint8_t *valid, int *wcnt) {
  const int n_all = P.na + P.nb, n_rows = P.a_len + P.b_len;
  int v[kMaxTiles];
#pragma unroll
  for (int i = 0; i < kMaxTiles; ++i) {  // every index of this CTA's tiles, loaded up front
    const int e = (k0 + i) * TILE + j;
    v[i] = -1;
    if (i < nk) v[i] = e < P.na ? P.idx_a[row * P.na + e] : (e < n_all ? P.idx_b[row * P.nb + (e - P.na)] : -1);
  }
#pragma unroll
  for (int i = 0; i < kMaxTiles; ++i) {
    if (i < nk) {
      const int e = (k0 + i) * TILE + j;
      if (e < n_all && (v[i] < -1 || v[i] >= n_rows)) atomicOr(P.status, kStatusBadIndex);
      const bool ok = e < n_all && v[i] >= 0 && v[i] < n_rows;
      const bf16 *p = nullptr;
      if (ok)
        p = v[i] < P.a_len ? P.rows_a + (b * P.a_seq_rows + v[i]) * HD
                           : P.rows_b + (b * P.b_seq_rows + (v[i] - P.a_len)) * HD;
      src_list[i * TILE + j] = p;
      valid[i * TILE + j] = ok;
      const unsigned bal = __ballot_sync(0xffffffffu, ok);
      if (lane == 0) wcnt[4 * i + iw] = __popc(bal);
    }
  }
}

// RoPE on q's last rd features, in place in the swizzled K-blocks (64 heads, [KB][64][128 B]): one
// 16-byte chunk (four adjacent pairs) of one head per unit, at most two units for each of 256 threads;
// the same f32 arithmetic as the separate pass.  rope_q_angles reads the angles (while q is still in
// flight), rope_q_apply turns q once it has landed.
__device__ __forceinline__ void rope_q_angles(const Params &P, int t, int tid, float4 (&qcs)[2][2]) {
  const int q_tail = HD - P.rd, q_nch = P.rd / 8;
  const float2 *tp = reinterpret_cast<const float2 *>(P.tab) + (int64_t)(P.start_pos + t) * (P.rd >> 1);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int u = tid + 256 * k;
    if (u < HG * q_nch) {
      const int f0 = q_tail + 8 * (u % q_nch);
      qcs[k][0] = *reinterpret_cast<const float4 *>(tp + (f0 - q_tail) / 2);
      qcs[k][1] = *reinterpret_cast<const float4 *>(tp + (f0 - q_tail) / 2 + 2);
    }
  }
}
// Turn one 16-byte chunk of q in shared memory (features f0 .. f0+7 of head h, four adjacent pairs)
// by the angles cs (cos, sin of each pair).
__device__ __forceinline__ void rope_q_chunk(uint8_t *sq, int h, int f0, const float (&cs)[8]) {
  uint8_t *cp = sq + (f0 / 64) * HG * 128 + h * 128 + ((((f0 % 64) / 8) ^ (h & 7)) << 4);
  uint4 x = *reinterpret_cast<const uint4 *>(cp);
  __nv_bfloat162 *pv = reinterpret_cast<__nv_bfloat162 *>(&x);
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const float a = __low2float(pv[jj]), bb = __high2float(pv[jj]), c = cs[2 * jj], sn = cs[2 * jj + 1];
    const float re = __fsub_rn(__fmul_rn(a, c), __fmul_rn(bb, sn));
    const float im = __fadd_rn(__fmul_rn(a, sn), __fmul_rn(bb, c));
    pv[jj] = __halves2bfloat162(__float2bfloat16_rn(re), __float2bfloat16_rn(im));
  }
  *reinterpret_cast<uint4 *>(cp) = x;
}
__device__ __forceinline__ void rope_q_apply(const Params &P, uint8_t *sq, int tid, const float4 (&qcs)[2][2]) {
  const int q_tail = HD - P.rd, q_nch = P.rd / 8;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int u = tid + 256 * k;
    if (u >= HG * q_nch) continue;
    const float cs[8] = {qcs[k][0].x, qcs[k][0].y, qcs[k][0].z, qcs[k][0].w,
                         qcs[k][1].x, qcs[k][1].y, qcs[k][1].z, qcs[k][1].w};
    rope_q_chunk(sq, u / q_nch, q_tail + 8 * (u % q_nch), cs);
  }
  fence_proxy_async();  // the turned q is read by the MMA (async proxy)
}

cudaError_t launch_sparse_attn_queries_tc(const Params &p, int units, int num_sms, cudaStream_t s);

}  // namespace attn
}  // namespace csa
