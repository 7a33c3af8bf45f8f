// k_gemm_simt.cu -- reference-shaped CUDA-core GEMM for linear_bf16 ("deepseek_v41_ref::attn"
// precision contract: f32 accumulation, bf16 result).  y[m][n] = sum_k x[m][k] W[n][k].
// 64x64 output tile per CTA, 256 threads with 4x4 outputs each, K staged through shared memory in
// slices of 32.  grid.z indexes the groups of the block-diagonal wo_a product.
#include "csa_internal.cuh"

namespace csa {

namespace {
constexpr int BM = 64, BN = 64, BK = 32;

__global__ void __launch_bounds__(256) k_gemm_simt(const bf16 *__restrict__ x, int M, int K, int ldx,
                                                   const bf16 *__restrict__ W, int N, int ldw, bf16 *__restrict__ y,
                                                   int ldy) {
  const int g = blockIdx.z;
  x += (int64_t)g * K;
  W += (int64_t)g * N * ldw;
  y += (int64_t)g * N;
  __shared__ float xs[BK][BM + 4];
  __shared__ float ws[BK][BN + 4];
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int tid = threadIdx.x;
  const int tm = (tid / 16) * 4, tn = (tid % 16) * 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BK) {
    // 64 rows x 32 k of each operand: 2048 elements, 8 per thread
    for (int e = tid; e < BM * BK; e += 256) {
      const int r = e / BK, kk = e % BK;
      const int gm = m0 + r, gn = n0 + r, gk = k0 + kk;
      xs[kk][r] = (gm < M && gk < K) ? __bfloat162float(x[(int64_t)gm * ldx + gk]) : 0.f;
      ws[kk][r] = (gn < N && gk < K) ? __bfloat162float(W[(int64_t)gn * ldw + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][tm + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = ws[kk][tn + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gm = m0 + tm + i, gn = n0 + tn + j;
      if (gm < M && gn < N) y[(int64_t)gm * ldy + gn] = __float2bfloat16_rn(acc[i][j]);
    }
}
}  // namespace

cudaError_t launch_linear_simt(const bf16 *x, int M, int K, int ldx, const bf16 *W, int N, int ldw, bf16 *y, int ldy,
                               int groups, cudaStream_t s) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM, groups);
  k_gemm_simt<<<grid, 256, 0, s>>>(x, M, K, ldx, W, N, ldw, y, ldy);
  return cudaGetLastError();
}

}  // namespace csa
