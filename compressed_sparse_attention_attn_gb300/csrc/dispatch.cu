// dispatch.cu -- picks the kernel for each step from the problem shape.
#include "csa_internal.cuh"

namespace csa {

cudaError_t launch_linear_simt(const bf16 *x, int M, int K, int ldx, const bf16 *W, int N, int ldw, bf16 *y, int ldy,
                               int groups, cudaStream_t s);
cudaError_t launch_sparse_attn_simt(const AttnArgs &a, cudaStream_t s);

cudaError_t launch_gemm_tc(const LinearProblem *probs, int nprob, float *ws, size_t ws_bytes, int num_sms,
                           int *status, cudaStream_t s, int *kernels);
bool gemm_tc_supported(const LinearProblem &q);

// Tensor-core Stream-K GEMM for every product TMA can address (16-byte aligned bases and strides);
// the CUDA-core kernel only for the rest.
cudaError_t launch_linear(const LinearProblem *probs, int n, float *ws, size_t ws_bytes, int num_sms, int *status,
                          cudaStream_t s, int *kernels) {
  LinearProblem batch[4];
  int nb = 0, nk = 0;
  if (kernels) *kernels = 0;
  // one tensor-core launch of the batch (its kernel count added when the caller counts)
  auto flush = [&]() -> cudaError_t {
    int k = 1;
    const cudaError_t e = launch_gemm_tc(batch, nb, ws, ws_bytes, num_sms, status, s, kernels ? &k : nullptr);
    nk += k;
    nb = 0;
    return e;
  };
  for (int i = 0; i < n; ++i) {
    const LinearProblem &q = probs[i];
    if (q.M <= 0) continue;
    if (gemm_tc_supported(q)) {
      if (nb == 4 || (nb > 0 && (batch[0].M != q.M || (batch[0].W8 != nullptr) != (q.W8 != nullptr)))) {
        cudaError_t e = flush();
        if (e != cudaSuccess) return e;
      }
      batch[nb++] = q;
    } else {
      if (q.W8) return cudaErrorInvalidValue;  // fp8 weights: tensor-core path only
      cudaError_t e = launch_linear_simt(q.x, q.M, q.K, q.ldx, q.W, q.N, q.ldw, q.y, q.ldy, q.groups, s);
      if (e != cudaSuccess) return e;
      ++nk;
    }
  }
  if (nb) {
    cudaError_t e = flush();
    if (e != cudaSuccess) return e;
  }
  if (kernels) *kernels = nk;
  return cudaSuccess;
}

bool sparse_attn_tc_supported(const AttnArgs &a);
cudaError_t launch_sparse_attn_tc(const AttnArgs &a, float *ws, size_t ws_bytes, int num_sms, cudaStream_t s,
                                  int *kernels);

// Tensor-core kernel for head_dim 512 (the model's); the CUDA-core kernel for other head sizes.
cudaError_t launch_sparse_attn(const AttnArgs &a, float *ws, size_t ws_bytes, int num_sms, cudaStream_t s,
                               int *kernels) {
  int k = 0;
  cudaError_t e;
  if (sparse_attn_tc_supported(a)) {
    e = launch_sparse_attn_tc(a, ws, ws_bytes, num_sms, s, &k);
  } else {
    if (a.rope_q) return cudaErrorInvalidValue;  // the CUDA-core kernel takes q as given
    e = launch_sparse_attn_simt(a, s);
    k = a.B * a.T > 0 ? 1 : 0;
  }
  if (kernels) *kernels = k;
  return e;
}

}  // namespace csa
