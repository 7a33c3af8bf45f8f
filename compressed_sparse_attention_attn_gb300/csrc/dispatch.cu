// dispatch.cu -- picks the kernel for each step from the problem shape.
#include "csa_internal.cuh"

namespace csa {

cudaError_t launch_linear_simt(const bf16 *x, int M, int K, int ldx, const bf16 *W, int N, int ldw, bf16 *y, int ldy,
                               int groups, cudaStream_t s);
cudaError_t launch_sparse_attn_simt(const AttnArgs &a, cudaStream_t s);

cudaError_t launch_linear(const bf16 *x, int M, int K, int ldx, const bf16 *W, int N, int ldw, bf16 *y, int ldy,
                          int groups, float *ws, size_t ws_bytes, int num_sms, cudaStream_t s) {
  (void)ws;
  (void)ws_bytes;
  (void)num_sms;
  return launch_linear_simt(x, M, K, ldx, W, N, ldw, y, ldy, groups, s);
}

cudaError_t launch_sparse_attn(const AttnArgs &a, float *ws, size_t ws_bytes, int num_sms, cudaStream_t s) {
  (void)ws;
  (void)ws_bytes;
  (void)num_sms;
  return launch_sparse_attn_simt(a, s);
}

}  // namespace csa
