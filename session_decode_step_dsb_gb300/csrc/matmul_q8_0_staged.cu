// The narrow q8_0 matmul reading activations that are already in its staged
// layout (sm_103a): the same kernel as matmul_q8_0.cu, instantiated with the
// staged source.  The decode step's q8_0-emitting kernels (RMSNorm, SiLU-gate,
// the attention merge) write that layout next to the q8_0 rows, so each CTA
// copies its k-range in with two bulk copies instead of copying the rows and
// unpacking them, and both weight stages of every warp are requested before
// the wait for the previous kernel.  Same plan, same codes and scales, so the
// outputs are bitwise those of the q8_0-row launch.
#include "matmul_q8_0_kernel.cuh"

namespace dsbk {

cudaError_t launch_matmul_q8_0_staged(const void* W, int64_t rows, int64_t cols, const void* staged, int n_tok,
                                      float* y, const float* residual, int num_sms, cudaStream_t st) {
  int G = 0;
  const int S = matmul_plan_of(rows, cols, num_sms, &G);
  const size_t smem = matmul_smem_bytes(rows, cols, n_tok, num_sms);
  ActSrc src;
  src.staged = static_cast<const uint32_t*>(staged);
  return dispatch<false, 3>(n_tok, static_cast<const uint8_t*>(W), (int)rows, (int)(cols / 32), src, y, residual,
                            nullptr, G, S, smem, st);
}

size_t matmul_staged_bytes(int n_tok, int64_t cols) { return staged_act_bytes(n_tok, (long long)(cols / 32)); }

unsigned int read_clear_error_matmul_staged() { return read_clear_error_unit(); }

}  // namespace dsbk
