// The narrow q8_0 matmul with its activation quantisation fused in front
// (sm_103a): the same kernel as matmul_q8_0.cu, instantiated with the RMSNorm
// + q8_0 prologue (the step's attention / FFN / final norms ahead of the QKV,
// gate|up and head matmuls) and the SiLU(gate) * up + q8_0 prologue (ahead of
// the down projection).  Each CTA quantises the activation blocks of its own
// k-range from the float rows; the RMSNorm prologue first sums every row's
// squares itself.  The plan (tiling, cluster split) is the q8_0-input plan of
// the same matrix, and the prologues repeat the standalone kernels'
// arithmetic, so the outputs are bitwise those of the two-kernel sequence.
#include "matmul_q8_0_kernel.cuh"

namespace dsbk {

size_t matmul_fused_smem_bytes(int64_t rows, int64_t cols, int n_tok, int pro, int num_sms) {
  int G = 0;
  const int S = matmul_plan_of(rows, cols, num_sms, &G);
  const int nks = (int)(cols / 256);
  return smem_bytes((nks + S - 1) / S, n_tok, G, S, pro);
}

cudaError_t launch_matmul_q8_0_fused(int pro, const void* W, int64_t rows, int64_t cols, const float* xf,
                                     int xf_stride, const float* norm_w, float eps, int n_tok, float* y,
                                     const float* residual, int num_sms, cudaStream_t st) {
  int G = 0;
  const int S = matmul_plan_of(rows, cols, num_sms, &G);
  const size_t smem = matmul_fused_smem_bytes(rows, cols, n_tok, pro, num_sms);
  const int nb = (int)(cols / 32);
  const uint8_t* w8 = static_cast<const uint8_t*>(W);
  ActSrc src;
  src.xf = xf;
  src.norm_w = norm_w;
  src.eps = eps;
  src.xf_stride = xf_stride;
  if (pro == 1) return dispatch<false, 1>(n_tok, w8, (int)rows, nb, src, y, residual, nullptr, G, S, smem, st);
  if (pro == 2) return dispatch<false, 2>(n_tok, w8, (int)rows, nb, src, y, residual, nullptr, G, S, smem, st);
  return cudaErrorInvalidValue;
}

unsigned int read_clear_error_matmul_fused() { return read_clear_error_unit(); }

}  // namespace dsbk
