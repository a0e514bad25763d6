// The narrow q8_0 matmul reading activations that are already in its staged
// layout (sm_103a): the same kernel as matmul_q8_0.cu, instantiated with the
// staged source.  The decode step's q8_0-emitting kernels (RMSNorm, SiLU-gate,
// the attention merge) write that layout next to the q8_0 rows, so each CTA
// copies its k-range in with two bulk copies instead of copying the rows and
// unpacking them, and both weight stages of every warp are requested before
// the wait for the previous kernel.  Same plan, same codes and scales, so the
// outputs are bitwise those of the q8_0-row launch.  A small kernel also
// writes the layout from q8_0 rows, for callers that hold the rows only.
#include "matmul_q8_0_kernel.cuh"

namespace dsbk {

namespace {

// One warp per (q8_0 block, token row) of xq: the block into the staged
// layout, lane = code.
__global__ void __launch_bounds__(256) stage_q8_0_kernel(const uint8_t* __restrict__ xq, int n_tok, int nb,
                                                         uint32_t* __restrict__ staged) {
  pdl_wait();
  pdl_trigger();
  const int warp = (int)(blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)), lane = threadIdx.x & 31;
  if (warp >= nb * n_tok) return;
  const int t = warp / nb, blk = warp - t * nb;
  const uint8_t* src = xq + ((size_t)t * nb + blk) * 34;
  const int q = (int)(signed char)src[2 + lane];
  const unsigned short dbits = (unsigned short)(src[0] | (src[1] << 8));
  staged_store_block(q, dbits, staged, nb, blk, t, n_tok, lane);
}

}  // namespace

cudaError_t launch_matmul_q8_0_staged(const void* W, int64_t rows, int64_t cols, const void* staged, int n_tok,
                                      float* y, const float* residual, int num_sms, cudaStream_t st) {
  int G = 0;
  const int S = matmul_plan_of(rows, cols, num_sms, &G);
  const int nks = (int)(cols / 256);
  const size_t smem = smem_bytes((nks + S - 1) / S, n_tok, G, S, 3);
  ActSrc src;
  src.staged = static_cast<const uint32_t*>(staged);
  return dispatch<false, 3>(n_tok, static_cast<const uint8_t*>(W), (int)rows, (int)(cols / 32), src, y, residual,
                            nullptr, G, S, smem, st);
}

cudaError_t launch_stage_q8_0(const void* xq, int n_tok, int64_t cols, void* staged, cudaStream_t st) {
  const int nb = (int)(cols / 32);
  const long long warps = (long long)nb * n_tok;
  if (warps <= 0) return cudaSuccess;
  return launch_kernel(stage_q8_0_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, st,
                       static_cast<const uint8_t*>(xq), n_tok, nb, static_cast<uint32_t*>(staged));
}

size_t matmul_staged_bytes(int n_tok, int64_t cols) { return staged_act_bytes(n_tok, (long long)(cols / 32)); }

unsigned int read_clear_error_matmul_staged() { return read_clear_error_unit(); }

}  // namespace dsbk
