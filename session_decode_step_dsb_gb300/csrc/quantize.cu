// q8_0 quantisation of float32 activation rows (sm_103a).
//
// Per 32 consecutive values (the pre-quantised "preq" activations that the
// narrow-batch matmul of antirez/ds4 PR #530 consumes; the workload's rule
// scale = max|x| / 127, code = round(x / scale)):
//     a = max|x_k|;  d = a / 127;  q_k = clamp(round(x_k / d), -127, 127)
// with IEEE float32 division (nvcc's default -prec-div=true), round half away
// from zero (roundf) and q = 0 when d == 0; the block stores fp16(d), round to
// nearest even, little-endian, then the 32 codes.  Every step is a single
// correctly rounded float32 operation, so the bytes equal the host codec's.
//
// One warp per block: lane k owns value k; the max is a butterfly over the
// warp; even lanes write two code bytes each and lane 0 the scale.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dsb_kernels.h"
#include "dsb_ptx.cuh"

namespace dsbk {

namespace {

__global__ void __launch_bounds__(256) quantize_q8_0_kernel(const float* __restrict__ x, long long n_blocks,
                                                           uint8_t* __restrict__ xq) {
  pdl_wait();
  pdl_trigger();
  const long long blk = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (blk >= n_blocks) return;
  const float v = __ldcg(x + blk * 32 + lane);
  float a = fabsf(v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const float d = __fdiv_rn(a, 127.0f);
  int q = 0;
  if (d != 0.0f) {
    const float r = roundf(__fdiv_rn(v, d));
    q = (int)fminf(fmaxf(r, -127.0f), 127.0f);
  }
  // Stores are 16-bit and 2-byte aligned (a block starts at an even byte):
  // lane 0 writes the fp16 scale, every even lane the code pair (l, l+1).
  const int q_next = __shfl_down_sync(0xffffffffu, q, 1);
  unsigned short* out16 = reinterpret_cast<unsigned short*>(xq + blk * 34);
  if ((lane & 1) == 0)
    out16[1 + (lane >> 1)] = (unsigned short)(((unsigned)q & 0xFFu) | (((unsigned)q_next & 0xFFu) << 8));
  if (lane == 0) out16[0] = __half_as_ushort(__float2half_rn(d));
}

}  // namespace

cudaError_t launch_quantize_q8_0(const float* x, int64_t n_rows, int64_t cols, void* xq, cudaStream_t st) {
  const long long n_blocks = (long long)n_rows * (cols / 32);
  if (n_blocks == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((n_blocks + 7) / 8);
  return launch_kernel(quantize_q8_0_kernel, dim3(grid), dim3(256), 0, st, x, n_blocks, static_cast<uint8_t*>(xq));
}

}  // namespace dsbk
