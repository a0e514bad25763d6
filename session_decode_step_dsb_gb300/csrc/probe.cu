// Measurement probes (sm_103a): micro-kernels that measure the issue rate and
// latency of the instructions the narrow q8_0 matmul can be built on -- the
// four-way int8 dot product (__dp4a) and the warp-level tensor-core products
// (mma.sync m16n8k16 f16 -> f32, m16n8k32 s8 -> s32) -- so the arithmetic
// ceiling of that kernel can be derived from measurements taken with
// committed code.
#include <cuda_runtime.h>

#include <cstdint>

#include "dsb.h"

namespace {

// mode 0 (rate): every thread advances 8 independent dp4a chains `iters`
// times, so a warp always has independent dp4a instructions ready; the
// caller divides blocks * 256 * 8 * iters by the measured time.
// mode 1 (latency): thread 0 of one warp advances one dependent chain and
// records the SM clock before and after; out[1] = cycles, out[2] = iters.
__global__ void __launch_bounds__(256) dp4a_probe_kernel(int mode, int iters, uint32_t seed, uint32_t* out) {
  const uint32_t t = threadIdx.x + blockIdx.x * blockDim.x;
  if (mode == 0) {
    int a[8];
    const int b = (int)(seed ^ (t * 2654435761u));
#pragma unroll
    for (int j = 0; j < 8; ++j) a[j] = (int)(t + 7u * j);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int j = 0; j < 8; ++j) a[j] = __dp4a(a[j], b, a[j]);
    }
    int s = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) s ^= a[j];
    if (s == 0x12345678) out[0] = (uint32_t)s;  // keeps the chains live
  } else if (threadIdx.x == 0 && blockIdx.x == 0) {
    int a = (int)seed;
    const int b = (int)(seed * 3u + 1u);
    const long long c0 = clock64();
    for (int i = 0; i < iters; ++i) a = __dp4a(a, b, a);
    const long long c1 = clock64();
    out[0] = (uint32_t)a;
    out[1] = (uint32_t)(c1 - c0);
    out[2] = (uint32_t)iters;
  }
}

// Tensor-core rate: every warp advances 8 independent accumulator tiles
// `iters` times (mode 2: m16n8k16 f16 x f16 -> f32; mode 3: m16n8k32
// s8 x s8 -> s32).  The caller divides blocks * 8 warps * 8 * iters products
// of 2*16*8*K flops by the measured time.
__global__ void __launch_bounds__(256) mma_probe_kernel(int mode, int iters, uint32_t seed, uint32_t* out) {
  const uint32_t t = threadIdx.x + blockIdx.x * blockDim.x;
  const uint32_t a0 = seed ^ t, a1 = a0 * 3u, a2 = a0 * 5u, a3 = a0 * 7u;
  const uint32_t b0 = (seed * 11u) ^ (t << 3), b1 = b0 * 13u;
  uint32_t acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[j][e] = 0u;
  if (mode == 2) {
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+r"(acc[j][0]), "+r"(acc[j][1]), "+r"(acc[j][2]), "+r"(acc[j][3])
            : "r"(a0 & 0x3C003C00u), "r"(a1 & 0x3C003C00u), "r"(a2 & 0x3C003C00u), "r"(a3 & 0x3C003C00u),
              "r"(b0 & 0x3C003C00u), "r"(b1 & 0x3C003C00u));
    }
  } else {
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+r"(acc[j][0]), "+r"(acc[j][1]), "+r"(acc[j][2]), "+r"(acc[j][3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
  }
  uint32_t s = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) s ^= acc[j][e];
  if (s == 0x12345678u) out[0] = s;  // keeps the accumulators live
}

}  // namespace

extern "C" dsb_status dsb_probe_mma(int mode, int blocks, int iters, uint32_t* out, void* stream) {
  if ((mode != 2 && mode != 3) || blocks < 1 || blocks > (1 << 20) || iters < 1 || !out) return DSB_ERR_INVALID_ARG;
  mma_probe_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(mode, iters, 0x9E3779B9u, out);
  return cudaGetLastError() == cudaSuccess ? DSB_OK : DSB_ERR_CUDA;
}

extern "C" dsb_status dsb_probe_dp4a(int mode, int blocks, int iters, uint32_t* out, void* stream) {
  if ((mode != 0 && mode != 1) || blocks < 1 || blocks > (1 << 20) || iters < 1 || !out) return DSB_ERR_INVALID_ARG;
  dp4a_probe_kernel<<<mode == 0 ? blocks : 1, mode == 0 ? 256 : 32, 0, static_cast<cudaStream_t>(stream)>>>(
      mode, iters, 0x9E3779B9u, out);
  return cudaGetLastError() == cudaSuccess ? DSB_OK : DSB_ERR_CUDA;
}
