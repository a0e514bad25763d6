// Measurement probes (sm_103a): micro-kernels that measure the issue rate and
// latency of the instruction the narrow q8_0 matmul is built on, the
// four-way int8 dot product (__dp4a), so the arithmetic ceiling of that
// kernel can be derived from measurements taken with committed code.
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

}  // namespace

extern "C" dsb_status dsb_probe_dp4a(int mode, int blocks, int iters, uint32_t* out, void* stream) {
  if ((mode != 0 && mode != 1) || blocks < 1 || blocks > (1 << 20) || iters < 1 || !out) return DSB_ERR_INVALID_ARG;
  dp4a_probe_kernel<<<mode == 0 ? blocks : 1, mode == 0 ? 256 : 32, 0, static_cast<cudaStream_t>(stream)>>>(
      mode, iters, 0x9E3779B9u, out);
  return cudaGetLastError() == cudaSuccess ? DSB_OK : DSB_ERR_CUDA;
}
