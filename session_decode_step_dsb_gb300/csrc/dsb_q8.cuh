// Device-side q8_0 block quantisation shared by the kernels that emit q8_0
// activations.  The steps are the codec's: a = max|x| (warp max), d = a / 127
// (IEEE float32 division), q = clamp(round-half-away(x / d), -127, 127), q = 0
// when d == 0, scale stored as fp16(d) round-to-nearest-even.
#pragma once
#include <cuda_fp16.h>

#include <cstdint>

namespace dsbk {

// One 32-value block held one value per lane of a full warp; 16-bit stores
// (a 34-byte block starts at an even byte): lane 0 the scale, even lanes a
// code pair.
__device__ __forceinline__ void q8_block_store(float v, uint8_t* out_block, int lane) {
  float a = fabsf(v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const float d = __fdiv_rn(a, 127.0f);
  int q = 0;
  if (d != 0.0f) q = (int)fminf(fmaxf(roundf(__fdiv_rn(v, d)), -127.0f), 127.0f);
  const int q_next = __shfl_down_sync(0xffffffffu, q, 1);
  unsigned short* out16 = reinterpret_cast<unsigned short*>(out_block);
  if ((lane & 1) == 0)
    out16[1 + (lane >> 1)] = (unsigned short)(((unsigned)q & 0xFFu) | (((unsigned)q_next & 0xFFu) << 8));
  if (lane == 0) out16[0] = __half_as_ushort(__float2half_rn(d));
}

}  // namespace dsbk
