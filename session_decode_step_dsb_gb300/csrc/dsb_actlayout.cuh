// The activation layout the narrow q8_0 matmul computes from, shared by the
// matmul (which builds it in shared memory from q8_0 rows) and by the step's
// q8_0-emitting kernels (which can write it straight to global memory, so the
// matmul that follows only copies its k-range in).
//
// For n_tok tokens and a row of nb q8_0 blocks:
//   codes  [nb][8][NTA] u32: code word k (codes 4k..4k+3) of block blk for
//          token t at slot act_pos(NTA, mma, k, t); on the warp-level
//          tensor-core path (n_tok >= kMmaMinNt) every byte is stored as
//          code + 128 (xor 0x80);
//   scales [nb][NTA] u32: the dp4a path stores the fp16 scale as a float; the
//          tensor-core path stores the fp16 scale bits in the low half and the
//          block's code sum (|sum| <= 32 * 127) as int16 in the high half.
// Slots NT..NTA-1 are padding: zero codes and scale 0, which contribute
// nothing.
#pragma once
#include <cuda_fp16.h>

#include <cstddef>
#include <cstdint>

namespace dsbk {

// From this many tokens on, the narrow matmul's k loop runs on the tensor
// cores instead of dp4a chains.
constexpr int kMmaMinNt = 8;
__host__ __device__ constexpr bool use_mma(int nt) { return nt >= kMmaMinNt; }

// Token slots per (block, word): rounded up to 4 so that four tokens load as
// one 16-byte word (dp4a path), or to 8, the tensor-core tile width.
__host__ __device__ constexpr int act_nta(int nt) { return use_mma(nt) ? (nt + 7) & ~7 : (nt + 3) & ~3; }

// Slot of token t in the row of activation word k.  In the mma layout with 16
// slots the two 8-token halves trade places in words 2, 3, 6 and 7, so that a
// warp's fragment loads (word 4h + c of token 8n + g for lane 4g + c) hit 32
// distinct banks.
__host__ __device__ inline int act_pos(int nta, bool mma, int k, int t) {
  return (mma && nta == 16) ? (t ^ (((k >> 1) & 1) << 3)) : t;
}

// Bytes of the byte form for n_tok tokens and nb blocks (codes, then scales).
__host__ __device__ inline size_t staged_act_bytes(int n_tok, long long nb) {
  return (size_t)nb * 36 * (size_t)act_nta(n_tok);
}

// Store one q8_0 block held one code per lane of a full warp (lane = code
// index, fp16 scale bits dbits) as block blk, token t of the staged layout of
// n_tok tokens x nb blocks.  The warp of the last token also writes the
// block's padding slots.
__device__ inline void staged_store_block(int q, unsigned short dbits, uint32_t* staged, long long nb, int blk, int t,
                                          int n_tok, int lane) {
  const bool mma = use_mma(n_tok);
  const int nta = act_nta(n_tok);
  const unsigned b0 = (unsigned)q & 0xFFu;
  const unsigned b1 = (unsigned)__shfl_down_sync(0xffffffffu, q, 1) & 0xFFu;
  const unsigned b2 = (unsigned)__shfl_down_sync(0xffffffffu, q, 2) & 0xFFu;
  const unsigned b3 = (unsigned)__shfl_down_sync(0xffffffffu, q, 3) & 0xFFu;
  int sum = q;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if ((lane & 3) == 0) {
    const int k = lane >> 2;
    const uint32_t word = (b0 | (b1 << 8) | (b2 << 16) | (b3 << 24)) ^ (mma ? 0x80808080u : 0u);
    staged[((size_t)blk * 8 + k) * nta + act_pos(nta, mma, k, t)] = word;
  }
  uint32_t* scales = staged + (size_t)nb * 8 * nta;
  if (lane == 0)
    scales[(size_t)blk * nta + t] =
        mma ? ((uint32_t)dbits | ((uint32_t)sum << 16)) : __float_as_uint(__half2float(__ushort_as_half(dbits)));
  // the last token's warp also fills the block's padding slots (codes 0,
  // scale 0)
  if (t == n_tok - 1) {
    for (int i = lane; i < (nta - n_tok) * 9; i += 32) {
      const int tp = n_tok + i / 9, k = i % 9;
      if (k < 8)
        staged[((size_t)blk * 8 + k) * nta + act_pos(nta, mma, k, tp)] = mma ? 0x80808080u : 0u;
      else
        scales[(size_t)blk * nta + tp] = 0u;
    }
  }
}

// q8_0-quantise one 32-value block held one value per lane of a full warp
// (the codec's steps: a = max|x|, d = a / 127 in float32, q =
// clamp(round-half-away(x / d), -127, 127), q = 0 when d == 0, scale fp16(d)
// round-to-nearest-even), and store it as the q8_0 block at out_block (when
// not null) and into the staged layout `staged` (when not null) of n_tok
// tokens x nb blocks at (block blk, token t).
__device__ inline void q8_block_store_staged(float v, uint8_t* out_block, uint32_t* staged, long long nb, int blk,
                                             int t, int n_tok, int lane) {
  float a = fabsf(v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const float d = __fdiv_rn(a, 127.0f);
  int q = 0;
  if (d != 0.0f) q = (int)fminf(fmaxf(roundf(__fdiv_rn(v, d)), -127.0f), 127.0f);
  const unsigned short dbits = __half_as_ushort(__float2half_rn(d));
  if (out_block) {
    const unsigned b1 = (unsigned)__shfl_down_sync(0xffffffffu, q, 1) & 0xFFu;
    unsigned short* out16 = reinterpret_cast<unsigned short*>(out_block);
    if ((lane & 1) == 0) out16[1 + (lane >> 1)] = (unsigned short)(((unsigned)q & 0xFFu) | (b1 << 8));
    if (lane == 0) out16[0] = dbits;
  }
  if (staged) staged_store_block(q, dbits, staged, nb, blk, t, n_tok, lane);
}

}  // namespace dsbk
