// Step glue of the batched decode step (sm_103a): the small per-token stages
// that sit between the matmuls.  antirez/ds4 PR #530 ("What") lists them among
// the dense stages a batched step runs once for all sessions (RoPE/norm around
// the attention projections and the output head); the forms used here are the
// plain llama ones:
//   rmsnorm(x) = x / sqrt(mean(x^2) + eps) * w      (fused with q8_0 quantise)
//   silu(g) * u = g / (1 + exp(-g)) * u              (fused with q8_0 quantise)
//   embedding  = the q8_0 row of the token id, dequantised
// The residual adds are fused into the matmul epilogue (y = residual + W x).
// Quantisation inside these kernels uses the same float32 codec steps as
// quantize.cu (max|x|/127, round half away from zero, fp16 scale).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dsb_actlayout.cuh"
#include "dsb_kernels.h"
#include "dsb_ptx.cuh"
#include "dsb_q8.cuh"

namespace dsbk {

namespace {

constexpr int kGlueThreads = 256;

constexpr int kMaxPerThread = 32;  // hidden <= 8192
constexpr int kMaxShare = 4;       // values per thread a RMSNorm CTA quantises

// A grid of (token row, split) CTAs.  Thread j holds elements j, j + 256, ...
// of the row in registers (one memory round trip); the sum of squares goes
// through a fixed tree, identical in every CTA of the row; then warp w
// quantises blocks w + 8k for the CTA's share of k (blockIdx.y-th of
// gridDim.y) -- element 32b + lane of block b is exactly the value thread
// 32w + lane already holds.  Splitting the blocks over CTAs keeps a 16-token
// step's norm from running on 16 SMs.
// With staged set, the rows also go to the narrow matmul's staged layout
// (n_tok = gridDim.x tokens, hidden / 32 blocks).
__global__ void __launch_bounds__(kGlueThreads) rmsnorm_quant_kernel(const float* __restrict__ x,
                                                                     const float* __restrict__ w, int hidden,
                                                                     float eps, uint8_t* __restrict__ xq,
                                                                     uint32_t* __restrict__ staged) {
  __shared__ float part[kGlueThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const float* xr = x + (size_t)t * hidden;
  const int n = hidden / kGlueThreads;  // hidden % 256 == 0 on this path
  float v[kMaxPerThread];
#pragma unroll
  for (int k = 0; k < kMaxPerThread; ++k)
    if (k < n) v[k] = __ldcg(xr + threadIdx.x + k * kGlueThreads);
  float ss = 0.0f;
#pragma unroll
  for (int k = 0; k < kMaxPerThread; ++k)
    if (k < n) ss = __fmaf_rn(v[k], v[k], ss);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
  if (lane == 0) part[warp] = ss;
  __syncthreads();
  float tot = 0.0f;
#pragma unroll
  for (int i = 0; i < kGlueThreads / 32; ++i) tot = __fadd_rn(tot, part[i]);
  const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)hidden), eps)));
  uint8_t* out = xq + (size_t)t * (hidden / 32) * 34;
  // this CTA's share k0 .. k0 + kper - 1 of the thread's values (kper <=
  // kMaxShare, as the launch sizes the split): picked out of the register
  // array by compile-time indices, so the quantise-and-store code below exists
  // kMaxShare times, not kMaxPerThread times
  const int kper = (n + (int)gridDim.y - 1) / (int)gridDim.y;
  const int k0 = (int)blockIdx.y * kper;
  float mine[kMaxShare];
#pragma unroll
  for (int j = 0; j < kMaxShare; ++j) mine[j] = 0.0f;
#pragma unroll
  for (int k = 0; k < kMaxPerThread; ++k)
#pragma unroll
    for (int j = 0; j < kMaxShare; ++j)
      if (k == k0 + j) mine[j] = v[k];
#pragma unroll
  for (int j = 0; j < kMaxShare; ++j) {
    const int k = k0 + j;
    if (j < kper && k < n) {
      const int e = threadIdx.x + k * kGlueThreads;
      const int b = e >> 5;
      const float y = __fmul_rn(__fmul_rn(mine[j], inv), w[e]);
      if (staged)
        q8_block_store_staged(y, out + (size_t)b * 34, staged, hidden / 32, b, t, (int)gridDim.x, lane);
      else
        q8_block_store(y, out + (size_t)b * 34, lane);
    }
  }
}

// gu: [n_tok][2*ffn] = [gate | up]; out: q8_0 [n_tok][ffn].  One warp per block.
// With staged set, the rows also go to the narrow matmul's staged layout.
__global__ void __launch_bounds__(kGlueThreads) silu_mul_quant_kernel(const float* __restrict__ gu, int ffn,
                                                                      long long n_blocks, uint8_t* __restrict__ xq,
                                                                      uint32_t* __restrict__ staged, int n_tok) {
  pdl_wait();
  pdl_trigger();
  const long long blk = (long long)blockIdx.x * (kGlueThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (blk >= n_blocks) return;
  const int per_row = ffn / 32;
  const long long t = blk / per_row;
  const int i = (int)(blk - t * per_row) * 32 + lane;
  const float g = __ldcg(gu + (size_t)t * 2 * ffn + i);
  const float u = __ldcg(gu + (size_t)t * 2 * ffn + ffn + i);
  const float s = __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
  if (staged)
    q8_block_store_staged(__fmul_rn(s, u), xq + (size_t)blk * 34, staged, per_row, (int)(blk - t * per_row), (int)t,
                          n_tok, lane);
  else
    q8_block_store(__fmul_rn(s, u), xq + (size_t)blk * 34, lane);
}

// h[t][:] = dequantised q8_0 row token[t] of the embedding table.  One warp per block.
// With meta_src set (the captured step reads its per-step metadata straight
// from mapped pinned host memory), the CTAs also copy the n_words metadata
// words to meta_dst for the kernels that follow; tokens then points into
// meta_src too.
__global__ void __launch_bounds__(kGlueThreads) embed_kernel(const uint8_t* __restrict__ table, int hidden,
                                                             const int32_t* __restrict__ tokens, long long n_blocks,
                                                             float* __restrict__ h, const int32_t* meta_src,
                                                             int32_t* meta_dst, int n_words) {
  pdl_wait();
  pdl_trigger();
  if (meta_src)
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_words; i += gridDim.x * blockDim.x)
      meta_dst[i] = meta_src[i];
  const long long blk = (long long)blockIdx.x * (kGlueThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (blk >= n_blocks) return;
  const int per_row = hidden / 32;
  const long long t = blk / per_row;
  const int b = (int)(blk - t * per_row);
  const uint8_t* src = table + ((size_t)tokens[t] * per_row + b) * 34;
  const unsigned short sbits = (unsigned short)(src[0] | (src[1] << 8));
  const float d = __half2float(__ushort_as_half(sbits));
  const int8_t q = (int8_t)src[2 + lane];
  h[(size_t)t * hidden + b * 32 + lane] = __fmul_rn(d, (float)q);
}

// The same gather with the step's metadata words carried in the kernel's own
// parameter block (a captured step rewrites them per replay), so no kernel
// reads host memory: the CTAs copy the n_words words to meta_dst for the
// kernels that follow, and the token ids are its first n_tok words.
template <int N>
__global__ void __launch_bounds__(kGlueThreads) embed_param_kernel(const uint8_t* __restrict__ table, int hidden,
                                                                   long long n_blocks, float* __restrict__ h,
                                                                   const __grid_constant__ StepMetaWords<N> meta,
                                                                   int32_t* meta_dst, int n_words) {
  pdl_wait();
  pdl_trigger();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_words; i += gridDim.x * blockDim.x) meta_dst[i] = meta.w[i];
  const long long blk = (long long)blockIdx.x * (kGlueThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (blk >= n_blocks) return;
  const int per_row = hidden / 32;
  const long long t = blk / per_row;
  const int b = (int)(blk - t * per_row);
  const uint8_t* src = table + ((size_t)meta.w[t] * per_row + b) * 34;
  const unsigned short sbits = (unsigned short)(src[0] | (src[1] << 8));
  const float d = __half2float(__ushort_as_half(sbits));
  const int8_t q = (int8_t)src[2 + lane];
  h[(size_t)t * hidden + b * 32 + lane] = __fmul_rn(d, (float)q);
}

template <int N>
cudaError_t launch_embed_param_n(const uint8_t* table, int hidden, int n_tok, float* h, const int32_t* words,
                                 int n_words, int32_t* meta_dst, cudaStream_t st, EmbedParamNode* node) {
  const long long n_blocks = (long long)n_tok * (hidden / 32);
  const unsigned grid = (unsigned)((n_blocks + 7) / 8);
  if (node) {
    node->func = reinterpret_cast<const void*>(embed_param_kernel<N>);
    node->grid = grid;
    node->block = kGlueThreads;
    node->n_blocks = n_blocks;
    node->capacity = N;
  }
  StepMetaWords<N> m;
  for (int i = 0; i < N; ++i) m.w[i] = i < n_words ? words[i] : 0;
  return launch_kernel(embed_param_kernel<N>, dim3(grid), dim3(kGlueThreads), 0, st, table, hidden, n_blocks, h, m,
                       meta_dst, n_words);
}

}  // namespace

cudaError_t launch_embed_params(const void* table, int hidden, int n_tok, float* h, const int32_t* words, int n_words,
                                int32_t* meta_dst, cudaStream_t st, EmbedParamNode* node) {
  if (n_tok == 0) return cudaSuccess;
  const uint8_t* t8 = static_cast<const uint8_t*>(table);
  if (n_words <= 256) return launch_embed_param_n<256>(t8, hidden, n_tok, h, words, n_words, meta_dst, st, node);
  if (n_words <= 1024) return launch_embed_param_n<1024>(t8, hidden, n_tok, h, words, n_words, meta_dst, st, node);
  if (n_words <= kEmbedParamMaxWords)
    return launch_embed_param_n<kEmbedParamMaxWords>(t8, hidden, n_tok, h, words, n_words, meta_dst, st, node);
  return cudaErrorInvalidValue;
}

cudaError_t launch_rmsnorm_quant(const float* x, const float* w, int n_tok, int hidden, float eps, void* xq,
                                 cudaStream_t st, void* staged) {
  if (n_tok == 0) return cudaSuccess;
  // about two blocks per warp (one block per warp up to 8 tokens, where
  // there are few rows to spread): hidden / 32 blocks over 8 warps per CTA
  const int n = hidden / kGlueThreads;
  int split = n_tok <= 8 ? (hidden / 32 + 7) / 8 : (hidden / 32 + 15) / 16;
  if (split > n) split = n;
  if (split < (n + kMaxShare - 1) / kMaxShare) split = (n + kMaxShare - 1) / kMaxShare;
  if (split < 1) split = 1;
  return launch_kernel(rmsnorm_quant_kernel, dim3(n_tok, split), dim3(kGlueThreads), 0, st, x, w, hidden, eps,
                       static_cast<uint8_t*>(xq), static_cast<uint32_t*>(staged));
}

cudaError_t launch_silu_mul_quant(const float* gu, int n_tok, int ffn, void* xq, cudaStream_t st, void* staged) {
  const long long n_blocks = (long long)n_tok * (ffn / 32);
  if (n_blocks == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((n_blocks + 7) / 8);
  return launch_kernel(silu_mul_quant_kernel, dim3(grid), dim3(kGlueThreads), 0, st, gu, ffn, n_blocks,
                       static_cast<uint8_t*>(xq), static_cast<uint32_t*>(staged), n_tok);
}

cudaError_t launch_embed(const void* table, int hidden, const int32_t* tokens, int n_tok, float* h,
                         const int32_t* meta_src, int32_t* meta_dst, int n_words, cudaStream_t st) {
  const long long n_blocks = (long long)n_tok * (hidden / 32);
  if (n_blocks == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((n_blocks + 7) / 8);
  return launch_kernel(embed_kernel, dim3(grid), dim3(kGlueThreads), 0, st, static_cast<const uint8_t*>(table), hidden,
                       tokens, n_blocks, h, meta_src, meta_dst, n_words);
}

}  // namespace dsbk
