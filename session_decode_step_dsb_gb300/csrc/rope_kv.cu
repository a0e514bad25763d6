// Pos-vector RoPE and the batch_index KV write (sm_103a).
//
// RoPE (antirez/ds4 PR #530, the pos-vector RoPE commit): a batched step
// evaluates each token row at its own position, so the kernel takes a position
// per token row instead of pos0 + t.  Rotate-half pairs (i, i + D/2) turn by
// pos[t] * theta^(-2i/D).  The angle, its reduction and its sine/cosine are
// evaluated in float64 (positions reach 65535 and a float32 product would be
// off by ~4e-3 rad there); the rotation itself is float32.  One CTA per token
// row, one thread per pair, looping over the heads of q and k, so each row's
// arithmetic is independent of n_tok (row t equals an n_tok = 1 launch).
//
// KV write (quic/efficient-transformers PR #1305, "Objective": the retained
// cache is sized for full_batch_size and the live batch addresses it through
// batch_index; antirez/ds4 PR #530: per-sequence KV append inside the batched
// step): K[batch_index[s]][h][pos[t]][:] = cvt(k[t][h][:]) for t = s*T + j,
// cvt = round to nearest even into fp16 or bf16.  Nothing else is written.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dsb_kernels.h"

namespace dsbk {

namespace {

__global__ void rope_posvec_kernel(float* __restrict__ q, long long q_stride, int n_q_heads, float* __restrict__ k,
                                   long long k_stride, int n_kv_heads, int head_dim, const int32_t* __restrict__ pos,
                                   double theta) {
  const int t = blockIdx.x;
  const int half = head_dim >> 1;
  const int i = threadIdx.x;
  if (i >= half) return;
  const double inv_freq = pow(theta, -2.0 * (double)i / (double)head_dim);
  const double ang = (double)pos[t] * inv_freq;
  double sd, cd;
  sincos(ang, &sd, &cd);
  const float s = (float)sd, c = (float)cd;
  float* qt = q + (size_t)t * q_stride;
  for (int h = 0; h < n_q_heads; ++h) {
    float* x = qt + (size_t)h * head_dim;
    const float x1 = x[i], x2 = x[i + half];
    x[i] = __fmaf_rn(x1, c, __fmul_rn(-x2, s));
    x[i + half] = __fmaf_rn(x1, s, __fmul_rn(x2, c));
  }
  if (k) {
    float* kt = k + (size_t)t * k_stride;
    for (int h = 0; h < n_kv_heads; ++h) {
      float* x = kt + (size_t)h * head_dim;
      const float x1 = x[i], x2 = x[i + half];
      x[i] = __fmaf_rn(x1, c, __fmul_rn(-x2, s));
      x[i + half] = __fmaf_rn(x1, s, __fmul_rn(x2, c));
    }
  }
}

template <typename T>
__device__ __forceinline__ T cvt_rn(float x);
template <>
__device__ __forceinline__ __half cvt_rn<__half>(float x) {
  return __float2half_rn(x);
}
template <>
__device__ __forceinline__ __nv_bfloat16 cvt_rn<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// grid (n_tok, n_kv_heads), one thread per element of a head row.
template <typename T>
__global__ void kv_scatter_kernel(T* __restrict__ kc, T* __restrict__ vc, int n_kv_heads, int ctx, int head_dim,
                                  const int32_t* __restrict__ batch_index, int tokens_per_seq,
                                  const int32_t* __restrict__ pos, const float* __restrict__ k,
                                  const float* __restrict__ v, long long kv_stride) {
  const int t = blockIdx.x, h = blockIdx.y;
  const int slot = batch_index[t / tokens_per_seq];
  const int p = pos[t];
  const size_t dst = (((size_t)slot * n_kv_heads + h) * ctx + p) * head_dim;
  const size_t src = (size_t)t * kv_stride + (size_t)h * head_dim;
  for (int d = threadIdx.x; d < head_dim; d += blockDim.x) {
    kc[dst + d] = cvt_rn<T>(k[src + d]);
    vc[dst + d] = cvt_rn<T>(v[src + d]);
  }
}

}  // namespace

cudaError_t launch_rope_posvec(float* q, long long q_stride, int n_q_heads, float* k, long long k_stride,
                               int n_kv_heads, int head_dim, int n_tok, const int32_t* pos_dev, float theta,
                               cudaStream_t st) {
  if (n_tok == 0) return cudaSuccess;
  const int half = head_dim / 2;
  const int threads = ((half + 31) / 32) * 32;
  if (dry_run()) return cudaSuccess;
  rope_posvec_kernel<<<n_tok, threads, 0, st>>>(q, q_stride, n_q_heads, k, k_stride, n_kv_heads, head_dim, pos_dev,
                                                 (double)theta);
  return cudaGetLastError();
}

cudaError_t launch_kv_scatter(void* kc, void* vc, int dtype, int n_kv_heads, int ctx, int head_dim,
                              const int32_t* batch_index_dev, int tokens_per_seq, const int32_t* pos_dev, int n_tok,
                              const float* k, const float* v, long long kv_stride, cudaStream_t st) {
  if (n_tok == 0) return cudaSuccess;
  const dim3 grid((unsigned)n_tok, (unsigned)n_kv_heads);
  const int threads = head_dim < 256 ? ((head_dim + 31) / 32) * 32 : 256;
  if (dry_run()) return cudaSuccess;
  if (dtype == 0)
    kv_scatter_kernel<__half><<<grid, threads, 0, st>>>(static_cast<__half*>(kc), static_cast<__half*>(vc),
                                                         n_kv_heads, ctx, head_dim, batch_index_dev, tokens_per_seq,
                                                         pos_dev, k, v, kv_stride);
  else
    kv_scatter_kernel<__nv_bfloat16><<<grid, threads, 0, st>>>(static_cast<__nv_bfloat16*>(kc),
                                                                static_cast<__nv_bfloat16*>(vc), n_kv_heads, ctx,
                                                                head_dim, batch_index_dev, tokens_per_seq, pos_dev,
                                                                k, v, kv_stride);
  return cudaGetLastError();
}

}  // namespace dsbk
