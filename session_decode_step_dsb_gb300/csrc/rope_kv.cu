// Pos-vector RoPE and the batch_index KV write (sm_103a).
//
// RoPE (antirez/ds4 PR #530, the pos-vector RoPE commit): a batched step
// evaluates each token row at its own position, so the kernel takes a position
// per token row instead of pos0 + t.  Rotate-half pairs (i, i + D/2) turn by
// a = pos[t] * theta^(-2i/D).  Positions reach 65535, where a float32 product
// would be off by ~4e-3 rad, so the angle is formed and reduced in float64:
// the per-pair frequency theta^(-2i/D) is a float64 table of the model (built
// on the host from theta and D), a = pos * f is one float64 multiply, and the
// reduction a - 2 pi k, k = rint(a / 2 pi), uses 2 pi split into two doubles
// (Cody and Waite's two-constant reduction) so that the remainder is exact to
// float64 rounding.  sincosf of the reduced float32 angle (|r| <= pi) and the
// float32 rotation follow.  Each token row's arithmetic is independent of
// n_tok, so row t equals an n_tok = 1 launch bitwise.
//
// KV write (quic/efficient-transformers PR #1305, "Objective": the retained
// cache is sized for full_batch_size and the live batch addresses it through
// batch_index; antirez/ds4 PR #530: per-sequence KV append inside the batched
// step): K[batch_index[s]][h][pos[t]][:] = cvt(k[t][h][:]) for t = s*T + j,
// cvt = round to nearest even into fp16 or bf16.  Nothing else is written.
// The decode step uses a fused kernel: RoPE of q and k and the KV write of
// the rotated k and of v in one pass over the token rows.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dsb_kernels.h"
#include "dsb_ptx.cuh"

namespace dsbk {

namespace {

// 2 pi = kTwoPiHi + kTwoPiLo to ~2^-106 (kTwoPiHi is the double nearest 2 pi).
constexpr double kTwoPiHi = 6.283185307179586232;
constexpr double kTwoPiLo = 2.4492935982947064e-16;
constexpr double kInvTwoPi = 0.15915494309189533577;

__device__ __forceinline__ void rope_cs(int pos, double freq, float* c, float* s) {
  const double a = (double)pos * freq;
  const double k = rint(a * kInvTwoPi);
  double r = fma(-k, kTwoPiHi, a);
  r = fma(-k, kTwoPiLo, r);
  sincosf((float)r, s, c);
}

// Heads handled per thread in one pass: every load of a pass is issued before
// any store, so the pass costs one memory round trip instead of one per head.
constexpr int kRopeHeads = 8;
constexpr int kRopeHeadsFew = 4;  // the step's RoPE + KV write up to 8 tokens: more, smaller CTAs
constexpr int kRopeMaxWarps = 16;  // head_dim <= 1024: at most 512 pair threads

// Optional per-head RMS norm before the rotation: for each of the block's
// heads, inv[u] = 1 / sqrt(mean(x^2) + eps) over the head's head_dim values
// (pair i of head u is (x1[u], x2[u]) in thread i; threads past the last
// pair hold zeros).  Sums go through a fixed xor tree per warp and the warps
// in order.  Every thread of the block must call it.
template <int HG = kRopeHeads>
__device__ __forceinline__ void head_inv_rms(const float (&x1)[HG], const float (&x2)[HG], int head_dim, float eps,
                                             float (&inv)[HG]) {
  __shared__ float part[HG][kRopeMaxWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n_warps = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int u = 0; u < HG; ++u) {
    float ss = __fmaf_rn(x2[u], x2[u], __fmul_rn(x1[u], x1[u]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    if (lane == 0) part[u][warp] = ss;
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < HG; ++u) {
    float tot = 0.0f;
    for (int w = 0; w < n_warps; ++w) tot = __fadd_rn(tot, part[u][w]);
    inv[u] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)head_dim), eps)));
  }
}

// grid (n_tok, ceil((Hq + Hkv) / kRopeHeads)), one thread per pair.  Head slot
// hs < Hq is query head hs, otherwise kv head hs - Hq of k.
__global__ void rope_posvec_kernel(float* __restrict__ q, long long q_stride, int n_q_heads, float* __restrict__ k,
                                   long long k_stride, int n_kv_heads, int head_dim, const int32_t* __restrict__ pos,
                                   const __grid_constant__ RopeFreqs freqs, const float* __restrict__ q_norm,
                                   const float* __restrict__ k_norm, float eps) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int half = head_dim >> 1;
  const int i = threadIdx.x;
  const bool pair = i < half;
  float c = 1.0f, s = 0.0f;
  if (pair) {
    rope_cs(pos[t], freqs.f[i], &c, &s);
    c = __fmul_rn(c, freqs.mscale);
    s = __fmul_rn(s, freqs.mscale);
  }
  const int h0 = blockIdx.y * kRopeHeads;
  float* ptr[kRopeHeads];
  float x1[kRopeHeads], x2[kRopeHeads];
#pragma unroll
  for (int u = 0; u < kRopeHeads; ++u) {
    const int hs = h0 + u;
    ptr[u] = nullptr;
    if (hs < n_q_heads)
      ptr[u] = q + (size_t)t * q_stride + (size_t)hs * head_dim;
    else if (k && hs < n_q_heads + n_kv_heads)
      ptr[u] = k + (size_t)t * k_stride + (size_t)(hs - n_q_heads) * head_dim;
    x1[u] = x2[u] = 0.0f;
    if (ptr[u] && pair) {
      x1[u] = __ldcg(ptr[u] + i);
      x2[u] = __ldcg(ptr[u] + i + half);
    }
  }
  if (q_norm || k_norm) {
    float inv[kRopeHeads];
    head_inv_rms(x1, x2, head_dim, eps, inv);
#pragma unroll
    for (int u = 0; u < kRopeHeads; ++u) {
      const float* w = h0 + u < n_q_heads ? q_norm : k_norm;
      if (w && pair) {
        x1[u] = __fmul_rn(__fmul_rn(x1[u], inv[u]), w[i]);
        x2[u] = __fmul_rn(__fmul_rn(x2[u], inv[u]), w[i + half]);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kRopeHeads; ++u) {
    if (ptr[u] && pair) {
      ptr[u][i] = __fmaf_rn(x1[u], c, __fmul_rn(-x2[u], s));
      ptr[u][i + half] = __fmaf_rn(x1[u], s, __fmul_rn(x2[u], c));
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
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x, h = blockIdx.y;
  const int slot = batch_index[t / tokens_per_seq];
  const int p = pos[t];
  const size_t dst = (((size_t)slot * n_kv_heads + h) * ctx + p) * head_dim;
  const size_t src = (size_t)t * kv_stride + (size_t)h * head_dim;
  for (int d = threadIdx.x; d < head_dim; d += blockDim.x) {
    kc[dst + d] = cvt_rn<T>(__ldcg(k + src + d));
    vc[dst + d] = cvt_rn<T>(__ldcg(v + src + d));
  }
}

// Paged KV write, grid (n_tok, n_kv_heads), one thread per element of a head row.
template <typename T>
__global__ void kv_scatter_paged_kernel(T* __restrict__ kp, T* __restrict__ vp, int n_kv_heads, int head_dim,
                                        const PagedView pv, int tokens_per_seq, const int32_t* __restrict__ pos,
                                        const float* __restrict__ k, const float* __restrict__ v,
                                        long long kv_stride) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x, h = blockIdx.y;
  const int s = t / tokens_per_seq;
  const int p = pos[t];
  int i = p >> 7;  // 128-key pages
  if (pv.window[s] > 0) i %= pv.n_blocks[s];
  const int page = pv.block_table[(size_t)s * pv.max_blocks + i];
  const size_t dst = (((size_t)page * n_kv_heads + h) * 128 + (p & 127)) * head_dim;
  const size_t src = (size_t)t * kv_stride + (size_t)h * head_dim;
  for (int d = threadIdx.x; d < head_dim; d += blockDim.x) {
    kp[dst + d] = cvt_rn<T>(__ldcg(k + src + d));
    vp[dst + d] = cvt_rn<T>(__ldcg(v + src + d));
  }
}

// The step's fused pass, grid (n_tok, ceil((Hq + Hkv) / HG)), one
// thread per pair.  Head slot hs < Hq rotates query head hs in place; slot
// Hq + g rotates kv head g of k and writes it, and kv head g of v, into the
// cache slot of the token's sequence.  Loads of a pass precede its stores.
template <typename T, int HG>
__global__ void rope_kv_write_kernel(float* __restrict__ qkv, long long stride, int n_q_heads, int n_kv_heads,
                                     int head_dim, const int32_t* __restrict__ pos,
                                     const int32_t* __restrict__ batch_index, int tokens_per_seq, T* __restrict__ kc,
                                     T* __restrict__ vc, int ctx, const __grid_constant__ RopeFreqs freqs,
                                     const float* __restrict__ q_norm, const float* __restrict__ k_norm, float eps,
                                     const PagedView pv) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int half = head_dim >> 1;
  const int i = threadIdx.x;
  const bool pair = i < half;
  const int p = pos[t];
  float c = 1.0f, s = 0.0f;
  if (pair) {
    rope_cs(p, freqs.f[i], &c, &s);
    c = __fmul_rn(c, freqs.mscale);
    s = __fmul_rn(s, freqs.mscale);
  }
  float* row = qkv + (size_t)t * stride;
  // the cache row of (token t, kv head g) is kv_row + g * kv_head_stride: the
  // token's slot at position p, or (paged view) row p mod 128 of the page its
  // block table names (the block index modulo the block count for a ring)
  const int sq = t / tokens_per_seq;
  size_t kv_row, kv_head_stride;
  if (pv.block_table) {
    int bi = p >> 7;
    if (pv.window[sq] > 0) bi %= pv.n_blocks[sq];
    const int page = pv.block_table[(size_t)sq * pv.max_blocks + bi];
    kv_row = ((size_t)page * n_kv_heads * 128 + (p & 127)) * head_dim;
    kv_head_stride = (size_t)128 * head_dim;
  } else {
    kv_row = ((size_t)batch_index[sq] * n_kv_heads * ctx + p) * head_dim;
    kv_head_stride = (size_t)ctx * head_dim;
  }
  const int h0 = blockIdx.y * HG;
  float x1[HG], x2[HG], v1[HG], v2[HG];
#pragma unroll
  for (int u = 0; u < HG; ++u) {
    const int hs = h0 + u;
    x1[u] = x2[u] = v1[u] = v2[u] = 0.0f;
    if (hs < n_q_heads + n_kv_heads && pair) {
      const float* src = row + (size_t)hs * head_dim;  // q heads, then k heads
      x1[u] = __ldcg(src + i);
      x2[u] = __ldcg(src + i + half);
      if (hs >= n_q_heads) {
        const float* vsrc = row + (size_t)(n_q_heads + n_kv_heads + hs - n_q_heads) * head_dim;
        v1[u] = __ldcg(vsrc + i);
        v2[u] = __ldcg(vsrc + i + half);
      }
    }
  }
  if (q_norm || k_norm) {
    float inv[HG];
    head_inv_rms<HG>(x1, x2, head_dim, eps, inv);
#pragma unroll
    for (int u = 0; u < HG; ++u) {
      const float* w = h0 + u < n_q_heads ? q_norm : k_norm;
      if (w && pair) {
        x1[u] = __fmul_rn(__fmul_rn(x1[u], inv[u]), w[i]);
        x2[u] = __fmul_rn(__fmul_rn(x2[u], inv[u]), w[i + half]);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < HG; ++u) {
    const int hs = h0 + u;
    if (hs >= n_q_heads + n_kv_heads || !pair) continue;
    const float y1 = __fmaf_rn(x1[u], c, __fmul_rn(-x2[u], s));
    const float y2 = __fmaf_rn(x1[u], s, __fmul_rn(x2[u], c));
    if (hs < n_q_heads) {
      float* dst = row + (size_t)hs * head_dim;
      dst[i] = y1;
      dst[i + half] = y2;
    } else {
      const int g = hs - n_q_heads;
      const size_t dst = kv_row + (size_t)g * kv_head_stride;
      kc[dst + i] = cvt_rn<T>(y1);
      kc[dst + i + half] = cvt_rn<T>(y2);
      vc[dst + i] = cvt_rn<T>(v1[u]);
      vc[dst + i + half] = cvt_rn<T>(v2[u]);
    }
  }
}

}  // namespace

cudaError_t launch_rope_posvec(float* q, long long q_stride, int n_q_heads, float* k, long long k_stride,
                               int n_kv_heads, int head_dim, int n_tok, const int32_t* pos_dev,
                               const RopeFreqs& freqs, cudaStream_t st, const float* q_norm, const float* k_norm,
                               float eps) {
  if (n_tok == 0) return cudaSuccess;
  const int half = head_dim / 2;
  const int threads = ((half + 31) / 32) * 32;
  const int groups = (n_q_heads + (k ? n_kv_heads : 0) + kRopeHeads - 1) / kRopeHeads;
  return launch_kernel(rope_posvec_kernel, dim3(n_tok, groups), dim3(threads), 0, st, q, q_stride, n_q_heads, k,
                       k_stride, n_kv_heads, head_dim, pos_dev, freqs, q_norm, k_norm, eps);
}

cudaError_t launch_kv_scatter(void* kc, void* vc, int dtype, int n_kv_heads, int ctx, int head_dim,
                              const int32_t* batch_index_dev, int tokens_per_seq, const int32_t* pos_dev, int n_tok,
                              const float* k, const float* v, long long kv_stride, cudaStream_t st) {
  if (n_tok == 0) return cudaSuccess;
  const dim3 grid((unsigned)n_tok, (unsigned)n_kv_heads);
  const int threads = head_dim < 256 ? ((head_dim + 31) / 32) * 32 : 256;
  if (dtype == 0)
    return launch_kernel(kv_scatter_kernel<__half>, grid, dim3(threads), 0, st, static_cast<__half*>(kc),
                         static_cast<__half*>(vc), n_kv_heads, ctx, head_dim, batch_index_dev, tokens_per_seq, pos_dev,
                         k, v, kv_stride);
  return launch_kernel(kv_scatter_kernel<__nv_bfloat16>, grid, dim3(threads), 0, st, static_cast<__nv_bfloat16*>(kc),
                       static_cast<__nv_bfloat16*>(vc), n_kv_heads, ctx, head_dim, batch_index_dev, tokens_per_seq,
                       pos_dev, k, v, kv_stride);
}

cudaError_t launch_kv_scatter_paged(void* kp, void* vp, int dtype, int n_kv_heads, int head_dim, PagedView pv,
                                    int tokens_per_seq, const int32_t* pos_dev, int n_tok, const float* k,
                                    const float* v, long long kv_stride, cudaStream_t st) {
  if (n_tok == 0) return cudaSuccess;
  const dim3 grid((unsigned)n_tok, (unsigned)n_kv_heads);
  const int threads = head_dim < 256 ? ((head_dim + 31) / 32) * 32 : 256;
  if (dtype == 0)
    return launch_kernel(kv_scatter_paged_kernel<__half>, grid, dim3(threads), 0, st, static_cast<__half*>(kp),
                         static_cast<__half*>(vp), n_kv_heads, head_dim, pv, tokens_per_seq, pos_dev, k, v, kv_stride);
  return launch_kernel(kv_scatter_paged_kernel<__nv_bfloat16>, grid, dim3(threads), 0, st,
                       static_cast<__nv_bfloat16*>(kp), static_cast<__nv_bfloat16*>(vp), n_kv_heads, head_dim, pv,
                       tokens_per_seq, pos_dev, k, v, kv_stride);
}

cudaError_t launch_rope_kv_write(float* qkv, long long stride, int n_q_heads, int n_kv_heads, int head_dim,
                                 const int32_t* pos_dev, const int32_t* batch_index_dev, int tokens_per_seq,
                                 int n_tok, void* kc, void* vc, int dtype, int ctx, const RopeFreqs& freqs,
                                 cudaStream_t st, const float* q_norm, const float* k_norm, float eps,
                                 PagedView pv) {
  if (n_tok == 0) return cudaSuccess;
  const int threads = ((head_dim / 2 + 31) / 32) * 32;
  // up to 8 tokens, groups of 4 heads (more CTAs for the few tokens); else 8
  const bool few = n_tok <= 8;
  const int hg = few ? kRopeHeadsFew : kRopeHeads;
  const dim3 grid((unsigned)n_tok, (unsigned)((n_q_heads + n_kv_heads + hg - 1) / hg));
  if (dtype == 0)
    return launch_kernel(few ? rope_kv_write_kernel<__half, kRopeHeadsFew> : rope_kv_write_kernel<__half, kRopeHeads>,
                         grid, dim3(threads), 0, st, qkv, stride, n_q_heads, n_kv_heads, head_dim, pos_dev,
                         batch_index_dev, tokens_per_seq, static_cast<__half*>(kc), static_cast<__half*>(vc), ctx,
                         freqs, q_norm, k_norm, eps, pv);
  return launch_kernel(
      few ? rope_kv_write_kernel<__nv_bfloat16, kRopeHeadsFew> : rope_kv_write_kernel<__nv_bfloat16, kRopeHeads>,
      grid, dim3(threads), 0, st, qkv, stride, n_q_heads, n_kv_heads, head_dim, pos_dev, batch_index_dev,
      tokens_per_seq, static_cast<__nv_bfloat16*>(kc), static_cast<__nv_bfloat16*>(vc), ctx, freqs, q_norm, k_norm,
      eps, pv);
}

// YaRN (Peng et al. 2023, "YaRN: Efficient Context Window Extension of Large
// Language Models", sections 3.2 "NTK-by-parts" and 3.3): pair i turns
// r_i = L f_i / (2 pi) times over the original context L.  Pairs that turn at
// least beta_fast times keep f_i, pairs that turn at most beta_slow times take
// f_i / s, and the pair indices in between blend the two linearly; the index
// where r = b is D ln(L / (2 pi b)) / (2 ln theta), rounded outward.  The
// attention temperature 0.1 ln s + 1 scales q and k through the rotation.
void rope_freqs(double theta, int head_dim, RopeFreqs* out, double yarn_factor, int yarn_orig_ctx,
                double yarn_beta_fast, double yarn_beta_slow) {
  const int half = head_dim / 2 < kRopeMaxPairs ? head_dim / 2 : kRopeMaxPairs;
  const bool yarn = yarn_factor > 1.0;
  double low = 0.0, span = 1.0;
  if (yarn) {
    const double log_theta2 = 2.0 * log(theta);
    const double two_pi = 6.283185307179586;
    const double c_fast = head_dim * log(yarn_orig_ctx / (two_pi * yarn_beta_fast)) / log_theta2;
    const double c_slow = head_dim * log(yarn_orig_ctx / (two_pi * yarn_beta_slow)) / log_theta2;
    low = floor(c_fast) > 0.0 ? floor(c_fast) : 0.0;
    const double high = ceil(c_slow) < head_dim - 1 ? ceil(c_slow) : (double)(head_dim - 1);
    span = high - low > 0.001 ? high - low : 0.001;
  }
  for (int i = 0; i < half; ++i) {
    const double f = pow(theta, -2.0 * i / head_dim);
    if (!yarn) {
      out->f[i] = f;
      continue;
    }
    double ramp = (i - low) / span;
    ramp = ramp < 0.0 ? 0.0 : (ramp > 1.0 ? 1.0 : ramp);
    out->f[i] = f * (1.0 - ramp) + (f / yarn_factor) * ramp;
  }
  out->mscale = yarn ? (float)(0.1 * log(yarn_factor) + 1.0) : 1.0f;
}

}  // namespace dsbk
