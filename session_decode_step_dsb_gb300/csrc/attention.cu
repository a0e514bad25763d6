// Multi-sequence GQA decode attention, split-K (flash-decode), sm_103a.
//
// What it computes (antirez/ds4 PR #530, "Batched decode: co-decode N live
// sessions in one GPU pass", the multi-sequence decode attention commit: one
// launch serves several sequences, each reading its own query rows and its own
// cache and writing its own output rows; hw-native-sys/pypto-lib PR #841: the
// live batch comes from the seq_lens descriptor).  For sequence s (cache slot
// batch_index[s], seq_lens[s] keys after this step's writes), draft token j of
// T (quic/efficient-transformers PR #1305, K+1 tokens per sequence) and query
// head h (kv head g = h / G):
//     score_k = q . K_k / sqrt(D)  for k <= seq_lens[s] - T + j
//     out     = sum_k softmax(score)_k V_k
//
// GB300 design.  The ds4 page's kernel keeps every score of a sequence in one
// shared buffer and gives up past ~31k compressed rows ("Known limitation");
// here the keys of each (sequence, kv head) are cut into DSB_ATTN_CHUNK = 128
// key chunks, so long contexts and b = 1 both fill the 152 SMs:
//  * partial kernel, one CTA per (sequence, chunk, kv head): the V chunk is
//    brought into shared memory by one 1-D TMA bulk copy (contiguous in the
//    [F][Hkv][C][D] cache) while the CTA computes scores; thread k owns key k,
//    holds its K row in registers (16-byte read-only loads) and dots it against
//    the G*T query rows of the GQA group, which are read from shared memory by
//    broadcast.  Every K/V byte is read once for all G*T query rows.  Per row
//    it writes (max, sum of exp, sum of exp * V) for the chunk.
//  * merge kernel, one warp per (token row, head): rescales the chunk partials
//    by exp(m_c - max_c m_c) and adds them in chunk order.
// No atomics and no inter-CTA waits; the chunking depends only on each
// sequence's own length, so a sequence's rows are bitwise equal whether it runs
// alone or inside a batch.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dsb_kernels.h"
#include "dsb_ptx.cuh"
#include "dsb_q8.cuh"

namespace dsbk {

namespace {

constexpr int kCh = 128;  // keys per chunk (DSB_ATTN_CHUNK)
constexpr int kThreads = 128;
// Query rows handled together in the score and P.V loops: the widest row
// group is 8, and each launch takes the narrowest power of two >= G*T, so a
// one-row item (MHA, T = 1) issues no predicated-off work for absent rows.
constexpr int kMaxRowGroup = 8;

__device__ unsigned int g_err_attention = 0;

template <typename T>
struct Cvt;
template <>
struct Cvt<__half> {
  static __device__ __forceinline__ float2 two(uint32_t w) { return __half22float2(*reinterpret_cast<__half2*>(&w)); }
};
template <>
struct Cvt<__nv_bfloat16> {
  static __device__ __forceinline__ float2 two(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w));
  }
};

template <int D, typename T, int kRowGroup>
__global__ void __launch_bounds__(kThreads) attention_partial_kernel(
    const float* __restrict__ q, long long q_stride, int n_q_heads, const T* kc, const T* __restrict__ vc,
    int n_kv_heads,
    int ctx, const int32_t* __restrict__ batch_index, const int32_t* __restrict__ seq_lens,
    const int32_t* __restrict__ chunk_off, int n_seq, int tps, int max_chunks, float scale,
    float* __restrict__ partials, const PagedView pv) {
  constexpr int NPAIR = D / 2;
  constexpr int NPART = kThreads / NPAIR;
  constexpr int KPP = kCh / NPART;
  extern __shared__ __align__(128) uint8_t smem[];
  const int G = n_q_heads / n_kv_heads, R = G * tps;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();  // q and the cache rows of this step come from the previous kernels
  pdl_trigger();

  T* Vs = reinterpret_cast<T*>(smem);                                        // [kCh][D]
  float* qs = reinterpret_cast<float*>(smem + (size_t)kCh * D * sizeof(T));  // [R][D]
  float* ps = qs + (size_t)R * D;                                            // [R][kCh]
  float* ms = ps + (size_t)R * kCh;                                          // [R]
  float* ls = ms + R;                                                        // [R]
  float* red = ls + R;                                                       // [NPART-1][kRowGroup][D]
  uint64_t* bar = reinterpret_cast<uint64_t*>(red + (NPART - 1) * kRowGroup * D);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }

  // Persistent loop over work items (chunk, kv head); the item count comes
  // from the device metadata, so a captured launch serves any seq_lens.
  const int total_items = chunk_off[n_seq] * n_kv_heads;
  uint32_t phase = 0;
  for (int item = blockIdx.x; item < total_items; item += gridDim.x, phase ^= 1u) {
  const int w = item / n_kv_heads, g = item - w * n_kv_heads;
  int lo = 0, hi = n_seq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (chunk_off[mid] <= w)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int s = lo, c_rel = w - chunk_off[s];  // c_rel: this sequence's chunk, counted from its first
  const int L = seq_lens[s];
  // Paged view: chunk c lives in one page (128 keys), found through the
  // block table (modulo the block count for a ring); a window hides keys
  // older than pos - W + 1, so the first chunks of a long ring are skipped.
  const int W = pv.block_table ? pv.window[s] : 0;
  const int c = (W > 0 ? max(0, L - tps + 1 - W) / kCh : 0) + c_rel;
  const int key0 = c * kCh;
  const int nkeys = min(kCh, L - key0);
  size_t chunk_row0;  // cache row of key key0 (rows of a chunk are consecutive)
  if (pv.block_table) {
    const int nb = pv.n_blocks[s];
    const int page = pv.block_table[(size_t)s * pv.max_blocks + (W > 0 ? c % nb : c)];
    chunk_row0 = ((size_t)page * n_kv_heads + g) * kCh;
  } else {
    chunk_row0 = ((size_t)batch_index[s] * n_kv_heads + g) * (size_t)ctx + key0;
  }
  __syncthreads();  // the previous item is done with every shared buffer
  if (tid == 0) {
    const uint32_t bytes = (uint32_t)nkeys * D * sizeof(T);
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(Vs, vc + chunk_row0 * D, bytes, bar);
  }
  // Thread tid owns key key0 + tid: its K row goes into registers first, so
  // that the K loads and the q staging below are in flight together.
  uint4 kreg[D / 8];
  if (tid < nkeys) {
    const uint4* kp = reinterpret_cast<const uint4*>(kc + (chunk_row0 + tid) * D);
#pragma unroll
    for (int cc = 0; cc < D / 8; ++cc) kreg[cc] = ld_v4(kp + cc);  // this step's rows were written by the previous kernel
  } else {
#pragma unroll
    for (int cc = 0; cc < D / 8; ++cc) kreg[cc] = make_uint4(0, 0, 0, 0);
  }
  for (int idx = tid; idx < R * D; idx += kThreads) {
    const int r = idx / D, d = idx - r * D;
    const int j = r / G, gi = r - j * G;
    qs[idx] = __ldcg(q + (size_t)(s * tps + j) * q_stride + (size_t)(g * G + gi) * D + d);
  }
  __syncthreads();

  // ---- scores
  {
    for (int r0 = 0; r0 < R; r0 += kRowGroup) {
      float dot[kRowGroup];
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r) dot[r] = 0.0f;
#pragma unroll
      for (int cc = 0; cc < D / 8; ++cc) {
        float kf[8];
        const float2 k01 = Cvt<T>::two(kreg[cc].x), k23 = Cvt<T>::two(kreg[cc].y);
        const float2 k45 = Cvt<T>::two(kreg[cc].z), k67 = Cvt<T>::two(kreg[cc].w);
        kf[0] = k01.x; kf[1] = k01.y; kf[2] = k23.x; kf[3] = k23.y;
        kf[4] = k45.x; kf[5] = k45.y; kf[6] = k67.x; kf[7] = k67.y;
#pragma unroll
        for (int r = 0; r < kRowGroup; ++r) {
          if (r0 + r < R) {
            const float4 qa = *reinterpret_cast<const float4*>(qs + (size_t)(r0 + r) * D + cc * 8);
            const float4 qb = *reinterpret_cast<const float4*>(qs + (size_t)(r0 + r) * D + cc * 8 + 4);
            float a = dot[r];
            a = __fmaf_rn(qa.x, kf[0], a); a = __fmaf_rn(qa.y, kf[1], a);
            a = __fmaf_rn(qa.z, kf[2], a); a = __fmaf_rn(qa.w, kf[3], a);
            a = __fmaf_rn(qb.x, kf[4], a); a = __fmaf_rn(qb.y, kf[5], a);
            a = __fmaf_rn(qb.z, kf[6], a); a = __fmaf_rn(qb.w, kf[7], a);
            dot[r] = a;
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r) {
        if (r0 + r < R) {
          const int j = (r0 + r) / G;
          const int vis = L - tps + j + 1;          // keys before vis are visible to draft token j ...
          const int vlo = W > 0 ? vis - W : 0;      // ... from vlo on under a window
          const int key = key0 + tid;
          ps[(size_t)(r0 + r) * kCh + tid] = (key < vis && key >= vlo) ? __fmul_rn(dot[r], scale) : -INFINITY;
        }
      }
    }
  }
  __syncthreads();

  // ---- chunk softmax statistics, one warp per row
  for (int r = warp; r < R; r += kThreads / 32) {
    float v[kCh / 32];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kCh / 32; ++i) {
      v[i] = ps[(size_t)r * kCh + lane + 32 * i];
      m = fmaxf(m, v[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.0f;
#pragma unroll
    for (int i = 0; i < kCh / 32; ++i) {
      const float p = (m == -INFINITY) ? 0.0f : expf(v[i] - m);
      ps[(size_t)r * kCh + lane + 32 * i] = p;
      l = __fadd_rn(l, p);
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) l = __fadd_rn(l, __shfl_xor_sync(0xffffffffu, l, o));
    if (lane == 0) {
      ms[r] = m;
      ls[r] = l;
    }
  }
  const bool ok = mbar_wait(bar, phase);
  if (!ok) g_err_attention = 1u;
  __syncthreads();

  // ---- P V: thread = (pair of dims, key part); parts added in order
  const int pr = tid % NPAIR, part = tid / NPAIR;
  for (int r0 = 0; r0 < R; r0 += kRowGroup) {
    float a0[kRowGroup], a1[kRowGroup];
#pragma unroll
    for (int r = 0; r < kRowGroup; ++r) a0[r] = a1[r] = 0.0f;
    for (int kk = 0; kk < KPP; ++kk) {
      const int key = part * KPP + kk;
      if (key < nkeys) {
        const float2 vf = Cvt<T>::two(*reinterpret_cast<const uint32_t*>(Vs + (size_t)key * D + 2 * pr));
#pragma unroll
        for (int r = 0; r < kRowGroup; ++r) {
          if (r0 + r < R) {
            const float p = ps[(size_t)(r0 + r) * kCh + key];
            a0[r] = __fmaf_rn(p, vf.x, a0[r]);
            a1[r] = __fmaf_rn(p, vf.y, a1[r]);
          }
        }
      }
    }
    if (part > 0) {
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r) {
        red[((part - 1) * kRowGroup + r) * D + 2 * pr] = a0[r];
        red[((part - 1) * kRowGroup + r) * D + 2 * pr + 1] = a1[r];
      }
    }
    __syncthreads();
    if (part == 0) {
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r) {
        if (r0 + r < R) {
          float x0 = a0[r], x1 = a1[r];
#pragma unroll
          for (int pp = 1; pp < NPART; ++pp) {
            x0 = __fadd_rn(x0, red[((pp - 1) * kRowGroup + r) * D + 2 * pr]);
            x1 = __fadd_rn(x1, red[((pp - 1) * kRowGroup + r) * D + 2 * pr + 1]);
          }
          const int j = (r0 + r) / G, gi = (r0 + r) - j * G;
          const int t = s * tps + j, h = g * G + gi;
          float* dst = partials + (((size_t)t * n_q_heads + h) * max_chunks + c_rel) * (D + 2);
          dst[2 + 2 * pr] = x0;
          dst[3 + 2 * pr] = x1;
          if (pr == 0) {
            dst[0] = ms[r0 + r];
            dst[1] = ls[r0 + r];
          }
        }
      }
    }
    __syncthreads();
  }
  }  // work items
}

// One warp per (token row, query head).  Lanes first take the chunks 32 at a
// time (max of m_c, then w_c = exp(m_c - M) and the partial sum of w_c l_c);
// the sums over lanes use a fixed xor tree; then the warp walks the chunks in
// order, lane d accumulating w_c * acc_c[d].  With QOUT the normalised row is
// q8_0-quantised (D / 32 blocks per head) straight into xq.
template <int D, bool QOUT>
__global__ void __launch_bounds__(128) attention_merge_kernel(const float* __restrict__ partials, int n_q_heads,
                                                              int tps, const int32_t* __restrict__ chunk_off,
                                                              int max_chunks, int n_tok, float* __restrict__ out,
                                                              uint8_t* __restrict__ xq) {
  pdl_wait();
  pdl_trigger();
  const int wg = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wg >= n_tok * n_q_heads) return;
  const int t = wg / n_q_heads, h = wg - t * n_q_heads;
  const int s = t / tps;
  // every chunk of the sequence; those that hide all of this row's keys hold
  // max = -inf and add exactly nothing
  const int nch = chunk_off[s + 1] - chunk_off[s];
  const float* base = partials + ((size_t)t * n_q_heads + h) * max_chunks * (D + 2);
  float M = -INFINITY;
  for (int c = lane; c < nch; c += 32) M = fmaxf(M, __ldcg(base + (size_t)c * (D + 2)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float lsum = 0.0f;
  float acc[D / 32];
#pragma unroll
  for (int e = 0; e < D / 32; ++e) acc[e] = 0.0f;
  for (int c0 = 0; c0 < nch; c0 += 32) {
    float wl = 0.0f;
    if (c0 + lane < nch) {
      const float* pc = base + (size_t)(c0 + lane) * (D + 2);
      const float mc = __ldcg(pc);
      wl = (mc == -INFINITY) ? 0.0f : expf(mc - M);
      lsum = __fmaf_rn(wl, __ldcg(pc + 1), lsum);
    }
    const int n = min(32, nch - c0);
#pragma unroll 4
    for (int cc = 0; cc < n; ++cc) {
      const float wc = __shfl_sync(0xffffffffu, wl, cc);
      const float* pc = base + (size_t)(c0 + cc) * (D + 2) + 2;
#pragma unroll
      for (int e = 0; e < D / 32; ++e) acc[e] = __fmaf_rn(wc, __ldcg(pc + lane + 32 * e), acc[e]);
    }
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) lsum = __fadd_rn(lsum, __shfl_xor_sync(0xffffffffu, lsum, o));
  if constexpr (QOUT) {
    uint8_t* dst = xq + ((size_t)t * n_q_heads + h) * (D / 32) * 34;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) q8_block_store(__fdiv_rn(acc[e], lsum), dst + (size_t)e * 34, lane);
  } else {
    float* o = out + ((size_t)t * n_q_heads + h) * D;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) o[lane + 32 * e] = __fdiv_rn(acc[e], lsum);
  }
}

template <int D, typename T, int kRowGroup>
size_t partial_smem(int R) {
  constexpr int NPART = kThreads / (D / 2);
  return (size_t)kCh * D * sizeof(T) + (size_t)R * D * 4 + (size_t)R * kCh * 4 + (size_t)2 * R * 4 +
         (size_t)(NPART - 1) * kRowGroup * D * 4 + 16;
}

template <int D, typename T, int kRowGroup>
cudaError_t launch_rg(const float* q, long long q_stride, int n_q_heads, const void* kc, const void* vc,
                         int n_kv_heads, int ctx,
                         MetaView meta, int n_seq, int tps, long long max_items, int max_chunks, float* partials,
                         float* out, void* xq_out, PagedView pv, cudaStream_t st) {
  const int R = (n_q_heads / n_kv_heads) * tps;
  const size_t smem = partial_smem<D, T, kRowGroup>(R);
  auto kern = attention_partial_kernel<D, T, kRowGroup>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const float scale = (float)(1.0 / sqrt((double)D));
  // Persistent grid: as many CTAs as fit at once, capped by the item count.
  static int resident = 0;
  static size_t resident_smem = 0;
  if (resident == 0 || resident_smem != smem) {
    int per_sm = 0, dev = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    resident = (per_sm > 0 ? per_sm : 1) * sms;
    resident_smem = smem;
  }
  const long long items = (long long)max_items;
  const unsigned grid = (unsigned)(items < resident ? (items > 0 ? items : 1) : resident);
  e = launch_kernel(kern, dim3(grid), dim3(kThreads), smem, st, q, q_stride, n_q_heads, static_cast<const T*>(kc),
                    static_cast<const T*>(vc), n_kv_heads, ctx, meta.batch_index, meta.seq_lens, meta.chunk_off,
                    n_seq, tps, max_chunks, scale, partials, pv);
  if (e != cudaSuccess) return e;
  const int n_tok = n_seq * tps;
  const unsigned mgrid = (unsigned)((n_tok * n_q_heads + 3) / 4);
  if (xq_out)
    return launch_kernel(attention_merge_kernel<D, true>, dim3(mgrid), dim3(128), 0, st, partials, n_q_heads, tps,
                         meta.chunk_off, max_chunks, n_tok, out, static_cast<uint8_t*>(xq_out));
  return launch_kernel(attention_merge_kernel<D, false>, dim3(mgrid), dim3(128), 0, st, partials, n_q_heads, tps,
                       meta.chunk_off, max_chunks, n_tok, out, static_cast<uint8_t*>(nullptr));
}

template <int D, typename T>
cudaError_t launch_typed(const float* q, long long q_stride, int n_q_heads, const void* kc, const void* vc,
                         int n_kv_heads, int ctx, MetaView meta, int n_seq, int tps, long long max_items,
                         int max_chunks, float* partials, float* out, void* xq_out, PagedView pv, cudaStream_t st) {
  const int R = (n_q_heads / n_kv_heads) * tps;
  if (R <= 1)
    return launch_rg<D, T, 1>(q, q_stride, n_q_heads, kc, vc, n_kv_heads, ctx, meta, n_seq, tps, max_items,
                              max_chunks, partials, out, xq_out, pv, st);
  if (R <= 2)
    return launch_rg<D, T, 2>(q, q_stride, n_q_heads, kc, vc, n_kv_heads, ctx, meta, n_seq, tps, max_items,
                              max_chunks, partials, out, xq_out, pv, st);
  if (R <= 4)
    return launch_rg<D, T, 4>(q, q_stride, n_q_heads, kc, vc, n_kv_heads, ctx, meta, n_seq, tps, max_items,
                              max_chunks, partials, out, xq_out, pv, st);
  return launch_rg<D, T, kMaxRowGroup>(q, q_stride, n_q_heads, kc, vc, n_kv_heads, ctx, meta, n_seq, tps,
                                       max_items, max_chunks, partials, out, xq_out, pv, st);
}

}  // namespace

size_t attention_partial_bytes(int n_tok, int n_q_heads, int head_dim, int ctx) {
  const size_t max_chunks = (size_t)(ctx + kCh - 1) / kCh;
  return (size_t)n_tok * n_q_heads * max_chunks * (head_dim + 2) * sizeof(float);
}

cudaError_t launch_attention_decode_multi(const float* q, long long q_stride, int n_q_heads, const void* kc,
                                          const void* vc, int dtype,
                                          int n_kv_heads, int ctx, int head_dim, MetaView meta, int n_seq,
                                          int tokens_per_seq, long long max_items, int max_chunks, float* partials,
                                          float* out, void* xq_out, cudaStream_t st, PagedView pv) {
  if (n_seq == 0) return cudaSuccess;
  if (head_dim == 128) {
    if (dtype == 0)
      return launch_typed<128, __half>(q, q_stride, n_q_heads, kc, vc, n_kv_heads, ctx, meta, n_seq, tokens_per_seq,
                                       max_items, max_chunks, partials, out, xq_out, pv, st);
    return launch_typed<128, __nv_bfloat16>(q, q_stride, n_q_heads, kc, vc, n_kv_heads, ctx, meta, n_seq, tokens_per_seq,
                                            max_items, max_chunks, partials, out, xq_out, pv, st);
  }
  if (head_dim == 64) {
    if (dtype == 0)
      return launch_typed<64, __half>(q, q_stride, n_q_heads, kc, vc, n_kv_heads, ctx, meta, n_seq, tokens_per_seq,
                                      max_items, max_chunks, partials, out, xq_out, pv, st);
    return launch_typed<64, __nv_bfloat16>(q, q_stride, n_q_heads, kc, vc, n_kv_heads, ctx, meta, n_seq, tokens_per_seq,
                                           max_items, max_chunks, partials, out, xq_out, pv, st);
  }
  return cudaErrorInvalidValue;
}

unsigned int read_clear_error_attention() {
  unsigned int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_attention, sizeof v) != cudaSuccess) return 0xFFFFFFFFu;
  cudaMemcpyToSymbol(g_err_attention, &z, sizeof z);
  return v;
}

}  // namespace dsbk
