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
//  * partial kernel, a persistent CTA loop over work items (sequence, chunk,
//    kv head).  The chunk's K and V rows (contiguous in the cache) come in by
//    TMA tensor copies with the 128-byte swizzle, in 64-key boxes, so thread k
//    reads key k's row 16 bytes at a time without bank conflicts while the
//    query rows are read by broadcast; the next item's K and V are requested
//    as soon as this item is done with the buffers.  Thread k dots key k
//    against the G*T query rows of the GQA group (packed f32x2 FMAs); the
//    chunk's per-row max and sum of exp are block reductions in a fixed
//    order; for P.V warp w takes keys 32w..32w+31 and each lane 4 (or 2)
//    dimensions, reading the probabilities key-major (four rows per load),
//    and the four warps' sums are added in warp order.  Every K/V byte is read
//    once for all G*T query rows.  Per row it writes (max, sum of exp,
//    sum of exp * V) for the chunk.  While an item is being computed, one
//    thread decodes the next item and the query rows of the next item are
//    loaded into registers, so an item starts with no dependent global reads.
//  * up to 32 query rows per kv head, the same partial kernel runs its two
//    contractions on the tensor cores (attention_partial_tc_kernel below):
//    the per-key CUDA-core dot products and the broadcast query reads they
//    need were the kernel's cost at decode sizes.
//  * merge kernel, one warp per (token row, head): rescales the chunk partials
//    by exp(m_c - max_c m_c) and adds them in chunk order.
// No atomics and no inter-CTA waits; the chunking depends only on each
// sequence's own length, so a sequence's rows are bitwise equal whether it runs
// alone or inside a batch.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "dsb_actlayout.cuh"
#include "dsb_kernels.h"
#include "dsb_ptx.cuh"
#include "dsb_q8.cuh"

namespace dsbk {

namespace {

constexpr int kCh = 128;  // keys per chunk (DSB_ATTN_CHUNK)
constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
// Query rows handled together in the score and P.V loops: the widest row
// group is 8, and each launch takes the narrowest power of two >= G*T, so a
// one-row item (MHA, T = 1) issues no predicated-off work for absent rows.
constexpr int kMaxRowGroup = 8;
constexpr int kBoxCols = 64;                   // elements per swizzled 128-byte row
constexpr int kBoxKeys = 64;                   // keys per TMA box
constexpr int kBoxBytes = kBoxKeys * 128;      // 8 KiB
constexpr int kColBoxBytes = kCh * 128;        // one 64-column slab of a chunk: 16 KiB

__device__ unsigned int g_err_attention = 0;

// Byte offset of 16-byte piece j (elements 8j..8j+7) of key k's row in a
// chunk tile [D/64][128 keys][128 bytes] written by TMA with the 128-byte
// swizzle: the piece index within a 128-byte row is XORed with k mod 8.
__device__ __forceinline__ uint32_t swz(int k, int j) {
  return (uint32_t)((j >> 3) * kColBoxBytes + k * 128 + (((j & 7) ^ (k & 7)) << 4));
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ unsigned long long pack2(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 unpack2(unsigned long long v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

template <typename T>
struct Cvt;
template <>
struct Cvt<__half> {
  static __device__ __forceinline__ float2 two(uint32_t w) { return __half22float2(*reinterpret_cast<__half2*>(&w)); }
  static __device__ __forceinline__ unsigned long long two_packed(uint32_t w) {
    const float2 f = two(w);
    return pack2(f.x, f.y);
  }
};
template <>
struct Cvt<__nv_bfloat16> {
  static __device__ __forceinline__ float2 two(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w));
  }
  // bf16 -> f32 is exact: the bf16 bits are the float's top half
  static __device__ __forceinline__ unsigned long long two_packed(uint32_t w) {
    return pack2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  }
};

// Work item -> (sequence, relative chunk, kv head), its first key, key count
// and first cache row (contiguous cache or paged pool).
struct Item {
  int s, c_rel, g, key0, nkeys, L, W;
  long long row0;
};

// kL2: the metadata is read through L2 (the tensor-core kernel decodes its
// first item before it waits for its predecessor); the items after it read
// it through L1, where the binary search's loads hit.
template <bool kL2 = false>
__device__ __forceinline__ Item decode_item(int item, int n_kv_heads, int ctx, const int32_t* batch_index,
                                            const int32_t* seq_lens, const int32_t* chunk_off, int n_seq, int tps,
                                            const PagedView& pv) {
  auto ld = [](const int32_t* p) { return kL2 ? __ldcg(p) : *p; };
  Item it;
  const int w = item / n_kv_heads;
  it.g = item - w * n_kv_heads;
  int lo = 0, hi = n_seq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ld(chunk_off + mid) <= w)
      lo = mid;
    else
      hi = mid - 1;
  }
  it.s = lo;
  it.c_rel = w - ld(chunk_off + lo);  // this sequence's chunk, counted from its first
  it.L = ld(seq_lens + lo);
  // Paged view: chunk c lives in one page (128 keys), found through the
  // block table (modulo the block count for a ring); a window hides keys
  // older than pos - W + 1, so the first chunks of a long ring are skipped.
  it.W = pv.block_table ? ld(pv.window + lo) : 0;
  const int c = (it.W > 0 ? max(0, it.L - tps + 1 - it.W) / kCh : 0) + it.c_rel;
  it.key0 = c * kCh;
  it.nkeys = min(kCh, it.L - it.key0);
  if (pv.block_table) {
    const int nb = ld(pv.n_blocks + lo);
    const int page = ld(pv.block_table + (size_t)lo * pv.max_blocks + (it.W > 0 ? c % nb : c));
    it.row0 = ((long long)page * n_kv_heads + it.g) * kCh;
  } else {
    it.row0 = ((long long)ld(batch_index + lo) * n_kv_heads + it.g) * (long long)ctx + it.key0;
  }
  return it;
}

// One thread issues the chunk's K (or V) boxes (64-key boxes, only as many as
// hold its keys) on one barrier.
template <int D>
__device__ __forceinline__ uint32_t tile_bytes(const Item& it) {
  return (uint32_t)((D / kBoxCols) * (it.nkeys > kBoxKeys ? 2 : 1) * kBoxBytes);
}

template <int D>
__device__ __forceinline__ void issue_boxes(const Item& it, const CUtensorMap* tm, uint8_t* dst, uint64_t* bar) {
  const int halves = it.nkeys > kBoxKeys ? 2 : 1;
#pragma unroll
  for (int cb = 0; cb < D / kBoxCols; ++cb)
    for (int h = 0; h < halves; ++h)
      tma_load_2d(dst + cb * kColBoxBytes + h * kBoxBytes, tm, cb * kBoxCols, (int)(it.row0 + h * kBoxKeys), bar);
}

template <int D>
__device__ __forceinline__ void issue_tile(const Item& it, const CUtensorMap* tm, uint8_t* dst, uint64_t* bar) {
  mbar_arrive_expect_tx(bar, tile_bytes<D>(it));
  issue_boxes<D>(it, tm, dst, bar);
}

template <int D>
__device__ __forceinline__ void issue_chunk(const Item& it, const CUtensorMap* tmk, const CUtensorMap* tmv, uint8_t* Ks,
                                            uint8_t* Vs, uint64_t* bar_k, uint64_t* bar_v) {
  issue_tile<D>(it, tmk, Ks, bar_k);
  issue_tile<D>(it, tmv, Vs, bar_v);
}

// kFull: R is a multiple of kRowGroup, so every row of every group is live and
// the per-row guards fold away at compile time.
template <int D, typename T, int kRowGroup, bool kFull>
__global__ void __launch_bounds__(kThreads) attention_partial_kernel(
    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, const float* __restrict__ q,
    long long q_stride, int n_q_heads, int n_kv_heads, int ctx, const int32_t* __restrict__ batch_index,
    const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ chunk_off, int n_seq, int tps, int max_chunks,
    float scale, float* __restrict__ partials, const PagedView pv) {
  constexpr int NJ = D / 8;  // 16-byte pieces of a key row
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int G = n_q_heads / n_kv_heads, R = G * tps;
  const int RP = (R + 3) & ~3;  // key-major probability row stride
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Shared layout (the swizzled tiles need 1024-byte alignment):
  // Ks | Vs [D/64][128][128 B] | qs [R][D] | ps [128][RP] | wstat [2][warps][8] |
  // ms, ls [R] | barriers.  After the scores Ks holds the P.V warp sums.
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Ks = smem;
  uint8_t* Vs = Ks + (size_t)D * kCh * sizeof(T);
  float* qs = reinterpret_cast<float*>(Vs + (size_t)D * kCh * sizeof(T));
  float* ps = qs + (size_t)R * D;
  float* wstat = ps + (size_t)kCh * RP;
  float* ms = wstat + 2 * kWarps * kRowGroup;
  float* ls = ms + R;
  uint64_t* bars = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(ls + R) + 7) & ~uintptr_t(7));
  Item* nx = reinterpret_cast<Item*>(bars + 2);  // the next item, decoded ahead by thread 0
  float* red = reinterpret_cast<float*>(Ks);  // [warps][kRowGroup][D], reused after the scores
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
  }
  pdl_wait();  // q and the cache rows of this step come from the previous kernels
  pdl_trigger();

  // Persistent loop over work items (chunk, kv head); the item count comes
  // from the device metadata, so a captured launch serves any seq_lens.
  const int total_items = chunk_off[n_seq] * n_kv_heads;
  // Query element idx of the item's [R][D] block, read from q.
  auto q_elem = [&](const Item& x, int idx) {
    const int r = idx / D, d = idx - r * D;
    const int j = r / G, gi = r - j * G;
    return __ldcg(q + (size_t)(x.s * tps + j) * q_stride + (size_t)(x.g * G + gi) * D + d);
  };
  constexpr int kQPre = 8;  // query elements per thread carried over from the previous item
  float qpre[kQPre];
  if ((int)blockIdx.x < total_items) {
    const Item first = decode_item(blockIdx.x, n_kv_heads, ctx, batch_index, seq_lens, chunk_off, n_seq, tps, pv);
    if (tid == 0) {
      *nx = first;
      issue_chunk<D>(first, &tmk, &tmv, Ks, Vs, &bars[0], &bars[1]);
    }
#pragma unroll
    for (int i = 0; i < kQPre; ++i)
      if (tid + i * kThreads < R * D) qpre[i] = q_elem(first, tid + i * kThreads);
  }
  __syncthreads();
  uint32_t phase = 0;
  for (int item = blockIdx.x; item < total_items; item += gridDim.x, phase ^= 1u) {
    const Item it = *nx;
#pragma unroll
    for (int i = 0; i < kQPre; ++i)
      if (tid + i * kThreads < R * D) qs[tid + i * kThreads] = qpre[i];
    for (int idx = tid + kQPre * kThreads; idx < R * D; idx += kThreads) qs[idx] = q_elem(it, idx);
    __syncthreads();
    const int next = item + gridDim.x;
    if (tid == 0 && next < total_items)
      *nx = decode_item(next, n_kv_heads, ctx, batch_index, seq_lens, chunk_off, n_seq, tps, pv);
    if (!mbar_wait(&bars[0], phase)) g_err_attention = 1u;

    // ---- scores and the chunk's softmax statistics, row group by row group
    const int k = tid;
    for (int r0 = 0; r0 < R; r0 += kRowGroup) {
      unsigned long long dot2[kRowGroup];
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r) dot2[r] = 0ull;
#pragma unroll
      for (int jj = 0; jj < NJ; ++jj) {
        const uint4 kw = *reinterpret_cast<const uint4*>(Ks + swz(k, jj));
        const unsigned long long k01 = Cvt<T>::two_packed(kw.x), k23 = Cvt<T>::two_packed(kw.y);
        const unsigned long long k45 = Cvt<T>::two_packed(kw.z), k67 = Cvt<T>::two_packed(kw.w);
#pragma unroll
        for (int r = 0; r < kRowGroup; ++r) {
          if ((kFull || r0 + r < R)) {
            const ulonglong2 qa = *reinterpret_cast<const ulonglong2*>(qs + (size_t)(r0 + r) * D + jj * 8);
            const ulonglong2 qb = *reinterpret_cast<const ulonglong2*>(qs + (size_t)(r0 + r) * D + jj * 8 + 4);
            unsigned long long a = dot2[r];
            a = fma2(qa.x, k01, a);
            a = fma2(qa.y, k23, a);
            a = fma2(qb.x, k45, a);
            a = fma2(qb.y, k67, a);
            dot2[r] = a;
          }
        }
      }
      float sc[kRowGroup];
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r) {
        const float2 d2 = unpack2(dot2[r]);
        const int j = (r0 + r) / G;
        const int vis = it.L - tps + j + 1;          // keys before vis are visible to draft token j ...
        const int vlo = it.W > 0 ? vis - it.W : 0;   // ... from vlo on under a window
        const int key = it.key0 + k;
        const bool ok = (kFull || r0 + r < R) && k < it.nkeys && key < vis && key >= vlo;
        sc[r] = ok ? __fmul_rn(__fadd_rn(d2.x, d2.y), scale) : -INFINITY;
      }
      // row max over the chunk: xor tree in each warp, then the warps in order
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r) {
        float m = sc[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) wstat[warp * kRowGroup + r] = m;
      }
      __syncthreads();
      float p[kRowGroup];
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r) {
        float M = wstat[r];
#pragma unroll
        for (int w2 = 1; w2 < kWarps; ++w2) M = fmaxf(M, wstat[w2 * kRowGroup + r]);
        p[r] = (M == -INFINITY) ? 0.0f : expf(sc[r] - M);
        if (tid == 0 && (kFull || r0 + r < R)) ms[r0 + r] = M;
        float l = p[r];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) l = __fadd_rn(l, __shfl_xor_sync(0xffffffffu, l, o));
        if (lane == 0) wstat[kWarps * kRowGroup + warp * kRowGroup + r] = l;
        if ((kFull || r0 + r < R)) ps[(size_t)k * RP + r0 + r] = p[r];
      }
      __syncthreads();
      if (tid < kRowGroup && (kFull || r0 + tid < R)) {
        float l = wstat[kWarps * kRowGroup + tid];
#pragma unroll
        for (int w2 = 1; w2 < kWarps; ++w2) l = __fadd_rn(l, wstat[kWarps * kRowGroup + w2 * kRowGroup + tid]);
        ls[r0 + tid] = l;
      }
    }
    // the next item's query rows (thread 0 decoded it before the barriers above)
    if (next < total_items) {
      const Item nxt = *nx;
#pragma unroll
      for (int i = 0; i < kQPre; ++i)
        if (tid + i * kThreads < R * D) qpre[i] = q_elem(nxt, tid + i * kThreads);
    }
    if (!mbar_wait(&bars[1], phase)) g_err_attention = 1u;

    // ---- P V: warp w takes keys 32w.., lane 4 (D = 128) or 2 (D = 64) dims
    constexpr int DPL = D / 32;  // dimensions per lane
    const int kb = warp * 32, ke = min(kb + 32, it.nkeys);
    int vj, vsub;  // this lane's 16-byte piece of a V row and the byte within it
    if constexpr (DPL == 4) {
      vj = lane >> 1;          // 16-byte piece (0..15)
      vsub = (lane & 1) * 8;   // byte within it
    } else {
      vj = lane >> 2;          // 0..7
      vsub = (lane & 3) * 4;
    }
    for (int r0 = 0; r0 < R; r0 += kRowGroup) {
      unsigned long long acc[kRowGroup][DPL / 2];
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r)
#pragma unroll
        for (int e = 0; e < DPL / 2; ++e) acc[r][e] = 0ull;
      for (int kk = kb; kk < ke; ++kk) {
        const uint8_t* vp = Vs + swz(kk, vj) + vsub;
        unsigned long long v2[DPL / 2];
        if constexpr (DPL == 4) {
          const uint2 vw = *reinterpret_cast<const uint2*>(vp);
          v2[0] = Cvt<T>::two_packed(vw.x);
          v2[1] = Cvt<T>::two_packed(vw.y);
        } else {
          v2[0] = Cvt<T>::two_packed(*reinterpret_cast<const uint32_t*>(vp));
        }
        const float* pk = ps + (size_t)kk * RP + r0;
#pragma unroll
        for (int r4 = 0; r4 < kRowGroup; r4 += 4) {
          if ((kFull || r0 + r4 < R)) {
            const float4 p4 = *reinterpret_cast<const float4*>(pk + r4);
            const float pr[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
            for (int i = 0; i < 4 && r4 + i < kRowGroup; ++i) {
              const unsigned long long pp = pack2(pr[i], pr[i]);
#pragma unroll
              for (int e = 0; e < DPL / 2; ++e) acc[r4 + i][e] = fma2(pp, v2[e], acc[r4 + i][e]);
            }
          }
        }
      }
      // the warps' sums, added in warp order (red overlays Ks: every thread is
      // past the scores)
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r) {
        float* dst = red + ((size_t)warp * kRowGroup + r) * D + lane * DPL;
        if constexpr (DPL == 4) {
          const float2 a = unpack2(acc[r][0]), b = unpack2(acc[r][1]);
          *reinterpret_cast<float4*>(dst) = make_float4(a.x, a.y, b.x, b.y);
        } else {
          *reinterpret_cast<float2*>(dst) = unpack2(acc[r][0]);
        }
      }
      __syncthreads();
      for (int idx = tid; idx < kRowGroup * D; idx += kThreads) {
        const int r = idx / D, d = idx - r * D;
        if ((kFull || r0 + r < R)) {
          float x = red[idx];
#pragma unroll
          for (int w2 = 1; w2 < kWarps; ++w2) x = __fadd_rn(x, red[(size_t)w2 * kRowGroup * D + idx]);
          const int j = (r0 + r) / G, gi = (r0 + r) - j * G;
          const int t = it.s * tps + j, h = it.g * G + gi;
          float* dst = partials + (((size_t)t * n_q_heads + h) * max_chunks + it.c_rel) * (D + 2);
          dst[2 + d] = x;
          if (d == 0) {
            dst[0] = ms[r0 + r];
            dst[1] = ls[r0 + r];
          }
        }
      }
      fence_proxy_async_smem();  // these generic accesses of Ks / Vs precede the next TMA writes
      __syncthreads();
    }
    // both buffers are free: request the next item's K and V
    if (tid == 0 && next < total_items) issue_chunk<D>(*nx, &tmk, &tmv, Ks, Vs, &bars[0], &bars[1]);
  }  // work items
}

// ---- the tensor-core partial kernel ----------------------------------------
//
// Same items, same partial records, same masks as the kernel above; the two
// contractions of an item run on the tensor cores (warp-level mma.sync
// m16n8k16 in the cache's 16-bit type, f32 accumulate):
//   S^T = K . Q^T   keys x query rows: warp w takes keys 32w..32w+31 (two
//                   16-key tiles), all rows (8-row tiles), K = D;
//   O^T = V^T . P^T dims x query rows: warp w takes dims D/4 * w.. (one or
//                   two 16-dim tiles), all rows, K = the chunk's keys.
// K and V fragments come straight from the swizzled TMA tiles by ldmatrix
// (V transposed on the way).  The float query rows and probabilities enter
// as hi + lo pairs of the 16-bit type (x = hi + lo to 2^-16 relative, 2^-22
// for f16), each product being two MMAs, so the scores and sums keep float
// accuracy; the cache values are exact in that type.  The query rows arrive
// by bulk copies issued just before the item's K boxes and on the same
// barrier (plain loads issued after the CTAs' K and V copies waited behind
// all of that traffic).  K's buffer is handed to the next item's query and K
// copies as soon as the scores are done, V's after P.V.
template <typename T>
struct Tc;
template <>
struct Tc<__half> {
  static __device__ __forceinline__ void split(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 f = __half22float2(h);
    const __half2 l = __floats2half2_rn(x0 - f.x, x1 - f.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
  }
  static __device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};
template <>
struct Tc<__nv_bfloat16> {
  static __device__ __forceinline__ void split(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 f = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - f.x, x1 - f.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
  }
  static __device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Shared memory of the tensor-core kernel (bytes past the 1024-byte aligned
// base): Ks | Vs [D/64][128][128 B] | Qf [R8][D + 8] f32 (the query rows as
// copied, one bulk copy per row) | Ph | Pl [R8][136] (16-bit) -- the row
// padding spreads a fragment load's 8 rows over the banks | per-warp row max
// and sum [2][4][R8] f32 | 2 barriers | two next-item slots.  About 74 KB at
// D = 128 and 8 rows: three CTAs per SM.
template <int D, int NRT>
__host__ __device__ constexpr size_t tc_smem_bytes() {
  return 1024 + 4 * (size_t)kCh * D + (size_t)(8 * NRT) * (D + 8) * 4 + 2 * (size_t)(8 * NRT) * (kCh + 8) * 2 +
         2 * (size_t)kWarps * (8 * NRT) * 4 + 2 * 8 + 2 * sizeof(Item) + 8;
}

template <int D, typename T, int NRT>
__global__ void __launch_bounds__(kThreads) attention_partial_tc_kernel(
    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, const float* __restrict__ q,
    long long q_stride, int n_q_heads, int n_kv_heads, int ctx, const int32_t* __restrict__ batch_index,
    const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ chunk_off, int n_seq, int tps, int max_chunks,
    float scale, float* __restrict__ partials, const PagedView pv) {
  constexpr int R8 = 8 * NRT;        // query rows, padded to whole 8-row tiles
  constexpr int QF = D + 8;          // query row stride (floats)
  constexpr int PS = kCh + 8;        // probability row stride (16-bit elements)
  constexpr int MTV = D / kWarps / 16;  // 16-dim tiles of P.V per warp
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int G = n_q_heads / n_kv_heads, R = G * tps;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Ks = smem;
  uint8_t* Vs = Ks + (size_t)D * kCh * 2;
  float* Qf = reinterpret_cast<float*>(Vs + (size_t)D * kCh * 2);
  uint16_t* Ph = reinterpret_cast<uint16_t*>(Qf + R8 * QF);
  uint16_t* Pl = Ph + R8 * PS;
  float* wmax = reinterpret_cast<float*>(Pl + R8 * PS);  // [warp][R8]
  float* wsum = wmax + kWarps * R8;
  uint64_t* bars = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(wsum + kWarps * R8) + 7) & ~uintptr_t(7));
  Item* nx2 = reinterpret_cast<Item*>(bars + 2);  // items alternate between two slots
  const uint32_t ks_addr = smem_addr(Ks), vs_addr = smem_addr(Vs);
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
  }
  // the padding query rows R..R8-1 stay zero (no copy writes them)
  for (int idx = tid; idx < (R8 - R) * QF; idx += kThreads) Qf[R * QF + idx] = 0.0f;

  // Thread 0 requests an item's query rows (one bulk copy of D floats per
  // row, into the padded rows of Qf) and then its K boxes, all on bars[0]:
  // the query rows are first in line behind no K or V traffic of this CTA.
  const uint32_t qb = (uint32_t)(D * 4);
  auto issue_q = [&](const Item& x) {
    for (int r = 0; r < R; ++r) {
      const int j = r / G, gi = r - j * G;
      bulk_g2s(Qf + (size_t)r * QF, q + (size_t)(x.s * tps + j) * q_stride + (size_t)(x.g * G + gi) * D, qb,
               &bars[0]);
    }
  };
  auto issue_qk = [&](const Item& x) {
    mbar_arrive_expect_tx(&bars[0], (uint32_t)R * qb + tile_bytes<D>(x));
    issue_q(x);
    issue_boxes<D>(x, &tmk, Ks, &bars[0]);
  };
  // With at most two items per CTA the start-up is a large part of a CTA's
  // time, so it moves ahead of the wait for the previous kernel.  The step's
  // metadata (lengths, slots, chunk offsets) is written by its first kernel,
  // which has completed before the previous kernel starts its own work (every
  // kernel waits for its predecessor before it lets the next one launch): the
  // first item is decoded before the wait, reading through L2.  So are its K
  // and V requested, when the cache is contiguous and none of the rows the
  // tile covers is one the previous kernel writes (the step's new rows
  // L - T .. L - 1 of this slot; slots are distinct).  The query rows always
  // follow the wait.  With more items per CTA the early start measured no
  // faster (the Qwen3-14B-shaped step at 16 sequences, 5 items per CTA).
  const int total_items = __ldcg(chunk_off + n_seq) * n_kv_heads;
  const bool start_early = total_items <= 2 * (int)gridDim.x;
  Item first{};
  bool early = false;
  if (start_early && (int)blockIdx.x < total_items && tid == 0) {
    first = decode_item<true>(blockIdx.x, n_kv_heads, ctx, batch_index, seq_lens, chunk_off, n_seq, tps, pv);
    const int tile_rows = (first.nkeys > kBoxKeys ? 2 : 1) * kBoxKeys;
    early = pv.block_table == nullptr && first.key0 + tile_rows <= first.L - tps;
    if (early) {
      mbar_arrive_expect_tx(&bars[0], (uint32_t)R * qb + tile_bytes<D>(first));
      issue_boxes<D>(first, &tmk, Ks, &bars[0]);
      issue_tile<D>(first, &tmv, Vs, &bars[1]);
    }
  }
  pdl_wait();  // q and the cache rows of this step come from the previous kernels
  pdl_trigger();
  if ((int)blockIdx.x < total_items && tid == 0) {
    if (!start_early)
      first = decode_item(blockIdx.x, n_kv_heads, ctx, batch_index, seq_lens, chunk_off, n_seq, tps, pv);
    nx2[0] = first;
    if (early) {
      issue_q(first);
    } else {
      issue_qk(first);
      issue_tile<D>(first, &tmv, Vs, &bars[1]);
    }
  }
  __syncthreads();
  uint32_t phase = 0;
  for (int item = blockIdx.x, slot = 0; item < total_items; item += gridDim.x, phase ^= 1u, slot ^= 1) {
    const Item it = nx2[slot];
    Item* nx = &nx2[slot ^ 1];  // the next item's slot, last read an item ago
    const int next = item + gridDim.x;
    if (tid == 0 && next < total_items)
      *nx = decode_item(next, n_kv_heads, ctx, batch_index, seq_lens, chunk_off, n_seq, tps, pv);
    if (!mbar_wait(&bars[0], phase)) g_err_attention = 1u;  // query rows and K
    __syncwarp();  // ldmatrix and mma.sync below run warp-converged

    // ---- S^T = K . Q^T: this warp's 32 keys x R8 rows
    float sacc[2][NRT][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NRT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[mt][nt][e] = 0.0f;
    {
      const int mi = lane >> 3;  // the ldmatrix sub-matrix this lane addresses
#pragma unroll
      for (int kq = 0; kq < D / 16; ++kq) {
        uint32_t a[2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
          ldsm_x4(a[mt], ks_addr + swz(32 * warp + 16 * mt + (lane & 7) + 8 * (mi & 1), 2 * kq + (mi >> 1)));
#pragma unroll
        for (int nt = 0; nt < NRT; ++nt) {
          // row 8nt + g, dims 16kq + 2c, +1 and 16kq + 8 + 2c, +1: hi and lo parts
          const float* qr = Qf + (8 * nt + g) * QF + 16 * kq + 2 * c;
          const float2 q0 = *reinterpret_cast<const float2*>(qr), q1 = *reinterpret_cast<const float2*>(qr + 8);
          uint32_t h0, l0, h1, l1;
          Tc<T>::split(q0.x, q0.y, h0, l0);
          Tc<T>::split(q1.x, q1.y, h1, l1);
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            Tc<T>::mma(sacc[mt][nt], a[mt], h0, h1);
            Tc<T>::mma(sacc[mt][nt], a[mt], l0, l1);
          }
        }
      }
    }
    // scale and mask: element e of tile (mt, nt) is key 32w + 16mt + g + 8(e >> 1),
    // row 8nt + 2c + (e & 1); then the chunk's row maxima
    float mx[NRT][2];
#pragma unroll
    for (int nt = 0; nt < NRT; ++nt) mx[nt][0] = mx[nt][1] = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NRT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kl = 32 * warp + 16 * mt + g + 8 * (e >> 1), row = 8 * nt + 2 * c + (e & 1);
          const int j = row / G;
          const int vis = it.L - tps + j + 1;         // keys before vis are visible to draft token j ...
          const int vlo = it.W > 0 ? vis - it.W : 0;  // ... from vlo on under a window
          const int key = it.key0 + kl;
          const bool ok = row < R && kl < it.nkeys && key < vis && key >= vlo;
          const float v = ok ? __fmul_rn(sacc[mt][nt][e], scale) : -INFINITY;
          sacc[mt][nt][e] = v;
          mx[nt][e & 1] = fmaxf(mx[nt][e & 1], v);
        }
#pragma unroll
    for (int nt = 0; nt < NRT; ++nt)
#pragma unroll
      for (int j2 = 0; j2 < 2; ++j2) {
        float m = mx[nt][j2];
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (g == 0) wmax[warp * R8 + 8 * nt + 2 * c + j2] = m;
      }
    fence_proxy_async_smem();  // the K and query reads precede the next item's copies
    __syncthreads();
    if (tid == 0 && next < total_items) issue_qk(*nx);

    // ---- probabilities (hi + lo into Ph / Pl) and the per-warp row sums
    float sm[NRT][2];
#pragma unroll
    for (int nt = 0; nt < NRT; ++nt)
#pragma unroll
      for (int j2 = 0; j2 < 2; ++j2) {
        const int row = 8 * nt + 2 * c + j2;
        float M = wmax[row];
#pragma unroll
        for (int w2 = 1; w2 < kWarps; ++w2) M = fmaxf(M, wmax[w2 * R8 + row]);
        mx[nt][j2] = M;
        sm[nt][j2] = 0.0f;
      }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NRT; ++nt)
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {  // keys g and g + 8 of the tile, rows 2c and 2c + 1
          const float M0 = mx[nt][0], M1 = mx[nt][1];
          const float p0 = (M0 == -INFINITY) ? 0.0f : expf(sacc[mt][nt][2 * e2] - M0);
          const float p1 = (M1 == -INFINITY) ? 0.0f : expf(sacc[mt][nt][2 * e2 + 1] - M1);
          sm[nt][0] = __fadd_rn(sm[nt][0], p0);
          sm[nt][1] = __fadd_rn(sm[nt][1], p1);
          const int kl = 32 * warp + 16 * mt + g + 8 * e2, row = 8 * nt + 2 * c;
          uint32_t hi, lo;
          Tc<T>::split(p0, p1, hi, lo);
          Ph[row * PS + kl] = (uint16_t)(hi & 0xFFFFu);
          Ph[(row + 1) * PS + kl] = (uint16_t)(hi >> 16);
          Pl[row * PS + kl] = (uint16_t)(lo & 0xFFFFu);
          Pl[(row + 1) * PS + kl] = (uint16_t)(lo >> 16);
        }
#pragma unroll
    for (int nt = 0; nt < NRT; ++nt)
#pragma unroll
      for (int j2 = 0; j2 < 2; ++j2) {
        float l = sm[nt][j2];
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) l = __fadd_rn(l, __shfl_xor_sync(0xffffffffu, l, o));
        if (g == 0) wsum[warp * R8 + 8 * nt + 2 * c + j2] = l;
      }
    __syncthreads();
    // row statistics of the chunk: (max, sum of exp), warps added in order
    if (tid < R) {
      float M = wmax[tid], l = wsum[tid];
#pragma unroll
      for (int w2 = 1; w2 < kWarps; ++w2) {
        M = fmaxf(M, wmax[w2 * R8 + tid]);
        l = __fadd_rn(l, wsum[w2 * R8 + tid]);
      }
      const int j = tid / G, gi = tid - j * G;
      float* dst = partials + (((size_t)(it.s * tps + j) * n_q_heads + it.g * G + gi) * max_chunks + it.c_rel) * (D + 2);
      dst[0] = M;
      dst[1] = l;
    }
    if (!mbar_wait(&bars[1], phase)) g_err_attention = 1u;
    __syncwarp();

    // ---- O^T = V^T . P^T: this warp's dims x R8 rows over the chunk's keys
    float oacc[MTV][NRT][4];
#pragma unroll
    for (int mv = 0; mv < MTV; ++mv)
#pragma unroll
      for (int nt = 0; nt < NRT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[mv][nt][e] = 0.0f;
    {
      const int mi = lane >> 3;
      const int nkk = (it.nkeys + 15) >> 4;
      for (int kk = 0; kk < nkk; ++kk) {
        uint32_t a[MTV][4];
#pragma unroll
        for (int mv = 0; mv < MTV; ++mv)
          ldsm_x4_trans(a[mv], vs_addr + swz(16 * kk + (lane & 7) + 8 * (mi >> 1), (D / kWarps / 8) * warp + 2 * mv +
                                                                                      (mi & 1)));
        if (16 * kk + 16 > it.nkeys) {
          // keys past the chunk's end: their rows may hold anything (the
          // probabilities there are zero, but 0 * inf is not), so zero them
          const int k0 = 16 * kk + 2 * c, k8 = k0 + 8;
          const uint32_t m0 = (k0 < it.nkeys ? 0xFFFFu : 0u) | (k0 + 1 < it.nkeys ? 0xFFFF0000u : 0u);
          const uint32_t m8 = (k8 < it.nkeys ? 0xFFFFu : 0u) | (k8 + 1 < it.nkeys ? 0xFFFF0000u : 0u);
#pragma unroll
          for (int mv = 0; mv < MTV; ++mv) {
            a[mv][0] &= m0;
            a[mv][1] &= m0;
            a[mv][2] &= m8;
            a[mv][3] &= m8;
          }
        }
#pragma unroll
        for (int nt = 0; nt < NRT; ++nt) {
          uint32_t b[4];  // Ph keys +0, +8, Pl keys +0, +8 of rows 8nt..8nt+7
          ldsm_x4(b, smem_addr((mi >> 1 ? Pl : Ph) + (8 * nt + (lane & 7)) * PS + 16 * kk + 8 * (mi & 1)));
#pragma unroll
          for (int mv = 0; mv < MTV; ++mv) {
            Tc<T>::mma(oacc[mv][nt], a[mv], b[0], b[1]);
            Tc<T>::mma(oacc[mv][nt], a[mv], b[2], b[3]);
          }
        }
      }
    }
    // element e of tile (mv, nt): dim D/4 * w + 16mv + g + 8(e >> 1), row 8nt + 2c + (e & 1)
#pragma unroll
    for (int nt = 0; nt < NRT; ++nt)
#pragma unroll
      for (int j2 = 0; j2 < 2; ++j2) {
        const int row = 8 * nt + 2 * c + j2;
        if (row < R) {
          const int j = row / G, gi = row - j * G;
          float* dst = partials +
                       (((size_t)(it.s * tps + j) * n_q_heads + it.g * G + gi) * max_chunks + it.c_rel) * (D + 2) + 2;
#pragma unroll
          for (int mv = 0; mv < MTV; ++mv) {
            const int d0 = (D / kWarps) * warp + 16 * mv + g;
            dst[d0] = oacc[mv][nt][j2];
            dst[d0 + 8] = oacc[mv][nt][2 + j2];
          }
        }
      }
    fence_proxy_async_smem();  // the V reads precede the next item's copy into Vs
    __syncthreads();
    if (tid == 0 && next < total_items) issue_tile<D>(*nx, &tmv, Vs, &bars[1]);
  }  // work items
}

// One CTA per (token row, query head), one warp per 32 dimensions of the head
// (warp q owns dims 32q .. 32q + 31, one q8_0 block).  Every warp first takes
// the chunks' (m, l) 32 at a time (max of m_c, then w_c = exp(m_c - M) and
// the partial sum of w_c l_c; the sums over lanes use a fixed xor tree), then
// walks the chunks in order, lane d accumulating w_c * acc_c[32q + d].  With
// QOUT the normalised block is q8_0-quantised straight into xq.
template <int D, bool QOUT>
__global__ void __launch_bounds__(D) attention_merge_kernel(const float* __restrict__ partials, int n_q_heads,
                                                            int tps, const int32_t* __restrict__ chunk_off,
                                                            int max_chunks, int n_tok, float* __restrict__ out,
                                                            uint8_t* __restrict__ xq,
                                                            uint32_t* __restrict__ xq_staged) {
  pdl_wait();
  pdl_trigger();
  const int wg = blockIdx.x;
  const int qd = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (wg >= n_tok * n_q_heads) return;
  const int t = wg / n_q_heads, h = wg - t * n_q_heads;
  const int s = t / tps;
  // every chunk of the sequence; those that hide all of this row's keys hold
  // max = -inf and add exactly nothing
  const int nch = chunk_off[s + 1] - chunk_off[s];
  const float* base = partials + ((size_t)t * n_q_heads + h) * max_chunks * (D + 2);
  const int dim = 32 * qd + lane;
  // The first 32 chunks' (m, l) and their sums are requested together,
  // before anything depends on them: at decode contexts (<= 32 chunks, 4096
  // keys) the merge waits for one round of loads.
  constexpr int kB = 32;  // chunks per batch of sum loads
  float v[kB];
  float m0 = -INFINITY, l0 = 0.0f;
  if (lane < nch) {
    const float* pc = base + (size_t)lane * (D + 2);
    m0 = __ldcg(pc);
    l0 = __ldcg(pc + 1);
  }
#pragma unroll
  for (int i = 0; i < kB; ++i)
    if (i < nch) v[i] = __ldcg(base + (size_t)i * (D + 2) + 2 + dim);
  float M = m0;
  for (int c = lane + 32; c < nch; c += 32) M = fmaxf(M, __ldcg(base + (size_t)c * (D + 2)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float lsum = 0.0f, acc = 0.0f;
  for (int c0 = 0; c0 < nch; c0 += 32) {
    float wl = 0.0f;
    if (c0 + lane < nch) {
      float mc = m0, lc = l0;
      if (c0 > 0) {
        const float* pc = base + (size_t)(c0 + lane) * (D + 2);
        mc = __ldcg(pc);
        lc = __ldcg(pc + 1);
      }
      wl = (mc == -INFINITY) ? 0.0f : expf(mc - M);
      lsum = __fmaf_rn(wl, lc, lsum);
    }
    const int n = min(32, nch - c0);
    // kB chunks' loads in flight, then their terms added in chunk order
    for (int cb = 0; cb < n; cb += kB) {
      if (c0 + cb > 0) {
#pragma unroll
        for (int i = 0; i < kB; ++i)
          if (cb + i < n) v[i] = __ldcg(base + (size_t)(c0 + cb + i) * (D + 2) + 2 + dim);
      }
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        const float wc = __shfl_sync(0xffffffffu, wl, (cb + i) & 31);
        if (cb + i < n) acc = __fmaf_rn(wc, v[i], acc);
      }
    }
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) lsum = __fadd_rn(lsum, __shfl_xor_sync(0xffffffffu, lsum, o));
  if constexpr (QOUT) {
    uint8_t* dst = xq + (((size_t)t * n_q_heads + h) * (D / 32) + qd) * 34;
    if (xq_staged)
      q8_block_store_staged(__fdiv_rn(acc, lsum), dst, xq_staged, (long long)n_q_heads * (D / 32),
                            h * (D / 32) + qd, t, n_tok, lane);
    else
      q8_block_store(__fdiv_rn(acc, lsum), dst, lane);
  } else {
    out[((size_t)t * n_q_heads + h) * D + dim] = __fdiv_rn(acc, lsum);
  }
}

template <int D, typename T, int kRowGroup>
size_t partial_smem(int R) {
  const int RP = (R + 3) & ~3;
  return 1024 + 2 * (size_t)kCh * D * sizeof(T) + (size_t)R * D * 4 + (size_t)kCh * RP * 4 +
         (size_t)2 * kWarps * kRowGroup * 4 + (size_t)2 * R * 4 + 8 + 2 * 8 + sizeof(Item);
}

// Tensor maps of the K and V caches viewed as [rows][D] 16-bit elements, with
// 64-column x 64-key boxes and the 128-byte swizzle.  Encoded on the host
// (no device work) and cached by address and shape.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

cudaError_t kv_tensor_map(const void* base, long long rows, int D, int dtype, CUtensorMap* out) {
  struct Entry {
    const void* base;
    long long rows;
    int D, dtype;
    CUtensorMap map;
  };
  static std::mutex mu;
  static Entry cache[16];
  static int n_cache = 0, next_slot = 0;
  static EncodeTiledFn encode = nullptr;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_cache; ++i)
    if (cache[i].base == base && cache[i].rows == rows && cache[i].D == D && cache[i].dtype == dtype) {
      *out = cache[i].map;
      return cudaSuccess;
    }
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBoxCols, (cuuint32_t)kBoxKeys};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  const CUresult r = encode(&m, dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const int slot = n_cache < 16 ? n_cache++ : (next_slot++ & 15);
  cache[slot] = Entry{base, rows, D, dtype, m};
  *out = m;
  return cudaSuccess;
}

// Launch a partial kernel as a persistent grid (as many CTAs as fit at once,
// capped by the item count), then the merge.
template <int D, typename Kern>
cudaError_t launch_partial_merge(Kern kern, size_t smem, const float* q, long long q_stride, int n_q_heads,
                                 const void* kc, const void* vc, int dtype, int n_kv_heads, int ctx, long long kv_rows,
                                 MetaView meta, int n_seq, int tps, long long max_items, int max_chunks,
                                 float* partials, float* out, void* xq_out, void* xq_staged, PagedView pv, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  CUtensorMap tmk, tmv;
  if ((e = kv_tensor_map(kc, kv_rows, D, dtype, &tmk)) != cudaSuccess) return e;
  if ((e = kv_tensor_map(vc, kv_rows, D, dtype, &tmv)) != cudaSuccess) return e;
  const float scale = (float)(1.0 / sqrt((double)D));
  int resident = 0;
  {
    struct Entry {
      const void* kern;
      size_t smem;
      int dev, ctas;
    };
    static std::mutex mu;
    static Entry cache[32];
    static int n_cache = 0;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_cache; ++i)
      if (cache[i].kern == reinterpret_cast<const void*>(kern) && cache[i].smem == smem && cache[i].dev == dev)
        resident = cache[i].ctas;
    if (resident == 0) {
      int per_sm = 0, sms = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
      if (e != cudaSuccess) return e;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      resident = (per_sm > 0 ? per_sm : 1) * sms;
      if (n_cache < 32) cache[n_cache++] = Entry{reinterpret_cast<const void*>(kern), smem, dev, resident};
    }
  }
  const long long items = (long long)max_items;
  const unsigned grid = (unsigned)(items < resident ? (items > 0 ? items : 1) : resident);
  e = launch_kernel(kern, dim3(grid), dim3(kThreads), smem, st, tmk, tmv, q, q_stride, n_q_heads, n_kv_heads, ctx,
                    meta.batch_index, meta.seq_lens, meta.chunk_off, n_seq, tps, max_chunks, scale, partials, pv);
  if (e != cudaSuccess) return e;
  const int n_tok = n_seq * tps;
  const unsigned mgrid = (unsigned)(n_tok * n_q_heads);
  if (xq_out)
    return launch_kernel(attention_merge_kernel<D, true>, dim3(mgrid), dim3(D), 0, st, partials, n_q_heads, tps,
                         meta.chunk_off, max_chunks, n_tok, out, static_cast<uint8_t*>(xq_out),
                         static_cast<uint32_t*>(xq_staged));
  return launch_kernel(attention_merge_kernel<D, false>, dim3(mgrid), dim3(D), 0, st, partials, n_q_heads, tps,
                       meta.chunk_off, max_chunks, n_tok, out, static_cast<uint8_t*>(nullptr),
                       static_cast<uint32_t*>(nullptr));
}

template <int D, typename T, int kRowGroup, bool kFull>
cudaError_t launch_rg_full(const float* q, long long q_stride, int n_q_heads, const void* kc, const void* vc, int dtype,
                           int n_kv_heads, int ctx, long long kv_rows, MetaView meta, int n_seq, int tps,
                           long long max_items, int max_chunks, float* partials, float* out, void* xq_out, void* xq_staged,
                           PagedView pv, cudaStream_t st) {
  const int R = (n_q_heads / n_kv_heads) * tps;
  return launch_partial_merge<D>(attention_partial_kernel<D, T, kRowGroup, kFull>, partial_smem<D, T, kRowGroup>(R), q,
                                 q_stride, n_q_heads, kc, vc, dtype, n_kv_heads, ctx, kv_rows, meta, n_seq, tps,
                                 max_items, max_chunks, partials, out, xq_out, xq_staged, pv, st);
}

template <int D, typename T, int NRT>
cudaError_t launch_tc(const float* q, long long q_stride, int n_q_heads, const void* kc, const void* vc, int dtype,
                      int n_kv_heads, int ctx, long long kv_rows, MetaView meta, int n_seq, int tps,
                      long long max_items, int max_chunks, float* partials, float* out, void* xq_out, void* xq_staged, PagedView pv,
                      cudaStream_t st) {
  return launch_partial_merge<D>(attention_partial_tc_kernel<D, T, NRT>, tc_smem_bytes<D, NRT>(), q, q_stride,
                                 n_q_heads, kc, vc, dtype, n_kv_heads, ctx, kv_rows, meta, n_seq, tps, max_items,
                                 max_chunks, partials, out, xq_out, xq_staged, pv, st);
}

// Row groups of 1, 2 and 5 serve R = 1, 2 and 5 only (always full); 4 and 8
// also serve R = 3 and R = 6, 7, 9.. (a partial last group).
template <int D, typename T, int kRowGroup>
cudaError_t launch_rg(const float* q, long long q_stride, int n_q_heads, const void* kc, const void* vc, int dtype,
                      int n_kv_heads, int ctx, long long kv_rows, MetaView meta, int n_seq, int tps,
                      long long max_items, int max_chunks, float* partials, float* out, void* xq_out, void* xq_staged, PagedView pv,
                      cudaStream_t st) {
  const int R = (n_q_heads / n_kv_heads) * tps;
  if (kRowGroup == 4 || kRowGroup == kMaxRowGroup) {
    if (R % kRowGroup != 0)
      return launch_rg_full<D, T, kRowGroup, false>(q, q_stride, n_q_heads, kc, vc, dtype, n_kv_heads, ctx, kv_rows,
                                                    meta, n_seq, tps, max_items, max_chunks, partials, out, xq_out, xq_staged, pv,
                                                    st);
  }
  return launch_rg_full<D, T, kRowGroup, true>(q, q_stride, n_q_heads, kc, vc, dtype, n_kv_heads, ctx, kv_rows, meta,
                                               n_seq, tps, max_items, max_chunks, partials, out, xq_out, xq_staged, pv, st);
}

template <int D, typename T>
cudaError_t launch_typed(const float* q, long long q_stride, int n_q_heads, const void* kc, const void* vc, int dtype,
                         int n_kv_heads, int ctx, long long kv_rows, MetaView meta, int n_seq, int tps,
                         long long max_items, int max_chunks, float* partials, float* out, void* xq_out, void* xq_staged, PagedView pv,
                         cudaStream_t st) {
  const int R = (n_q_heads / n_kv_heads) * tps;
  // up to 32 query rows per kv head: the tensor-core kernel (1, 2 or 4
  // eight-row tiles), which copies the query rows in bulk (16-byte aligned
  // rows); wider groups or unaligned query rows: the row-group kernel
  const bool tc_ok = (reinterpret_cast<uintptr_t>(q) & 15) == 0 && (q_stride & 3) == 0;
  if (tc_ok && R <= 8)
    return launch_tc<D, T, 1>(q, q_stride, n_q_heads, kc, vc, dtype, n_kv_heads, ctx, kv_rows, meta, n_seq, tps,
                              max_items, max_chunks, partials, out, xq_out, xq_staged, pv, st);
  if (tc_ok && R <= 16)
    return launch_tc<D, T, 2>(q, q_stride, n_q_heads, kc, vc, dtype, n_kv_heads, ctx, kv_rows, meta, n_seq, tps,
                              max_items, max_chunks, partials, out, xq_out, xq_staged, pv, st);
  if (tc_ok && R <= 32)
    return launch_tc<D, T, 4>(q, q_stride, n_q_heads, kc, vc, dtype, n_kv_heads, ctx, kv_rows, meta, n_seq, tps,
                              max_items, max_chunks, partials, out, xq_out, xq_staged, pv, st);
  if (R <= 1)
    return launch_rg<D, T, 1>(q, q_stride, n_q_heads, kc, vc, dtype, n_kv_heads, ctx, kv_rows, meta, n_seq, tps,
                              max_items, max_chunks, partials, out, xq_out, xq_staged, pv, st);
  if (R <= 2)
    return launch_rg<D, T, 2>(q, q_stride, n_q_heads, kc, vc, dtype, n_kv_heads, ctx, kv_rows, meta, n_seq, tps,
                              max_items, max_chunks, partials, out, xq_out, xq_staged, pv, st);
  if (R <= 4)
    return launch_rg<D, T, 4>(q, q_stride, n_q_heads, kc, vc, dtype, n_kv_heads, ctx, kv_rows, meta, n_seq, tps,
                              max_items, max_chunks, partials, out, xq_out, xq_staged, pv, st);
  // five query rows per kv head: GQA 5:1 at one token per sequence (the
  // Qwen3-14B shape), where a group of eight would carry three idle rows
  if (R == 5)
    return launch_rg<D, T, 5>(q, q_stride, n_q_heads, kc, vc, dtype, n_kv_heads, ctx, kv_rows, meta, n_seq, tps,
                              max_items, max_chunks, partials, out, xq_out, xq_staged, pv, st);
  return launch_rg<D, T, kMaxRowGroup>(q, q_stride, n_q_heads, kc, vc, dtype, n_kv_heads, ctx, kv_rows, meta, n_seq,
                                       tps, max_items, max_chunks, partials, out, xq_out, xq_staged, pv, st);
}

}  // namespace

size_t attention_partial_bytes(int n_tok, int n_q_heads, int head_dim, int ctx) {
  const size_t max_chunks = (size_t)(ctx + kCh - 1) / kCh;
  return (size_t)n_tok * n_q_heads * max_chunks * (head_dim + 2) * sizeof(float);
}

cudaError_t launch_attention_decode_multi(const float* q, long long q_stride, int n_q_heads, const void* kc,
                                          const void* vc, int dtype, int n_kv_heads, int ctx, int head_dim,
                                          long long kv_rows, MetaView meta, int n_seq, int tokens_per_seq,
                                          long long max_items, int max_chunks, float* partials, float* out,
                                          void* xq_out, cudaStream_t st, PagedView pv, void* xq_staged) {
  if (n_seq == 0) return cudaSuccess;
  if (head_dim == 128) {
    if (dtype == 0)
      return launch_typed<128, __half>(q, q_stride, n_q_heads, kc, vc, dtype, n_kv_heads, ctx, kv_rows, meta, n_seq,
                                       tokens_per_seq, max_items, max_chunks, partials, out, xq_out, xq_staged, pv, st);
    return launch_typed<128, __nv_bfloat16>(q, q_stride, n_q_heads, kc, vc, dtype, n_kv_heads, ctx, kv_rows, meta,
                                            n_seq, tokens_per_seq, max_items, max_chunks, partials, out, xq_out, xq_staged, pv,
                                            st);
  }
  if (head_dim == 64) {
    if (dtype == 0)
      return launch_typed<64, __half>(q, q_stride, n_q_heads, kc, vc, dtype, n_kv_heads, ctx, kv_rows, meta, n_seq,
                                      tokens_per_seq, max_items, max_chunks, partials, out, xq_out, xq_staged, pv, st);
    return launch_typed<64, __nv_bfloat16>(q, q_stride, n_q_heads, kc, vc, dtype, n_kv_heads, ctx, kv_rows, meta,
                                           n_seq, tokens_per_seq, max_items, max_chunks, partials, out, xq_out, xq_staged, pv,
                                           st);
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
