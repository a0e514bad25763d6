// The narrow-batch q8_0 matmul kernel template and its launch helpers, shared
// by the translation units that instantiate it (q8_0 activations in one, the
// fused RMSNorm / SiLU-gate activation prologues in another, compiled in
// parallel).  Everything here has internal linkage: each unit holds its own
// instances, host caches and device error flag.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <type_traits>

#include "dsb_actlayout.cuh"
#include "dsb_kernels.h"
#include "dsb_ptx.cuh"

namespace dsbk {

namespace {

constexpr int kWarps = 8;              // warps of a CTA; one CTA per SM
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerWarp = 32;        // lane = weight row
constexpr int kChunkBytes = 272;        // one k-step of a row: 8 blocks of 34 bytes
constexpr int kStage = kRowsPerWarp * kChunkBytes;
constexpr int kNStage = 2;              // weight stages per warp
constexpr int kMaxCluster = 16;         // k-split CTAs per cluster (above 8: a non-portable cluster size)
constexpr uint32_t kMagic = 0x4B400000u;  // bits of 12582912.0f = 1.5 * 2^23
constexpr unsigned long long kMagic2 = 0x4B4000004B400000ull;

__device__ unsigned int g_err_matmul = 0;

// One 2-D tensor copy of a weight stage: 32 rows x 272 bytes (x in 16-bit
// elements: the k-step times 136; y: the first row), counted on `bar`.
__device__ __forceinline__ void tma_stage_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

struct Split {
  int ks0, ks1;
};

__device__ __forceinline__ Split kstep_range(int nks, int S, int rank) {
  // balanced contiguous split of nks k-steps over S CTAs
  Split s;
  s.ks0 = (int)(((long long)nks * rank) / S);
  s.ks1 = (int)(((long long)nks * (rank + 1)) / S);
  return s;
}

// acc2 += (bits2 - magic2) * s2 for two tokens with packed f32x2 instructions.
__device__ __forceinline__ unsigned long long acc_pair(unsigned long long acc2, int bits_a, int bits_b,
                                                       unsigned long long s2) {
  unsigned long long f2;
  asm("{\n .reg .b64 b;\n mov.b64 b, {%1, %2};\n sub.rn.f32x2 %0, b, %3;\n}\n"
      : "=l"(f2)
      : "r"(bits_a), "r"(bits_b), "l"(kMagic2));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2) : "l"(f2), "l"(s2));
  return acc2;
}

__device__ __forceinline__ unsigned long long mul_pair(unsigned long long a2, unsigned long long b2) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a2), "l"(b2));
  return r;
}

__device__ __forceinline__ unsigned long long dup_pair(float x) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ unsigned long long make_pair(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ float2 unpack_pair(unsigned long long v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}

// The kernel.  A CTA (one per SM, 8 warps) works through tiles of G row
// groups of 32 rows (lane = row); the KW = 8 / G warps of a row group take
// interleaved k-steps of the CTA's k-range, and the S CTAs of a cluster split
// the k-range of the matrix.  Every warp handles all n_tok tokens of its rows
// and owns a 2-stage ring of weight stages (32 rows x 272 bytes, one 2-D
// tensor copy per stage): it loads a stage into registers (17 conflict-free 16-byte
// shared loads per lane; the 272-byte stride is an odd number of 16-byte bank
// groups), releases it to the copy two units ahead, and computes from
// registers while both stages are in flight.  No warp waits on another warp
// inside the k loop.
//
// Sums per token: each warp adds its blocks in k order; the KW warps of a row
// group are added in warp order (shared memory), then the S CTAs of a cluster
// in rank order (distributed shared memory).  None of this depends on n_tok,
// so column t of an n_tok = k call is bitwise the n_tok = 1 call.
//
// Activation source of a launch.  PRO 0: q8_0 rows xq.  PRO 3: the same
// activations already in the staged layout (written by the kernel that
// produced them), copied in as they are.  PRO 1: float rows xf
// (row stride xf_stride) that the kernel RMS-normalises (weight norm_w, eps)
// and quantises itself; PRO 2: float rows [gate | up] (gate at column c, up at
// column c + cols) that it turns into silu(gate) * up and quantises.  The
// prologues repeat the arithmetic of the standalone RMSNorm / SiLU-gate q8_0
// kernels step by step (the same sum-of-squares order, the same codec), so
// their codes and scales are bitwise those kernels' output.
struct ActSrc {
  const uint32_t* staged = nullptr;  // PRO 3: the activations already in the staged layout
  const uint8_t* xq = nullptr;
  const float* xf = nullptr;
  const float* norm_w = nullptr;
  float eps = 0.0f;
  int xf_stride = 0;
};

// From kMmaMinNt tokens on, the k loop runs on the tensor cores (warp-level
// mma.sync m16n8k16, f16 x f16 -> f32) instead of dp4a chains.  A q8_0 block
// is K = 32, two products: the weight codes enter as the f16 values 1152 + q
// (exact: integers below 2048), the activation codes as f16 q, and the
// accumulator starts at -1152 * sum(q_x) of the block, so the result is the
// exact integer block dot (every partial sum is an integer below 2^24).  The
// scaling that follows is the dp4a path's, operation for operation, so both
// paths give bitwise the same outputs.  The activation layout both paths read
// (use_mma, act_nta, act_pos) is in dsb_actlayout.cuh.

// d = a * b + c for f32 pairs.
__device__ __forceinline__ unsigned long long fma_pair(unsigned long long a, unsigned long long b,
                                                       unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// Four signed codes (bytes of x ^ 0x80808080) as two f16 pairs of 1152 + q:
// bytes 0, 1 -> lo, bytes 2, 3 -> hi.
__device__ __forceinline__ void codes_to_f16_offset(uint32_t xu, uint32_t& lo, uint32_t& hi) {
  lo = __byte_perm(xu, 0x64646464u, 0x4140);
  hi = __byte_perm(xu, 0x64646464u, 0x4342);
}

// The same, minus 1152: the codes themselves as f16 pairs (exact).
__device__ __forceinline__ void codes_to_f16(uint32_t xu, uint32_t& lo, uint32_t& hi) {
  codes_to_f16_offset(xu, lo, hi);
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x64806480u));
}

// D += A * B, one m16n8k16 tile (A row-major 16 x 16, B column-major 16 x 8).
__device__ __forceinline__ void mma_16816(float& d0, float& d1, float& d2, float& d3, uint32_t a0, uint32_t a1,
                                          uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Shared-memory layout (bytes), identical in every CTA of a cluster (the
// distributed-shared-memory reads rely on the sums sitting at one offset):
//   act codes [kr_alloc*8][8][NTA] u32 | act scales [kr_alloc*8][NTA] f32
//   (mma path: u32 = fp16 scale bits | int16 code sum << 16) |
//   stages [2][8 warps][8704] | warp partials [8][NT][32] f32 (G < 8) |
//   CTA sums [2][G][NT][32] f32 (S > 1) | mbarriers [8][2] + 1 | prologue scratch
struct SmemLayout {
  size_t act_s, stages, red, red_sum, bars, pro, total;
};

__host__ __device__ inline SmemLayout smem_layout(int kr_alloc, int nt, int G, int S, int pro) {
  SmemLayout L;
  const size_t nta = (size_t)act_nta(nt);
  size_t off = (size_t)kr_alloc * 8 * 8 * nta * 4;
  L.act_s = off;
  off += (size_t)kr_alloc * 8 * nta * 4;
  off = (off + 127) & ~(size_t)127;
  L.stages = off;
  off += (size_t)kWarps * kNStage * kStage;
  L.red = off;
  if (G < kWarps) off += (size_t)kWarps * nt * 32 * 4;
  L.red_sum = off;
  if (S > 1) off += (size_t)2 * G * nt * 32 * 4;
  L.bars = off;
  off += (size_t)(kWarps * kNStage + 1) * 8;
  L.pro = off;
  if (pro == 1) off += (size_t)nt * (kWarps + 1) * 4;
  L.total = off;
  return L;
}

template <int NT, bool EMIT, int PRO>
__global__ void __launch_bounds__(kThreads, 1)
    matmul_q8_0_narrow_kernel(const __grid_constant__ CUtensorMap tmw, int rows, int nb, const ActSrc src, float* y,
                              const float* residual, int32_t* __restrict__ isum_out, int G) {
  constexpr int NTA = act_nta(NT);
  constexpr int NP = (NT + 1) / 2;  // token pairs
  constexpr bool kMma = use_mma(NT);
  constexpr int NTN = NTA / 8;                               // mma path: 8-token tiles
  constexpr uint32_t kActXor = kMma ? 0x80808080u : 0u;  // mma path stores codes + 128 per byte
  extern __shared__ __align__(128) uint8_t smem[];
  const int nks = nb >> 3;
  const int S = gridDim.y;
  const int rank = blockIdx.y;  // cluster dims (1, S, 1): rank within the cluster
  const int n_clusters = gridDim.x;
  const Split ksr = kstep_range(nks, S, rank);
  const int kr = ksr.ks1 - ksr.ks0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KW = kWarps / G;
  const int grp = warp % G, kph = warp / G;
  const int tile_rows = G * kRowsPerWarp;
  const int tiles = (rows + tile_rows - 1) / tile_rows;
  const int n_tiles = (int)blockIdx.x < tiles ? (tiles - 1 - (int)blockIdx.x) / n_clusters + 1 : 0;
  const int kr_alloc = (nks + S - 1) / S;
  const SmemLayout L = smem_layout(kr_alloc, NT, G, S, PRO);
  uint32_t* act_q = reinterpret_cast<uint32_t*>(smem);
  float* act_s = reinterpret_cast<float*>(smem + L.act_s);
  uint32_t* act_su = reinterpret_cast<uint32_t*>(smem + L.act_s);  // mma path view
  // the fp16 scale (bits) of activation block idx = blk * NTA + t: as a float
  // (dp4a path), or kept as bits with the block's code sum (|sum| <= 4064) as
  // int16 in the high half (mma path: -1152 * sum starts the block's
  // tensor-core accumulator)
  auto store_scale = [&](size_t idx, uint32_t bits16, int code_sum) {
    if constexpr (kMma)
      act_su[idx] = (bits16 & 0xFFFFu) | ((uint32_t)code_sum << 16);
    else
      act_s[idx] = half_bits_to_float(bits16);
  };
  // activation word k of block blk (CTA-local) for token t
  auto act_word = [&](int blk, int k, int t) -> uint32_t& {
    return act_q[(size_t)(blk * 8 + k) * NTA + act_pos(NTA, kMma, k, t)];
  };
  // stage s of this warp at stages + (s * 8 + warp) * 8704: the second stages
  // of all warps are contiguous, and hold the raw activations at start-up
  auto stage_ptr = [&](int s) { return smem + L.stages + ((size_t)s * kWarps + warp) * kStage; };
  float* red = reinterpret_cast<float*>(smem + L.red);
  float* red_sum = reinterpret_cast<float*>(smem + L.red_sum);
  uint64_t* my_bars = reinterpret_cast<uint64_t*>(smem + L.bars) + warp * kNStage;
  uint64_t* act_bar = reinterpret_cast<uint64_t*>(smem + L.bars) + kWarps * kNStage;
  const int kSum = G * NT * 32;  // one CTA sum buffer (floats)

  if (lane == 0) {
    for (int s = 0; s < kNStage; ++s) mbar_init(&my_bars[s], 1);
    if (warp == 0) mbar_init(act_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // This warp's units: for each of the CTA's tiles m, the k-steps
  // ks0 + kph, ks0 + kph + KW, ... of the CTA's k-range.  Unit u = m*n_mine + i.
  const int n_mine = kr > kph ? (kr - kph + KW - 1) / KW : 0;
  const int n_units = n_tiles * n_mine;
  // Lane 0 requests unit u's stage with one 2-D tensor copy (rows past the
  // matrix read as zeros and are never stored); a row group wholly past the
  // end only arrives.
  auto issue = [&](int u) {
    if (lane != 0) return;
    const int m = u / n_mine, i = u - m * n_mine;
    const int row0 = ((int)blockIdx.x + m * n_clusters) * tile_rows + grp * kRowsPerWarp;
    const int ks = ksr.ks0 + kph + KW * i;
    uint64_t* bar = &my_bars[u % kNStage];
    if (row0 < rows) {
      mbar_arrive_expect_tx(bar, (uint32_t)kStage);
      tma_stage_2d(stage_ptr(u % kNStage), &tmw, ks * (kChunkBytes / 2), row0, bar);
    } else {
      mbar_arrive_expect_tx(bar, 0u);
    }
  };
  int issued = 0;  // units whose copies were requested
  // Weights do not depend on the previous kernel.  The second stages hold the
  // raw activation rows during start-up except when they arrive staged.
  for (int i = 0; i < (PRO == 3 ? kNStage : 1); ++i)
    if (issued < n_units) issue(issued++);
  pdl_wait();  // the activations (and y / residual) may be the previous kernel's results
  pdl_trigger();
  bool dead = false;

  if constexpr (PRO == 3) {
    // The CTA's k-range of the staged layout: codes [ks0*8, ks1*8) x 8 x NTA
    // and their scale words, two bulk copies (sizes multiples of 128 bytes).
    if (threadIdx.x == 0) {
      const uint32_t cb = (uint32_t)kr * 8 * 8 * NTA * 4, sb = (uint32_t)kr * 8 * NTA * 4;
      mbar_arrive_expect_tx(act_bar, cb + sb);
      bulk_g2s(act_q, src.staged + (size_t)ksr.ks0 * 8 * 8 * NTA, cb, act_bar);
      bulk_g2s(act_su, src.staged + (size_t)nb * 8 * NTA + (size_t)ksr.ks0 * 8 * NTA, sb, act_bar);
    }
    const bool ok = mbar_wait(act_bar, 0u);
    dead = __syncthreads_or(!ok) != 0;
    if (dead && threadIdx.x == 0) g_err_matmul = 1u;
  } else if constexpr (PRO == 0) {
    // Unpack the CTA's activation blocks [ks0*8, ks1*8) x NT into the
    // word-major form.  The rows arrive by one 1-D bulk copy per token (kr *
    // 272 bytes, 16-byte aligned) into the second weight stages, which no copy
    // uses yet, in as many rounds of tokens as that region needs.  Item
    // (k-step j, token t), tokens fastest: the 272 bytes of token t's row for
    // k-step ks0 + j (8 blocks), split into codes and scales as the weight
    // chunks are, and stored word-major (consecutive threads write consecutive
    // tokens).
    uint8_t* raw = smem + L.stages + (size_t)kWarps * kStage;
    const int row_raw = kr * kChunkBytes;
    int per_round = (kWarps * kStage) / row_raw;
    if (per_round > NT) per_round = NT;
    for (int t0 = 0, rd = 0; t0 < NT && !dead; t0 += per_round, ++rd) {
      const int tn = NT - t0 < per_round ? NT - t0 : per_round;
      if (rd > 0) {
        // the previous round's reads of the raw rows precede the next copies
        fence_proxy_async_smem();
        __syncthreads();
      }
      if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(act_bar, (uint32_t)(tn * row_raw));
        for (int t = 0; t < tn; ++t)
          bulk_g2s(raw + (size_t)t * row_raw, src.xq + (size_t)(t0 + t) * nb * 34 + (size_t)ksr.ks0 * kChunkBytes,
                   (uint32_t)row_raw, act_bar);
      }
      const bool ok = mbar_wait(act_bar, (uint32_t)(rd & 1));
      dead = __syncthreads_or(!ok) != 0;
      if (dead) {
        if (threadIdx.x == 0) g_err_matmul = 1u;
        break;
      }
      for (int it = threadIdx.x; it < kr * tn; it += kThreads) {
        const int j = it / tn, tl = it - j * tn, t = t0 + tl;
        const uint4* rp = reinterpret_cast<const uint4*>(raw + (size_t)tl * row_raw + (size_t)j * kChunkBytes);
        uint32_t wv[68];
#pragma unroll
        for (int c = 0; c < 17; ++c) {
          const uint4 v = rp[c];
          wv[4 * c + 0] = v.x;
          wv[4 * c + 1] = v.y;
          wv[4 * c + 2] = v.z;
          wv[4 * c + 3] = v.w;
        }
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          int sx = 0;  // the block's code sum (mma path)
          if ((b & 1) == 0) {
            const int base = (17 * b) / 2;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t x = __funnelshift_r(wv[base + k], wv[base + k + 1], 16);
              if constexpr (kMma) sx = __dp4a((int)x, 0x01010101, sx);
              act_word(j * 8 + b, k, t) = x ^ kActXor;
            }
            store_scale((size_t)(j * 8 + b) * NTA + t, wv[base], sx);
          } else {
            const int base = (17 * b - 1) / 2;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t x = wv[base + 1 + k];
              if constexpr (kMma) sx = __dp4a((int)x, 0x01010101, sx);
              act_word(j * 8 + b, k, t) = x ^ kActXor;
            }
            store_scale((size_t)(j * 8 + b) * NTA + t, wv[base] >> 16, sx);
          }
        }
      }
    }
    if constexpr (NTA > NT) {
      // the pad tokens NT..NTA-1 hold zero words and scales
      for (int idx = threadIdx.x; idx < kr * 8 * 9 * (NTA - NT); idx += kThreads) {
        const int bw = idx / (NTA - NT), t = NT + idx - bw * (NTA - NT);  // bw: (block, word 0..7 | scale 8)
        const int b = bw / 9, k = bw - b * 9;
        if (k < 8)
          act_word(b, k, t) = kActXor;
        else
          act_su[(size_t)b * NTA + t] = 0u;  // 0.0f in either form
      }
    }
  } else {
    // The pad tokens NT..NTA-1 hold zero words and scales.
    for (int idx = threadIdx.x; idx < kr * 8 * 8; idx += kThreads)
      for (int t = NT; t < NTA; ++t) act_word(idx >> 3, idx & 7, t) = kActXor;
    for (int idx = threadIdx.x; idx < kr * 8; idx += kThreads)
      for (int t = NT; t < NTA; ++t) act_su[(size_t)idx * NTA + t] = 0u;  // 0.0f in either form
    const int cols = nb * 32;
    float* inv_s = reinterpret_cast<float*>(smem + L.pro);  // [NT]
    float* part_s = inv_s + NT;                              // [NT][8]
    if constexpr (PRO == 1) {
      // each token row's 1 / sqrt(mean(x^2) + eps): thread j sums elements
      // j, j + 256, ... (fused multiply-adds in that order), an xor tree in
      // the warp, then the 8 warps in order
      const int n = cols / kThreads;
      float ss[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) ss[t] = 0.0f;
      for (int k = 0; k < n; ++k) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const float v = __ldcg(src.xf + (size_t)t * src.xf_stride + threadIdx.x + k * kThreads);
          ss[t] = __fmaf_rn(v, v, ss[t]);
        }
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        float v = ss[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) part_s[t * 8 + warp] = v;
      }
      __syncthreads();
      if (threadIdx.x < NT) {
        float tot = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) tot = __fadd_rn(tot, part_s[threadIdx.x * 8 + i]);
        inv_s[threadIdx.x] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)cols), src.eps)));
      }
      __syncthreads();
    }
    // one thread per (block, token) of the CTA's k-range: its 32 values in
    // eight 16-byte loads, then the q8_0 codec as the standalone kernels
    // apply it (the block maximum does not depend on the order)
    for (int pi = threadIdx.x; pi < kr * 8 * NT; pi += kThreads) {
      const int b = pi / NT, t = pi - b * NT;
      const int e0 = (ksr.ks0 * 8 + b) * 32;
      const float4* row = reinterpret_cast<const float4*>(src.xf + (size_t)t * src.xf_stride + e0);
      float v[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 f = __ldcg(row + i);
        v[4 * i] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
      }
      if constexpr (PRO == 1) {
        const float inv = inv_s[t];
        const float4* wr = reinterpret_cast<const float4*>(src.norm_w + e0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 wv = __ldg(wr + i);
          v[4 * i] = __fmul_rn(__fmul_rn(v[4 * i], inv), wv.x);
          v[4 * i + 1] = __fmul_rn(__fmul_rn(v[4 * i + 1], inv), wv.y);
          v[4 * i + 2] = __fmul_rn(__fmul_rn(v[4 * i + 2], inv), wv.z);
          v[4 * i + 3] = __fmul_rn(__fmul_rn(v[4 * i + 3], inv), wv.w);
        }
      } else {
        const float4* up = row + cols / 4;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 u = __ldcg(up + i);
          const float uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float gg = v[4 * i + j];
            v[4 * i + j] = __fmul_rn(__fdiv_rn(gg, __fadd_rn(1.0f, expf(-gg))), uu[j]);
          }
        }
      }
      float a = 0.0f;
#pragma unroll
      for (int j = 0; j < 32; ++j) a = fmaxf(a, fabsf(v[j]));
      const float d = __fdiv_rn(a, 127.0f);
      int sx = 0;  // the block's code sum (mma path)
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          int q = 0;
          if (d != 0.0f) q = (int)fminf(fmaxf(roundf(__fdiv_rn(v[4 * k + j], d)), -127.0f), 127.0f);
          word |= ((uint32_t)q & 0xFFu) << (8 * j);
        }
        if constexpr (kMma) sx = __dp4a((int)word, 0x01010101, sx);
        act_word(b, k, t) = word ^ kActXor;
      }
      store_scale((size_t)b * NTA + t, __half_as_ushort(__float2half_rn(d)), sx);
    }
  }
  // every thread's reads of the raw rows precede the copies into those stages
  fence_proxy_async_smem();
  __syncthreads();
  while (!dead && issued < n_units && issued < kNStage) issue(issued++);

  // Cross-CTA sums: the CTA sum of tile m goes to buffer m & 1 and the CTA
  // arrives on the cluster barrier; it waits, and adds the cluster's sums of
  // tile m (its slice, ranks in order), only after computing tile m + 1.  A
  // buffer is rewritten two tiles later, after the next wait, which no CTA
  // passes before every CTA has read it.
  const bool cluster_sums = !EMIT && S > 1;
  // A tile's cluster sums are finished in two halves: gather_tile reads the
  // S ranks' sums of this CTA's slice over distributed shared memory and adds
  // them in rank order into registers (before this CTA's next arrive, which
  // releases the buffer); finish_tile adds the residual and stores y after
  // that arrive, so the arrive never waits for global stores.  A slice holds
  // at most G*NT*32 / (2*256) <= 8 outputs per thread.
  // A slice holds at most G*NT*32 / (2*256) <= 8 outputs per thread, read as
  // 16-byte quads (4 consecutive rows of one token).
  constexpr int kMaxQuad = 2;
  float4 vsum[kMaxQuad];
  auto gather_tile = [&](int m) {
    const float* rs = red_sum + (m & 1) * kSum;
    uint32_t base[kMaxCluster];  // this buffer in each rank's shared window
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r)
      if (r < S) base[r] = cluster_map(rs, (uint32_t)r);
#pragma unroll
    for (int jq = 0; jq < kMaxQuad; ++jq) {
      const int qd = rank * kThreads + (int)threadIdx.x + jq * S * kThreads;
      if (qd < kSum / 4) {
        float4 part[kMaxCluster];  // every rank's load in flight before the adds
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r)
          if (r < S) part[r] = ld_cluster_v4(base[r] + 16u * (uint32_t)qd);
        float4 v = part[0];
#pragma unroll
        for (int r = 1; r < kMaxCluster; ++r)
          if (r < S) {
            v.x = __fadd_rn(v.x, part[r].x);
            v.y = __fadd_rn(v.y, part[r].y);
            v.z = __fadd_rn(v.z, part[r].z);
            v.w = __fadd_rn(v.w, part[r].w);
          }
        vsum[jq] = v;
      }
    }
  };
  auto finish_tile = [&](int m) {
    const int row0 = ((int)blockIdx.x + m * n_clusters) * tile_rows;
#pragma unroll
    for (int jq = 0; jq < kMaxQuad; ++jq) {
      const int qd = rank * kThreads + (int)threadIdx.x + jq * S * kThreads;
      if (qd < kSum / 4) {
        const int idx = 4 * qd;
        const int gq = idx / (NT * 32);  // row group of this output
        const int t = (idx / 32) % NT, r0 = row0 + gq * kRowsPerWarp + (idx & 31);
        const float vv[4] = {vsum[jq].x, vsum[jq].y, vsum[jq].z, vsum[jq].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (r0 + e < rows) {
            const size_t o = (size_t)t * rows + r0 + e;
            y[o] = residual ? __fadd_rn(__ldcg(residual + o), vv[e]) : vv[e];  // residual may alias y
          }
        }
      }
    }
  };

  int u = 0, landed = 0;  // landed: units whose stage wait succeeded
  for (int m = 0; m < n_tiles; ++m) {
    const int row0 = ((int)blockIdx.x + m * n_clusters) * tile_rows;
    const int row = row0 + grp * kRowsPerWarp + lane;
    unsigned long long acc2[kMma ? 1 : NP];
    unsigned long long accm[kMma ? 4 : 1][kMma ? NTN : 1];
    if constexpr (kMma) {
#pragma unroll
      for (int ri = 0; ri < 4; ++ri)
#pragma unroll
        for (int n = 0; n < NTN; ++n) accm[ri][n] = 0ull;
    } else {
#pragma unroll
      for (int p = 0; p < NP; ++p) acc2[p] = 0ull;
    }

    for (int i = 0; i < n_mine; ++i, ++u) {
      const int ks = ksr.ks0 + kph + KW * i;
      const int kl = ks - ksr.ks0;
      uint64_t* bar = &my_bars[u % kNStage];
      if (!dead) {
        const bool ok = mbar_wait(bar, (uint32_t)((u / kNStage) & 1));
        dead = __any_sync(0xffffffffu, !ok);  // warp-uniform
        if (dead && lane == 0) g_err_matmul = 1u;
        if (!dead) landed = u + 1;
      }
      // Every lane's reads of the stage are ordered before the copy that
      // overwrites it (the copy writes through the async proxy).
      auto release = [&]() {
        fence_proxy_async_smem();
        __syncwarp();
        if (!dead && u + kNStage < n_units) {
          issue(u + kNStage);
          issued = u + kNStage + 1;
        }
      };
      if constexpr (kMma) {
        // Lane 4g + c holds, for rows 8ri + g (ri = 0..3: the two 16-row
        // tiles' upper and lower halves), code words c and 4 + c of every
        // block of the k-step (the K order inside a block is permuted the same
        // way for weights and activations), plus the rows' scales.  Block b
        // starts at byte 34b of a row: an even block's codes start 2 bytes
        // past a word boundary (two words per code word, byte_perm), an odd
        // block's on one.  Row r's words start at bank 4r, so every load hits
        // 32 distinct banks.
        const int g = lane >> 2, c = lane & 3;
        const uint32_t* st = reinterpret_cast<const uint32_t*>(stage_ptr(u % kNStage));
        uint32_t wq[4][8][2];
        uint32_t wsc[4][4];  // scales of blocks 2j (low half) and 2j + 1 (high half)
#pragma unroll
        for (int ri = 0; ri < 4; ++ri) {
          const uint32_t* rp = st + (8 * ri + g) * (kChunkBytes / 4);
#pragma unroll
          for (int b = 0; b < 8; b += 2) {
            const int w0 = (34 * b) / 4;            // even block: scale in the low half of word w0
            const int w1 = (34 * (b + 1) + 2) / 4;  // odd block: codes from word w1, scale in the high half of w1 - 1
            const uint32_t v0 = rp[w0 + c], v1 = rp[w0 + c + 1], v4 = rp[w0 + c + 4], v5 = rp[w0 + c + 5];
            wq[ri][b][0] = __byte_perm(v0, v1, 0x5432);
            wq[ri][b][1] = __byte_perm(v4, v5, 0x5432);
            wq[ri][b + 1][0] = rp[w1 + c];
            wq[ri][b + 1][1] = rp[w1 + c + 4];
            wsc[ri][b / 2] = __byte_perm(rp[w0], rp[w1 - 1], 0x7610);
          }
        }
        release();
        __syncwarp();  // the warp-wide tensor-core products below run converged

#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const int kb = kl * 8 + b;
          uint32_t af[4][2][2];  // [row ri][half h][slots 2c, 2c+1 | 2c+8, 2c+9]
          float dw[4];
#pragma unroll
          for (int ri = 0; ri < 4; ++ri) {
#pragma unroll
            for (int h = 0; h < 2; ++h) codes_to_f16_offset(wq[ri][b][h] ^ 0x80808080u, af[ri][h][0], af[ri][h][1]);
            dw[ri] = half_bits_to_float((b & 1) ? (wsc[ri][b / 2] >> 16) : wsc[ri][b / 2]);
          }
#pragma unroll
          for (int n = 0; n < NTN; ++n) {
            const int tb = 8 * n;
            uint32_t bf[2][2];
#pragma unroll
            for (int h = 0; h < 2; ++h) codes_to_f16(act_word(kb, 4 * h + c, tb + g), bf[h][0], bf[h][1]);
            // tokens tb + 2c, tb + 2c + 1: scales and -1152 * code sums
            const uint2 sc = *reinterpret_cast<const uint2*>(act_su + (size_t)kb * NTA + tb + 2 * c);
            const unsigned long long sx2 = make_pair(half_bits_to_float(sc.x), half_bits_to_float(sc.y));
            const float cx0 = -1152.0f * (float)((int)sc.x >> 16), cx1 = -1152.0f * (float)((int)sc.y >> 16);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              float d0 = cx0, d1 = cx1, d2 = cx0, d3 = cx1;
              mma_16816(d0, d1, d2, d3, af[2 * mt][0][0], af[2 * mt + 1][0][0], af[2 * mt][0][1],
                        af[2 * mt + 1][0][1], bf[0][0], bf[0][1]);
              mma_16816(d0, d1, d2, d3, af[2 * mt][1][0], af[2 * mt + 1][1][0], af[2 * mt][1][1],
                        af[2 * mt + 1][1][1], bf[1][0], bf[1][1]);
              if constexpr (EMIT) {
                const float dd[4] = {d0, d1, d2, d3};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int r = row0 + grp * kRowsPerWarp + 16 * mt + 8 * (e >> 1) + g, t = tb + 2 * c + (e & 1);
                  if (r < rows && t < NT)
                    isum_out[((size_t)t * rows + r) * nb + (size_t)ks * 8 + b] = __float2int_rn(dd[e]);
                }
              } else {
                accm[2 * mt][n] = fma_pair(make_pair(d0, d1), mul_pair(dup_pair(dw[2 * mt]), sx2), accm[2 * mt][n]);
                accm[2 * mt + 1][n] =
                    fma_pair(make_pair(d2, d3), mul_pair(dup_pair(dw[2 * mt + 1]), sx2), accm[2 * mt + 1][n]);
              }
            }
          }
        }
      } else {
        const uint4* stg =
            reinterpret_cast<const uint4*>(stage_ptr(u % kNStage) + lane * kChunkBytes);
        uint32_t w[68];
#pragma unroll
        for (int c = 0; c < 17; ++c) {
          const uint4 v = stg[c];
          w[4 * c + 0] = v.x;
          w[4 * c + 1] = v.y;
          w[4 * c + 2] = v.z;
          w[4 * c + 3] = v.w;
        }
        release();

#pragma unroll
        for (int b = 0; b < 8; ++b) {
          uint32_t q[8];
          float dw;
          if ((b & 1) == 0) {
            const int base = (17 * b) / 2;
#pragma unroll
            for (int k = 0; k < 8; ++k) q[k] = __funnelshift_r(w[base + k], w[base + k + 1], 16);
            dw = half_bits_to_float(w[base]);
          } else {
            const int base = (17 * b - 1) / 2;
#pragma unroll
            for (int k = 0; k < 8; ++k) q[k] = w[base + 1 + k];
            dw = half_bits_to_float(w[base] >> 16);
          }
          const uint32_t* aq = act_q + (size_t)(kl * 8 + b) * 8 * NTA;
          const float* as = act_s + (size_t)(kl * 8 + b) * NTA;
          const unsigned long long dw2 = dup_pair(dw);
          // every token's chain advances word by word together (NT independent
          // dp4a chains); one broadcast 16-byte load gives word k of four tokens
          int sd[NT];
#pragma unroll
          for (int t = 0; t < NT; ++t) sd[t] = (int)kMagic;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
#pragma unroll
            for (int t4 = 0; t4 < NT; t4 += 4) {
              const int cnt = NT - t4 < 4 ? NT - t4 : 4;
              if (cnt >= 3) {
                const uint4 a = *reinterpret_cast<const uint4*>(aq + k * NTA + t4);
                sd[t4] = __dp4a((int)q[k], (int)a.x, sd[t4]);
                sd[t4 + 1] = __dp4a((int)q[k], (int)a.y, sd[t4 + 1]);
                sd[t4 + 2] = __dp4a((int)q[k], (int)a.z, sd[t4 + 2]);
                if (cnt == 4) sd[t4 + 3] = __dp4a((int)q[k], (int)a.w, sd[t4 + 3]);
              } else if (cnt == 2) {
                const uint2 a = *reinterpret_cast<const uint2*>(aq + k * NTA + t4);
                sd[t4] = __dp4a((int)q[k], (int)a.x, sd[t4]);
                sd[t4 + 1] = __dp4a((int)q[k], (int)a.y, sd[t4 + 1]);
              } else {
                sd[t4] = __dp4a((int)q[k], (int)aq[k * NTA + t4], sd[t4]);
              }
            }
          }
          if constexpr (EMIT) {
            if (row < rows) {
#pragma unroll
              for (int t = 0; t < NT; ++t)
                isum_out[((size_t)t * rows + row) * nb + (size_t)ks * 8 + b] = sd[t] - (int)kMagic;
            }
          } else {
#pragma unroll
            for (int t4 = 0; t4 < NT; t4 += 4) {
              const int cnt = NT - t4 < 4 ? NT - t4 : 4;
              if (cnt >= 3) {
                const float4 sx = *reinterpret_cast<const float4*>(as + t4);
                acc2[t4 / 2] = acc_pair(acc2[t4 / 2], sd[t4], sd[t4 + 1], mul_pair(dw2, make_pair(sx.x, sx.y)));
                acc2[t4 / 2 + 1] = acc_pair(acc2[t4 / 2 + 1], sd[t4 + 2], cnt == 4 ? sd[t4 + 3] : (int)kMagic,
                                            mul_pair(dw2, make_pair(sx.z, sx.w)));
              } else if (cnt == 2) {
                const float2 sx = *reinterpret_cast<const float2*>(as + t4);
                acc2[t4 / 2] = acc_pair(acc2[t4 / 2], sd[t4], sd[t4 + 1], mul_pair(dw2, make_pair(sx.x, sx.y)));
              } else {
                acc2[t4 / 2] = acc_pair(acc2[t4 / 2], sd[t4], (int)kMagic, mul_pair(dw2, dup_pair(as[t4])));
              }
            }
          }
        }
      }
    }

    if constexpr (!EMIT) {
      // this thread's outputs as (row within the warp's 32, token, value)
      float acc[kMma ? 1 : NT];
      if constexpr (!kMma) {
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          const float2 v = unpack_pair(acc2[p]);
          acc[2 * p] = v.x;
          if (2 * p + 1 < NT) acc[2 * p + 1] = v.y;
        }
      }
      auto for_outputs = [&](auto&& f) {
        if constexpr (kMma) {
          const int g = lane >> 2, c = lane & 3;
#pragma unroll
          for (int ri = 0; ri < 4; ++ri)
#pragma unroll
            for (int n = 0; n < NTN; ++n) {
              const float2 v = unpack_pair(accm[ri][n]);
              const int t = 8 * n + 2 * c;
              if (t < NT) f(8 * ri + g, t, v.x);
              if (t + 1 < NT) f(8 * ri + g, t + 1, v.y);
            }
        } else {
#pragma unroll
          for (int t = 0; t < NT; ++t) f(lane, t, acc[t]);
        }
      };
      if (KW == 1 && S == 1) {
        // One warp owns these rows over the whole k: write them directly.
        for_outputs([&](int rl, int t, float v) {
          const int r = row0 + grp * kRowsPerWarp + rl;
          if (r < rows) {
            const size_t o = (size_t)t * rows + r;
            y[o] = residual ? __fadd_rn(__ldcg(residual + o), v) : v;  // residual may alias y
          }
        });
      } else {
        // the previous tile's cluster sums, now that this tile is computed
        if (cluster_sums && m > 0) {
          cluster_wait();
          gather_tile(m - 1);
        }
        float* rs = red_sum + (m & 1) * kSum;
        if (KW == 1) {
          for_outputs([&](int rl, int t, float v) { rs[(grp * NT + t) * 32 + rl] = v; });
        } else {
          // the KW warps of each row group, added in warp (k-phase) order
          for_outputs([&](int rl, int t, float v) { red[(warp * NT + t) * 32 + rl] = v; });
          __syncthreads();
          for (int idx = threadIdx.x; idx < kSum; idx += kThreads) {
            const int gq = idx / (NT * 32), rest = idx - gq * NT * 32;
            float v = red[gq * NT * 32 + rest];
            for (int p2 = 1; p2 < KW; ++p2) v = __fadd_rn(v, red[(p2 * G + gq) * NT * 32 + rest]);
            if (cluster_sums) {
              rs[idx] = v;
            } else {
              const int t = rest / 32, rr = row0 + gq * kRowsPerWarp + (rest & 31);
              if (rr < rows) {
                const size_t o = (size_t)t * rows + rr;
                y[o] = residual ? __fadd_rn(__ldcg(residual + o), v) : v;
              }
            }
          }
          __syncthreads();  // every partial read before the next tile rewrites them
        }
        if (cluster_sums) {
          cluster_arrive();
          if (m > 0) finish_tile(m - 1);
        }
      }
    }
  }
  if (cluster_sums && n_tiles > 0) {
    cluster_wait();
    gather_tile(n_tiles - 1);
    // keep this CTA's sums alive until every CTA of the cluster has read them
    cluster_arrive();
    finish_tile(n_tiles - 1);
    cluster_wait();
  }
  if (dead) {
    // A wait ran out: give the copies still in flight (units landed ..
    // issued - 1) a bounded chance to land before the CTA's shared memory is
    // released.
    for (int v = landed; v < issued; ++v) (void)mbar_wait(&my_bars[v % kNStage], (uint32_t)((v / kNStage) & 1));
  }
}

size_t smem_bytes(int kr, int nt, int G, int S, int pro = 0) { return smem_layout(kr, nt, G, S, pro).total; }

// The weight matrix as a 2-D tensor of 16-bit elements, [rows][cols/32*17],
// read in boxes of 136 x 32 (one k-step of 32 rows, 8704 bytes, no swizzle).
// Encoded on the host and cached by (address, shape).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

cudaError_t weight_tensor_map(const void* W, int rows, int nb, CUtensorMap* out) {
  struct Entry {
    const void* base;
    int rows, nb;
    CUtensorMap map;
  };
  static std::mutex mu;
  static Entry cache[64];
  static int n_cache = 0, next_slot = 0;
  static EncodeTiledFn encode = nullptr;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_cache; ++i)
    if (cache[i].base == W && cache[i].rows == rows && cache[i].nb == nb) {
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
  const cuuint64_t dims[2] = {(cuuint64_t)nb * 17, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)nb * 34};
  const cuuint32_t box[2] = {(cuuint32_t)(kChunkBytes / 2), (cuuint32_t)kRowsPerWarp};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  const CUresult r = encode(&m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(W), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const int slot = n_cache < 64 ? n_cache++ : (next_slot++ & 63);
  cache[slot] = Entry{W, rows, nb, m};
  *out = m;
  return cudaSuccess;
}

// Per-instantiation host caches, each behind its own lock: the largest
// dynamic shared memory granted so far, and the number of co-resident clusters
// for each (S, smem) seen.  The attributes are per function, the same for every
// device of one architecture.
template <int NT, bool EMIT, int PRO>
cudaError_t grant_smem(size_t smem) {
  static std::mutex mu;
  static size_t granted = 0;
  static bool non_portable = false;
  std::lock_guard<std::mutex> lock(mu);
  if (!non_portable) {
    cudaError_t e = cudaFuncSetAttribute(matmul_q8_0_narrow_kernel<NT, EMIT, PRO>,
                                         cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    non_portable = true;
  }
  if (smem <= granted) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(matmul_q8_0_narrow_kernel<NT, EMIT, PRO>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) granted = smem;
  return e;
}

template <int NT, bool EMIT, int PRO>
cudaError_t cluster_capacity(int S, size_t smem, int* clusters) {
  struct Entry {
    int S;
    size_t smem;
    int clusters;
  };
  static std::mutex mu;
  static Entry cache[32];
  static int n_cache = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_cache; ++i)
    if (cache[i].S == S && cache[i].smem == smem) {
      *clusters = cache[i].clusters;
      return cudaSuccess;
    }
  cudaError_t e = grant_smem<NT, EMIT, PRO>(smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)S;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.gridDim = dim3(1, (unsigned)S, 1);
  int c = 0;
  e = cudaOccupancyMaxActiveClusters(&c, matmul_q8_0_narrow_kernel<NT, EMIT, PRO>, &cfg);
  if (e != cudaSuccess) return e;
  cache[n_cache < 32 ? n_cache++ : 31] = Entry{S, smem, c};
  *clusters = c;
  return cudaSuccess;
}

template <int NT, bool EMIT, int PRO>
cudaError_t launch_nt(const uint8_t* W, int rows, int nb, const ActSrc& src, float* y, const float* residual,
                      int32_t* isum, int G, int S, size_t smem, cudaStream_t st) {
  auto kern = matmul_q8_0_narrow_kernel<NT, EMIT, PRO>;
  // The persistent grid: as many clusters as fit at once, up to one per tile.
  int resident = 0;
  cudaError_t e = cluster_capacity<NT, EMIT, PRO>(S, smem, &resident);
  if (e != cudaSuccess) return e;
  if (resident < 1) return cudaErrorInvalidConfiguration;
  CUtensorMap tmw;
  if ((e = weight_tensor_map(W, rows, nb, &tmw)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)S;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  const int tile = G * kRowsPerWarp;
  const int tiles = (rows + tile - 1) / tile;
  const int n_clusters = tiles < resident ? tiles : resident;
  cfg.gridDim = dim3((unsigned)n_clusters, (unsigned)S, 1);
  cfg.numAttrs = pdl() ? 2 : 1;
  if (dry_run()) return cudaSuccess;
  return cudaLaunchKernelEx(&cfg, kern, tmw, rows, nb, src, y, residual, isum, G);
}

template <bool EMIT, int PRO>
cudaError_t dispatch(int nt, const uint8_t* W, int rows, int nb, const ActSrc& src, float* y, const float* residual,
                     int32_t* isum, int G, int S, size_t smem, cudaStream_t st) {
  switch (nt) {
#define DSB_CASE(N) \
  case N:           \
    return launch_nt<N, EMIT, PRO>(W, rows, nb, src, y, residual, isum, G, S, smem, st);
    DSB_CASE(1) DSB_CASE(2) DSB_CASE(3) DSB_CASE(4) DSB_CASE(5) DSB_CASE(6) DSB_CASE(7) DSB_CASE(8)
    DSB_CASE(9) DSB_CASE(10) DSB_CASE(11) DSB_CASE(12) DSB_CASE(13) DSB_CASE(14) DSB_CASE(15) DSB_CASE(16)
#undef DSB_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

// This unit's device error flag (a bounded wait ran out), read and cleared.
inline unsigned int read_clear_error_unit() {
  unsigned int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_matmul, sizeof v) != cudaSuccess) return 0xFFFFFFFFu;
  cudaMemcpyToSymbol(g_err_matmul, &z, sizeof z);
  return v;
}

}  // namespace
}  // namespace dsbk
