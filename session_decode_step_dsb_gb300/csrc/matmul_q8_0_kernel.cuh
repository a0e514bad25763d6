// The narrow-batch q8_0 matmul kernel template and its launch helpers, shared
// by the translation units that instantiate it (q8_0 activations in one, the
// fused RMSNorm / SiLU-gate activation prologues in another, compiled in
// parallel).  Everything here has internal linkage: each unit holds its own
// instances, host caches and device error flag.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <type_traits>

#include "dsb_kernels.h"
#include "dsb_ptx.cuh"

namespace dsbk {

namespace {

constexpr int kPairs = 4;             // row groups (or k-step lanes) of a CTA
constexpr int kWarps = 2 * kPairs;     // two warps per row group: one per token half
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerCta = 32;
constexpr int kChunkBytes = 272;  // 8 blocks of 34 bytes
constexpr int kStage = kRowsPerCta * kChunkBytes;
constexpr int kNStage = 2;
constexpr int kMaxCluster = 16;  // k-split CTAs per cluster (above 8: a non-portable cluster size)
constexpr uint32_t kMagic = 0x4B400000u;  // bits of 12582912.0f = 1.5 * 2^23
constexpr unsigned long long kMagic2 = 0x4B4000004B400000ull;

__device__ unsigned int g_err_matmul = 0;

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

__device__ __forceinline__ float2 unpack_pair(unsigned long long v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}

// The 8 warps form 4 pairs; the two warps of a pair read the same weight
// stages (one 2-stage ring per pair) and take the first and second half of the
// tokens, so a weight byte crosses shared memory once per pair while twice as
// many warps hide the latencies.  The first warp of a pair refills a stage once
// both hold it in registers (a 64-thread named barrier per k-step; it let the
// refill go out earlier than polled "empty" mbarriers did).
// ROWS = false (few-row matrices): a CTA tile is 32 rows and its 4 pairs
//   take interleaved k-steps of the CTA's k-range; pair partials are added in
//   pair order at each tile end.
// ROWS = true (many-row matrices): a CTA tile is 128 rows, pair p owns rows
//   32p..32p+31 over the whole k-range; no partials are exchanged between
//   pairs, and with S = 1 no CTA-wide barrier is taken after start-up.
// In both modes the S CTAs of a cluster split k and their sums are added in
// rank order through distributed shared memory.  Token t's arithmetic (block
// order, k-step order, pair and rank order) does not depend on n_tok.
// Activation source of a launch.  PRO 0: q8_0 rows xq.  PRO 1: float rows xf
// (row stride xf_stride) that the kernel RMS-normalises (weight norm_w, eps)
// and quantises itself; PRO 2: float rows [gate | up] (gate at column c, up at
// column c + cols) that it turns into silu(gate) * up and quantises.  The
// prologues repeat the arithmetic of the standalone RMSNorm / SiLU-gate q8_0
// kernels step by step (the same sum-of-squares order, the same codec), so
// their codes and scales are bitwise those kernels' output.
struct ActSrc {
  const uint8_t* xq = nullptr;
  const float* xf = nullptr;
  const float* norm_w = nullptr;
  float eps = 0.0f;
  int xf_stride = 0;
};

template <int NT, bool EMIT, bool ROWS, int PRO>
__global__ void __launch_bounds__(kThreads, 2)
    matmul_q8_0_narrow_kernel(const uint8_t* __restrict__ W, int rows, int nb, const ActSrc src,
                              float* y, const float* residual, int32_t* __restrict__ isum_out) {
  const uint8_t* xq = src.xq;
  constexpr int kTile = ROWS ? kPairs * kRowsPerCta : kRowsPerCta;
  constexpr int kRed = ROWS ? 0 : kPairs * NT * 32;          // pair partials (k-split mode)
  constexpr int kSum = (ROWS ? kPairs : 1) * NT * 32;        // one CTA sum buffer
  // Token halves: the first warp of a pair takes NTH0 tokens, the second the
  // rest.  NTH is even, so both halves start on an even token and their word
  // and scale pairs load as aligned 8-byte words; n_tok <= 2 is not split.
  constexpr int NTH = ((NT + 1) / 2 + 1) & ~1;
  constexpr int NTH0 = NTH < NT ? NTH : NT;
  constexpr int NTP = 2 * NTH;            // scale row stride: both halves' pairs within the row
  constexpr int NTA = (NT + 3) & ~3;      // word row stride: four tokens per 16-byte load
  extern __shared__ __align__(128) uint8_t smem[];
  const int nks = nb >> 3;
  const int S = gridDim.y;
  const int rank = blockIdx.y;  // cluster dims (1, S, 1): rank within the cluster
  const int n_clusters = gridDim.x;
  const Split ksr = kstep_range(nks, S, rank);
  const int kr = ksr.ks1 - ksr.ks0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = warp & (kPairs - 1), half = warp / kPairs;
  const int t0 = half ? NTH0 : 0;                  // this warp's first token
  const size_t row_bytes = (size_t)nb * 34;
  const int tiles = (rows + kTile - 1) / kTile;
  const int n_tiles = (int)blockIdx.x < tiles ? (tiles - 1 - (int)blockIdx.x) / n_clusters + 1 : 0;
  const int warp_row = ROWS ? pair * kRowsPerCta : 0;

  // Shared layout: act codes | act scales | stage rings | warp partials |
  // CTA sums (double-buffered) | barriers.  The act region is sized for the
  // largest k-range of the cluster in every CTA, so all CTAs of a cluster put
  // the CTA sums at the same offset -- the distributed-shared-memory reads of
  // rank 0 rely on that.
  const int kr_alloc = (nks + S - 1) / S;
  uint32_t* act_q = reinterpret_cast<uint32_t*>(smem);                               // [kr*8][8][NTA]
  float* act_s = reinterpret_cast<float*>(act_q + (size_t)kr_alloc * 8 * 8 * NTA);  // [kr*8][NTP]
  uint8_t* stages = reinterpret_cast<uint8_t*>(act_s + (size_t)kr_alloc * 8 * NTP);  // [kPairs][kNStage][kStage]
  float* red = reinterpret_cast<float*>(stages + (size_t)kPairs * kNStage * kStage);  // [kPairs][NT][32]
  float* red_sum = red + kRed;                                                        // [2][kSum]
  uint64_t* bars = reinterpret_cast<uint64_t*>(red_sum + 2 * kSum);                  // [kPairs][kNStage]
  uint8_t* my_stages = stages + (size_t)pair * kNStage * kStage;
  uint64_t* my_bars = bars + pair * kNStage;
  constexpr int kReaders = NT > NTH0 ? 2 : 1;       // warps of a pair with tokens

  if (half == 0 && lane == 0) {
    for (int s = 0; s < kNStage; ++s) mbar_init(&my_bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // This pair's units: for each of the CTA's tiles m, its k-steps (all of the
  // k-range in ROWS mode, every kPairs-th otherwise).  Unit u = m*n_mine + i.
  const int n_mine = ROWS ? kr : (kr > pair ? (kr - pair + kPairs - 1) / kPairs : 0);
  const int n_units = n_tiles * n_mine;
  auto kstep = [&](int i) { return ROWS ? ksr.ks0 + i : ksr.ks0 + pair + kPairs * i; };
  auto issue = [&](int u) {
    const int m = u / n_mine, i = u - m * n_mine;
    const int row0 = ((int)blockIdx.x + m * n_clusters) * kTile + warp_row;
    const int row = row0 + lane;
    const int ks = kstep(i);
    uint64_t* bar = &my_bars[u % kNStage];
    uint8_t* dst = my_stages + (size_t)(u % kNStage) * kStage;
    const int live = rows - row0 < kRowsPerCta ? rows - row0 : kRowsPerCta;
    if (lane == 0 && live > 0) mbar_arrive_expect_tx(bar, (uint32_t)(live * kChunkBytes));
    if (lane == 0 && live <= 0) mbar_arrive_expect_tx(bar, 0u);
    __syncwarp();
    if (row < rows)
      bulk_g2s(dst + lane * kChunkBytes, W + (size_t)row * row_bytes + (size_t)ks * kChunkBytes, kChunkBytes, bar);
  };
  if (half == 0)
    for (int u = 0; u < kNStage && u < n_units; ++u) issue(u);  // weights do not depend on the previous kernel
  pdl_wait();  // the activations (and y / residual) may be the previous kernel's results
  pdl_trigger();

  if constexpr (PRO == 0) {
    // Unpack the CTA's activation blocks [ks0*8, ks1*8) x NT into the
    // word-major form (unrolled so that several blocks' loads are in flight at
    // once); the pad tokens NT..NTA-1 hold zero words.
  #pragma unroll 4
    for (int idx = threadIdx.x; idx < kr * 8 * NTA; idx += kThreads) {
      const int b = idx / NTA, t = idx - b * NTA;
      uint32_t* dq = act_q + (size_t)b * 8 * NTA + t;
      if (t >= NT) {
  #pragma unroll
        for (int k = 0; k < 8; ++k) dq[k * NTA] = 0u;
        for (int tp = t; tp < NTP; tp += NTA) act_s[(size_t)b * NTP + tp] = 0.0f;
        continue;
      }
      const long long g = (long long)t * nb + (long long)ksr.ks0 * 8 + b;  // global block index
      const uint32_t* src = reinterpret_cast<const uint32_t*>(xq + ((34 * g) & ~3LL));
      uint32_t wv[9];
  #pragma unroll
      for (int k = 0; k < 9; ++k) wv[k] = ld_u32(src + k);  // written by the previous kernel
      const bool odd = (g & 1) != 0;  // odd blocks start 2 bytes into a word
      const uint32_t sh = odd ? 32u : 16u;
  #pragma unroll
      for (int k = 0; k < 8; ++k) dq[k * NTA] = __funnelshift_rc(wv[k], wv[k + 1], sh);
      act_s[(size_t)b * NTP + t] = half_bits_to_float(odd ? (wv[0] >> 16) : wv[0]);
    }
  } else {
    // The pad tokens NT..NTA-1 hold zero words and scales.
    for (int idx = threadIdx.x; idx < kr * 8 * 8; idx += kThreads)
      for (int t = NT; t < NTA; ++t) act_q[(size_t)idx * NTA + t] = 0u;
    for (int idx = threadIdx.x; idx < kr * 8; idx += kThreads)
      for (int t = NT; t < NTP; ++t) act_s[(size_t)idx * NTP + t] = 0.0f;
    const int cols = nb * 32;
    float* inv_s = reinterpret_cast<float*>(bars + kPairs * kNStage);  // [NT]
    float* part_s = inv_s + NT;                                         // [NT][8]
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
            const float g = v[4 * i + j];
            v[4 * i + j] = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), uu[j]);
          }
        }
      }
      float a = 0.0f;
#pragma unroll
      for (int j = 0; j < 32; ++j) a = fmaxf(a, fabsf(v[j]));
      const float d = __fdiv_rn(a, 127.0f);
      uint32_t* dq = act_q + (size_t)b * 8 * NTA + t;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          int q = 0;
          if (d != 0.0f) q = (int)fminf(fmaxf(roundf(__fdiv_rn(v[4 * k + j], d)), -127.0f), 127.0f);
          word |= ((uint32_t)q & 0xFFu) << (8 * j);
        }
        dq[k * NTA] = word;
      }
      act_s[(size_t)b * NTP + t] = __half2float(__float2half_rn(d));
    }
  }
  __syncthreads();

  // Cross-CTA sums: the CTA sum of tile m goes to buffer m & 1 and the CTA
  // arrives on the cluster barrier; it waits, and adds the cluster's sums of
  // tile m (its slice, ranks in order), only after computing tile m + 1.  A
  // buffer is rewritten two tiles later, after the next wait, which no CTA
  // passes before every CTA has read it.
  constexpr bool kCluster = !EMIT;  // ROWS && S == 1 writes directly instead (runtime)
  const bool cluster_sums = kCluster && !(ROWS && S == 1);
  auto reduce_tile = [&](int m) {
    const float* rs = red_sum + (m & 1) * kSum;
    const int row0 = ((int)blockIdx.x + m * n_clusters) * kTile;
    for (int idx = rank * kThreads + (int)threadIdx.x; idx < kSum; idx += S * kThreads) {
      float part[kMaxCluster];
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < S) part[r] = ld_dsmem_f32(&rs[idx], (uint32_t)r);
      float v = part[0];
#pragma unroll
      for (int r = 1; r < kMaxCluster; ++r)
        if (r < S) v = __fadd_rn(v, part[r]);
      const int wq = ROWS ? idx / (NT * 32) : 0;  // the pair (row group) of this output
      const int t = (idx / 32) % NT, rr = row0 + wq * kRowsPerCta + (idx & 31);
      if (rr < rows) {
        const size_t o = (size_t)t * rows + rr;
        y[o] = residual ? __fadd_rn(__ldcg(residual + o), v) : v;  // residual may alias y
      }
    }
  };

  bool dead = false;
  int u = 0;
  // The tile loop, specialised on this warp's token count NTM (compile time):
  // the two halves of a pair run their own instance.
  auto run = [&](auto ntm_c) {
    constexpr int NTM = decltype(ntm_c)::value;
    constexpr int NTMA = NTM > 0 ? NTM : 1;  // array extents
    for (int m = 0; m < n_tiles; ++m) {
      const int row0 = ((int)blockIdx.x + m * n_clusters) * kTile;
      const int row = row0 + warp_row + lane;
      unsigned long long acc2[(NTMA + 1) / 2];
#pragma unroll
      for (int p = 0; p < (NTMA + 1) / 2; ++p) acc2[p] = 0ull;

      if constexpr (NTM > 0) {
        for (int i = 0; i < n_mine; ++i, ++u) {
          const int ks = kstep(i);
          const int kl = ks - ksr.ks0;
          uint64_t* bar = &my_bars[u % kNStage];
          if (!dead) {
            const bool ok = mbar_wait(bar, (uint32_t)((u / kNStage) & 1));
            dead = __any_sync(0xffffffffu, !ok);  // warp-uniform
            if (dead && lane == 0) g_err_matmul = 1u;
          }
          const uint4* src =
              reinterpret_cast<const uint4*>(my_stages + (size_t)(u % kNStage) * kStage + lane * kChunkBytes);
          uint32_t w[68];
#pragma unroll
          for (int c = 0; c < 17; ++c) {
            const uint4 v = src[c];
            w[4 * c + 0] = v.x;
            w[4 * c + 1] = v.y;
            w[4 * c + 2] = v.z;
            w[4 * c + 3] = v.w;
          }
          // every reader of the pair holds the stage: it may be refilled
          if constexpr (kReaders == 2)
            asm volatile("bar.sync %0, 64;" ::"r"(1 + pair) : "memory");
          else
            __syncwarp();
          if (half == 0 && !dead && u + kNStage < n_units) issue(u + kNStage);

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
            const uint32_t* aq = act_q + (size_t)(kl * 8 + b) * 8 * NTA + t0;
            // this warp's block dots advance word by word together (two
            // words per 8-byte load; t0 is even)
            int sd[NTM];
#pragma unroll
            for (int t = 0; t < NTM; ++t) sd[t] = (int)kMagic;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
#pragma unroll
              for (int t2 = 0; t2 < NTM; t2 += 2) {
                if (t2 + 1 < NTM) {
                  const uint2 a = *reinterpret_cast<const uint2*>(aq + k * NTA + t2);
                  sd[t2] = __dp4a((int)q[k], (int)a.x, sd[t2]);
                  sd[t2 + 1] = __dp4a((int)q[k], (int)a.y, sd[t2 + 1]);
                } else {
                  sd[t2] = __dp4a((int)q[k], (int)aq[k * NTA + t2], sd[t2]);
                }
              }
            }
            if constexpr (EMIT) {
              if (row < rows) {
#pragma unroll
                for (int t = 0; t < NTM; ++t)
                  isum_out[((size_t)(t0 + t) * rows + row) * nb + (size_t)ks * 8 + b] = sd[t] - (int)kMagic;
              }
            } else {
              const float* as = act_s + (size_t)(kl * 8 + b) * NTP + t0;
              const unsigned long long dw2 = dup_pair(dw);
#pragma unroll
              for (int t = 0; t < NTM; t += 2) {
                unsigned long long sx2;
                if (t + 1 < NTM)
                  sx2 = *reinterpret_cast<const unsigned long long*>(as + t);
                else
                  sx2 = dup_pair(as[t]);
                acc2[t / 2] =
                    acc_pair(acc2[t / 2], sd[t], t + 1 < NTM ? sd[t + 1] : (int)kMagic, mul_pair(dw2, sx2));
              }
            }
          }
        }
      }

      if constexpr (!EMIT) {
        float acc[NTMA];
#pragma unroll
        for (int p = 0; p < (NTMA + 1) / 2; ++p) {
          const float2 v = unpack_pair(acc2[p]);
          acc[2 * p] = v.x;
          if (2 * p + 1 < NTMA) acc[2 * p + 1] = v.y;
        }
        if (!cluster_sums) {
          // One pair owns these rows over the whole k: write them directly.
          if (row < rows) {
#pragma unroll
            for (int t = 0; t < NTM; ++t) {
              const size_t o = (size_t)(t0 + t) * rows + row;
              y[o] = residual ? __fadd_rn(__ldcg(residual + o), acc[t]) : acc[t];  // residual may alias y
            }
          }
        } else {
          // the previous tile's cluster sums, now that this tile is computed
          if (m > 0) {
            cluster_wait();
            reduce_tile(m - 1);
          }
          // this tile's CTA sum (k-split mode: pair partials in pair order)
          float* rs = red_sum + (m & 1) * kSum;
          if constexpr (ROWS) {
#pragma unroll
            for (int t = 0; t < NTM; ++t) rs[(pair * NT + t0 + t) * 32 + lane] = acc[t];
          } else {
#pragma unroll
            for (int t = 0; t < NTM; ++t) red[(pair * NT + t0 + t) * 32 + lane] = acc[t];
            __syncthreads();
            for (int idx = threadIdx.x; idx < NT * 32; idx += kThreads) {
              float v = red[idx];
#pragma unroll
              for (int p2 = 1; p2 < kPairs; ++p2) v = __fadd_rn(v, red[p2 * NT * 32 + idx]);
              rs[idx] = v;
            }
          }
          cluster_arrive();
        }
      }
    }
    if (cluster_sums && n_tiles > 0) {
      cluster_wait();
      reduce_tile(n_tiles - 1);
      // keep this CTA's sums alive until every CTA of the cluster has read them
      cluster_sync();
    }
  };
  if (half == 0)
    run(std::integral_constant<int, NTH0>{});
  else
    run(std::integral_constant<int, NT - NTH0>{});
}

size_t smem_bytes(int kr, int nt, bool rows_mode, int pro = 0) {
  const size_t red = rows_mode ? 0 : (size_t)kPairs * nt * 32 * 4;
  const size_t sums = 2 * (rows_mode ? (size_t)kPairs : 1) * nt * 32 * 4;
  const size_t ntp = 2 * ((((size_t)nt + 1) / 2 + 1) & ~(size_t)1);  // the kernel's NTP
  const size_t nta = ((size_t)nt + 3) & ~(size_t)3;
  return (size_t)kr * 8 * (nta * 32 + ntp * 4) + (size_t)kPairs * kNStage * kStage + red + sums +
         (size_t)kPairs * kNStage * 8 + (pro == 1 ? (size_t)nt * 9 * 4 : 0);
}

// Per-instantiation host caches, each behind its own lock: the largest
// dynamic shared memory granted so far, and the number of co-resident clusters
// for each (S, smem) seen.  The attributes are per function, the same for every
// device of one architecture.
template <int NT, bool EMIT, bool ROWS, int PRO>
cudaError_t grant_smem(size_t smem) {
  static std::mutex mu;
  static size_t granted = 0;
  static bool non_portable = false;
  std::lock_guard<std::mutex> lock(mu);
  if (!non_portable) {
    cudaError_t e = cudaFuncSetAttribute(matmul_q8_0_narrow_kernel<NT, EMIT, ROWS, PRO>,
                                         cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    non_portable = true;
  }
  if (smem <= granted) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(matmul_q8_0_narrow_kernel<NT, EMIT, ROWS, PRO>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) granted = smem;
  return e;
}

template <int NT, bool EMIT, bool ROWS, int PRO>
cudaError_t cluster_capacity(int S, size_t smem, int* clusters) {
  struct Entry {
    int S;
    size_t smem;
    int clusters;
  };
  static std::mutex mu;
  static Entry cache[16];
  static int n_cache = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_cache; ++i)
    if (cache[i].S == S && cache[i].smem == smem) {
      *clusters = cache[i].clusters;
      return cudaSuccess;
    }
  cudaError_t e = grant_smem<NT, EMIT, ROWS, PRO>(smem);
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
  e = cudaOccupancyMaxActiveClusters(&c, matmul_q8_0_narrow_kernel<NT, EMIT, ROWS, PRO>, &cfg);
  if (e != cudaSuccess) return e;
  cache[n_cache < 16 ? n_cache++ : 15] = Entry{S, smem, c};
  *clusters = c;
  return cudaSuccess;
}

template <int NT, bool EMIT, bool ROWS, int PRO>
cudaError_t launch_nt(const uint8_t* W, int rows, int nb, const ActSrc& src, float* y, const float* residual,
                      int32_t* isum, int S, size_t smem, cudaStream_t st) {
  auto kern = matmul_q8_0_narrow_kernel<NT, EMIT, ROWS, PRO>;
  // The persistent grid: as many clusters as fit at once, up to one per tile.
  int resident = 0;
  cudaError_t e = cluster_capacity<NT, EMIT, ROWS, PRO>(S, smem, &resident);
  if (e != cudaSuccess) return e;
  if (resident < 1) return cudaErrorInvalidConfiguration;
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
  const int tile = ROWS ? kPairs * kRowsPerCta : kRowsPerCta;
  const int tiles = (rows + tile - 1) / tile;
  const int n_clusters = tiles < resident ? tiles : resident;
  cfg.gridDim = dim3((unsigned)n_clusters, (unsigned)S, 1);
  cfg.numAttrs = pdl() ? 2 : 1;
  if (dry_run()) return cudaSuccess;
  return cudaLaunchKernelEx(&cfg, kern, W, rows, nb, src, y, residual, isum);
}

template <bool EMIT, bool ROWS, int PRO>
cudaError_t dispatch(int nt, const uint8_t* W, int rows, int nb, const ActSrc& src, float* y, const float* residual,
                     int32_t* isum, int S, size_t smem, cudaStream_t st) {
  switch (nt) {
#define DSB_CASE(N) \
  case N:           \
    return launch_nt<N, EMIT, ROWS, PRO>(W, rows, nb, src, y, residual, isum, S, smem, st);
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
