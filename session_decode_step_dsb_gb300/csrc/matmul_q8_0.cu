// Narrow-batch q8_0 matmul for sm_103a.
//
// What it computes (antirez/ds4 PR #530, "Batched decode: co-decode N live
// sessions in one GPU pass", section "Why it's worth it -- the narrow-batch
// matmul", and the narrow-batch q8_0 matmul commit): for n_tok <= 16
// pre-quantised q8_0 activation rows,
//     y[t][r] = sum_i dW[r,i] * dX[t,i] * sum_k qW[r,i,k] * qX[t,i,k].
// The page's point is that in decode the weights are the whole cost, so each
// weight block must cross HBM once and serve every token.
//
// GB300 design (differs from the page's one-warp-per-row kernel):
//  * A CTA owns 32 weight rows (lane = row) and a contiguous range of 8-block
//    k-steps; its 4 warps take interleaved k-steps.  A k-step of one row is
//    8 blocks = 272 bytes = 17 x 16 bytes, so every row chunk is 16-byte
//    aligned whenever cols % 256 == 0.
//  * Each warp streams its 32 row chunks with 1-D TMA bulk copies
//    (cp.async.bulk, one 272-byte copy per lane) into a private NSTAGE-deep
//    shared-memory ring guarded by mbarriers; no thread spends instructions on
//    global loads of weights.  A lane reads its chunk back with 17 conflict-free
//    16-byte shared loads (the 272-byte stride is an odd number of 16-byte
//    bank groups) and unpacks the 34-byte blocks with funnel shifts.
//  * Activation blocks of the CTA's k-range are unpacked once, at kernel start,
//    into an aligned layout (32 code bytes + fp32 scale per block and token),
//    so the inner loop reads them with warp-uniform (broadcast) 16-byte loads.
//  * Block dots are __dp4a chains started from the bit pattern of 1.5 * 2^23:
//    |isum| <= 32*127*127 < 2^22, so the int32 result read as a float is
//    1.5*2^23 + isum exactly and one FADD converts it (no I2F).
//  * When rows alone give too few CTAs, k is split over the CTAs of a thread
//    block cluster (<= 8) and the partial sums are added through distributed
//    shared memory in cluster-rank order.  No atomics; every reduction order
//    depends only on (rows, cols) and the device's SM count, never on n_tok,
//    so column t of an n_tok = k call is bitwise equal to the n_tok = 1 call.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dsb_kernels.h"
#include "dsb_ptx.cuh"

namespace dsbk {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerCta = 32;
constexpr int kChunkBytes = 272;  // 8 blocks of 34 bytes
constexpr int kStage = kRowsPerCta * kChunkBytes;
constexpr int kNStage = 2;
constexpr uint32_t kMagic = 0x4B400000u;  // bits of 12582912.0f = 1.5 * 2^23
constexpr unsigned long long kMagic2 = 0x4B4000004B400000ull;
constexpr float kMagicF = 12582912.0f;

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

// ROWS = false (few-row matrices): a CTA tile is 32 rows and its 4 warps
//   take interleaved k-steps of the CTA's k-range; warp partials are added in
//   warp order at each tile end.
// ROWS = true (many-row matrices): a CTA tile is 128 rows, warp w owns rows
//   32w..32w+31 over the whole k-range; no partials are exchanged between
//   warps, and with S = 1 no barrier of any kind is taken after start-up.
// In both modes the S CTAs of a cluster split k and rank 0 adds their sums in
// rank order through distributed shared memory.
template <int NT, bool EMIT, bool ROWS>
__global__ void __launch_bounds__(kThreads, 2)
    matmul_q8_0_narrow_kernel(const uint8_t* __restrict__ W, int rows, int nb, const uint8_t* xq,
                              float* y, const float* residual, int32_t* __restrict__ isum_out) {
  constexpr int kTile = ROWS ? kWarps * kRowsPerCta : kRowsPerCta;
  constexpr int kRed = ROWS ? 0 : kWarps * NT * 32;          // warp partials (k-split mode)
  constexpr int kSum = (ROWS ? kWarps : 1) * NT * 32;        // one CTA sum buffer
  constexpr int kSumBufs = ROWS ? 1 : 2;  // rows mode: one buffer, a second barrier per tile
  constexpr int NTP = NT + (NT & 1);      // scale row stride: even, so token pairs load as 8 bytes
  extern __shared__ __align__(128) uint8_t smem[];
  const int nks = nb >> 3;
  const int S = gridDim.y;
  const int rank = blockIdx.y;  // cluster dims (1, S, 1): rank within the cluster
  const int n_clusters = gridDim.x;
  const Split ksr = kstep_range(nks, S, rank);
  const int kr = ksr.ks1 - ksr.ks0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row_bytes = (size_t)nb * 34;
  const int tiles = (rows + kTile - 1) / kTile;
  const int n_tiles = (int)blockIdx.x < tiles ? (tiles - 1 - (int)blockIdx.x) / n_clusters + 1 : 0;
  const int warp_row = ROWS ? warp * kRowsPerCta : 0;

  // Shared layout: act codes | act scales | stage rings | warp partials |
  // CTA sums (double-buffered) | barriers.  The act region is sized for the
  // largest k-range of the cluster in every CTA, so all CTAs of a cluster put
  // the CTA sums at the same offset -- the distributed-shared-memory reads of
  // rank 0 rely on that.
  const int kr_alloc = (nks + S - 1) / S;
  uint32_t* act_q = reinterpret_cast<uint32_t*>(smem);                              // [kr*8][NT][8]
  float* act_s = reinterpret_cast<float*>(act_q + (size_t)kr_alloc * 8 * NT * 8);  // [kr*8][NTP]
  uint8_t* stages = reinterpret_cast<uint8_t*>(act_s + (size_t)kr_alloc * 8 * NTP);  // [kWarps][kNStage][kStage]
  float* red = reinterpret_cast<float*>(stages + (size_t)kWarps * kNStage * kStage);  // [kWarps][NT][32]
  float* red_sum = red + kRed;                                                        // [kSumBufs][kSum]
  uint64_t* bars = reinterpret_cast<uint64_t*>(red_sum + kSumBufs * kSum);           // [kWarps][kNStage]
  uint8_t* my_stages = stages + (size_t)warp * kNStage * kStage;
  uint64_t* my_bars = bars + warp * kNStage;

  if (lane == 0) {
    for (int s = 0; s < kNStage; ++s) mbar_init(&my_bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // This warp's units: for each of the CTA's tiles m, its k-steps (all of the
  // k-range in ROWS mode, every kWarps-th otherwise).  Unit u = m*n_mine + i.
  const int n_mine = ROWS ? kr : (kr > warp ? (kr - warp + kWarps - 1) / kWarps : 0);
  const int n_units = n_tiles * n_mine;
  auto kstep = [&](int i) { return ROWS ? ksr.ks0 + i : ksr.ks0 + warp + kWarps * i; };
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
  for (int u = 0; u < kNStage && u < n_units; ++u) issue(u);  // weights do not depend on the previous kernel
  pdl_wait();  // the activations (and y / residual) may be the previous kernel's results
  pdl_trigger();

  // Unpack the CTA's activation blocks [ks0*8, ks1*8) x NT into aligned form
  // (unrolled so that several blocks' loads are in flight at once).
#pragma unroll 4
  for (int idx = threadIdx.x; idx < kr * 8 * NT; idx += kThreads) {
    const int b = idx / NT, t = idx - b * NT;
    const long long g = (long long)t * nb + (long long)ksr.ks0 * 8 + b;  // global block index
    const uint32_t* src = reinterpret_cast<const uint32_t*>(xq + ((34 * g) & ~3LL));
    uint32_t wv[9];
#pragma unroll
    for (int k = 0; k < 9; ++k) wv[k] = ld_u32(src + k);  // written by the previous kernel
    const bool odd = (g & 1) != 0;  // odd blocks start 2 bytes into a word
    const uint32_t sh = odd ? 32u : 16u;
    uint32_t* dq = act_q + ((size_t)b * NT + t) * 8;
#pragma unroll
    for (int k = 0; k < 8; ++k) dq[k] = __funnelshift_rc(wv[k], wv[k + 1], sh);
    act_s[(size_t)b * NTP + t] = half_bits_to_float(odd ? (wv[0] >> 16) : wv[0]);
  }
  __syncthreads();

  bool dead = false;
  int u = 0;
  for (int m = 0; m < n_tiles; ++m) {
    const int row0 = ((int)blockIdx.x + m * n_clusters) * kTile;
    const int row = row0 + warp_row + lane;
    unsigned long long acc2[(NT + 1) / 2];
#pragma unroll
    for (int p = 0; p < (NT + 1) / 2; ++p) acc2[p] = 0ull;

    for (int i = 0; i < n_mine; ++i, ++u) {
      const int ks = kstep(i);
      const int kl = ks - ksr.ks0;
      uint64_t* bar = &my_bars[u % kNStage];
      if (!dead) {
        const bool ok = mbar_wait(bar, (uint32_t)((u / kNStage) & 1));
        dead = __any_sync(0xffffffffu, !ok);  // warp-uniform
        if (dead && lane == 0) g_err_matmul = 1u;
      }
      const uint4* src = reinterpret_cast<const uint4*>(my_stages + (size_t)(u % kNStage) * kStage + lane * kChunkBytes);
      uint32_t w[68];
#pragma unroll
      for (int c = 0; c < 17; ++c) {
        const uint4 v = src[c];
        w[4 * c + 0] = v.x;
        w[4 * c + 1] = v.y;
        w[4 * c + 2] = v.z;
        w[4 * c + 3] = v.w;
      }
      __syncwarp();  // every lane has read the stage: it may be refilled
      if (!dead && u + kNStage < n_units) issue(u + kNStage);

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
        const uint32_t* aq = act_q + ((size_t)(kl * 8 + b) * NT) * 8;
        const float* as = act_s + (size_t)(kl * 8 + b) * NTP;  // 8-byte aligned row
        const unsigned long long dw2 = dup_pair(dw);
#pragma unroll
        for (int t = 0; t < NT; t += 2) {
          // two tokens' dp4a chains interleaved
          const uint4 a0 = *reinterpret_cast<const uint4*>(aq + t * 8);
          const uint4 a1 = *reinterpret_cast<const uint4*>(aq + t * 8 + 4);
          uint4 b0 = make_uint4(0, 0, 0, 0), b1 = make_uint4(0, 0, 0, 0);
          if (t + 1 < NT) {
            b0 = *reinterpret_cast<const uint4*>(aq + (t + 1) * 8);
            b1 = *reinterpret_cast<const uint4*>(aq + (t + 1) * 8 + 4);
          }
          int sa = (int)kMagic, sb = (int)kMagic;
          sa = __dp4a((int)q[0], (int)a0.x, sa);
          sb = __dp4a((int)q[0], (int)b0.x, sb);
          sa = __dp4a((int)q[1], (int)a0.y, sa);
          sb = __dp4a((int)q[1], (int)b0.y, sb);
          sa = __dp4a((int)q[2], (int)a0.z, sa);
          sb = __dp4a((int)q[2], (int)b0.z, sb);
          sa = __dp4a((int)q[3], (int)a0.w, sa);
          sb = __dp4a((int)q[3], (int)b0.w, sb);
          sa = __dp4a((int)q[4], (int)a1.x, sa);
          sb = __dp4a((int)q[4], (int)b1.x, sb);
          sa = __dp4a((int)q[5], (int)a1.y, sa);
          sb = __dp4a((int)q[5], (int)b1.y, sb);
          sa = __dp4a((int)q[6], (int)a1.z, sa);
          sb = __dp4a((int)q[6], (int)b1.z, sb);
          sa = __dp4a((int)q[7], (int)a1.w, sa);
          sb = __dp4a((int)q[7], (int)b1.w, sb);
          if constexpr (EMIT) {
            if (row < rows) {
              isum_out[((size_t)t * rows + row) * nb + (size_t)ks * 8 + b] = sa - (int)kMagic;
              if (t + 1 < NT) isum_out[((size_t)(t + 1) * rows + row) * nb + (size_t)ks * 8 + b] = sb - (int)kMagic;
            }
          } else {
            unsigned long long sx2;
            if (t + 1 < NT)
              sx2 = *reinterpret_cast<const unsigned long long*>(as + t);
            else
              sx2 = dup_pair(as[t]);
            acc2[t / 2] = acc_pair(acc2[t / 2], sa, sb, mul_pair(dw2, sx2));
          }
        }
      }
    }

    if constexpr (!EMIT) {
      float acc[NT];
#pragma unroll
      for (int p = 0; p < (NT + 1) / 2; ++p) {
        const float2 v = unpack_pair(acc2[p]);
        acc[2 * p] = v.x;
        if (2 * p + 1 < NT) acc[2 * p + 1] = v.y;
      }
      if (ROWS && S == 1) {
        // One warp owns these rows over the whole k: write them directly.
        if (row < rows) {
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const size_t o = (size_t)t * rows + row;
            y[o] = residual ? __fadd_rn(__ldcg(residual + o), acc[t]) : acc[t];  // residual may alias y
          }
        }
      } else {
        // The CTA's sum for this tile (k-split mode: warp partials added in
        // warp order), then rank 0 adds the cluster's CTA sums in rank order.
        // k-split mode double-buffers the sums by tile parity, so one cluster
        // barrier per tile suffices (a buffer is rewritten two tiles later,
        // after the next barrier, which rank 0 reaches only once it has read
        // this one); rows mode keeps one larger buffer and takes a second
        // barrier after rank 0's reads.
        float* rs = red_sum + (kSumBufs == 2 ? (m & 1) : 0) * kSum;
        if constexpr (ROWS) {
#pragma unroll
          for (int t = 0; t < NT; ++t) rs[(warp * NT + t) * 32 + lane] = acc[t];
        } else {
#pragma unroll
          for (int t = 0; t < NT; ++t) red[(warp * NT + t) * 32 + lane] = acc[t];
          __syncthreads();
          for (int idx = threadIdx.x; idx < NT * 32; idx += kThreads) {
            float v = red[idx];
#pragma unroll
            for (int w2 = 1; w2 < kWarps; ++w2) v = __fadd_rn(v, red[w2 * NT * 32 + idx]);
            rs[idx] = v;
          }
        }
        cluster_sync();
        if (rank == 0) {
          for (int idx = threadIdx.x; idx < kSum; idx += kThreads) {
            float v = rs[idx];
            for (int r = 1; r < S; ++r) v = __fadd_rn(v, ld_dsmem_f32(&rs[idx], (uint32_t)r));
            const int wq = ROWS ? idx / (NT * 32) : 0;
            const int t = (idx / 32) % NT, rr = row0 + wq * kRowsPerCta + (idx & 31);
            if (rr < rows) {
              const size_t o = (size_t)t * rows + rr;
              y[o] = residual ? __fadd_rn(__ldcg(residual + o), v) : v;  // residual may alias y
            }
          }
        }
        if constexpr (ROWS) cluster_sync();  // rank 0 is done with every CTA's buffer
      }
    }
  }
  // keep this CTA's sums alive until rank 0 has read them
  if (!EMIT && !ROWS) cluster_sync();
}

size_t smem_bytes(int kr, int nt, bool rows_mode) {
  const size_t red = rows_mode ? 0 : (size_t)kWarps * nt * 32 * 4;
  const size_t sums = rows_mode ? (size_t)kWarps * nt * 32 * 4 : 2 * (size_t)nt * 32 * 4;
  const size_t ntp = (size_t)nt + (nt & 1);
  return (size_t)kr * 8 * (nt * 32 + ntp * 4) + (size_t)kWarps * kNStage * kStage + red + sums +
         (size_t)kWarps * kNStage * 8;
}

template <int NT, bool EMIT, bool ROWS>
cudaError_t launch_nt(const uint8_t* W, int rows, int nb, const uint8_t* xq, float* y, const float* residual,
                      int32_t* isum, int S, size_t smem, cudaStream_t st) {
  auto kern = matmul_q8_0_narrow_kernel<NT, EMIT, ROWS>;
  // Per-instantiation caches (not thread-safe; one host thread drives a
  // device): the largest dynamic shared memory granted so far, and the number
  // of co-resident clusters for each (S, smem) seen -- the persistent grid.
  struct Entry {
    int S;
    size_t smem;
    int clusters;
  };
  static Entry cache[8];
  static int n_cache = 0;
  static size_t granted = 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)S;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  if (smem > granted) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    granted = smem;
  }
  int resident = 0;
  for (int i = 0; i < n_cache; ++i)
    if (cache[i].S == S && cache[i].smem == smem) resident = cache[i].clusters;
  if (resident == 0) {
    cfg.gridDim = dim3(1, (unsigned)S, 1);
    cudaError_t e = cudaOccupancyMaxActiveClusters(&resident, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (resident < 1) return cudaErrorInvalidConfiguration;
    cache[n_cache < 8 ? n_cache++ : 7] = Entry{S, smem, resident};
  }
  const int tile = ROWS ? kWarps * kRowsPerCta : kRowsPerCta;
  const int tiles = (rows + tile - 1) / tile;
  const int n_clusters = tiles < resident ? tiles : resident;
  cfg.gridDim = dim3((unsigned)n_clusters, (unsigned)S, 1);
  cfg.numAttrs = pdl() ? 2 : 1;
  if (dry_run()) return cudaSuccess;
  return cudaLaunchKernelEx(&cfg, kern, W, rows, nb, xq, y, residual, isum);
}

template <bool EMIT, bool ROWS>
cudaError_t dispatch(int nt, const uint8_t* W, int rows, int nb, const uint8_t* xq, float* y, const float* residual,
                     int32_t* isum, int S, size_t smem, cudaStream_t st) {
  switch (nt) {
#define DSB_CASE(N) \
  case N:           \
    return launch_nt<N, EMIT, ROWS>(W, rows, nb, xq, y, residual, isum, S, smem, st);
    DSB_CASE(1) DSB_CASE(2) DSB_CASE(3) DSB_CASE(4) DSB_CASE(5) DSB_CASE(6) DSB_CASE(7) DSB_CASE(8)
    DSB_CASE(9) DSB_CASE(10) DSB_CASE(11) DSB_CASE(12) DSB_CASE(13) DSB_CASE(14) DSB_CASE(15) DSB_CASE(16)
#undef DSB_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

struct Plan {
  bool rows_mode;
  int S;
};

// Depends on (rows, cols, SM count) only -- never on n_tok -- so that the
// summation order of every output is the same for every n_tok.  Each CTA of
// a cluster keeps the activations of its k-range in shared memory, which at
// n_tok = 16 allows at most 8 k-steps (36 KiB) next to the weight rings.
// Rows mode (128-row tiles, no cross-warp sums) when there are at least as
// many 128-row tiles per cluster slot as SMs; otherwise k-split mode on
// 32-row tiles.  Among the admissible S the smallest estimated makespan (tiles
// per cluster x k-steps per CTA, plus a per-tile reduction cost) wins,
// assuming two resident CTAs per SM.
Plan matmul_plan(int64_t rows, int64_t cols, int num_sms) {
  const int nks = (int)(cols / 256);
  int s_max = nks < 8 ? nks : 8;
  int s_min = (nks + 7) / 8;
  if (s_min > s_max) s_min = s_max;
  if (s_min < 1) s_min = 1;
  const int P = 2 * num_sms;
  Plan best{false, s_min};
  double best_cost = 1e30;
  for (int mode = 0; mode < 2; ++mode) {
    const bool rm = mode == 1;
    const int tile = rm ? kWarps * kRowsPerCta : kRowsPerCta;
    const int tiles = (int)((rows + tile - 1) / tile);
    for (int S = s_min; S <= s_max; ++S) {
      const int clusters = P / S > 0 ? P / S : 1;
      const int per = (tiles + clusters - 1) / clusters;
      const int ksteps = (nks + S - 1) / S;
      // time ~ tiles per cluster x (k-steps each warp runs + per-tile sync cost)
      const double sync = (rm && S == 1) ? 0.0 : 0.5;
      const double warp_steps = rm ? (double)ksteps : (double)((ksteps + kWarps - 1) / kWarps);
      const double c = per * (warp_steps + sync);
      if (c < best_cost - 1e-9) {
        best_cost = c;
        best = Plan{rm, S};
      }
    }
  }
  return best;
}

}  // namespace

int matmul_split(int64_t rows, int64_t cols, int num_sms) { return matmul_plan(rows, cols, num_sms).S; }

size_t matmul_smem_bytes(int64_t rows, int64_t cols, int n_tok, int num_sms) {
  const Plan pl = matmul_plan(rows, cols, num_sms);
  const int nks = (int)(cols / 256);
  const int kr_max = (nks + pl.S - 1) / pl.S;
  return smem_bytes(kr_max, n_tok, pl.rows_mode);
}

cudaError_t launch_matmul_q8_0_narrow(const void* W, int64_t rows, int64_t cols, const void* xq, int n_tok,
                                      float* y, const float* residual, int32_t* isum, int num_sms, cudaStream_t st) {
  const Plan pl = matmul_plan(rows, cols, num_sms);
  const size_t smem = matmul_smem_bytes(rows, cols, n_tok, num_sms);
  const int nb = (int)(cols / 32);
  const uint8_t* w8 = static_cast<const uint8_t*>(W);
  const uint8_t* x8 = static_cast<const uint8_t*>(xq);
  if (isum)
    return pl.rows_mode ? dispatch<true, true>(n_tok, w8, (int)rows, nb, x8, y, residual, isum, pl.S, smem, st)
                        : dispatch<true, false>(n_tok, w8, (int)rows, nb, x8, y, residual, isum, pl.S, smem, st);
  return pl.rows_mode ? dispatch<false, true>(n_tok, w8, (int)rows, nb, x8, y, residual, isum, pl.S, smem, st)
                      : dispatch<false, false>(n_tok, w8, (int)rows, nb, x8, y, residual, isum, pl.S, smem, st);
}

namespace {
thread_local bool g_dry_run = false;
}
thread_local bool g_pdl = false;
void set_dry_run(bool on) { g_dry_run = on; }
bool dry_run() { return g_dry_run; }
void set_pdl(bool on) { g_pdl = on; }
bool pdl() { return g_pdl; }

unsigned int read_clear_error_matmul() {
  unsigned int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_matmul, sizeof v) != cudaSuccess) return 0xFFFFFFFFu;
  cudaMemcpyToSymbol(g_err_matmul, &z, sizeof z);
  return v;
}

}  // namespace dsbk
