// Wide-batch q8_0 matmul on the 5th-generation tensor cores (sm_103a), for
// n_tok > 16 token rows: speculative decode with K+1 drafts per sequence over
// many sequences (quic/efficient-transformers PR #1305, "Assumptions and
// limitations": K+1 tokens per sequence), where the narrow kernel's dp4a pipe,
// not HBM, would bound the step (antirez/ds4 PR #530, "Why it's worth it -- the
// narrow-batch matmul": past 16 tokens the page hands the batch to its
// batched path).
//
// Math (the product of the narrow kernel, accumulated in another order):
//   y[t][r] = sum_i sum_k (dW[r,i] qW[r,i,k]) (dX[t,i] qX[t,i,k]).
// Each dequantised value v = d*q (fp16 scale d, int8 code q) is split exactly
// into two f16 values, hi = RN(d*q) and lo = d*q - hi: lo is a multiple of
// ulp(d) no larger than ulp(hi)/2, so it has at most 7 significant bits and is
// exact in f16 (subnormal or not).  Then
//   v_w v_x = hi_w hi_x + hi_w lo_x + lo_w hi_x + lo_w lo_x,
// every product exact in float32.  Three kind::f16 MMAs per K step (the last
// term, below 2^-22 of the first, is dropped) accumulate a chunk of 8 q8_0
// blocks (K = 256) in a float32 TMEM accumulator; the scales are folded into
// the operands, so no per-block work follows the MMAs.  The tensor core's
// accumulation rounds toward zero, a bias of about 2^-24 of the partial sum
// per accumulation, so chunks stay short: two accumulators alternate, and the
// workers add each finished chunk into float32 registers (round to nearest).
// Values must satisfy |d*q| <= 65504 (scales up to 65504/127); a larger scale
// is flagged as a device error.
//
// CTA tile: 128 weight rows (TMEM lanes) x 128 token rows (TMEM columns).
// Narrow matrices are split along K over the S CTAs of a thread-block
// cluster (grid z, S <= 8, each CTA a contiguous range of 8-block chunks) so
// that the grid fills the SMs; rank 0 then adds the other ranks' float32
// partial tiles through distributed shared memory in rank order (no atomics,
// the same order on every run).  Warp roles (10 warps):
//   0..7  workers.  Warps w and w + 4 own TMEM lane quarter w % 4 (weight
//         rows 32(w%4) .. +31, lane = row) and convert its rows for the
//         q8_0 blocks of even and odd index respectively: the odd warp stages
//         the quarter's raw q8_0 bytes by 1-D bulk copies (8 blocks = 272 B per
//         row, 16-byte aligned when cols % 256 == 0) into a two-stage ring
//         that both read, refilling a stage once both are done with it; each
//         lane splits its row's 32 values into hi and lo and stores them into
//         the block's weight operand slot in tensor memory (tcgen05.st, 16
//         columns each), so the MMAs read only the token operand from shared
//         memory.  Every worker also drains the chunk accumulators for its
//         lane quarter and columns 64*(w/4).. into registers, a few blocks
//         behind the MMAs, and at the end stores y (+ residual).  Warp 0 also
//         allocates and frees the TMEM.
//   8     producer: bulk copies of the token operands (hi and lo), which a
//         pack kernel laid out once per call.
//   9     MMA issuer (one thread); A from tensor memory, B from shared memory.
// Tensor memory (512 columns): the two chunk accumulators (columns 0..255),
// then eight weight operand slots of 32 columns (hi, then lo; a 128 x 16 f16
// operand is 8 columns of two f16 values per lane).
// Token operand layout (no swizzle, K-major): element (m, k) of a 128 x 32 f16
// operand at byte (m/8)*512 + (k/8)*128 + (m%8)*16 + (k%8)*2, i.e. 8x8 core
// matrices of 128 contiguous bytes, 128 B apart along K (LBO) and 512 B apart
// along M/N (SBO).
//
// Every mbarrier wait is bounded and sleeps in mbarrier.try_wait (with a
// suspend-time hint) rather than spinning; on a timeout the CTA records a
// device error, every role leaves its loop, the MMA thread and the copy
// issuers wait (bounded) for what they issued, and the TMEM is freed before
// exit.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "dsb_kernels.h"
#include "dsb_ptx.cuh"

namespace dsbk {

namespace {

constexpr int kTcM = 128;            // weight rows per CTA
constexpr int kTcN = 128;            // token rows per CTA
constexpr int kTcStageBlocks = 8;    // q8_0 blocks per raw weight stage
constexpr int kTcRawStages = 2;
constexpr int kTcSlots = 8;          // operand slots, one q8_0 block each
constexpr int kTcWorkWarps = 8;
constexpr int kTcProducerWarp = kTcWorkWarps;                 // 8
constexpr int kTcMmaWarp = kTcProducerWarp + 1;               // 9
constexpr int kTcThreads = (kTcMmaWarp + 1) * 32;             // 320
constexpr int kTcChunk = 8;                                   // blocks per TMEM accumulation chunk
constexpr int kTcAccRegions = 2;
constexpr int kTcQuarters = kTcM / 32;                        // TMEM lane quarters (32 rows each)
constexpr int kTcACol0 = kTcAccRegions * kTcN;                // 256: first column of the weight operand slots
constexpr int kTcASlotCols = 32;                              // one slot: hi (16 columns), then lo (16)
constexpr int kTcTmemCols = 512;                              // accumulators + operand slots, a power of two
static_assert(kTcACol0 + kTcSlots * kTcASlotCols <= kTcTmemCols, "tensor memory holds the operand slots");
static_assert(kTcSlots % 2 == 0, "a slot always holds blocks of one parity");
constexpr int kOpBytes = kTcM * 32 * 2;                       // 8192: one 128 x 32 f16 operand
constexpr int kRawRowBytes = kTcStageBlocks * 34;             // 272
constexpr int kRawStageBytes = kTcM * kRawRowBytes;           // 34816
constexpr uint32_t kLbo = 128;
constexpr uint32_t kSbo = 512;
constexpr uint32_t kSuspendHintNs = 100000;                   // per try_wait
static_assert(kTcN == kTcM, "token operands share the weight operands' geometry");

struct __align__(1024) TcSmem {
  uint8_t b[kTcSlots][2][kOpBytes];            // token hi, lo (bulk-copied from the pack)
  uint8_t raw[kTcRawStages][kRawStageBytes];   // raw q8_0 weight rows, 32 rows per lane quarter
  uint64_t raw_full[kTcRawStages][kTcQuarters], raw_empty[kTcRawStages][kTcQuarters];
  uint64_t slot_full[kTcSlots], slot_empty[kTcSlots];
  uint64_t acc_full[kTcAccRegions], acc_empty[kTcAccRegions];
  uint32_t tmem_base;
  int abort_flag;
  int cta_ok;
};
static_assert(sizeof(((TcSmem*)nullptr)->b) >= (size_t)kTcM * kTcN * 4, "the partial tile reuses the token slots");

__device__ unsigned int g_err_matmul_tc = 0;

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One poll that may suspend the thread for up to kSuspendHintNs; it resumes as
// soon as the phase completes.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Bounded wait that also gives up as soon as another role of the CTA has.
__device__ __forceinline__ bool tc_wait(TcSmem& s, uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if ((i & 15u) == 15u) {
      if (*reinterpret_cast<volatile int*>(&s.abort_flag)) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
  }
  *reinterpret_cast<volatile int*>(&s.abort_flag) = 1;
  atomicOr(&g_err_matmul_tc, 1u);
  return false;
}

// Short bounded wait used only on the way out (for copies or MMAs issued).
__device__ __forceinline__ void tc_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait_sleep(bar, parity)) return;
    if ((i & 15u) == 15u && globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

__device__ __forceinline__ uint32_t ld_dsmem_u32(const void* p, uint32_t rank) {
  uint32_t remote, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(p)), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: start address, LBO, SBO (all >> 4), the
// descriptor version (1) at bit 46, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(const void* p) {
  const uint32_t a = smem_addr(p);
  return (uint64_t)((a & 0x3FFFFu) >> 4) | ((uint64_t)(kLbo >> 4) << 16) | ((uint64_t)(kSbo >> 4) << 32) |
         (1ull << 46);
}

// Instruction descriptor of kind::f16: f32 accumulator (bits 4-5 = 1), f16 A
// and B (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bit
// 17, M >> 4 at bit 24.
__device__ __forceinline__ uint32_t idesc_f16(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D (tensor memory) (+)= A (tensor memory) x B (shared-memory descriptor).
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// 16 consecutive TMEM columns of this warp's 32 lanes, one 32-bit word each.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// 32 consecutive TMEM columns of this warp's 32 lanes, one 32-bit word each.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Four int8 codes (one 32-bit word) -> two f16x2 words, exactly: the byte
// q ^ 0x80 = q + 128 becomes the low mantissa byte of the f16 1024 + (q+128)
// (exponent of 1024, unit spacing), and subtracting 1152 leaves q.
__device__ __forceinline__ void codes_to_f16(uint32_t w, uint32_t& c01, uint32_t& c23) {
  const uint32_t x = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(x, 0x64646464u, 0x4140);
  const uint32_t b = __byte_perm(x, 0x64646464u, 0x4342);
  const uint32_t bias = 0x64806480u;  // f16x2 (1152, 1152)
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(c01) : "r"(a), "r"(bias));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(c23) : "r"(b), "r"(bias));
}

// The value d*q of a code pair, split exactly into f16 hi + lo: hi = RN(d*q)
// and lo = d*q - hi, which the fused multiply-add forms exactly (the
// remainder is a multiple of ulp(d) below ulp(hi)/2: at most 7 significant
// bits, representable in f16, subnormal or not).
__device__ __forceinline__ void split_pair(uint32_t d2, uint32_t q2, uint32_t& hi, uint32_t& lo) {
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(d2), "r"(q2));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(lo) : "r"(d2), "r"(q2), "r"(hi ^ 0x80008000u));
}

// Eight codes (two words) of a block with scale d2 = (d, d) -> hi and lo
// halves of its 16-byte operand chunk.
__device__ __forceinline__ void split8(uint32_t w0, uint32_t w1, uint32_t d2, uint4& hi, uint4& lo) {
  uint32_t q0, q1, q2, q3;
  codes_to_f16(w0, q0, q1);
  codes_to_f16(w1, q2, q3);
  split_pair(d2, q0, hi.x, lo.x);
  split_pair(d2, q1, hi.y, lo.y);
  split_pair(d2, q2, hi.z, lo.z);
  split_pair(d2, q3, hi.w, lo.w);
}

// |d*q| <= 127 d must stay below the f16 maximum 65504.
constexpr float kMaxScale = 65504.0f / 127.0f;

__device__ __forceinline__ float half_bits_to_float_tc(uint32_t bits) {
  return __half2float(__ushort_as_half((unsigned short)(bits & 0xFFFFu)));
}


__global__ void __launch_bounds__(kTcThreads, 1)
    matmul_q8_0_tc_kernel(const uint8_t* __restrict__ W, int rows, int nb, const uint8_t* pack, int n_tok,
                          float* y, const float* residual) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // Align by pointer arithmetic on the shared array itself (not through an
  // integer round trip), so that every access below stays a shared-memory one.
  TcSmem& s = *reinterpret_cast<TcSmem*>(smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = (int)blockIdx.x * kTcM;
  const int tile = (int)blockIdx.y;
  const int tok0 = tile * kTcN;
  const int n_valid = min(kTcN, n_tok - tok0);
  const int n_cols = (n_valid + 15) & ~15;
  const int rows_valid = min(kTcM, rows - row0);
  const size_t row_bytes = (size_t)nb * 34;
  // this CTA's chunks of the K range (cluster rank = blockIdx.z)
  const int S = (int)gridDim.z, rank = (int)blockIdx.z;
  const int n_chunks_all = nb / kTcChunk;
  const int c_lo = (int)((long long)n_chunks_all * rank / S);
  const int c_hi = (int)((long long)n_chunks_all * (rank + 1) / S);
  const int kb0 = c_lo * kTcChunk;           // first q8_0 block
  const int nbl = (c_hi - c_lo) * kTcChunk;  // blocks of this CTA
  const int n_stages = nbl / kTcStageBlocks;
  static_assert(kTcStageBlocks == kTcChunk, "a raw stage is one accumulation chunk");
  bool ok = true;
  float acc[64];
#pragma unroll
  for (int j = 0; j < 64; ++j) acc[j] = 0.0f;
  const int q = warp & 3, c0 = (warp >> 2) * 64;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcRawStages; ++i)
      for (int c = 0; c < kTcQuarters; ++c) {
        mbar_init(&s.raw_full[i][c], 1);
        mbar_init(&s.raw_empty[i][c], 2);  // both warps of the quarter are done with the stage
      }
    for (int i = 0; i < kTcSlots; ++i) {
      mbar_init(&s.slot_full[i], kTcWorkWarps / 2 + 1);  // the four warps of the block's parity + the producer
      mbar_init(&s.slot_empty[i], 1);
    }
    for (int i = 0; i < kTcAccRegions; ++i) {
      mbar_init(&s.acc_full[i], 1);
      mbar_init(&s.acc_empty[i], kTcWorkWarps);
    }
    s.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&s.tmem_base)),
                 "r"(kTcTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  if (warp == kTcProducerWarp) {
    // ---------------------------------------------------------------- producer
    int issued = 0;
    pdl_wait();  // the packed token operands are the previous kernel's output
    pdl_trigger();
    for (int i = 0; i < nbl; ++i) {
      const int sl = i % kTcSlots;
      if (i >= kTcSlots) ok = tc_wait(s, &s.slot_empty[sl], (uint32_t)((i / kTcSlots - 1) & 1));
      ok = __all_sync(0xffffffffu, ok);  // the warp leaves together
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&s.slot_full[sl], (uint32_t)(2 * kOpBytes));
        bulk_g2s(s.b[sl][0], pack + ((size_t)tile * nb + kb0 + i) * (2 * kOpBytes), 2 * kOpBytes, &s.slot_full[sl]);
      }
      ++issued;
      __syncwarp();
    }
    // on the way out: every copy issued has landed (already so unless a wait gave up)
    if (lane == 0)
      for (int i = issued - kTcSlots; i < issued; ++i)
        if (i >= 0) tc_drain(&s.slot_full[i % kTcSlots], (uint32_t)((i / kTcSlots) & 1));
    __syncwarp();
  } else if (warp == kTcMmaWarp) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kTcM, n_cols);
      int issued = 0;
      for (int i = 0; i < nbl; ++i) {
        const int sl = i % kTcSlots;
        const int c = i / kTcChunk, jc = i % kTcChunk, ac = c % kTcAccRegions;
        if (jc == 0 && c >= kTcAccRegions &&
            !tc_wait(s, &s.acc_empty[ac], (uint32_t)((c / kTcAccRegions - 1) & 1))) {
          ok = false;
          break;
        }
        if (!tc_wait(s, &s.slot_full[sl], (uint32_t)((i / kTcSlots) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(ac * kTcN);
        const uint32_t a_hi = tmem + (uint32_t)(kTcACol0 + sl * kTcASlotCols), a_lo = a_hi + 16u;
        const uint64_t b_hi = smem_desc(s.b[sl][0]), b_lo = smem_desc(s.b[sl][1]);
#pragma unroll
        for (int kh = 0; kh < 2; ++kh) {
          // k = 16*kh .. +15: the operands' TMEM columns 8kh .. 8kh + 7 (two
          // f16 per column), core matrices 2kh, 2kh+1 of the token operand
          // (2 * LBO = 256 bytes per half)
          const uint64_t dk = (uint64_t)(kh * (256u >> 4));
          const uint32_t ak = (uint32_t)(8 * kh);
          mma_f16_ta(d, a_hi + ak, b_hi + dk, idesc, (jc > 0 || kh > 0) ? 1u : 0u);
          mma_f16_ta(d, a_hi + ak, b_lo + dk, idesc, 1u);
          mma_f16_ta(d, a_lo + ak, b_hi + dk, idesc, 1u);
        }
        mma_commit(&s.slot_empty[sl]);
        if (jc == kTcChunk - 1 || i == nbl - 1) mma_commit(&s.acc_full[ac]);
        issued = i + 1;
      }
      // on the way out: the MMAs issued have completed
      if (issued > 0) tc_drain(&s.slot_empty[(issued - 1) % kTcSlots], (uint32_t)(((issued - 1) / kTcSlots) & 1));
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
  } else {
    // ---------------------------------------------------------------- workers
    // Warp w converts the rows of TMEM lane quarter qw = w % 4 (rows 32qw ..
    // 32qw + 31, lane = row) for the blocks of parity w / 4; the two warps of a
    // quarter share its raw stages, which the odd one refills once both are
    // done with them.
    const int qw = warp & 3, par = warp >> 2;
    const int my_row = qw * 32 + lane;
    const int quarter_rows = max(0, min(32, rows_valid - qw * 32));
    const uint32_t lane_base = (uint32_t)(qw * 32) << 16;
    int raw_issued = 0;
    const int n_chunks = nbl / kTcChunk;
    int drained = 0;
    // Add the finished accumulator of chunk c (this warp's lanes and columns)
    // into acc, then hand the accumulator back to the MMA issuer.
    auto drain = [&](int c) -> bool {
      const int ac = c % kTcAccRegions;
      bool w_ok = __all_sync(0xffffffffu, tc_wait(s, &s.acc_full[ac], (uint32_t)((c / kTcAccRegions) & 1)));
      if (!w_ok) return false;
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (c0 + 32 * h < n_cols) {  // warp-uniform
          uint32_t v[32];
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ac * kTcN + c0 + 32 * h), v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[32 * h + j] = __fadd_rn(acc[32 * h + j], __uint_as_float(v[j]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.acc_empty[ac]);
      return true;
    };
    // this quarter's rows of raw stage st, one row per lane (the odd warp)
    auto issue_raw = [&](int st) {
      uint64_t* bar = &s.raw_full[st & 1][qw];
      if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(quarter_rows * kRawRowBytes));
      __syncwarp();
      if (lane < quarter_rows)
        bulk_g2s(s.raw[st & 1] + (qw * 32 + lane) * kRawRowBytes,
                 W + (size_t)(row0 + qw * 32 + lane) * row_bytes + (size_t)(c_lo + st) * kRawRowBytes, kRawRowBytes,
                 bar);
    };
    // the weights do not depend on the previous kernel: start them first
    if (par == 1)
      for (; raw_issued < kTcRawStages && raw_issued < n_stages; ++raw_issued) issue_raw(raw_issued);
    bool range_ok = true;
    // Stage by stage; this warp's four blocks of a stage are jb = 2jj + par.
    // Block jb's 34 bytes start at byte 34jb = 68jj + 34par of the row's
    // stage chunk, i.e. 2par bytes into word jj of the three 16-byte pieces
    // from byte 64jj + 32par on (16-byte loads at the 272-byte row stride
    // touch eight distinct bank groups per quarter-warp).
    for (int st = 0; st < n_stages && ok; ++st) {
      const int rb = st & 1;
      ok = __all_sync(0xffffffffu, tc_wait(s, &s.raw_full[rb][qw], (uint32_t)((st >> 1) & 1)));
      if (!ok) break;
      const uint8_t* row_raw = s.raw[rb] + my_row * kRawRowBytes + 32 * par;
#pragma unroll
      for (int jj = 0; jj < kTcStageBlocks / 2; ++jj) {
        const int i = st * kTcStageBlocks + 2 * jj + par, sl = i % kTcSlots;
        if (i >= kTcSlots) ok = tc_wait(s, &s.slot_empty[sl], (uint32_t)((i / kTcSlots - 1) & 1));
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();  // the slot's previous MMAs have read its operands
        uint32_t hi[16], lo[16];
        uint32_t dbits = 0u;
        if (lane < quarter_rows) {
          const uint4* src = reinterpret_cast<const uint4*>(row_raw + 64 * jj);
          const uint4 p0 = src[0], p1 = src[1], p2 = src[2];
          const uint32_t wd[12] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w, p2.x, p2.y, p2.z, p2.w};
          uint32_t bw[9];  // the block's bytes 4k .. 4k + 3
#pragma unroll
          for (int k = 0; k < 9; ++k) bw[k] = __funnelshift_r(wd[jj + k], wd[jj + k + 1 < 12 ? jj + k + 1 : 11], 16 * par);
          dbits = bw[0] & 0xFFFFu;
          const uint32_t d2 = dbits | (dbits << 16);
          // codes 4k .. 4k + 3 are bytes 2 + 4k .. 5 + 4k of the block
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            uint32_t c01, c23;
            codes_to_f16(__funnelshift_r(bw[k], bw[k + 1], 16), c01, c23);
            split_pair(d2, c01, hi[2 * k], lo[2 * k]);
            split_pair(d2, c23, hi[2 * k + 1], lo[2 * k + 1]);
          }
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k) hi[k] = lo[k] = 0u;
        }
        range_ok &= half_bits_to_float_tc(dbits) <= kMaxScale;
        const uint32_t acol = tmem + lane_base + (uint32_t)(kTcACol0 + sl * kTcASlotCols);
        tmem_st16(acol, hi);
        tmem_st16(acol + 16u, lo);
        tmem_st_wait();
        tc_fence_before();  // the operand stores precede the MMAs the barrier releases
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.slot_full[sl]);
      }
      if (!ok) break;
      // both warps of the quarter are done with the stage: the odd one refills it
      fence_proxy_async_smem();  // this warp's reads of the stage precede the refill's writes
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.raw_empty[rb][qw]);
      if (par == 1 && raw_issued < n_stages) {
        ok = __all_sync(0xffffffffu, tc_wait(s, &s.raw_empty[rb][qw], (uint32_t)((st >> 1) & 1)));
        if (!ok) break;
        issue_raw(raw_issued);
        ++raw_issued;
      }
      // the chunk before this stage: its MMAs trail the conversions by at most the slot depth
      if (st >= 1) {
        ok = drain(drained);
        ++drained;
      }
    }
    if (!range_ok) atomicOr(&g_err_matmul_tc, 2u);
    // on the way out: every raw copy issued has landed
    if (lane == 0 && par == 1)
      for (int st = raw_issued - kTcRawStages; st < raw_issued; ++st)
        if (st >= 0) tc_drain(&s.raw_full[st & 1][qw], (uint32_t)((st >> 1) & 1));
    __syncwarp();

    while (ok && drained < n_chunks) {
      ok = drain(drained);
      ++drained;
    }
  }

  // ---------------------------------------------------------------- epilogue
  // Every role is done and every MMA has completed (the workers drained the
  // last chunk).  Workers hold this CTA's partial sums in acc.
  tc_fence_before();
  const bool cta_ok = __syncthreads_and(ok ? 1 : 0) != 0;
  const bool worker = warp < kTcWorkWarps;
  const int row_l = q * 32 + lane, row = row0 + row_l;
  auto store = [&](const float (&v)[64]) {
    pdl_wait();  // y and the residual may be the previous kernels' data
    pdl_trigger();
    if (row < rows) {
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const int t = c0 + j;
        if (t < n_valid) {
          const size_t o = (size_t)(tok0 + t) * rows + row;
          y[o] = residual ? __fadd_rn(__ldcg(residual + o), v[j]) : v[j];
        }
      }
    }
  };
  if (S == 1) {
    if (worker && cta_ok) store(acc);
  } else {
    float* part = reinterpret_cast<float*>(&s.b[0][0][0]);  // [kTcN][kTcM], free once the MMAs are done
    if (worker && rank > 0) {
#pragma unroll
      for (int j = 0; j < 64; ++j) part[(c0 + j) * kTcM + row_l] = acc[j];
    }
    if (threadIdx.x == 0) s.cta_ok = cta_ok ? 1 : 0;
    cluster_sync();
    if (worker && rank == 0) {
      bool all_ok = cta_ok;
      for (int r = 1; r < S; ++r) all_ok = all_ok && ld_dsmem_u32(&s.cta_ok, (uint32_t)r) != 0u;
      if (all_ok) {
        for (int r = 1; r < S; ++r) {
#pragma unroll
          for (int j = 0; j < 64; ++j) acc[j] = __fadd_rn(acc[j], ld_dsmem_f32(part + (c0 + j) * kTcM + row_l, (uint32_t)r));
        }
        store(acc);
      }
    }
    cluster_sync();  // the other ranks keep their shared memory until rank 0 has read it
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols) : "memory");
  }
}

// Token operand pack: for token tile T (128 rows, zero past n_tok) and q8_0
// block i, the hi and lo f16 operands (8 KiB each, hi first) in the layout
// above.  Thread j of a CTA writes the j-th 16 bytes of each: token
// (j>>5)*8 + (j&7), codes 8*((j>>3)&3) .. +7.
__global__ void __launch_bounds__(512) pack_tokens_tc_kernel(const uint8_t* xq, int n_tok, int nb,
                                                             uint8_t* __restrict__ pack) {
  pdl_wait();
  pdl_trigger();
  const int i = (int)blockIdx.x, tile = (int)blockIdx.y;
  const int j = threadIdx.x;
  const int t_loc = (j >> 5) * 8 + (j & 7), g = (j >> 3) & 3;
  const int t = tile * kTcN + t_loc;
  uint4 hi = make_uint4(0u, 0u, 0u, 0u), lo = hi;
  if (t < n_tok) {
    const uint8_t* blk = xq + ((size_t)t * nb + i) * 34;
    const uint16_t* c = reinterpret_cast<const uint16_t*>(blk + 2 + 8 * g);  // blocks are 34 B: 2-aligned
    uint32_t h[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      unsigned short v;
      asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(v) : "l"(c + k) : "memory");
      h[k] = v;
    }
    unsigned short sb;
    asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(sb) : "l"(blk) : "memory");
    if (half_bits_to_float_tc(sb) > kMaxScale) atomicOr(&g_err_matmul_tc, 2u);
    split8(h[0] | (h[1] << 16), h[2] | (h[3] << 16), (uint32_t)sb | ((uint32_t)sb << 16), hi, lo);
  }
  uint8_t* slot = pack + ((size_t)tile * nb + i) * (2 * kOpBytes);
  reinterpret_cast<uint4*>(slot)[j] = hi;
  reinterpret_cast<uint4*>(slot + kOpBytes)[j] = lo;
}

std::mutex g_tc_mu;
bool g_tc_attr = false;
int g_tc_clusters[9] = {0};  // co-resident clusters of size S (0: not yet queried)

// Co-resident CTAs when clusters have S CTAs each.
cudaError_t tc_capacity(int S, size_t smem, int* out) {
  std::lock_guard<std::mutex> lock(g_tc_mu);
  if (!g_tc_attr) {
    cudaError_t e = cudaFuncSetAttribute(matmul_q8_0_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    g_tc_attr = true;
  }
  if (g_tc_clusters[S] == 0) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)S;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(1, 1, (unsigned)S);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, matmul_q8_0_tc_kernel, &cfg);
    if (e != cudaSuccess) return e;
    g_tc_clusters[S] = n > 0 ? n : -1;
  }
  *out = g_tc_clusters[S] > 0 ? g_tc_clusters[S] * S : 0;
  return cudaSuccess;
}

// K split: the S (1..8, at most one per chunk) that minimises waves x (chunks
// per CTA + one chunk's worth of fixed cost per CTA: TMEM and barrier set-up,
// pipeline fill), with a small charge per extra rank for the reduction.
cudaError_t tc_split(int tiles, int n_chunks, size_t smem, int* S_out) {
  int best = 1;
  double best_t = 1e30;
  for (int S = 1; S <= 8 && S <= n_chunks; ++S) {
    int cap = 0;
    cudaError_t e = tc_capacity(S, smem, &cap);
    if (e != cudaSuccess) return e;
    if (cap < S) continue;
    const long long ctas = (long long)tiles * S;
    const double waves = (double)((ctas + cap - 1) / cap);
    const double t = waves * (double)((n_chunks + S - 1) / S + 1) + 0.25 * (S - 1);
    if (t < best_t - 1e-9) {
      best_t = t;
      best = S;
    }
  }
  *S_out = best;
  return cudaSuccess;
}

}  // namespace

size_t matmul_tc_scratch_bytes(int n_tok, int64_t cols) {
  if (n_tok < 1 || cols < 32) return 0;
  const size_t tiles = (size_t)((n_tok + kTcN - 1) / kTcN);
  return tiles * (size_t)(cols / 32) * 2 * kOpBytes;
}

size_t matmul_tc_smem_bytes() { return sizeof(TcSmem) + 1024; }

cudaError_t launch_matmul_q8_0_tc(const void* W, int64_t rows, int64_t cols, const void* xq, int n_tok, float* y,
                                  const float* residual, void* scratch, cudaStream_t st) {
  if (n_tok <= 0 || rows <= 0) return cudaSuccess;
  const size_t smem = matmul_tc_smem_bytes();
  const int nb = (int)(cols / 32);
  const int tiles = (n_tok + kTcN - 1) / kTcN;
  const int row_tiles = (int)((rows + kTcM - 1) / kTcM);
  int S = 1;
  cudaError_t es = tc_split(row_tiles * tiles, nb / kTcChunk, smem, &S);
  if (es != cudaSuccess) return es;
  uint8_t* pack = static_cast<uint8_t*>(scratch);
  cudaError_t e = launch_kernel(pack_tokens_tc_kernel, dim3((unsigned)nb, (unsigned)tiles), dim3(512), 0, st,
                                static_cast<const uint8_t*>(xq), n_tok, nb, pack);
  if (e != cudaSuccess) return e;
  if (dry_run()) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int n_attr = 0;
  attr[n_attr].id = cudaLaunchAttributeClusterDimension;
  attr[n_attr].val.clusterDim.x = 1;
  attr[n_attr].val.clusterDim.y = 1;
  attr[n_attr].val.clusterDim.z = (unsigned)S;
  ++n_attr;
  if (pdl()) {
    attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
    ++n_attr;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n_attr;
  cfg.gridDim = dim3((unsigned)row_tiles, (unsigned)tiles, (unsigned)S);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  return cudaLaunchKernelEx(&cfg, matmul_q8_0_tc_kernel, static_cast<const uint8_t*>(W), (int)rows, nb,
                            static_cast<const uint8_t*>(pack), n_tok, y, residual);
}

unsigned int read_clear_error_matmul_tc() {
  unsigned int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_matmul_tc, sizeof v) != cudaSuccess) return 0xFFFFFFFFu;
  cudaMemcpyToSymbol(g_err_matmul_tc, &z, sizeof z);
  return v;
}

}  // namespace dsbk
