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
//    into a word-major layout: for each block and each of its eight 4-code
//    words, that word of every token side by side (then the fp32 scales), so
//    the inner loop reads four tokens' words with one warp-uniform (broadcast)
//    16-byte load.
//  * Block dots are __dp4a chains started from the bit pattern of 1.5 * 2^23:
//    |isum| <= 32*127*127 < 2^22, so the int32 result read as a float is
//    1.5*2^23 + isum exactly and one FADD converts it (no I2F).  The chains
//    of all n_tok tokens advance word by word together, so consecutive dp4a
//    instructions never depend on each other.
//  * When rows alone give too few CTAs, k is split over the CTAs of a thread
//    block cluster (<= 16 CTAs) and the partial sums are added through distributed
//    shared memory in cluster-rank order; every CTA of the cluster sums a
//    slice of the tile, from double-buffered sums, one cluster barrier per
//    tile.  No atomics; every reduction order depends only on (rows, cols) and
//    the device, never on n_tok, so column t of an n_tok = k call is bitwise
//    equal to the n_tok = 1 call.
#include "matmul_q8_0_kernel.cuh"

namespace dsbk {

namespace {

struct Plan {
  bool rows_mode;
  int S;
};

// Depends on (rows, cols) and the device only -- never on n_tok -- so that
// the summation order of every output is the same for every n_tok.  Each CTA
// of a cluster keeps the activations of its k-range in shared memory, which at
// n_tok = 16 allows at most 8 k-steps (36 KiB) next to the weight rings.
// Rows mode: 128-row tiles, warps own 32 rows over the CTA's whole k-range;
// k-split mode: 32-row tiles whose k-steps the 4 warps share.  Among the
// admissible (mode, S) the smallest estimated makespan (tiles per cluster x
// k-steps per warp, plus a per-tile reduction cost) wins, with the number of
// clusters that fit on the device at once taken from the occupancy query of
// the n_tok = 16 instance (the largest shared memory).
Plan matmul_plan(int64_t rows, int64_t cols, int num_sms) {
  struct Memo {
    int64_t rows, cols;
    int num_sms;
    Plan plan;
  };
  static std::mutex mu;
  static Memo memo[64];
  static int n_memo = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_memo; ++i)
    if (memo[i].rows == rows && memo[i].cols == cols && memo[i].num_sms == num_sms) return memo[i].plan;
  const int nks = (int)(cols / 256);
  int s_max = nks < kMaxCluster ? nks : kMaxCluster;
  int s_min = (nks + 7) / 8;
  if (s_min > s_max) s_min = s_max;
  if (s_min < 1) s_min = 1;
  Plan best{false, s_min};
  double best_cost = 1e30;
  bool queried = true;
  for (int mode = 0; mode < 2; ++mode) {
    const bool rm = mode == 1;
    const int tile = rm ? kPairs * kRowsPerCta : kRowsPerCta;
    const int tiles = (int)((rows + tile - 1) / tile);
    for (int S = s_min; S <= s_max; ++S) {
      const size_t smem = smem_bytes((nks + S - 1) / S, 16, rm);
      int clusters = 0;
      const cudaError_t e = rm ? cluster_capacity<16, false, true, 0>(S, smem, &clusters)
                               : cluster_capacity<16, false, false, 0>(S, smem, &clusters);
      if (e != cudaSuccess) {
        (void)cudaGetLastError();
        queried = false;
        clusters = (2 * num_sms) / S;  // estimate: two CTAs per SM
      }
      if (clusters < 1) continue;
      const int per = (tiles + clusters - 1) / clusters;
      const int ksteps = (nks + S - 1) / S;
      // time ~ tiles per cluster x (k-steps each warp runs + per-tile sync cost)
      const double sync = (rm && S == 1) ? 0.0 : 0.5;
      const double warp_steps = rm ? (double)ksteps : (double)((ksteps + kPairs - 1) / kPairs);
      const double c = per * (warp_steps + sync);
      if (c < best_cost - 1e-9) {
        best_cost = c;
        best = Plan{rm, S};
      }
    }
  }
  if (queried && n_memo < 64) memo[n_memo++] = Memo{rows, cols, num_sms, best};
  return best;
}

}  // namespace

int matmul_split(int64_t rows, int64_t cols, int num_sms) { return matmul_plan(rows, cols, num_sms).S; }

int matmul_plan_of(int64_t rows, int64_t cols, int num_sms, bool* rows_mode) {
  const Plan pl = matmul_plan(rows, cols, num_sms);
  *rows_mode = pl.rows_mode;
  return pl.S;
}

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
  ActSrc src;
  src.xq = static_cast<const uint8_t*>(xq);
  if (isum)
    return pl.rows_mode ? dispatch<true, true, 0>(n_tok, w8, (int)rows, nb, src, y, residual, isum, pl.S, smem, st)
                        : dispatch<true, false, 0>(n_tok, w8, (int)rows, nb, src, y, residual, isum, pl.S, smem, st);
  return pl.rows_mode ? dispatch<false, true, 0>(n_tok, w8, (int)rows, nb, src, y, residual, isum, pl.S, smem, st)
                      : dispatch<false, false, 0>(n_tok, w8, (int)rows, nb, src, y, residual, isum, pl.S, smem, st);
}

namespace {
thread_local bool g_dry_run = false;
}
thread_local bool g_pdl = false;
void set_dry_run(bool on) { g_dry_run = on; }
bool dry_run() { return g_dry_run; }
void set_pdl(bool on) { g_pdl = on; }
bool pdl() { return g_pdl; }

unsigned int read_clear_error_matmul() { return read_clear_error_unit(); }

}  // namespace dsbk
