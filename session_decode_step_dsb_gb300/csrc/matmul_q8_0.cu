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
//  * One persistent CTA per SM, 8 warps.  A warp owns 32 weight rows (lane =
//    row) and every token; k-steps of 8 blocks = 272 bytes = 17 x 16 bytes,
//    so every row chunk is 16-byte aligned whenever cols % 256 == 0.
//  * Each warp streams its 32 row chunks with one 2-D TMA tensor copy per
//    stage (cp.async.bulk.tensor over the matrix viewed as rows x (cols/32 *
//    17) 16-bit elements, box 136 x 32, so one copy moves 32 rows x 272
//    bytes) into its own 2-stage shared-memory ring guarded by mbarriers
//    (one copy per stage rather than one per row: the copy engine's issue
//    rate, not HBM, bounded the per-row form); it reads a stage back into
//    registers (17 conflict-free 16-byte shared loads per lane), hands the
//    stage to the copy two units ahead and computes from registers, so two
//    copies stay in flight per warp and no warp waits on another in the k loop.
//  * Activation blocks of the CTA's k-range arrive by one bulk copy per token
//    and are unpacked once, at kernel start, into a word-major layout: for each block and each of its eight 4-code
//    words, that word of every token side by side (then the fp32 scales), so
//    the inner loop reads four tokens' words with one warp-uniform (broadcast)
//    16-byte load.
//  * Up to 7 tokens, block dots are __dp4a chains started from the bit pattern
//    of 1.5 * 2^23: |isum| <= 32*127*127 < 2^22, so the int32 result read as a
//    float is 1.5*2^23 + isum exactly and one FADD converts it (no I2F).  Four
//    tokens' chains advance word by word together, so consecutive dp4a
//    instructions never depend on each other.
//  * From 8 tokens on, the block dots run on the tensor cores: a warp's 32
//    rows x 8-token tiles x one q8_0 block are two mma.sync m16n8k16 (f16 in,
//    f32 accumulate).  Weight codes enter as the exact f16 values 1152 + q
//    (one xor and two byte permutes per four codes), activation codes as f16
//    q, and the accumulator starts at -1152 * (the block's activation code
//    sum), so the product is the exact integer block dot.  dp4a's issue rate
//    (64 per clock per SM, measured) and the shared-memory broadcasts that feed
//    it bound the dp4a form at 16 tokens; the tensor-core form reads each
//    activation word once per warp and fragment.  Both forms scale and add the
//    block dots with the same float operations in the same order, so their
//    outputs are bitwise equal.
//  * A CTA tile is G row groups; the 8 / G warps of a group take interleaved
//    k-steps, and k is further split over the CTAs of a thread block cluster
//    (<= 16 CTAs).  Partial sums are added in warp order in shared memory and
//    in cluster-rank order through distributed shared memory, one cluster
//    barrier per tile (double-buffered sums).  No atomics; every reduction
//    order depends only on (rows, cols) and the device, never on n_tok, so
//    column t of an n_tok = k call is bitwise equal to the n_tok = 1 call.
#include "matmul_q8_0_kernel.cuh"

namespace dsbk {

namespace {

struct Plan {
  int G;  // row groups (of 32 rows) per CTA tile; 8 / G warps per group
  int S;  // CTAs per cluster along k
};

int max_smem_optin() {
  static std::mutex mu;
  static int dev_cached = -1, value = 0;
  std::lock_guard<std::mutex> lock(mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev != dev_cached) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
    value = v;
    dev_cached = dev;
  }
  return value;
}

// Depends on (rows, cols) and the device only -- never on n_tok -- so that
// the summation order of every output is the same for every n_tok.  Each CTA
// keeps the activations of its k-range in shared memory, so at n_tok = 16 the
// k-range of one CTA is bounded (about 12 k-steps next to the weight rings);
// longer rows are split over a cluster.  Among the admissible (G, S) the
// smallest estimated makespan wins: rounds of tiles over the clusters that fit
// on the device at once (occupancy query of the n_tok = 16 instance, the
// largest shared memory) x the k-steps of one warp per tile plus the tile's
// reduction costs, stretched when too few SMs are busy to draw the HBM
// bandwidth (each SM keeps ~140 KB of weights in flight).
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
  const int s_max = nks < kMaxCluster ? nks : kMaxCluster;
  const size_t cap = (size_t)max_smem_optin();
  Plan best{kWarps, s_max};
  double best_cost = 1e30;
  bool queried = cap > 0;
  for (int G = kWarps; G >= 1; G /= 2) {
    const int KW = kWarps / G;
    const long long tiles = (rows + 32LL * G - 1) / (32LL * G);
    for (int S = 1; S <= s_max; ++S) {
      const int kr = (nks + S - 1) / S;
      const size_t smem = smem_bytes(kr, 16, G, S);
      if (cap > 0 && smem > cap) continue;
      int clusters = 0;
      const cudaError_t e = cluster_capacity<16, false, 0>(S, smem, &clusters);
      if (e != cudaSuccess) {
        (void)cudaGetLastError();
        queried = false;
        clusters = num_sms / S;  // estimate: one CTA per SM
      }
      if (clusters < 1) continue;
      const long long rounds = (tiles + clusters - 1) / clusters;
      const double per_tile = (double)((kr + KW - 1) / KW) + (KW > 1 ? 0.3 : 0.0) + (S > 1 ? 0.4 : 0.0);
      const long long busy = (tiles < clusters ? tiles : clusters) * S;
      const double stretch = busy >= 96 ? 1.0 : 96.0 / (double)busy;
      const double c = (double)rounds * per_tile * stretch;
      if (c < best_cost - 1e-9) {
        best_cost = c;
        best = Plan{G, S};
      }
    }
  }
  if (queried && n_memo < 64) memo[n_memo++] = Memo{rows, cols, num_sms, best};
  return best;
}

}  // namespace

int matmul_split(int64_t rows, int64_t cols, int num_sms) { return matmul_plan(rows, cols, num_sms).S; }

int matmul_plan_of(int64_t rows, int64_t cols, int num_sms, int* G) {
  const Plan pl = matmul_plan(rows, cols, num_sms);
  *G = pl.G;
  return pl.S;
}

size_t matmul_smem_bytes(int64_t rows, int64_t cols, int n_tok, int num_sms) {
  const Plan pl = matmul_plan(rows, cols, num_sms);
  const int nks = (int)(cols / 256);
  const int kr_max = (nks + pl.S - 1) / pl.S;
  return smem_bytes(kr_max, n_tok, pl.G, pl.S);
}

cudaError_t launch_matmul_q8_0_narrow(const void* W, int64_t rows, int64_t cols, const void* xq, int n_tok,
                                      float* y, const float* residual, int32_t* isum, int num_sms, cudaStream_t st) {
  const Plan pl = matmul_plan(rows, cols, num_sms);
  const size_t smem = matmul_smem_bytes(rows, cols, n_tok, num_sms);
  const int nb = (int)(cols / 32);
  const uint8_t* w8 = static_cast<const uint8_t*>(W);
  ActSrc src;
  src.xq = static_cast<const uint8_t*>(xq);
  if (isum) return dispatch<true, 0>(n_tok, w8, (int)rows, nb, src, y, residual, isum, pl.G, pl.S, smem, st);
  return dispatch<false, 0>(n_tok, w8, (int)rows, nb, src, y, residual, isum, pl.G, pl.S, smem, st);
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
