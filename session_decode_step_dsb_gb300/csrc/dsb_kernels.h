// Internal interface between the C ABI (dsb.cpp) and the CUDA translation
// units.  Host-side launch functions only; no device code here.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace dsbk {

// When set (per host thread), every launch_* function performs its one-time
// set-up (shared-memory attribute, occupancy query) but enqueues nothing.
// Used to warm those caches before a CUDA graph capture.
void set_dry_run(bool on);
bool dry_run();

// When set (per host thread), kernels launched through launch_kernel carry the
// programmatic-stream-serialization attribute, so that each kernel of the
// decode step may be scheduled while its predecessor finishes (its CTAs wait
// in pdl_wait() before touching the predecessor's results).
void set_pdl(bool on);
bool pdl();

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                 Args... args) {
  if (dry_run()) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (pdl()) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Per-call metadata staged in device memory (workspace), int32 words:
//   [0] n_seq  [1] tokens_per_seq  [2] n_tok  [3] total attention chunks
//   then batch_index[n_seq], seq_lens[n_seq], chunk_off[n_seq + 1], pos[n_tok]
// Offsets of the arrays are given explicitly to each kernel.
struct MetaView {
  const int32_t* batch_index;  // [n_seq]
  const int32_t* seq_lens;     // [n_seq]
  const int32_t* chunk_off;    // [n_seq + 1] prefix sums of ceil(seq_len / chunk)
  const int32_t* pos;          // [n_tok]
};

// Paged KV geometry per sequence (device arrays): the cache is a pool of
// 128-key pages [n_pages][Hkv][128][D]; sequence s finds key position p in
// page block_table[s * max_blocks + i], row p % 128, with i = p / 128
// (window[s] == 0) or i = (p / 128) % n_blocks[s] (a ring; window[s] > 0 also
// hides keys older than pos - window + 1).  block_table == NULL: the
// contiguous [F][Hkv][ctx][D] cache addressed through batch_index.
struct PagedView {
  const int32_t* block_table = nullptr;
  int max_blocks = 0;
  const int32_t* n_blocks = nullptr;
  const int32_t* window = nullptr;
};

int matmul_split(int64_t rows, int64_t cols, int num_sms);
// The (tiling, cluster split) plan of a matrix: returns S (CTAs per cluster
// along k), sets *G (row groups of 32 rows per CTA tile).
int matmul_plan_of(int64_t rows, int64_t cols, int num_sms, int* G);
// Narrow matmul (n_tok <= 16) whose activations are float rows quantised in
// the kernel: pro 1 = RMSNorm (norm_w, eps) of xf[n_tok][xf_stride] over cols
// values then q8_0; pro 2 = silu(gate) * up of xf = [gate | up] (stride
// xf_stride, up at column cols + c) then q8_0.  Outputs bitwise those of the
// standalone quantising kernel followed by launch_matmul_q8_0_narrow.
size_t matmul_fused_smem_bytes(int64_t rows, int64_t cols, int n_tok, int pro, int num_sms);
cudaError_t launch_matmul_q8_0_fused(int pro, const void* W, int64_t rows, int64_t cols, const float* xf,
                                     int xf_stride, const float* norm_w, float eps, int n_tok, float* y,
                                     const float* residual, int num_sms, cudaStream_t st);
unsigned int read_clear_error_matmul_fused();
size_t matmul_smem_bytes(int64_t rows, int64_t cols, int n_tok, int num_sms);
// Narrow matmul (n_tok <= 16) whose activations are already in the staged
// layout of dsb_actlayout.cuh (matmul_staged_bytes(n_tok, cols) bytes,
// 256-byte aligned), as the step's q8_0-emitting kernels write it; outputs
// bitwise those of launch_matmul_q8_0_narrow on the same activations.
cudaError_t launch_matmul_q8_0_staged(const void* W, int64_t rows, int64_t cols, const void* staged, int n_tok,
                                      float* y, const float* residual, int num_sms, cudaStream_t st);
size_t matmul_staged_bytes(int n_tok, int64_t cols);  // staged_act_bytes(n_tok, cols / 32)
// q8_0 rows xq [n_tok][cols/32] into the staged layout.
cudaError_t launch_stage_q8_0(const void* xq, int n_tok, int64_t cols, void* staged, cudaStream_t st);
unsigned int read_clear_error_matmul_staged();
// residual (may alias y, may be NULL): y = residual + W x.
cudaError_t launch_matmul_q8_0_narrow(const void* W, int64_t rows, int64_t cols, const void* xq, int n_tok, float* y,
                                      const float* residual, int32_t* isum, int num_sms, cudaStream_t st);

// Wide-batch matmul on the tensor cores (csrc/matmul_q8_0_tc.cu), any n_tok
// >= 1, cols % 256 == 0.  scratch: matmul_tc_scratch_bytes(n_tok, cols) bytes,
// 16-byte aligned (the packed token operands).  residual (may alias y, may be
// NULL): y = residual + W x.
size_t matmul_tc_scratch_bytes(int n_tok, int64_t cols);
size_t matmul_tc_smem_bytes();
cudaError_t launch_matmul_q8_0_tc(const void* W, int64_t rows, int64_t cols, const void* xq, int n_tok, float* y,
                                  const float* residual, void* scratch, cudaStream_t st);
unsigned int read_clear_error_matmul_tc();

cudaError_t launch_quantize_q8_0(const float* x, int64_t n_rows, int64_t cols, void* xq, cudaStream_t st);

// Float64 frequencies of the rotate-half pairs (a model constant) and the
// float32 factor every rotated value is multiplied by, passed to the RoPE
// kernels by value.  Plain RoPE: f_i = theta^(-2i/D), mscale 1.  YaRN
// (yarn_factor s > 1, original context yarn_orig_ctx): f_i blended between
// f_i and f_i / s by a ramp over the pair index, mscale 0.1 ln s + 1.
constexpr int kRopeMaxPairs = 512;
struct RopeFreqs {
  double f[kRopeMaxPairs];
  float mscale;
};
void rope_freqs(double theta, int head_dim, RopeFreqs* out, double yarn_factor = 0.0, int yarn_orig_ctx = 0,
                double yarn_beta_fast = 32.0, double yarn_beta_slow = 1.0);

// q_stride / k_stride: floats between consecutive token rows.
cudaError_t launch_rope_posvec(float* q, long long q_stride, int n_q_heads, float* k, long long k_stride,
                               int n_kv_heads, int head_dim, int n_tok, const int32_t* pos_dev,
                               const RopeFreqs& freqs, cudaStream_t st, const float* q_norm = nullptr,
                               const float* k_norm = nullptr, float eps = 0.0f);
// Step-fused RoPE + KV write on the [q | k | v] rows of qkv (row stride `stride`).
// q_norm / k_norm (float32 [head_dim], may be NULL): per-head RMS norm of the
// q / k heads before the rotation, with eps.
cudaError_t launch_rope_kv_write(float* qkv, long long stride, int n_q_heads, int n_kv_heads, int head_dim,
                                 const int32_t* pos_dev, const int32_t* batch_index_dev, int tokens_per_seq,
                                 int n_tok, void* kc, void* vc, int dtype, int ctx, const RopeFreqs& freqs,
                                 cudaStream_t st, const float* q_norm = nullptr, const float* k_norm = nullptr,
                                 float eps = 0.0f, PagedView pv = PagedView{});
cudaError_t launch_kv_scatter(void* kc, void* vc, int dtype, int n_kv_heads, int ctx, int head_dim,
                              const int32_t* batch_index_dev, int tokens_per_seq, const int32_t* pos_dev, int n_tok,
                              const float* k, const float* v, long long kv_stride, cudaStream_t st);

// Split-K decode attention: persistent partial kernel over the (chunk, kv head)
// items listed by meta.chunk_off (count read on the device), then the
// chunk-order merge.  max_items bounds the item count (sizes the grid);
// partials: float [n_tok][n_q_heads][max_chunks][head_dim + 2].  With xq_out
// non-NULL the merge writes q8_0 rows [n_tok][n_q_heads*head_dim/32 blocks]
// instead of float32 out.
// With pv.block_table set, kc / vc are page pools and ctx is unused; a
// sequence's work items are its chunks from the first one a window leaves
// visible (meta.chunk_off counts those).
// kv_rows: rows of the K / V tensors viewed as [kv_rows][head_dim] (F*Hkv*ctx
// for a contiguous cache, n_pages*Hkv*128 for a page pool); the kernels read
// them through TMA tensor maps of exactly that extent.
cudaError_t launch_attention_decode_multi(const float* q, long long q_stride, int n_q_heads, const void* kc,
                                          const void* vc, int dtype, int n_kv_heads, int ctx, int head_dim,
                                          long long kv_rows, MetaView meta, int n_seq, int tokens_per_seq,
                                          long long max_items, int max_chunks, float* partials, float* out,
                                          void* xq_out, cudaStream_t st, PagedView pv = PagedView{},
                                          void* xq_staged = nullptr);
// KV write through the paged view: token t of sequence t / T at pos[t].
cudaError_t launch_kv_scatter_paged(void* kp, void* vp, int dtype, int n_kv_heads, int head_dim, PagedView pv,
                                    int tokens_per_seq, const int32_t* pos_dev, int n_tok, const float* k,
                                    const float* v, long long kv_stride, cudaStream_t st);

size_t attention_partial_bytes(int n_tok, int n_q_heads, int head_dim, int ctx);

// staged (optional): also write the narrow matmul's staged layout of the rows.
cudaError_t launch_rmsnorm_quant(const float* x, const float* w, int n_tok, int hidden, float eps, void* xq,
                                 cudaStream_t st, void* staged = nullptr);
cudaError_t launch_silu_mul_quant(const float* gu, int n_tok, int ffn, void* xq, cudaStream_t st,
                                  void* staged = nullptr);
// tokens: device-readable token ids.  meta_src non-NULL: the kernel also
// copies n_words words from meta_src (device-readable, e.g. mapped pinned
// host memory) to meta_dst.
// The step's metadata words as a kernel parameter block (N words).
template <int N>
struct StepMetaWords {
  int32_t w[N];
};
constexpr int kEmbedParamMaxWords = 4096;  // 16 KiB of kernel parameters
// What a captured launch of the parameter-block embedding needs to rebuild
// its node parameters: the kernel, its launch shape and the block capacity.
struct EmbedParamNode {
  const void* func = nullptr;
  unsigned grid = 0, block = 0;
  long long n_blocks = 0;
  int capacity = 0;
};
// Embedding gather with the step's n_words metadata words (tokens first)
// passed by value in the kernel's parameters (n_words <= kEmbedParamMaxWords)
// and copied to meta_dst; `node`, if given, receives the launch description.
cudaError_t launch_embed_params(const void* table, int hidden, int n_tok, float* h, const int32_t* words, int n_words,
                                int32_t* meta_dst, cudaStream_t st, EmbedParamNode* node = nullptr);
cudaError_t launch_embed(const void* table, int hidden, const int32_t* tokens, int n_tok, float* h,
                         const int32_t* meta_src, int32_t* meta_dst, int n_words, cudaStream_t st);

// Scratch of dsb_attention_decode_multi_noalloc (csrc/noalloc.cu): a static
// device array, looked up once per device.
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;
constexpr int kNoAllocMaxSeqs = 256;
constexpr size_t kNoAllocTableBytes = 4096;  // the sequence table at the start of the array
cudaError_t noalloc_scratch(void** out);
cudaError_t launch_noalloc_table(const int32_t* batch_index, const int32_t* seq_lens, int n_seq, void* scratch,
                                 long long* total_chunks, cudaStream_t st);

unsigned int read_clear_error_matmul();
unsigned int read_clear_error_attention();

}  // namespace dsbk
