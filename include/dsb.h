/*
 * dsb.h -- C ABI of libdsb.so: the batched multi-session decode step on
 * GB300 (sm_103a).
 *
 * One decode step advances b live sessions (1 <= b <= full_batch_size) by one
 * token each, or by T = K+1 tokens each under speculative decode, in one GPU
 * pass.  Sources of the operations (the pages this library restates):
 *
 *   [DS4]  antirez/ds4 PR #530, "Batched decode: co-decode N live sessions in
 *          one GPU pass (opt-in)": the narrow-batch q8_0 matmul ("Why it's
 *          worth it -- the narrow-batch matmul"), the pos-vector RoPE, the
 *          multi-sequence decode attention and the engine-owned scratch vs
 *          per-session state split (commit bodies of the walk-through).
 *   [QAIC] quic/efficient-transformers PR #1305, "[feature] Enable Dynamic
 *          Batching": KV cache always sized for full_batch_size, addressed by
 *          batch_index ("Objective"); K+1 speculative tokens per sequence and
 *          rejecting bad combinations with clear errors before execution
 *          ("Assumptions and limitations").
 *   [PTO]  hw-native-sys/pypto-lib PR #841, "Add: dynamic public batch (1..16)
 *          for Qwen3-14B decode": live batch taken from the seq_lens
 *          descriptor; contract 1 <= batch <= batch_pad (commit message).
 *
 * Conventions for every call
 *   - Device pointers point to memory the caller owns (e.g. torch tensors);
 *     the library never frees them.  Host arrays (batch_index, pos, seq_lens)
 *     are read during the call only; the caller may reuse them on return.
 *   - Every call validates all arguments on the host BEFORE any CUDA call and
 *     returns a status; on a non-OK status no device memory has been written.
 *     It never aborts.  dsb_last_error() gives a message for the last non-OK
 *     status of the calling thread.
 *   - Work is enqueued on the given stream (a cudaStream_t; NULL = legacy
 *     default stream) and runs asynchronously.  Device pointers must be 16-byte
 *     aligned.  Kernels never spin on flags other CTAs set: CTAs of one
 *     launch meet only at the hardware barrier of their thread-block cluster
 *     (co-scheduled by construction), and the mbarrier waits inside a CTA are
 *     bounded and, if exceeded, set a device error word reported by
 *     dsb_device_error().
 *   - A workspace serves one stream at a time (the engine-owned scratch shared
 *     by the sessions one thread drives, [DS4] session-split commit).
 *   - Host threads may call concurrently when each passes its own workspace
 *     (and model, step graph, batch former): the library's own host state --
 *     launch plans, tensor maps, occupancy and device queries -- is memoised
 *     behind locks.  The one exception is the shared scratch of
 *     dsb_attention_decode_multi_noalloc, described there.
 */
#ifndef DSB_H
#define DSB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSB_OK = 0,
  DSB_ERR_INVALID_ARG = 1, /* bad pointer, size, index or combination     */
  DSB_ERR_UNSUPPORTED = 2, /* valid but not served by this library        */
  DSB_ERR_WORKSPACE = 3,   /* workspace missing or too small              */
  DSB_ERR_CUDA = 4,        /* a CUDA runtime call failed (see last_error) */
  DSB_ERR_TIMEOUT = 5,     /* a bounded host wait ran out                 */
  DSB_ERR_DEVICE = 6       /* a kernel reported a bounded wait that ran out */
} dsb_status;

typedef enum { DSB_F16 = 0, DSB_BF16 = 1 } dsb_dtype;

/* Largest live batch and token count one call accepts (metadata capacity). */
#define DSB_MAX_SEQS 1024
#define DSB_MAX_TOKENS 8192
/* Largest n_tok of the narrow matmul (one weight read serves all tokens). */
#define DSB_NARROW_MAX 16
/* Keys per split-K chunk of the decode attention (independent of b, n_tok). */
#define DSB_ATTN_CHUNK 128

/* A q8_0 matrix on the device: rows x cols values, cols % 32 == 0, stored as
 * rows x (cols/32) blocks of 34 bytes laid end to end; block i of row r sits
 * at byte (r*(cols/32) + i)*34 and holds the fp16 scale d (little-endian)
 * followed by 32 int8 codes; value k of the block is d * q[k].
 * ([DS4] "Why it's worth it": 32-weight blocks, int8 plus an fp16 scale.) */
typedef struct {
  const void* blocks;
  int64_t rows;
  int64_t cols;
} dsb_q8_0_mat;

/* A retained KV cache on the device ([QAIC] "Objective"): K and V each
 * [full_batch_size][n_kv_heads][ctx][head_dim] in dtype, row-major.  The
 * attention names a row (slot, kv head, position) by a 32-bit tensor
 * coordinate: full_batch_size * n_kv_heads * ctx above 2^31 - 129 is
 * DSB_ERR_UNSUPPORTED (no such cache fits in one GPU's memory at
 * head_dim >= 64). */
typedef struct {
  void* k;
  void* v;
  int32_t dtype; /* dsb_dtype */
  int32_t full_batch_size;
  int32_t n_kv_heads;
  int32_t ctx;
  int32_t head_dim;
} dsb_kv_cache;

/* Opaque caller-sized scratch: split-K attention partials and the staged
 * per-call metadata ([DS4] session-split commit: engine-owned scratch). */
typedef struct dsb_workspace dsb_workspace;

/* ---- library / workspace ------------------------------------------------ */

/* Message for the calling thread's last non-OK status ("" if none). */
const char* dsb_last_error(void);

/* Build string: compile-time architecture and version. */
const char* dsb_version(void);

/* Device bytes a workspace needs to serve calls with up to max_tokens token
 * rows, n_q_heads query heads of width head_dim, against caches of length
 * ctx.  Returns 0 if an argument is out of range. */
size_t dsb_workspace_bytes(int max_tokens, int n_q_heads, int head_dim, int ctx);

/* Wrap caller-owned device memory [device_ptr, device_ptr + device_bytes) as a
 * workspace bound to the current CUDA device.  Allocates the workspace's small
 * pinned host staging ring and its events (set-up time only).  *out is NULL on
 * failure. */
dsb_status dsb_workspace_create(void* device_ptr, size_t device_bytes, dsb_workspace** out);

/* Waits (bounded) for the workspace's staged copies, then frees the host-side
 * resources.  Does not free the device memory. */
dsb_status dsb_workspace_destroy(dsb_workspace* ws);

/* Reads and clears the device error word set by a kernel whose bounded
 * mbarrier wait ran out (synchronises the current device).  DSB_OK if none. */
dsb_status dsb_device_error(void);

/* ---- the hot path --------------------------------------------------------- */

/* q8_0-quantise n_rows float32 rows of length cols (cols % 32 == 0) into
 * xq (n_rows * cols/32 blocks of 34 bytes).  Per 32 values: d = max|x|/127 in
 * float32, q = round-half-away(x/d) clamped to [-127,127] (0 if d == 0), scale
 * stored as fp16(d) round-to-nearest-even.  Bit-identical to the host codec.
 * x: device float32 [n_rows][cols].  xq: device, 16-byte aligned. */
dsb_status dsb_quantize_q8_0(const float* x, int64_t n_rows, int64_t cols, void* xq, void* stream);

/* Narrow-batch q8_0 matmul ([DS4] "Why it's worth it -- the narrow-batch
 * matmul"; the narrow-batch q8_0 matmul commit):
 *   y[t][r] = sum_i fp32(dW[r,i]) * fp32(dX[t,i]) * sum_k qW[r,i,k] qX[t,i,k]
 * for 1 <= n_tok <= DSB_NARROW_MAX.  Each weight block is read from HBM once
 * per call and dotted against all n_tok activation blocks.  xq: device q8_0
 * [n_tok][cols/32 blocks]; y: device float32 [n_tok][rows] (token-major).
 * Column t of y is bitwise equal to the same input run with n_tok = 1.
 * Requires cols % 256 == 0 (rows of 16-byte-aligned 8-block chunks). */
dsb_status dsb_matmul_q8_0_narrow(const dsb_q8_0_mat* w, const void* xq, int n_tok, float* y,
                                  void* stream);

/* Same product for any n_tok >= 1: tokens in chunks of DSB_NARROW_MAX through
 * the narrow kernel (weights re-read ceil(n_tok/16) times).  Columns are
 * bitwise equal to the narrow call's. */
dsb_status dsb_matmul_q8_0(const dsb_q8_0_mat* w, const void* xq, int n_tok, float* y, void* stream);

/* Debug emission of the narrow kernel: instead of y it writes the exact int32
 * block dot products isum[t][r][i] = sum_k qW[r,i,k] qX[t,i,k]
 * (device int32 [n_tok][rows][cols/32]), through the same loads and dp4a
 * chain as dsb_matmul_q8_0_narrow. */
dsb_status dsb_matmul_q8_0_block_dots(const dsb_q8_0_mat* w, const void* xq, int n_tok,
                                      int32_t* isum, void* stream);

/* The narrow product from activations already in a staged layout: the path
 * the decode step takes, where the kernel that produces the q8_0 activations
 * writes this layout too ([DS4] "Why it's worth it -- the narrow-batch
 * matmul": each weight block crosses HBM once for every token).
 * dsb_stage_q8_0 writes the staged layout of xq (device q8_0 [n_tok][cols/32])
 * that the narrow kernel reads at n_tok tokens: per block and 4-code word the
 * words of every token side by side, then the scales (with the blocks' code
 * sums from 8 tokens on); dsb_matmul_q8_0_staged computes y (device float32
 * [n_tok][rows], 16-byte aligned) from it, bitwise equal to
 * dsb_matmul_q8_0_narrow on xq.
 * staged: device, 16-byte aligned, at least dsb_matmul_q8_0_staged_bytes(
 * n_tok, cols) bytes, owned by the caller; its contents are only meaningful
 * to the staged matmul at the same cols and n_tok.  n_tok in [1, 16]
 * (DSB_ERR_INVALID_ARG otherwise); a short or unaligned staged buffer is
 * DSB_ERR_WORKSPACE; cols % 256 != 0 is DSB_ERR_UNSUPPORTED.
 * dsb_matmul_q8_0_staged_bytes is 0 for arguments out of range. */
size_t dsb_matmul_q8_0_staged_bytes(int n_tok, int64_t cols);
dsb_status dsb_stage_q8_0(const dsb_q8_0_mat* w, const void* xq, int n_tok, void* staged, size_t staged_bytes,
                          void* stream);
dsb_status dsb_matmul_q8_0_staged(const dsb_q8_0_mat* w, const void* staged, size_t staged_bytes, int n_tok, float* y,
                                  void* stream);

/* Scratch bytes dsb_matmul_q8_0_wide needs: the token operands packed for the
 * tensor cores, ceil(n_tok/128) * cols/32 * 16384 bytes.  0 if n_tok is out
 * of [1, DSB_MAX_TOKENS] or cols is not a positive multiple of 256. */
size_t dsb_matmul_q8_0_wide_scratch_bytes(int n_tok, int64_t cols);

/* Wide-batch q8_0 matmul on the tensor cores: the product of
 * dsb_matmul_q8_0_narrow for any 1 <= n_tok <= DSB_MAX_TOKENS.  Speculative
 * decode puts K+1 token rows per sequence through every matmul ([QAIC]
 * "Assumptions and limitations"), beyond the narrow kernel's 16 ([DS4] "Why
 * it's worth it -- the narrow-batch matmul").  Every dequantised value d*q is
 * split exactly into two f16 values and the products accumulate in float32
 * over the whole row (so the result differs from the narrow kernel's in
 * rounding order only).  Weights are read once per 128 token rows.  Values
 * must satisfy |d*q| <= 65504, i.e. q8_0 scales up to 65504/127; a larger
 * scale makes dsb_device_error report DSB_ERR_DEVICE.  xq: device q8_0
 * [n_tok][cols/32 blocks]; y: device float32 [n_tok][rows]; scratch: device,
 * 16-byte aligned, at least dsb_matmul_q8_0_wide_scratch_bytes(n_tok, cols)
 * bytes, owned by the caller and free again once the stream has passed the
 * call.  Requires cols % 256 == 0 (DSB_ERR_UNSUPPORTED otherwise); a short
 * scratch is DSB_ERR_WORKSPACE. */
dsb_status dsb_matmul_q8_0_wide(const dsb_q8_0_mat* w, const void* xq, int n_tok, float* y,
                                void* scratch, size_t scratch_bytes, void* stream);

/* Pos-vector RoPE ([DS4] pos-vector RoPE commit): every token row t carries
 * its own position pos[t] (host int32[n_tok], each in [0, 2^24)).  In place
 * on q (device float32 [n_tok][n_q_heads][head_dim]) and k (device float32
 * [n_tok][n_kv_heads][head_dim]; may be NULL with n_kv_heads = 0).  Rotate-half
 * pairs (i, i + D/2), angle pos * theta^(-2i/D), angle and its sine/cosine in
 * float64, rotation in float32.  Row t is bitwise equal to an n_tok = 1 call. */
dsb_status dsb_rope_posvec(float* q, int n_q_heads, float* k, int n_kv_heads, int head_dim,
                           int n_tok, const int32_t* pos, float theta, dsb_workspace* ws,
                           void* stream);

/* RoPE parameters.  yarn_factor <= 1 (e.g. a zeroed struct with theta set):
 * the plain pos-vector RoPE of dsb_rope_posvec.  yarn_factor = s > 1: the
 * YaRN variant ([DS4] pos-vector RoPE commit, "plain and YaRN paths"; read as
 * published by Peng et al. 2023, "YaRN: Efficient Context Window Extension of
 * Large Language Models", sections 3.2-3.3): with L = yarn_orig_ctx and
 * corr(b) = D ln(L / (2 pi b)) / (2 ln theta), low = max(floor(corr(beta_fast)), 0),
 * high = min(ceil(corr(beta_slow)), D - 1), pair i's frequency
 * f_i = theta^(-2i/D) becomes f_i (1 - ramp_i) + (f_i / s) ramp_i with
 * ramp_i = clamp((i - low) / max(high - low, 0.001), 0, 1), and every rotated
 * value is multiplied by 0.1 ln s + 1 (float32).  Frequencies and the
 * correction range in float64.  Requires theta > 0 finite; with yarn:
 * yarn_orig_ctx >= 1 and 0 < beta_slow < beta_fast (typically 32 and 1). */
typedef struct {
  float theta;
  float yarn_factor;
  int32_t yarn_orig_ctx;
  float yarn_beta_fast;
  float yarn_beta_slow;
} dsb_rope;

/* Per-head RMS norm, then the pos-vector RoPE ([DS4] the fused head norm +
 * RoPE tail and its position-vector twin): every head vector x of q (and of k)
 * becomes x / sqrt(mean(x^2) + eps) * w elementwise, w = q_norm (k_norm) a
 * device float32 [head_dim] weight, and is then rotated as dsb_rope_posvec
 * with the parameters in rope (host struct, read during the call).
 * Either weight may be NULL: those heads are only rotated.  Sum of squares,
 * root and division in float32 (round to nearest).  Other arguments and errors
 * as dsb_rope_posvec; eps must be finite and >= 0. */
dsb_status dsb_head_rmsnorm_rope(float* q, int n_q_heads, float* k, int n_kv_heads, int head_dim, int n_tok,
                                 const int32_t* pos, const dsb_rope* rope, const float* q_norm, const float* k_norm,
                                 float eps, dsb_workspace* ws, void* stream);

/* KV write through batch_index ([QAIC] "Objective"; [DS4] batched-decode
 * encoder commit).  For s < n_seq, j < tokens_per_seq, t = s*T + j:
 *   K[batch_index[s]][h][pos[t]][:] = cvt(k[t][h][:]),  same for V,
 * cvt = float32 -> cache dtype, round to nearest even.  Nothing else in the
 * cache is written.  batch_index: host int32[n_seq], distinct, in
 * [0, full_batch_size); pos: host int32[n_seq*T] in [0, ctx).  k, v: device
 * float32 [n_tok][n_kv_heads][head_dim]. */
dsb_status dsb_kv_scatter(const dsb_kv_cache* kv, const int32_t* batch_index, int n_seq,
                          int tokens_per_seq, const int32_t* pos, const float* k, const float* v,
                          dsb_workspace* ws, void* stream);

/* Multi-sequence GQA decode attention ([DS4] multi-sequence decode attention
 * commit; [PTO] live batch from seq_lens).  Sequence s (cache slot
 * batch_index[s], KV length seq_lens[s] after this step's writes) has query
 * rows t = s*T + j; token j sees keys 0 .. seq_lens[s]-T+j.  Query head h
 * reads kv head h / (n_q_heads / n_kv_heads).  score = q.k / sqrt(head_dim);
 * out = softmax(score) V.  Split-K: keys are cut into DSB_ATTN_CHUNK chunks,
 * one partial (max, sum, acc) per chunk, merged in chunk order by a second
 * kernel; no atomics, so row t is bitwise equal to a single-sequence call.
 * q: device float32 [n_tok][n_q_heads][head_dim]; out: device float32, same
 * shape.  seq_lens: host int32[n_seq], each in [T, ctx].  head_dim in
 * {64, 128}; n_q_heads/n_kv_heads * T <= 64. */
dsb_status dsb_attention_decode_multi(const float* q, int n_q_heads, const dsb_kv_cache* kv,
                                      const int32_t* batch_index, int n_seq, int tokens_per_seq,
                                      const int32_t* seq_lens, float* out, dsb_workspace* ws,
                                      void* stream);

/* The same attention with its output q8_0-quantised in the merge, as the
 * decode step feeds the O projection ([DS4] "What": activations enter every
 * matmul pre-quantised): xq receives n_tok rows of n_q_heads*head_dim/32
 * q8_0 blocks (device, 16-byte aligned), row t holding heads 0..Hq-1 in order.
 * Arguments and errors otherwise as dsb_attention_decode_multi. */
dsb_status dsb_attention_decode_multi_q8_0(const float* q, int n_q_heads, const dsb_kv_cache* kv,
                                           const int32_t* batch_index, int n_seq, int tokens_per_seq,
                                           const int32_t* seq_lens, void* xq, dsb_workspace* ws,
                                           void* stream);

/* ---- paged / ring KV geometry ([PTO] paged attention with a block table,
 * pa_max_blocks; [DS4] multi-sequence decode attention commit: each sequence
 * carries its own cache view and ring geometry). ----------------------------
 *
 * The cache is a pool of pages of DSB_KV_PAGE keys, K and V each
 * [n_pages][n_kv_heads][DSB_KV_PAGE][head_dim] in the cache dtype.  Sequence s
 * (host arrays): block_table[s * max_blocks + i] (page indices, the first
 * n_blocks[s] used) and window[s].  The key at absolute position p is row
 * p % DSB_KV_PAGE of page block_table[s][i] with i = p / DSB_KV_PAGE
 * (window[s] == 0: a linear table, which must cover the sequence) or
 * i = (p / DSB_KV_PAGE) % n_blocks[s] (window[s] > 0: a ring holding the newest
 * n_blocks[s] * DSB_KV_PAGE positions, at least window[s] + T - 1).  Draft
 * token j of T sits at pos = seq_lens[s] - T + j and sees keys
 * max(0, pos - window + 1) .. pos (all keys 0 .. pos without a window).
 * Sequences may share pages for reading.  Violations are DSB_ERR_INVALID_ARG
 * before any launch. */
#define DSB_KV_PAGE 128

typedef struct {
  void* k;          /* device page pool */
  void* v;          /* device page pool */
  dsb_dtype dtype;
  int32_t n_pages;  /* n_pages * n_kv_heads * DSB_KV_PAGE <= 2^31 - 129 */
  int32_t n_kv_heads;
  int32_t head_dim;
} dsb_kv_pages;

/* KV write through the paged geometry: the k and v rows of token t
 * (sequence t / T) at pos[t] (host int32[n_seq*T], >= 0), converted to the
 * cache dtype (round to nearest even).  Two tokens of one call writing the same
 * page row are rejected.  k, v: device float32 [n_tok][n_kv_heads][head_dim]. */
dsb_status dsb_kv_scatter_paged(const dsb_kv_pages* kv, const int32_t* block_table, int max_blocks,
                                const int32_t* n_blocks, const int32_t* window, int n_seq,
                                int tokens_per_seq, const int32_t* pos, const float* k,
                                const float* v, dsb_workspace* ws, void* stream);

/* Multi-sequence GQA decode attention through the paged geometry; q, out and
 * the result as dsb_attention_decode_multi.  The workspace must hold the
 * split-K partials of the longest visited key range (a workspace made for a
 * ctx of max_blocks * DSB_KV_PAGE does). */
dsb_status dsb_attention_decode_paged(const float* q, int n_q_heads, const dsb_kv_pages* kv,
                                      const int32_t* block_table, int max_blocks, const int32_t* n_blocks,
                                      const int32_t* window, int n_seq, int tokens_per_seq,
                                      const int32_t* seq_lens, float* out, dsb_workspace* ws,
                                      void* stream);

/* ---- step glue, one fused kernel per call ([DS4] "What": RoPE/norm around
 * the attention projections and the dense stages run once for all sessions;
 * each emits the pre-quantised q8_0 activations the next matmul reads). ---- */

/* xq[t] = q8_0(x[t] / sqrt(mean(x[t]^2) + eps) * w), float32 arithmetic, the
 * q8_0 codec of dsb_quantize_q8_0.  x: device float32 [n_tok][hidden]; w:
 * device float32 [hidden]; xq: device q8_0 [n_tok][hidden/32].  hidden must be
 * a multiple of 256 in [256, 8192] (DSB_ERR_UNSUPPORTED otherwise). */
dsb_status dsb_rmsnorm_q8_0(const float* x, const float* w, int n_tok, int hidden, float eps, void* xq,
                            void* stream);

/* xq[t] = q8_0(silu(g) * u) with g = gu[t][0:ffn], u = gu[t][ffn:2*ffn],
 * silu(g) = g / (1 + exp(-g)) in float32.  gu: device float32 [n_tok][2*ffn];
 * xq: device q8_0 [n_tok][ffn/32]; ffn % 32 == 0. */
dsb_status dsb_silu_mul_q8_0(const float* gu, int n_tok, int ffn, void* xq, void* stream);

/* The narrow matmul with its activation quantisation in the same kernel: each
 * CTA quantises the activation blocks of its own k-range from float rows, so
 * no q8_0 activation array round-trips through memory and one launch replaces
 * two.  Outputs are bitwise those of the two-call sequence.
 *   dsb_rmsnorm_matmul_q8_0: y = W q8(rmsnorm(x) * norm_w) as
 *     dsb_rmsnorm_q8_0(x, norm_w, n_tok, w->cols, eps) then
 *     dsb_matmul_q8_0_narrow; x: device float32 [n_tok][w->cols].
 *   dsb_silu_matmul_q8_0: y = W q8(silu(g) * u) as dsb_silu_mul_q8_0(gu,
 *     n_tok, w->cols) then dsb_matmul_q8_0_narrow; gu: device float32
 *     [n_tok][2 * w->cols] = [gate | up].
 * y: device float32 [n_tok][w->rows].  n_tok in [1, 16]; w->cols a multiple of
 * 256 (and <= 8192 for the RMSNorm); errors as those calls. */
dsb_status dsb_rmsnorm_matmul_q8_0(const dsb_q8_0_mat* w, const float* x, const float* norm_w, float eps, int n_tok,
                                   float* y, void* stream);
dsb_status dsb_silu_matmul_q8_0(const dsb_q8_0_mat* w, const float* gu, int n_tok, float* y, void* stream);

/* h[t] = the dequantised q8_0 row token_ids[t] of the embedding table
 * (device q8_0 [vocab][hidden/32]); exact in float32.  token_ids: host int32
 * [n_tok], each in [0, vocab) (DSB_ERR_INVALID_ARG otherwise); staged through
 * the workspace.  h: device float32 [n_tok][hidden]. */
dsb_status dsb_embed_q8_0(const void* table, int vocab, int hidden, const int32_t* token_ids, int n_tok,
                          float* h, dsb_workspace* ws, void* stream);

/* The step's fused RoPE + KV write on the [q | k | v] rows of a QKV
 * projection: qkv is device float32 [n_tok][(n_q_heads + 2*Hkv) * head_dim].
 * q heads are rotated in place (as dsb_rope_posvec); k rotated and v as is are
 * written, converted to the cache dtype, at K/V[batch_index[s]][h][pos[t]]
 * (as dsb_kv_scatter).  The k and v parts of qkv are left as they were.
 * rope: the RoPE parameters (plain or YaRN) as dsb_head_rmsnorm_rope.
 * q_norm / k_norm (device float32 [head_dim], each may be NULL): the per-head
 * RMS norm of dsb_head_rmsnorm_rope, with eps, before the rotation.
 * Arguments and errors as those calls. */
dsb_status dsb_rope_kv_write(float* qkv, int n_q_heads, const dsb_kv_cache* kv, const int32_t* batch_index,
                             int n_seq, int tokens_per_seq, const int32_t* pos, const dsb_rope* rope,
                             const float* q_norm, const float* k_norm, float eps, dsb_workspace* ws,
                             void* stream);

/* Decode attention for callers that cannot allocate device memory: code
 * running inside an allocator hook or memory-pool callback, processes whose
 * device allocator belongs to another framework that forbids outside
 * allocations, or latency-critical loops that must not take allocator locks.
 * The pages describe no such entry point; it is an addition of this library.
 * Same arguments, result and error behaviour as dsb_attention_decode_multi, but
 * no workspace: the split-K partials and the sequence table live in one static
 * 16 MiB device array that every device holds while the library is loaded.
 *   - The first call on a device looks up that array's address (with the
 *     device current) and may load the library's kernels onto the device,
 *     which the driver backs with device memory (lazy module loading): make
 *     that first call outside the no-allocation context (e.g. at start-up)
 *     and before any stream capture.  Later calls allocate nothing.
 *   - The address is kept for the life of the process: resetting the device
 *     (cudaDeviceReset) after the first call on it is not supported.
 *   - Limits: n_seq <= 256, and n_tok * n_q_heads * ceil(ctx/128) *
 *     (head_dim + 2) * 4 bytes of partials must fit in 16 MiB - 4 KiB;
 *     larger calls return DSB_ERR_UNSUPPORTED with a message.
 *   - All calls share the array: calls that overlap on the GPU (other streams,
 *     other threads) race; serialise them.  Nothing in it needs zeroing.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine, and uses no
 *     heap memory per call: the sequence table is built on the stack. */
dsb_status dsb_attention_decode_multi_noalloc(const float* q, int n_q_heads, const dsb_kv_cache* kv,
                                              const int32_t* batch_index, int n_seq, int tokens_per_seq,
                                              const int32_t* seq_lens, float* out, void* stream);

/* ---- measurement probe -------------------------------------------------------
 * The issue rate and latency of the four-way int8 dot product (__dp4a) the
 * narrow q8_0 matmul is built on, so that its arithmetic ceiling comes from a
 * measurement of committed code.  Not part of the decode step.
 *   mode 0: `blocks` CTAs of 256 threads, each thread 8 independent chains of
 *           `iters` dp4a (8 * iters * 256 * blocks in total); time the call
 *           with events on `stream`.
 *   mode 1: one thread runs one dependent chain of `iters` dp4a; out[1] = SM
 *           clock cycles it took, out[2] = iters.
 * out: device uint32[3].  DSB_ERR_INVALID_ARG for another mode or sizes out of
 * range; DSB_ERR_CUDA if the launch fails. */
dsb_status dsb_probe_dp4a(int mode, int blocks, int iters, uint32_t* out, void* stream);

/* The issue rate of the warp-level tensor-core products a narrow q8_0 matmul
 * can use in place of dp4a.  `blocks` CTAs of 256 threads; every warp runs 8
 * independent accumulator tiles for `iters` iterations, i.e. 64 * iters *
 * blocks products in total:
 *   mode 2: mma.sync m16n8k16, f16 x f16 -> f32 (4096 flops each);
 *   mode 3: mma.sync m16n8k32, s8 x s8 -> s32 (8192 ops each).
 * Time the call with events on `stream`.  out: device uint32[1] (written only
 * to keep the results live).  DSB_ERR_INVALID_ARG for another mode or sizes
 * out of range; DSB_ERR_CUDA if the launch fails. */
dsb_status dsb_probe_mma(int mode, int blocks, int iters, uint32_t* out, void* stream);

/* ---- the whole decode step -------------------------------------------------
 * A llama-style pre-norm decoder driven through the kernels above, one pass
 * for all live sessions ([DS4] "What" and "Design note": dense stages batched
 * with n_tokens = n_seqs, KV append and attention per sequence; [QAIC]
 * "Objective": cache slots addressed by batch_index).  Per layer:
 *   x = q8(rmsnorm(h)); [q|k|v] = Wqkv x; rope(q, k, pos); KV write;
 *   a = attention; h += Wo q8(a); x = q8(rmsnorm(h)); [g|u] = Wgu x;
 *   h += Wdown q8(silu(g) u)
 * then logits = Whead q8(rmsnorm(h)).  Token row t = s*T + j of sequence s
 * sits at position seq_lens[s] - T + j.  Embedding, head and every matrix are
 * q8_0; norms are float32 weights; the step's float32 activations live in the
 * workspace.  A layer with q_norm / k_norm weights applies the per-head RMS
 * norm of dsb_head_rmsnorm_rope (eps = rms_eps) to q / k before the rope. */
typedef struct {
  int32_t hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab, n_layers;
  float rms_eps; /* e.g. 1e-6 */
  dsb_rope rope; /* theta e.g. 10000; plain RoPE or YaRN */
} dsb_model_shape;

typedef struct {
  dsb_q8_0_mat wqkv;      /* rows (Hq + 2 Hkv) * D (q rows, then k, then v), cols hidden */
  dsb_q8_0_mat wo;        /* rows hidden, cols Hq * D */
  dsb_q8_0_mat wgu;       /* rows 2 * ffn (gate rows, then up rows), cols hidden */
  dsb_q8_0_mat wdown;     /* rows hidden, cols ffn */
  const float* attn_norm; /* device [hidden] */
  const float* ffn_norm;  /* device [hidden] */
  dsb_kv_cache kv;        /* this layer's retained cache */
  const float* q_norm;    /* device [head_dim] per-head q RMS-norm weight, or NULL (no norm) */
  const float* k_norm;    /* device [head_dim] per-head k RMS-norm weight, or NULL (no norm) */
} dsb_layer;

typedef struct {
  dsb_model_shape shape;
  const void* embed;        /* device q8_0 [vocab][hidden] */
  const dsb_layer* layers;  /* HOST array [n_layers], read during the call */
  const float* final_norm;  /* device [hidden] */
  dsb_q8_0_mat head;        /* rows vocab, cols hidden */
} dsb_model;

/* Device bytes a workspace needs for decode steps of up to max_tokens token
 * rows against caches of length ctx (activations + attention partials +
 * staged metadata).  0 if an argument is out of range. */
size_t dsb_step_workspace_bytes(const dsb_model_shape* shape, int max_tokens, int ctx);

/* One batched decode step.  token_ids: host int32[n_seq*T] in [0, vocab);
 * batch_index: host int32[n_seq], distinct; seq_lens: host int32[n_seq] in
 * [T, ctx] (KV length after this step).  Writes the step's K/V rows into each
 * layer's cache and logits (device float32 [n_seq*T][vocab]).  Shapes must
 * satisfy hidden, Hq*D and ffn % 256 == 0, head_dim in {64, 128}. */
dsb_status dsb_decode_step(const dsb_model* model, const int32_t* token_ids, const int32_t* batch_index, int n_seq,
                           int tokens_per_seq, const int32_t* seq_lens, float* logits, dsb_workspace* ws,
                           void* stream);

/* Stage trace of the step, for parity checking.  dsb_decode_step_trace runs
 * the kernels of dsb_decode_step, in the same order and with the same launch
 * plans, and after each stage copies that stage's result (on the same stream)
 * into the caller's device buffers below; a NULL pointer skips that copy.  The
 * copies change no value the step computes, so a test can hold every stage of
 * every layer to its own operation's tolerance, fed the GPU's own inputs to
 * that stage ([DS4] "Correctness": the batched step must agree with its
 * parts).  Sizes with n_tok = n_seq*T; q8_0 rows are cols/32 blocks of 34 B. */
typedef struct {
  void* x_attn;    /* q8_0 [n_tok][hidden/32]: q8(rmsnorm(h_in, attn_norm)) */
  float* qkv;      /* [n_tok][(Hq + 2 Hkv) D]: Wqkv x_attn, before the rope */
  float* qkv_rope; /* the same after the rope + KV write kernel: q heads rotated (and normed) */
  void* att_q8;    /* q8_0 [n_tok][Hq D/32]: q8(attention) */
  float* h_attn;   /* [n_tok][hidden]: h_in + Wo att_q8 */
  void* x_ffn;     /* q8_0 [n_tok][hidden/32]: q8(rmsnorm(h_attn, ffn_norm)) */
  float* gu;       /* [n_tok][2 ffn]: Wgu x_ffn (gate columns, then up) */
  void* act_q8;    /* q8_0 [n_tok][ffn/32]: q8(silu(gate) * up) */
  float* h_out;    /* [n_tok][hidden]: h_attn + Wdown act_q8, the next layer's h_in */
} dsb_layer_trace;

typedef struct {
  float* h_embed;                /* [n_tok][hidden]: the embedded tokens */
  const dsb_layer_trace* layers; /* HOST array [n_layers], or NULL */
  void* x_final;                 /* q8_0 [n_tok][hidden/32]: q8(rmsnorm(h_out, final_norm)) */
} dsb_step_trace;

dsb_status dsb_decode_step_trace(const dsb_model* model, const int32_t* token_ids, const int32_t* batch_index,
                                 int n_seq, int tokens_per_seq, const int32_t* seq_lens, float* logits,
                                 dsb_workspace* ws, const dsb_step_trace* trace, void* stream);

/* The same step on paged and ring KV ([DS4] the multi-sequence decode
 * attention commit: per-sequence cache views with ring geometry; [PTO] the
 * paged attention it serves): layer l's K/V live in the page pool pages[l]
 * (HOST array [n_layers]; every pool of one n_pages, dtype, n_kv_heads =
 * shape.n_kv_heads and head_dim = shape.head_dim; the layers' contiguous kv
 * fields are ignored), addressed through one block geometry for all layers
 * as in dsb_attention_decode_paged: sequence s's key p sits in page
 * block_table[s][p / 128] (ring, window[s] > 0: block (p / 128) mod
 * n_blocks[s]), row p mod 128, and a window W shows draft token j only the
 * keys (pos_j - W, pos_j].  block_table: host int32[n_seq][max_blocks];
 * n_blocks, window: host int32[n_seq]; seq_lens as dsb_decode_step (the ring
 * must hold W + T - 1 keys, a linear table must cover seq_lens[s]).  Two
 * tokens of the step writing the same page row are rejected.  The workspace
 * must hold the partials of 128 x (the most chunks a sequence visits) keys
 * (dsb_step_workspace_bytes with ctx = 128 * (max_blocks + 1) always does).
 * Same kernels and results as dsb_decode_step on a cache holding the same
 * keys; DSB_ERR_UNSUPPORTED when the block tables do not fit the staging
 * slot. */
dsb_status dsb_decode_step_paged(const dsb_model* model, const dsb_kv_pages* pages, const int32_t* token_ids,
                                 int n_seq, int tokens_per_seq, const int32_t* seq_lens, const int32_t* block_table,
                                 int max_blocks, const int32_t* n_blocks, const int32_t* window, float* logits,
                                 dsb_workspace* ws, void* stream);

/* The same step captured once into a CUDA graph for a fixed (n_seq, T) and
 * replayed.  The step's metadata (token ids, slots, seq_lens and what follows
 * from them) reaches the graph's first kernel, which copies it to the
 * workspace for the others: in that kernel's parameters, rewritten on the host
 * for each replay with new metadata, when it fits 4096 int32 words (2*n_seq*T
 * + 3*n_seq + 1); otherwise from a mapped pinned host copy the graph owns.  So
 * a replay serves new token ids, slots and seq_lens without re-capture; the
 * attention kernel reads its work count on the device.  The model, logits and
 * workspace must stay valid for the graph's lifetime; one graph per workspace
 * at a time. */
typedef struct dsb_step_graph dsb_step_graph;
dsb_status dsb_step_graph_create(const dsb_model* model, int n_seq, int tokens_per_seq, float* logits,
                                 dsb_workspace* ws, void* stream, dsb_step_graph** out);
/* Validates and stages the metadata, then launches the graph.  When the
 * metadata changes: parameter form, the first kernel's parameters are
 * rewritten (no wait); mapped form, the host waits (bounded) until the previous
 * replay has read the pinned copy before rewriting it. */
dsb_status dsb_step_graph_launch(dsb_step_graph* g, const int32_t* token_ids, const int32_t* batch_index,
                                 const int32_t* seq_lens, void* stream);
/* The paged step (dsb_decode_step_paged) captured the same way, for a fixed
 * (n_seq, T) and block-table width max_blocks: the pools' device memory is
 * bound at capture (pages: host array [n_layers], read during the call only;
 * the pools must outlive the graph), while every replay takes new token ids,
 * seq_lens, block tables, block counts and windows in its metadata (mapped
 * form once the block tables pass 4096 words).  The attention is captured for
 * max_blocks + 1 chunks per sequence, the most any geometry of that width
 * visits, and reads the actual count on the device; the workspace must hold
 * dsb_step_workspace_bytes(shape, n_seq*T, 128 * (max_blocks + 1)).
 * DSB_ERR_UNSUPPORTED when 2*n_seq*T + 3*n_seq + 1 + n_seq*(max_blocks + 2)
 * words exceed the staging slot. */
dsb_status dsb_step_graph_create_paged(const dsb_model* model, const dsb_kv_pages* pages, int max_blocks, int n_seq,
                                       int tokens_per_seq, float* logits, dsb_workspace* ws, void* stream,
                                       dsb_step_graph** out);
/* Validates the step's geometry as dsb_decode_step_paged does (against the
 * pools bound at capture) and launches the graph; the metadata handling is
 * that of dsb_step_graph_launch.  Each launch function rejects a graph of the
 * other kind with DSB_ERR_INVALID_ARG. */
dsb_status dsb_step_graph_launch_paged(dsb_step_graph* g, const int32_t* token_ids, const int32_t* seq_lens,
                                       const int32_t* block_table, const int32_t* n_blocks, const int32_t* window,
                                       void* stream);
dsb_status dsb_step_graph_destroy(dsb_step_graph* g);

/* ---- live-batch former (host only) -----------------------------------------
 * Hands out the retained cache's slots to sessions and builds each step's
 * metadata ([QAIC] "Objective": cache sized for full_batch_size, addressed by
 * batch_index; [PTO] commit message: the live batch is the seq_lens
 * descriptor; [DS4] "What": sessions join and leave between steps).  A session
 * is named by its slot.  Not thread-safe; pure host code, no CUDA calls. */
typedef struct dsb_batch_former dsb_batch_former;
/* All arguments in range (full_batch_size <= DSB_MAX_SEQS, T <= ctx, F*T <=
 * DSB_MAX_TOKENS) or DSB_ERR_INVALID_ARG. */
dsb_status dsb_batch_former_create(int full_batch_size, int ctx, int tokens_per_seq, dsb_batch_former** out);
void dsb_batch_former_destroy(dsb_batch_former* b);
/* Gives a free slot (the lowest) to a session whose first prefill_length KV
 * rows are already in the cache; DSB_ERR_UNSUPPORTED if every slot is live. */
dsb_status dsb_batch_join(dsb_batch_former* b, int prefill_length, int32_t* slot_out);
/* Frees the slot (its KV rows become garbage); DSB_ERR_INVALID_ARG if not live. */
dsb_status dsb_batch_leave(dsb_batch_former* b, int slot);
/* Queues the session's next T token ids (host int32[T], copied);
 * DSB_ERR_UNSUPPORTED if its KV length + T would exceed ctx. */
dsb_status dsb_batch_submit(dsb_batch_former* b, int slot, const int32_t* token_ids);
/* Lists the live sessions with queued tokens in slot order: batch_index[n],
 * seq_lens[n] (length after the step) and token_ids[n*T]; host arrays of
 * capacity full_batch_size (and full_batch_size*T).  Does not change state. */
dsb_status dsb_batch_form(const dsb_batch_former* b, int32_t* batch_index, int32_t* seq_lens, int32_t* token_ids,
                          int32_t* n_seq_out);
/* After the step ran: advances the listed sessions' KV lengths by T and
 * clears their queued tokens.  Checks every slot before changing anything. */
dsb_status dsb_batch_commit(dsb_batch_former* b, const int32_t* batch_index, int n_seq);
/* KV length of a live slot, or -1. */
int dsb_batch_length(const dsb_batch_former* b, int slot);

#ifdef __cplusplus
}
#endif
#endif /* DSB_H */
