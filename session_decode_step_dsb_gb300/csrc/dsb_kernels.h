// Internal interface between the C ABI (dsb.cpp) and the CUDA translation
// units.  Host-side launch functions only; no device code here.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace dsbk {

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

int matmul_split(int64_t rows, int64_t cols, int num_sms);
size_t matmul_smem_bytes(int64_t rows, int64_t cols, int n_tok, int num_sms);
cudaError_t launch_matmul_q8_0_narrow(const void* W, int64_t rows, int64_t cols, const void* xq, int n_tok, float* y,
                                      int32_t* isum, int num_sms, cudaStream_t st);

cudaError_t launch_quantize_q8_0(const float* x, int64_t n_rows, int64_t cols, void* xq, cudaStream_t st);

cudaError_t launch_rope_posvec(float* q, int n_q_heads, float* k, int n_kv_heads, int head_dim, int n_tok,
                               const int32_t* pos_dev, float theta, cudaStream_t st);

cudaError_t launch_kv_scatter(void* kc, void* vc, int dtype, int n_kv_heads, int ctx, int head_dim,
                              const int32_t* batch_index_dev, int tokens_per_seq, const int32_t* pos_dev, int n_tok,
                              const float* k, const float* v, cudaStream_t st);

// Split-K decode attention: partial kernel over (sequence, chunk) x kv head,
// then the chunk-order merge.  partials: float [n_tok][n_q_heads][max_chunks][head_dim + 2].
cudaError_t launch_attention_decode_multi(const float* q, int n_q_heads, const void* kc, const void* vc, int dtype,
                                          int n_kv_heads, int ctx, int head_dim, MetaView meta, int n_seq,
                                          int tokens_per_seq, int total_chunks, int max_chunks, float* partials,
                                          float* out, cudaStream_t st);

size_t attention_partial_bytes(int n_tok, int n_q_heads, int head_dim, int ctx);

unsigned int read_clear_error_matmul();
unsigned int read_clear_error_attention();

}  // namespace dsbk
