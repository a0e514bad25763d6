// C ABI of libdsb.so (declared in include/dsb.h): argument validation,
// workspace management and kernel launches.  Every entry point checks all of
// its arguments on the host before it makes any CUDA call, so a rejected call
// leaves device memory untouched; host metadata (batch_index, pos, seq_lens)
// is validated, copied into a pinned staging slot of the workspace and sent to
// the device on the caller's stream.
#include "dsb.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "dsb_kernels.h"

namespace {

thread_local std::string g_last_error;

dsb_status fail(dsb_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

dsb_status cuda_fail(cudaError_t e, const char* where) {
  return fail(DSB_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorString(e), cudaGetErrorName(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kSlots = 16;
constexpr size_t kMetaHeader = 16;
constexpr size_t kMetaWords = kMetaHeader + 3 * (size_t)DSB_MAX_SEQS + 1 + (size_t)DSB_MAX_TOKENS;
constexpr size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
constexpr size_t kMetaSlotBytes = round_up(kMetaWords * sizeof(int32_t), 256);
constexpr size_t kMetaBytes = kSlots * kMetaSlotBytes;
constexpr double kHostWaitSeconds = 30.0;

struct DeviceInfo {
  int sms = 0;
  int max_smem_optin = 0;
};

dsb_status device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  static DeviceInfo cache[64];
  if (dev >= 0 && dev < 64 && cache[dev].sms > 0) {
    *out = cache[dev];
    return DSB_OK;
  }
  DeviceInfo d;
  e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
  e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(shared memory)");
  if (dev >= 0 && dev < 64) cache[dev] = d;
  *out = d;
  return DSB_OK;
}

}  // namespace

struct dsb_workspace {
  int device = -1;
  char* dev = nullptr;
  size_t dev_bytes = 0;
  char* host = nullptr;  // pinned, kSlots * kMetaSlotBytes
  cudaEvent_t ev[kSlots] = {};
  bool pending[kSlots] = {};
  int next = 0;
};

namespace {

// Copy `n` int32 words of metadata into the next staging slot and enqueue
// the host -> device copy.  Returns the device address of the slot.
dsb_status stage(dsb_workspace* ws, const std::vector<int32_t>& words, cudaStream_t st, const int32_t** dev_out) {
  if (words.size() > kMetaWords) return fail(DSB_ERR_INVALID_ARG, "metadata exceeds the staging slot");
  const int slot = ws->next;
  ws->next = (slot + 1) % kSlots;
  if (ws->pending[slot]) {
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
      cudaError_t q = cudaEventQuery(ws->ev[slot]);
      if (q == cudaSuccess) break;
      if (q != cudaErrorNotReady) return cuda_fail(q, "cudaEventQuery(staging slot)");
      if (std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count() > kHostWaitSeconds)
        return fail(DSB_ERR_TIMEOUT, "staging slot still in use after %.0f s", kHostWaitSeconds);
      std::this_thread::yield();
    }
    ws->pending[slot] = false;
  }
  char* h = ws->host + (size_t)slot * kMetaSlotBytes;
  char* d = ws->dev + (size_t)slot * kMetaSlotBytes;
  std::memcpy(h, words.data(), words.size() * sizeof(int32_t));
  cudaError_t e = cudaMemcpyAsync(d, h, words.size() * sizeof(int32_t), cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(metadata)");
  e = cudaEventRecord(ws->ev[slot], st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(metadata)");
  ws->pending[slot] = true;
  *dev_out = reinterpret_cast<const int32_t*>(d);
  return DSB_OK;
}

char* partial_base(dsb_workspace* ws) { return ws->dev + kMetaBytes; }
size_t partial_capacity(const dsb_workspace* ws) { return ws->dev_bytes > kMetaBytes ? ws->dev_bytes - kMetaBytes : 0; }

dsb_status check_mat(const dsb_q8_0_mat* w) {
  if (!w) return fail(DSB_ERR_INVALID_ARG, "w is NULL");
  if (!w->blocks) return fail(DSB_ERR_INVALID_ARG, "w->blocks is NULL");
  if (!aligned16(w->blocks)) return fail(DSB_ERR_INVALID_ARG, "w->blocks is not 16-byte aligned");
  if (w->rows < 1 || w->rows > INT_MAX) return fail(DSB_ERR_INVALID_ARG, "w->rows=%lld out of [1, INT_MAX]", (long long)w->rows);
  if (w->cols < 32 || w->cols % 32) return fail(DSB_ERR_INVALID_ARG, "w->cols=%lld is not a positive multiple of 32", (long long)w->cols);
  if (w->cols % 256) return fail(DSB_ERR_UNSUPPORTED, "w->cols=%lld: the narrow kernel needs cols %% 256 == 0", (long long)w->cols);
  if (w->cols / 32 > INT_MAX / 64) return fail(DSB_ERR_INVALID_ARG, "w->cols too large");
  return DSB_OK;
}

dsb_status check_kv(const dsb_kv_cache* kv) {
  if (!kv) return fail(DSB_ERR_INVALID_ARG, "kv is NULL");
  if (!kv->k || !kv->v) return fail(DSB_ERR_INVALID_ARG, "kv->k / kv->v is NULL");
  if (!aligned16(kv->k) || !aligned16(kv->v)) return fail(DSB_ERR_INVALID_ARG, "kv->k / kv->v not 16-byte aligned");
  if (kv->dtype != DSB_F16 && kv->dtype != DSB_BF16) return fail(DSB_ERR_INVALID_ARG, "kv->dtype=%d", kv->dtype);
  if (kv->full_batch_size < 1) return fail(DSB_ERR_INVALID_ARG, "kv->full_batch_size=%d", kv->full_batch_size);
  if (kv->n_kv_heads < 1) return fail(DSB_ERR_INVALID_ARG, "kv->n_kv_heads=%d", kv->n_kv_heads);
  if (kv->ctx < 1) return fail(DSB_ERR_INVALID_ARG, "kv->ctx=%d", kv->ctx);
  if (kv->head_dim < 2 || kv->head_dim % 2 || kv->head_dim > 1024)
    return fail(DSB_ERR_INVALID_ARG, "kv->head_dim=%d must be even in [2, 1024]", kv->head_dim);
  return DSB_OK;
}

dsb_status check_batch(const dsb_kv_cache* kv, const int32_t* batch_index, int n_seq, int tps) {
  if (n_seq < 1 || n_seq > kv->full_batch_size || n_seq > DSB_MAX_SEQS)
    return fail(DSB_ERR_INVALID_ARG, "n_seq=%d out of [1, min(full_batch_size=%d, %d)]", n_seq, kv->full_batch_size,
                DSB_MAX_SEQS);
  if (tps < 1) return fail(DSB_ERR_INVALID_ARG, "tokens_per_seq=%d < 1", tps);
  if ((long long)n_seq * tps > DSB_MAX_TOKENS)
    return fail(DSB_ERR_INVALID_ARG, "n_seq*tokens_per_seq=%lld exceeds %d", (long long)n_seq * tps, DSB_MAX_TOKENS);
  if (!batch_index) return fail(DSB_ERR_INVALID_ARG, "batch_index is NULL");
  std::vector<char> seen((size_t)kv->full_batch_size, 0);
  for (int s = 0; s < n_seq; ++s) {
    const int b = batch_index[s];
    if (b < 0 || b >= kv->full_batch_size)
      return fail(DSB_ERR_INVALID_ARG, "batch_index[%d]=%d out of [0, %d)", s, b, kv->full_batch_size);
    if (seen[(size_t)b]) return fail(DSB_ERR_INVALID_ARG, "batch_index[%d]=%d is duplicated", s, b);
    seen[(size_t)b] = 1;
  }
  return DSB_OK;
}

}  // namespace

extern "C" {

const char* dsb_last_error(void) { return g_last_error.c_str(); }

const char* dsb_version(void) { return "dsb 0.1 (sm_103a)"; }

size_t dsb_workspace_bytes(int max_tokens, int n_q_heads, int head_dim, int ctx) {
  if (max_tokens < 0 || max_tokens > DSB_MAX_TOKENS || n_q_heads < 0 || head_dim < 0 || head_dim > 1024 || ctx < 0)
    return 0;
  return kMetaBytes + round_up(dsbk::attention_partial_bytes(max_tokens, n_q_heads, head_dim, ctx), 256);
}

dsb_status dsb_workspace_create(void* device_ptr, size_t device_bytes, dsb_workspace** out) {
  if (!out) return fail(DSB_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!device_ptr) return fail(DSB_ERR_INVALID_ARG, "device_ptr is NULL");
  if (reinterpret_cast<uintptr_t>(device_ptr) & 255u) return fail(DSB_ERR_INVALID_ARG, "device_ptr not 256-byte aligned");
  if (device_bytes < kMetaBytes)
    return fail(DSB_ERR_WORKSPACE, "device_bytes=%zu below the %zu-byte metadata area", device_bytes, kMetaBytes);
  dsb_workspace* ws = new (std::nothrow) dsb_workspace();
  if (!ws) return fail(DSB_ERR_INVALID_ARG, "out of host memory");
  cudaError_t e = cudaGetDevice(&ws->device);
  if (e == cudaSuccess) e = cudaHostAlloc(reinterpret_cast<void**>(&ws->host), kMetaBytes, cudaHostAllocDefault);
  int made = 0;
  for (; e == cudaSuccess && made < kSlots; ++made) e = cudaEventCreateWithFlags(&ws->ev[made], cudaEventDisableTiming);
  if (e != cudaSuccess) {
    for (int i = 0; i < made; ++i) cudaEventDestroy(ws->ev[i]);
    if (ws->host) cudaFreeHost(ws->host);
    delete ws;
    return cuda_fail(e, "dsb_workspace_create");
  }
  ws->dev = static_cast<char*>(device_ptr);
  ws->dev_bytes = device_bytes;
  *out = ws;
  return DSB_OK;
}

dsb_status dsb_workspace_destroy(dsb_workspace* ws) {
  if (!ws) return DSB_OK;
  dsb_status st = DSB_OK;
  for (int i = 0; i < kSlots; ++i) {
    if (ws->pending[i]) {
      const auto t0 = std::chrono::steady_clock::now();
      while (cudaEventQuery(ws->ev[i]) == cudaErrorNotReady) {
        if (std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count() > kHostWaitSeconds) {
          st = fail(DSB_ERR_TIMEOUT, "staged copy still pending at destroy");
          break;
        }
        std::this_thread::yield();
      }
    }
    cudaEventDestroy(ws->ev[i]);
  }
  if (ws->host) cudaFreeHost(ws->host);
  delete ws;
  return st;
}

dsb_status dsb_device_error(void) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  const unsigned int m = dsbk::read_clear_error_matmul();
  const unsigned int a = dsbk::read_clear_error_attention();
  if (m || a)
    return fail(DSB_ERR_DEVICE, "a kernel's bounded wait ran out (matmul=%u attention=%u)", m, a);
  return DSB_OK;
}

dsb_status dsb_quantize_q8_0(const float* x, int64_t n_rows, int64_t cols, void* xq, void* stream) {
  if (n_rows < 0) return fail(DSB_ERR_INVALID_ARG, "n_rows=%lld < 0", (long long)n_rows);
  if (cols < 32 || cols % 32) return fail(DSB_ERR_INVALID_ARG, "cols=%lld is not a positive multiple of 32", (long long)cols);
  if (n_rows == 0) return DSB_OK;
  if (!x || !xq) return fail(DSB_ERR_INVALID_ARG, "x / xq is NULL");
  if (!aligned16(x) || !aligned16(xq)) return fail(DSB_ERR_INVALID_ARG, "x / xq not 16-byte aligned");
  if (n_rows > (1LL << 40) / cols) return fail(DSB_ERR_INVALID_ARG, "n_rows*cols too large");
  cudaError_t e = dsbk::launch_quantize_q8_0(x, n_rows, cols, xq, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "quantize_q8_0 launch");
}

static dsb_status matmul_common(const dsb_q8_0_mat* w, const void* xq, int n_tok, float* y, int32_t* isum,
                                void* stream, bool narrow) {
  dsb_status st = check_mat(w);
  if (st != DSB_OK) return st;
  if (narrow && (n_tok < 1 || n_tok > DSB_NARROW_MAX))
    return fail(DSB_ERR_INVALID_ARG, "n_tok=%d out of [1, %d]", n_tok, DSB_NARROW_MAX);
  if (!narrow && (n_tok < 1 || n_tok > DSB_MAX_TOKENS))
    return fail(DSB_ERR_INVALID_ARG, "n_tok=%d out of [1, %d]", n_tok, DSB_MAX_TOKENS);
  if (!xq) return fail(DSB_ERR_INVALID_ARG, "xq is NULL");
  if (!aligned16(xq)) return fail(DSB_ERR_INVALID_ARG, "xq not 16-byte aligned");
  if (!y && !isum) return fail(DSB_ERR_INVALID_ARG, "output is NULL");
  if ((y && !aligned16(y)) || (isum && !aligned16(isum))) return fail(DSB_ERR_INVALID_ARG, "output not 16-byte aligned");
  DeviceInfo di;
  st = device_info(&di);
  if (st != DSB_OK) return st;
  const int nt_max = n_tok < DSB_NARROW_MAX ? n_tok : DSB_NARROW_MAX;
  const size_t smem = dsbk::matmul_smem_bytes(w->rows, w->cols, nt_max, di.sms);
  if (smem > (size_t)di.max_smem_optin)
    return fail(DSB_ERR_UNSUPPORTED, "matmul %lldx%lld needs %zu bytes of shared memory (max %d)", (long long)w->rows,
                (long long)w->cols, smem, di.max_smem_optin);
  const size_t blk_row = (size_t)(w->cols / 32) * 34;
  for (int t0 = 0; t0 < n_tok; t0 += DSB_NARROW_MAX) {
    const int nt = std::min(DSB_NARROW_MAX, n_tok - t0);
    cudaError_t e = dsbk::launch_matmul_q8_0_narrow(
        w->blocks, w->rows, w->cols, static_cast<const char*>(xq) + (size_t)t0 * blk_row, nt,
        y ? y + (size_t)t0 * w->rows : nullptr, isum ? isum + (size_t)t0 * w->rows * (w->cols / 32) : nullptr,
        di.sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "matmul_q8_0 launch");
  }
  return DSB_OK;
}

dsb_status dsb_matmul_q8_0_narrow(const dsb_q8_0_mat* w, const void* xq, int n_tok, float* y, void* stream) {
  if (!y) return fail(DSB_ERR_INVALID_ARG, "y is NULL");
  return matmul_common(w, xq, n_tok, y, nullptr, stream, true);
}

dsb_status dsb_matmul_q8_0(const dsb_q8_0_mat* w, const void* xq, int n_tok, float* y, void* stream) {
  if (!y) return fail(DSB_ERR_INVALID_ARG, "y is NULL");
  return matmul_common(w, xq, n_tok, y, nullptr, stream, false);
}

dsb_status dsb_matmul_q8_0_block_dots(const dsb_q8_0_mat* w, const void* xq, int n_tok, int32_t* isum, void* stream) {
  if (!isum) return fail(DSB_ERR_INVALID_ARG, "isum is NULL");
  return matmul_common(w, xq, n_tok, nullptr, isum, stream, true);
}

dsb_status dsb_rope_posvec(float* q, int n_q_heads, float* k, int n_kv_heads, int head_dim, int n_tok,
                           const int32_t* pos, float theta, dsb_workspace* ws, void* stream) {
  if (n_tok < 0 || n_tok > DSB_MAX_TOKENS) return fail(DSB_ERR_INVALID_ARG, "n_tok=%d out of [0, %d]", n_tok, DSB_MAX_TOKENS);
  if (head_dim < 2 || head_dim % 2 || head_dim > 1024)
    return fail(DSB_ERR_INVALID_ARG, "head_dim=%d must be even in [2, 1024]", head_dim);
  if (n_q_heads < 1) return fail(DSB_ERR_INVALID_ARG, "n_q_heads=%d < 1", n_q_heads);
  if (n_kv_heads < 0 || (n_kv_heads == 0) != (k == nullptr))
    return fail(DSB_ERR_INVALID_ARG, "k must be NULL exactly when n_kv_heads == 0");
  if (!(theta > 0.0f) || !std::isfinite(theta)) return fail(DSB_ERR_INVALID_ARG, "theta must be finite and > 0");
  if (!ws) return fail(DSB_ERR_WORKSPACE, "workspace is NULL");
  if (n_tok == 0) return DSB_OK;
  if (!q || !pos) return fail(DSB_ERR_INVALID_ARG, "q / pos is NULL");
  if (!aligned16(q) || (k && !aligned16(k))) return fail(DSB_ERR_INVALID_ARG, "q / k not 16-byte aligned");
  for (int t = 0; t < n_tok; ++t)
    if (pos[t] < 0 || pos[t] >= (1 << 24)) return fail(DSB_ERR_INVALID_ARG, "pos[%d]=%d out of [0, 2^24)", t, pos[t]);
  std::vector<int32_t> words(pos, pos + n_tok);
  const int32_t* dev = nullptr;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  dsb_status s = stage(ws, words, st, &dev);
  if (s != DSB_OK) return s;
  cudaError_t e = dsbk::launch_rope_posvec(q, n_q_heads, k, n_kv_heads, head_dim, n_tok, dev, theta, st);
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "rope_posvec launch");
}

dsb_status dsb_kv_scatter(const dsb_kv_cache* kv, const int32_t* batch_index, int n_seq, int tokens_per_seq,
                          const int32_t* pos, const float* k, const float* v, dsb_workspace* ws, void* stream) {
  dsb_status st = check_kv(kv);
  if (st != DSB_OK) return st;
  st = check_batch(kv, batch_index, n_seq, tokens_per_seq);
  if (st != DSB_OK) return st;
  if (!pos) return fail(DSB_ERR_INVALID_ARG, "pos is NULL");
  if (!k || !v) return fail(DSB_ERR_INVALID_ARG, "k / v is NULL");
  if (!aligned16(k) || !aligned16(v)) return fail(DSB_ERR_INVALID_ARG, "k / v not 16-byte aligned");
  if (!ws) return fail(DSB_ERR_WORKSPACE, "workspace is NULL");
  const int n_tok = n_seq * tokens_per_seq;
  for (int s = 0; s < n_seq; ++s) {
    for (int j = 0; j < tokens_per_seq; ++j) {
      const int p = pos[s * tokens_per_seq + j];
      if (p < 0 || p >= kv->ctx) return fail(DSB_ERR_INVALID_ARG, "pos[%d]=%d out of [0, ctx=%d)", s * tokens_per_seq + j, p, kv->ctx);
      for (int j2 = 0; j2 < j; ++j2)
        if (pos[s * tokens_per_seq + j2] == p)
          return fail(DSB_ERR_INVALID_ARG, "sequence %d writes position %d twice", s, p);
    }
  }
  std::vector<int32_t> words;
  words.reserve((size_t)n_seq + n_tok);
  words.insert(words.end(), batch_index, batch_index + n_seq);
  words.insert(words.end(), pos, pos + n_tok);
  const int32_t* dev = nullptr;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  st = stage(ws, words, cs, &dev);
  if (st != DSB_OK) return st;
  cudaError_t e = dsbk::launch_kv_scatter(kv->k, kv->v, kv->dtype, kv->n_kv_heads, kv->ctx, kv->head_dim, dev,
                                          tokens_per_seq, dev + n_seq, n_tok, k, v, cs);
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "kv_scatter launch");
}

dsb_status dsb_attention_decode_multi(const float* q, int n_q_heads, const dsb_kv_cache* kv,
                                      const int32_t* batch_index, int n_seq, int tokens_per_seq,
                                      const int32_t* seq_lens, float* out, dsb_workspace* ws, void* stream) {
  dsb_status st = check_kv(kv);
  if (st != DSB_OK) return st;
  if (n_q_heads < 1 || n_q_heads % kv->n_kv_heads)
    return fail(DSB_ERR_INVALID_ARG, "n_q_heads=%d is not a positive multiple of n_kv_heads=%d", n_q_heads,
                kv->n_kv_heads);
  st = check_batch(kv, batch_index, n_seq, tokens_per_seq);
  if (st != DSB_OK) return st;
  if (kv->head_dim != 64 && kv->head_dim != 128)
    return fail(DSB_ERR_UNSUPPORTED, "head_dim=%d: attention serves 64 and 128", kv->head_dim);
  const long long R = (long long)(n_q_heads / kv->n_kv_heads) * tokens_per_seq;
  if (R > 64) return fail(DSB_ERR_UNSUPPORTED, "query rows per kv head (G*T=%lld) exceed 64", R);
  if (!q || !out || !seq_lens) return fail(DSB_ERR_INVALID_ARG, "q / out / seq_lens is NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(DSB_ERR_INVALID_ARG, "q / out not 16-byte aligned");
  if (!ws) return fail(DSB_ERR_WORKSPACE, "workspace is NULL");
  for (int s = 0; s < n_seq; ++s)
    if (seq_lens[s] < tokens_per_seq || seq_lens[s] > kv->ctx)
      return fail(DSB_ERR_INVALID_ARG, "seq_lens[%d]=%d out of [T=%d, ctx=%d]", s, seq_lens[s], tokens_per_seq, kv->ctx);
  const int n_tok = n_seq * tokens_per_seq;
  const size_t need = dsbk::attention_partial_bytes(n_tok, n_q_heads, kv->head_dim, kv->ctx);
  if (need > partial_capacity(ws))
    return fail(DSB_ERR_WORKSPACE, "attention needs %zu workspace bytes for partials, have %zu", need,
                partial_capacity(ws));
  std::vector<int32_t> words;
  words.reserve(3 * (size_t)n_seq + 1);
  words.insert(words.end(), batch_index, batch_index + n_seq);
  words.insert(words.end(), seq_lens, seq_lens + n_seq);
  long long total = 0;
  words.push_back(0);
  for (int s = 0; s < n_seq; ++s) {
    total += (seq_lens[s] + DSB_ATTN_CHUNK - 1) / DSB_ATTN_CHUNK;
    words.push_back((int32_t)total);
  }
  if (total > INT_MAX) return fail(DSB_ERR_INVALID_ARG, "too many attention chunks");
  const int32_t* dev = nullptr;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  st = stage(ws, words, cs, &dev);
  if (st != DSB_OK) return st;
  dsbk::MetaView mv{dev, dev + n_seq, dev + 2 * n_seq, nullptr};
  const int max_chunks = (kv->ctx + DSB_ATTN_CHUNK - 1) / DSB_ATTN_CHUNK;
  cudaError_t e = dsbk::launch_attention_decode_multi(
      q, n_q_heads, kv->k, kv->v, kv->dtype, kv->n_kv_heads, kv->ctx, kv->head_dim, mv, n_seq, tokens_per_seq,
      (int)total, max_chunks, reinterpret_cast<float*>(partial_base(ws)), out, cs);
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "attention_decode_multi launch");
}

}  // extern "C"
