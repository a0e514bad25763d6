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
#include <mutex>
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
  static std::mutex mu;
  static DeviceInfo cache[64];
  if (dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].sms > 0) {
      *out = cache[dev];
      return DSB_OK;
    }
  }
  DeviceInfo d;
  e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
  e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(shared memory)");
  if (dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lock(mu);
    cache[dev] = d;
  }
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
  // the attention addresses cache rows (slot, kv head, position) by a 32-bit
  // tensor coordinate
  if ((long long)kv->full_batch_size * kv->n_kv_heads * kv->ctx > (long long)INT_MAX - 128)
    return fail(DSB_ERR_UNSUPPORTED, "cache of %lld rows (full_batch_size*n_kv_heads*ctx) exceeds 2^31 - 129",
                (long long)kv->full_batch_size * kv->n_kv_heads * kv->ctx);
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

dsb_status check_rope(const dsb_rope* r) {
  if (!r) return fail(DSB_ERR_INVALID_ARG, "rope is NULL");
  if (!(r->theta > 0.0f) || !std::isfinite(r->theta)) return fail(DSB_ERR_INVALID_ARG, "theta must be finite and > 0");
  if (std::isnan(r->yarn_factor) || std::isinf(r->yarn_factor))
    return fail(DSB_ERR_INVALID_ARG, "yarn_factor must be finite");
  if (r->yarn_factor > 1.0f) {
    if (r->yarn_orig_ctx < 1) return fail(DSB_ERR_INVALID_ARG, "yarn_orig_ctx=%d < 1", r->yarn_orig_ctx);
    if (!(r->yarn_beta_slow > 0.0f) || !(r->yarn_beta_fast > r->yarn_beta_slow) || !std::isfinite(r->yarn_beta_fast))
      return fail(DSB_ERR_INVALID_ARG, "yarn betas must satisfy 0 < beta_slow < beta_fast, finite");
  }
  return DSB_OK;
}

void fill_rope_freqs(const dsb_rope& r, int head_dim, dsbk::RopeFreqs* out) {
  if (r.yarn_factor > 1.0f)
    dsbk::rope_freqs((double)r.theta, head_dim, out, (double)r.yarn_factor, r.yarn_orig_ctx, (double)r.yarn_beta_fast,
                     (double)r.yarn_beta_slow);
  else
    dsbk::rope_freqs((double)r.theta, head_dim, out);
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
  const unsigned int mt = dsbk::read_clear_error_matmul_tc() | dsbk::read_clear_error_matmul_fused() |
                           dsbk::read_clear_error_matmul_staged();
  const unsigned int a = dsbk::read_clear_error_attention();
  if (m || mt || a)
    return fail(DSB_ERR_DEVICE, "a kernel's bounded wait ran out (matmul=%u matmul_tc=%u attention=%u)", m, mt, a);
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
        y ? y + (size_t)t0 * w->rows : nullptr, nullptr,
        isum ? isum + (size_t)t0 * w->rows * (w->cols / 32) : nullptr,
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

size_t dsb_matmul_q8_0_staged_bytes(int n_tok, int64_t cols) {
  if (n_tok < 1 || n_tok > DSB_NARROW_MAX || cols < 256 || cols % 256) return 0;
  return dsbk::matmul_staged_bytes(n_tok, cols);
}

static dsb_status staged_common(const dsb_q8_0_mat* w, int n_tok, const void* staged, size_t staged_bytes,
                                DeviceInfo* di) {
  dsb_status st = check_mat(w);
  if (st != DSB_OK) return st;
  if (n_tok < 1 || n_tok > DSB_NARROW_MAX)
    return fail(DSB_ERR_INVALID_ARG, "n_tok=%d out of [1, %d]", n_tok, DSB_NARROW_MAX);
  const size_t need = dsbk::matmul_staged_bytes(n_tok, w->cols);
  if (!staged || !aligned16(staged)) return fail(DSB_ERR_WORKSPACE, "staged is NULL or not 16-byte aligned");
  if (staged_bytes < need) return fail(DSB_ERR_WORKSPACE, "staged has %zu bytes, needs %zu", staged_bytes, need);
  st = device_info(di);
  if (st != DSB_OK) return st;
  const size_t smem = dsbk::matmul_smem_bytes(w->rows, w->cols, n_tok, di->sms);
  if (smem > (size_t)di->max_smem_optin)
    return fail(DSB_ERR_UNSUPPORTED, "matmul %lldx%lld needs %zu bytes of shared memory (max %d)", (long long)w->rows,
                (long long)w->cols, smem, di->max_smem_optin);
  return DSB_OK;
}

dsb_status dsb_stage_q8_0(const dsb_q8_0_mat* w, const void* xq, int n_tok, void* staged, size_t staged_bytes,
                          void* stream) {
  if (!xq || !aligned16(xq)) return fail(DSB_ERR_INVALID_ARG, "xq is NULL or not 16-byte aligned");
  DeviceInfo di;
  dsb_status st = staged_common(w, n_tok, staged, staged_bytes, &di);
  if (st != DSB_OK) return st;
  cudaError_t e = dsbk::launch_stage_q8_0(xq, n_tok, w->cols, staged, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "stage_q8_0 launch");
}

dsb_status dsb_matmul_q8_0_staged(const dsb_q8_0_mat* w, const void* staged, size_t staged_bytes, int n_tok, float* y,
                                  void* stream) {
  if (!y || !aligned16(y)) return fail(DSB_ERR_INVALID_ARG, "y is NULL or not 16-byte aligned");
  DeviceInfo di;
  dsb_status st = staged_common(w, n_tok, staged, staged_bytes, &di);
  if (st != DSB_OK) return st;
  cudaError_t e = dsbk::launch_matmul_q8_0_staged(w->blocks, w->rows, w->cols, staged, n_tok, y, nullptr, di.sms,
                                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "matmul_q8_0_staged launch");
}

size_t dsb_matmul_q8_0_wide_scratch_bytes(int n_tok, int64_t cols) {
  if (n_tok < 1 || n_tok > DSB_MAX_TOKENS || cols < 256 || cols % 256) return 0;
  return dsbk::matmul_tc_scratch_bytes(n_tok, cols);
}

dsb_status dsb_matmul_q8_0_wide(const dsb_q8_0_mat* w, const void* xq, int n_tok, float* y, void* scratch,
                                size_t scratch_bytes, void* stream) {
  dsb_status st = check_mat(w);
  if (st != DSB_OK) return st;
  if (n_tok < 1 || n_tok > DSB_MAX_TOKENS)
    return fail(DSB_ERR_INVALID_ARG, "n_tok=%d out of [1, %d]", n_tok, DSB_MAX_TOKENS);
  if (w->rows > (1LL << 31) - 128) return fail(DSB_ERR_UNSUPPORTED, "rows=%lld too large", (long long)w->rows);
  if (!xq || !aligned16(xq)) return fail(DSB_ERR_INVALID_ARG, "xq is NULL or not 16-byte aligned");
  if (!y || !aligned16(y)) return fail(DSB_ERR_INVALID_ARG, "y is NULL or not 16-byte aligned");
  const size_t need = dsbk::matmul_tc_scratch_bytes(n_tok, w->cols);
  if (!scratch || !aligned16(scratch)) return fail(DSB_ERR_WORKSPACE, "scratch is NULL or not 16-byte aligned");
  if (scratch_bytes < need) return fail(DSB_ERR_WORKSPACE, "scratch has %zu bytes, needs %zu", scratch_bytes, need);
  DeviceInfo di;
  st = device_info(&di);
  if (st != DSB_OK) return st;
  if (dsbk::matmul_tc_smem_bytes() > (size_t)di.max_smem_optin)
    return fail(DSB_ERR_UNSUPPORTED, "the tensor-core matmul needs %zu bytes of shared memory (max %d)",
                dsbk::matmul_tc_smem_bytes(), di.max_smem_optin);
  cudaError_t e = dsbk::launch_matmul_q8_0_tc(w->blocks, w->rows, w->cols, xq, n_tok, y, nullptr, scratch,
                                              static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "matmul_q8_0_wide launch");
}

dsb_status dsb_head_rmsnorm_rope(float* q, int n_q_heads, float* k, int n_kv_heads, int head_dim, int n_tok,
                                 const int32_t* pos, const dsb_rope* rope, const float* q_norm, const float* k_norm,
                                 float eps,
                                 dsb_workspace* ws, void* stream) {
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return fail(DSB_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (k_norm && !k) return fail(DSB_ERR_INVALID_ARG, "k_norm given without k");
  if (n_tok < 0 || n_tok > DSB_MAX_TOKENS) return fail(DSB_ERR_INVALID_ARG, "n_tok=%d out of [0, %d]", n_tok, DSB_MAX_TOKENS);
  if (head_dim < 2 || head_dim % 2 || head_dim > 1024)
    return fail(DSB_ERR_INVALID_ARG, "head_dim=%d must be even in [2, 1024]", head_dim);
  if (n_q_heads < 1) return fail(DSB_ERR_INVALID_ARG, "n_q_heads=%d < 1", n_q_heads);
  if (n_kv_heads < 0 || (n_kv_heads == 0) != (k == nullptr))
    return fail(DSB_ERR_INVALID_ARG, "k must be NULL exactly when n_kv_heads == 0");
  if (check_rope(rope) != DSB_OK) return DSB_ERR_INVALID_ARG;
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
  static thread_local dsbk::RopeFreqs freqs;
  fill_rope_freqs(*rope, head_dim, &freqs);
  cudaError_t e = dsbk::launch_rope_posvec(q, (long long)n_q_heads * head_dim, n_q_heads, k,
                                           (long long)n_kv_heads * head_dim, n_kv_heads, head_dim, n_tok, dev, freqs, st,
                                           q_norm, k_norm, eps);
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "rope_posvec launch");
}

dsb_status dsb_rope_posvec(float* q, int n_q_heads, float* k, int n_kv_heads, int head_dim, int n_tok,
                           const int32_t* pos, float theta, dsb_workspace* ws, void* stream) {
  const dsb_rope rope{theta, 0.0f, 0, 0.0f, 0.0f};
  return dsb_head_rmsnorm_rope(q, n_q_heads, k, n_kv_heads, head_dim, n_tok, pos, &rope, nullptr, nullptr, 0.0f, ws,
                               stream);
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
                                          tokens_per_seq, dev + n_seq, n_tok, k, v,
                                          (long long)kv->n_kv_heads * kv->head_dim, cs);
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "kv_scatter launch");
}

static dsb_status attention_common(const float* q, int n_q_heads, const dsb_kv_cache* kv,
                                   const int32_t* batch_index, int n_seq, int tokens_per_seq,
                                   const int32_t* seq_lens, float* out, void* xq, dsb_workspace* ws, void* stream) {
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
  if (!q || !(out || xq) || !seq_lens) return fail(DSB_ERR_INVALID_ARG, "q / out / seq_lens is NULL");
  if (!aligned16(q) || (out && !aligned16(out)) || (xq && !aligned16(xq)))
    return fail(DSB_ERR_INVALID_ARG, "q / out not 16-byte aligned");
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
      q, (long long)n_q_heads * kv->head_dim, n_q_heads, kv->k, kv->v, kv->dtype, kv->n_kv_heads, kv->ctx, kv->head_dim,
      (long long)kv->full_batch_size * kv->n_kv_heads * kv->ctx, mv, n_seq, tokens_per_seq,
      total * kv->n_kv_heads, max_chunks, reinterpret_cast<float*>(partial_base(ws)), out, xq, cs);
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "attention_decode_multi launch");
}

// ---- paged / ring KV geometry ----------------------------------------------

static dsb_status check_pages(const dsb_kv_pages* kv) {
  if (!kv) return fail(DSB_ERR_INVALID_ARG, "kv is NULL");
  if (!kv->k || !kv->v) return fail(DSB_ERR_INVALID_ARG, "kv->k / kv->v is NULL");
  if (!aligned16(kv->k) || !aligned16(kv->v)) return fail(DSB_ERR_INVALID_ARG, "page pools not 16-byte aligned");
  if (kv->dtype != DSB_F16 && kv->dtype != DSB_BF16) return fail(DSB_ERR_INVALID_ARG, "dtype must be DSB_F16 or DSB_BF16");
  if (kv->n_pages < 1 || kv->n_kv_heads < 1) return fail(DSB_ERR_INVALID_ARG, "n_pages / n_kv_heads < 1");
  if (kv->head_dim < 8 || kv->head_dim % 8 || kv->head_dim > 1024)
    return fail(DSB_ERR_INVALID_ARG, "head_dim=%d must be a multiple of 8 in [8, 1024]", kv->head_dim);
  if ((long long)kv->n_pages * kv->n_kv_heads * DSB_KV_PAGE > (long long)INT_MAX - 128)
    return fail(DSB_ERR_UNSUPPORTED, "page pools of %lld rows (n_pages*n_kv_heads*%d) exceed 2^31 - 129",
                (long long)kv->n_pages * kv->n_kv_heads * DSB_KV_PAGE, DSB_KV_PAGE);
  return DSB_OK;
}

// Block tables, block counts, windows and lengths of one call; lens: the KV
// lengths after the step (NULL when only positions are known).
static dsb_status check_paged_geometry(const dsb_kv_pages* kv, const int32_t* block_table, int max_blocks,
                                       const int32_t* n_blocks, const int32_t* window, int n_seq, int tps,
                                       const int32_t* lens) {
  if (n_seq < 1 || n_seq > DSB_MAX_SEQS) return fail(DSB_ERR_INVALID_ARG, "n_seq=%d out of [1, %d]", n_seq, DSB_MAX_SEQS);
  if (tps < 1 || (long long)n_seq * tps > DSB_MAX_TOKENS)
    return fail(DSB_ERR_INVALID_ARG, "tokens_per_seq=%d out of range", tps);
  if (max_blocks < 1) return fail(DSB_ERR_INVALID_ARG, "max_blocks=%d < 1", max_blocks);
  if (!block_table || !n_blocks || !window) return fail(DSB_ERR_INVALID_ARG, "block_table / n_blocks / window is NULL");
  for (int s = 0; s < n_seq; ++s) {
    const int nb = n_blocks[s], w = window[s];
    if (nb < 1 || nb > max_blocks) return fail(DSB_ERR_INVALID_ARG, "n_blocks[%d]=%d out of [1, %d]", s, nb, max_blocks);
    if (w < 0) return fail(DSB_ERR_INVALID_ARG, "window[%d]=%d < 0", s, w);
    for (int i = 0; i < nb; ++i) {
      const int page = block_table[(size_t)s * max_blocks + i];
      if (page < 0 || page >= kv->n_pages)
        return fail(DSB_ERR_INVALID_ARG, "block_table[%d][%d]=%d out of [0, %d)", s, i, page, kv->n_pages);
    }
    if (w > 0 && (long long)nb * DSB_KV_PAGE < (long long)w + tps - 1)
      return fail(DSB_ERR_INVALID_ARG, "sequence %d: a ring of %d pages cannot hold window %d + T - 1", s, nb, w);
    if (lens) {
      if (lens[s] < tps) return fail(DSB_ERR_INVALID_ARG, "seq_lens[%d]=%d < T=%d", s, lens[s], tps);
      if (w == 0 && ((long long)lens[s] + DSB_KV_PAGE - 1) / DSB_KV_PAGE > nb)
        return fail(DSB_ERR_INVALID_ARG, "sequence %d: %d blocks do not cover %d keys", s, nb, lens[s]);
    }
  }
  return DSB_OK;
}

// Chunks of sequence s the attention visits: from the first one a window
// leaves visible to the last.
static int paged_first_chunk(int len, int tps, int w) {
  return w > 0 ? std::max(0, len - tps + 1 - w) / DSB_ATTN_CHUNK : 0;
}

dsb_status dsb_kv_scatter_paged(const dsb_kv_pages* kv, const int32_t* block_table, int max_blocks,
                                const int32_t* n_blocks, const int32_t* window, int n_seq, int tokens_per_seq,
                                const int32_t* pos, const float* k, const float* v, dsb_workspace* ws, void* stream) {
  dsb_status st = check_pages(kv);
  if (st != DSB_OK) return st;
  st = check_paged_geometry(kv, block_table, max_blocks, n_blocks, window, n_seq, tokens_per_seq, nullptr);
  if (st != DSB_OK) return st;
  if (!pos || !k || !v) return fail(DSB_ERR_INVALID_ARG, "pos / k / v is NULL");
  if (!aligned16(k) || !aligned16(v)) return fail(DSB_ERR_INVALID_ARG, "k / v not 16-byte aligned");
  if (!ws) return fail(DSB_ERR_WORKSPACE, "workspace is NULL");
  const int n_tok = n_seq * tokens_per_seq;
  std::vector<long long> rows;  // (page, row) of every write: two writes of one row would race
  rows.reserve((size_t)n_tok);
  for (int t = 0; t < n_tok; ++t) {
    const int s = t / tokens_per_seq, p = pos[t];
    if (p < 0) return fail(DSB_ERR_INVALID_ARG, "pos[%d]=%d < 0", t, p);
    int i = p / DSB_KV_PAGE;
    if (window[s] > 0) {
      i %= n_blocks[s];
    } else if (i >= n_blocks[s]) {
      return fail(DSB_ERR_INVALID_ARG, "pos[%d]=%d beyond sequence %d's %d blocks", t, p, s, n_blocks[s]);
    }
    rows.push_back((long long)block_table[(size_t)s * max_blocks + i] * DSB_KV_PAGE + p % DSB_KV_PAGE);
  }
  std::vector<long long> sorted = rows;
  std::sort(sorted.begin(), sorted.end());
  if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end())
    return fail(DSB_ERR_INVALID_ARG, "two tokens of the call write the same page row");
  std::vector<int32_t> words;
  words.reserve((size_t)n_seq * max_blocks + 2 * (size_t)n_seq + n_tok);
  words.insert(words.end(), block_table, block_table + (size_t)n_seq * max_blocks);
  words.insert(words.end(), n_blocks, n_blocks + n_seq);
  words.insert(words.end(), window, window + n_seq);
  words.insert(words.end(), pos, pos + n_tok);
  if (words.size() > kMetaWords) return fail(DSB_ERR_UNSUPPORTED, "block tables exceed the staging slot");
  const int32_t* dev = nullptr;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  st = stage(ws, words, cs, &dev);
  if (st != DSB_OK) return st;
  dsbk::PagedView pv;
  pv.block_table = dev;
  pv.max_blocks = max_blocks;
  pv.n_blocks = dev + (size_t)n_seq * max_blocks;
  pv.window = pv.n_blocks + n_seq;
  cudaError_t e = dsbk::launch_kv_scatter_paged(kv->k, kv->v, kv->dtype, kv->n_kv_heads, kv->head_dim, pv,
                                                tokens_per_seq, pv.window + n_seq, n_tok, k, v,
                                                (long long)kv->n_kv_heads * kv->head_dim, cs);
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "kv_scatter_paged launch");
}

dsb_status dsb_attention_decode_paged(const float* q, int n_q_heads, const dsb_kv_pages* kv,
                                      const int32_t* block_table, int max_blocks, const int32_t* n_blocks,
                                      const int32_t* window, int n_seq, int tokens_per_seq, const int32_t* seq_lens,
                                      float* out, dsb_workspace* ws, void* stream) {
  dsb_status st = check_pages(kv);
  if (st != DSB_OK) return st;
  if (kv->head_dim != 64 && kv->head_dim != 128)
    return fail(DSB_ERR_UNSUPPORTED, "head_dim=%d: attention serves 64 and 128", kv->head_dim);
  if (n_q_heads < 1 || n_q_heads % kv->n_kv_heads)
    return fail(DSB_ERR_INVALID_ARG, "n_q_heads=%d is not a positive multiple of n_kv_heads=%d", n_q_heads,
                kv->n_kv_heads);
  if ((long long)(n_q_heads / kv->n_kv_heads) * tokens_per_seq > 64)
    return fail(DSB_ERR_UNSUPPORTED, "query rows per kv head (G*T) exceed 64");
  if (!seq_lens) return fail(DSB_ERR_INVALID_ARG, "seq_lens is NULL");
  st = check_paged_geometry(kv, block_table, max_blocks, n_blocks, window, n_seq, tokens_per_seq, seq_lens);
  if (st != DSB_OK) return st;
  if (!q || !out) return fail(DSB_ERR_INVALID_ARG, "q / out is NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(DSB_ERR_INVALID_ARG, "q / out not 16-byte aligned");
  if (!ws) return fail(DSB_ERR_WORKSPACE, "workspace is NULL");
  const int n_tok = n_seq * tokens_per_seq;
  std::vector<int32_t> words;
  words.reserve(3 * (size_t)n_seq + 1 + (size_t)n_seq * max_blocks + 2 * (size_t)n_seq);
  words.insert(words.end(), (size_t)n_seq, 0);  // batch_index: unused by the paged view
  words.insert(words.end(), seq_lens, seq_lens + n_seq);
  long long total = 0;
  int max_chunks = 1;
  words.push_back(0);
  for (int s = 0; s < n_seq; ++s) {
    const int c0 = paged_first_chunk(seq_lens[s], tokens_per_seq, window[s]);
    const int n = (seq_lens[s] - 1) / DSB_ATTN_CHUNK - c0 + 1;
    max_chunks = std::max(max_chunks, n);
    total += n;
    words.push_back((int32_t)total);
  }
  if (total * kv->n_kv_heads > INT_MAX) return fail(DSB_ERR_INVALID_ARG, "too many attention chunks");
  words.insert(words.end(), block_table, block_table + (size_t)n_seq * max_blocks);
  words.insert(words.end(), n_blocks, n_blocks + n_seq);
  words.insert(words.end(), window, window + n_seq);
  if (words.size() > kMetaWords) return fail(DSB_ERR_UNSUPPORTED, "block tables exceed the staging slot");
  const size_t need = (size_t)n_tok * n_q_heads * max_chunks * (kv->head_dim + 2) * sizeof(float);
  if (need > partial_capacity(ws))
    return fail(DSB_ERR_WORKSPACE, "attention needs %zu workspace bytes for partials, have %zu", need,
                partial_capacity(ws));
  const int32_t* dev = nullptr;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  st = stage(ws, words, cs, &dev);
  if (st != DSB_OK) return st;
  dsbk::MetaView mv{dev, dev + n_seq, dev + 2 * n_seq, nullptr};
  dsbk::PagedView pv;
  pv.block_table = dev + 3 * (size_t)n_seq + 1;
  pv.max_blocks = max_blocks;
  pv.n_blocks = pv.block_table + (size_t)n_seq * max_blocks;
  pv.window = pv.n_blocks + n_seq;
  cudaError_t e = dsbk::launch_attention_decode_multi(
      q, (long long)n_q_heads * kv->head_dim, n_q_heads, kv->k, kv->v, kv->dtype, kv->n_kv_heads, 0, kv->head_dim,
      (long long)kv->n_pages * kv->n_kv_heads * DSB_KV_PAGE, mv, n_seq, tokens_per_seq, total * kv->n_kv_heads, max_chunks, reinterpret_cast<float*>(partial_base(ws)), out,
      nullptr, cs, pv);
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "attention_decode_paged launch");
}

dsb_status dsb_attention_decode_multi(const float* q, int n_q_heads, const dsb_kv_cache* kv,
                                      const int32_t* batch_index, int n_seq, int tokens_per_seq,
                                      const int32_t* seq_lens, float* out, dsb_workspace* ws, void* stream) {
  if (!out) return fail(DSB_ERR_INVALID_ARG, "out is NULL");
  return attention_common(q, n_q_heads, kv, batch_index, n_seq, tokens_per_seq, seq_lens, out, nullptr, ws, stream);
}

dsb_status dsb_attention_decode_multi_q8_0(const float* q, int n_q_heads, const dsb_kv_cache* kv,
                                           const int32_t* batch_index, int n_seq, int tokens_per_seq,
                                           const int32_t* seq_lens, void* xq, dsb_workspace* ws, void* stream) {
  if (!xq) return fail(DSB_ERR_INVALID_ARG, "xq is NULL");
  return attention_common(q, n_q_heads, kv, batch_index, n_seq, tokens_per_seq, seq_lens, nullptr, xq, ws, stream);
}

// ---- step glue, exposed one kernel at a time --------------------------------

dsb_status dsb_rmsnorm_q8_0(const float* x, const float* w, int n_tok, int hidden, float eps, void* xq,
                            void* stream) {
  if (n_tok < 0 || n_tok > DSB_MAX_TOKENS) return fail(DSB_ERR_INVALID_ARG, "n_tok=%d out of [0, %d]", n_tok, DSB_MAX_TOKENS);
  if (hidden < 256 || hidden % 256 || hidden > 8192)
    return fail(DSB_ERR_UNSUPPORTED, "hidden=%d: RMSNorm serves multiples of 256 up to 8192", hidden);
  if (!(eps > 0.0f) || !std::isfinite(eps)) return fail(DSB_ERR_INVALID_ARG, "eps must be finite and > 0");
  if (n_tok == 0) return DSB_OK;
  if (!x || !w || !xq) return fail(DSB_ERR_INVALID_ARG, "x / w / xq is NULL");
  if (!aligned16(x) || !aligned16(w) || !aligned16(xq)) return fail(DSB_ERR_INVALID_ARG, "x / w / xq not 16-byte aligned");
  cudaError_t e = dsbk::launch_rmsnorm_quant(x, w, n_tok, hidden, eps, xq, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "rmsnorm_q8_0 launch");
}

dsb_status dsb_silu_mul_q8_0(const float* gu, int n_tok, int ffn, void* xq, void* stream) {
  if (n_tok < 0 || n_tok > DSB_MAX_TOKENS) return fail(DSB_ERR_INVALID_ARG, "n_tok=%d out of [0, %d]", n_tok, DSB_MAX_TOKENS);
  if (ffn < 32 || ffn % 32) return fail(DSB_ERR_INVALID_ARG, "ffn=%d is not a positive multiple of 32", ffn);
  if (n_tok == 0) return DSB_OK;
  if (!gu || !xq) return fail(DSB_ERR_INVALID_ARG, "gu / xq is NULL");
  if (!aligned16(gu) || !aligned16(xq)) return fail(DSB_ERR_INVALID_ARG, "gu / xq not 16-byte aligned");
  cudaError_t e = dsbk::launch_silu_mul_quant(gu, n_tok, ffn, xq, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "silu_mul_q8_0 launch");
}

static dsb_status fused_matmul_common(int pro, const dsb_q8_0_mat* w, const float* xf, const float* norm_w,
                                      float eps, int n_tok, float* y, void* stream) {
  dsb_status st = check_mat(w);
  if (st != DSB_OK) return st;
  if (n_tok < 1 || n_tok > DSB_NARROW_MAX)
    return fail(DSB_ERR_INVALID_ARG, "n_tok=%d out of [1, %d]", n_tok, DSB_NARROW_MAX);
  if (pro == 1) {
    if (w->cols > 8192) return fail(DSB_ERR_UNSUPPORTED, "cols=%lld: RMSNorm serves up to 8192", (long long)w->cols);
    if (!(eps > 0.0f) || !std::isfinite(eps)) return fail(DSB_ERR_INVALID_ARG, "eps must be finite and > 0");
    if (!norm_w) return fail(DSB_ERR_INVALID_ARG, "norm_w is NULL");
    if (!aligned16(norm_w)) return fail(DSB_ERR_INVALID_ARG, "norm_w not 16-byte aligned");
  }
  if (!xf || !y) return fail(DSB_ERR_INVALID_ARG, "input / y is NULL");
  if (!aligned16(xf) || !aligned16(y)) return fail(DSB_ERR_INVALID_ARG, "input / y not 16-byte aligned");
  DeviceInfo di;
  st = device_info(&di);
  if (st != DSB_OK) return st;
  if (dsbk::matmul_fused_smem_bytes(w->rows, w->cols, n_tok, pro, di.sms) > (size_t)di.max_smem_optin)
    return fail(DSB_ERR_UNSUPPORTED, "matmul %lldx%lld exceeds the shared memory", (long long)w->rows,
                (long long)w->cols);
  const int stride = pro == 1 ? (int)w->cols : 2 * (int)w->cols;
  cudaError_t e = dsbk::launch_matmul_q8_0_fused(pro, w->blocks, w->rows, w->cols, xf, stride, norm_w, eps, n_tok, y,
                                                 nullptr, di.sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "fused matmul launch");
}

dsb_status dsb_rmsnorm_matmul_q8_0(const dsb_q8_0_mat* w, const float* x, const float* norm_w, float eps, int n_tok,
                                   float* y, void* stream) {
  return fused_matmul_common(1, w, x, norm_w, eps, n_tok, y, stream);
}

dsb_status dsb_silu_matmul_q8_0(const dsb_q8_0_mat* w, const float* gu, int n_tok, float* y, void* stream) {
  return fused_matmul_common(2, w, gu, nullptr, 0.0f, n_tok, y, stream);
}

dsb_status dsb_embed_q8_0(const void* table, int vocab, int hidden, const int32_t* token_ids, int n_tok, float* h,
                          dsb_workspace* ws, void* stream) {
  if (n_tok < 0 || n_tok > DSB_MAX_TOKENS) return fail(DSB_ERR_INVALID_ARG, "n_tok=%d out of [0, %d]", n_tok, DSB_MAX_TOKENS);
  if (vocab < 1) return fail(DSB_ERR_INVALID_ARG, "vocab=%d < 1", vocab);
  if (hidden < 32 || hidden % 32) return fail(DSB_ERR_INVALID_ARG, "hidden=%d is not a positive multiple of 32", hidden);
  if (!ws) return fail(DSB_ERR_WORKSPACE, "workspace is NULL");
  if (n_tok == 0) return DSB_OK;
  if (!table || !token_ids || !h) return fail(DSB_ERR_INVALID_ARG, "table / token_ids / h is NULL");
  if (!aligned16(table) || !aligned16(h)) return fail(DSB_ERR_INVALID_ARG, "table / h not 16-byte aligned");
  for (int t = 0; t < n_tok; ++t)
    if (token_ids[t] < 0 || token_ids[t] >= vocab)
      return fail(DSB_ERR_INVALID_ARG, "token_ids[%d]=%d out of [0, vocab=%d)", t, token_ids[t], vocab);
  std::vector<int32_t> words(token_ids, token_ids + n_tok);
  const int32_t* dev = nullptr;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  dsb_status st = stage(ws, words, cs, &dev);
  if (st != DSB_OK) return st;
  cudaError_t e = dsbk::launch_embed(table, hidden, dev, n_tok, h, nullptr, nullptr, 0, cs);
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "embed_q8_0 launch");
}

dsb_status dsb_rope_kv_write(float* qkv, int n_q_heads, const dsb_kv_cache* kv, const int32_t* batch_index,
                             int n_seq, int tokens_per_seq, const int32_t* pos, const dsb_rope* rope,
                             const float* q_norm,
                             const float* k_norm, float eps, dsb_workspace* ws, void* stream) {
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return fail(DSB_ERR_INVALID_ARG, "eps must be finite and >= 0");
  dsb_status st = check_kv(kv);
  if (st != DSB_OK) return st;
  if (n_q_heads < 1 || n_q_heads % kv->n_kv_heads)
    return fail(DSB_ERR_INVALID_ARG, "n_q_heads=%d is not a positive multiple of n_kv_heads=%d", n_q_heads,
                kv->n_kv_heads);
  if (kv->head_dim % 2 || kv->head_dim > 1024) return fail(DSB_ERR_INVALID_ARG, "head_dim=%d must be even, <= 1024", kv->head_dim);
  st = check_batch(kv, batch_index, n_seq, tokens_per_seq);
  if (st != DSB_OK) return st;
  if (check_rope(rope) != DSB_OK) return DSB_ERR_INVALID_ARG;
  if (!qkv || !pos) return fail(DSB_ERR_INVALID_ARG, "qkv / pos is NULL");
  if (!aligned16(qkv)) return fail(DSB_ERR_INVALID_ARG, "qkv not 16-byte aligned");
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
  static thread_local dsbk::RopeFreqs freqs;
  fill_rope_freqs(*rope, kv->head_dim, &freqs);
  const long long stride = (long long)(n_q_heads + 2 * kv->n_kv_heads) * kv->head_dim;
  cudaError_t e = dsbk::launch_rope_kv_write(qkv, stride, n_q_heads, kv->n_kv_heads, kv->head_dim, dev + n_seq, dev,
                                             tokens_per_seq, n_tok, kv->k, kv->v, kv->dtype, kv->ctx, freqs, cs, q_norm,
                                             k_norm, eps);
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "rope_kv_write launch");
}

}  // extern "C"

// ===========================================================================
// The whole decode step (declared at the end of include/dsb.h).
// ===========================================================================
namespace {

struct StepLayout {
  size_t h = 0, qkv = 0, att = 0, gu = 0, xq = 0, staged = 0, graph_meta = 0, partials = 0, pack = 0, total = 0;
};

StepLayout step_layout(const dsb_model_shape& sh, int n_tok, int ctx) {
  StepLayout L;
  size_t off = kMetaBytes;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += round_up(bytes, 256);
    return o;
  };
  const size_t nt = (size_t)n_tok;
  const size_t qkv_cols = (size_t)(sh.n_q_heads + 2 * sh.n_kv_heads) * sh.head_dim;
  const size_t att_cols = (size_t)sh.n_q_heads * sh.head_dim;
  size_t max_cols = (size_t)sh.hidden;
  if (att_cols > max_cols) max_cols = att_cols;
  if ((size_t)sh.ffn > max_cols) max_cols = (size_t)sh.ffn;
  L.h = take(nt * sh.hidden * 4);
  L.qkv = take(nt * qkv_cols * 4);
  L.att = take(nt * att_cols * 4);
  L.gu = take(nt * 2 * (size_t)sh.ffn * 4);
  L.xq = take(nt * (max_cols / 32) * 34);
  // the narrow matmul's staged activation layout, written by the q8_0-emitting
  // kernels next to the q8_0 rows (n_tok <= DSB_NARROW_MAX)
  L.staged = take(n_tok <= DSB_NARROW_MAX ? dsbk::matmul_staged_bytes(n_tok, (int64_t)max_cols) : 0);
  L.graph_meta = take(kMetaSlotBytes);
  L.partials = take(dsbk::attention_partial_bytes(n_tok, sh.n_q_heads, sh.head_dim, ctx));
  // packed token operands of the tensor-core matmul (n_tok > DSB_NARROW_MAX)
  L.pack = take(n_tok > DSB_NARROW_MAX ? dsbk::matmul_tc_scratch_bytes(n_tok, (int64_t)max_cols) : 0);
  L.total = off;
  return L;
}

dsb_status check_mat_shape(const dsb_q8_0_mat& m, long long rows, long long cols, const char* what, int layer) {
  dsb_status st = check_mat(&m);
  if (st != DSB_OK) return fail(st, "layer %d %s: %s", layer, what, dsb_last_error());
  if (m.rows != rows || m.cols != cols)
    return fail(DSB_ERR_INVALID_ARG, "layer %d %s is %lldx%lld, expected %lldx%lld", layer, what, (long long)m.rows,
                (long long)m.cols, rows, cols);
  return DSB_OK;
}

// Validates the model description; on success *kv0 is layer 0's cache (all
// layers share its geometry).
// need_kv: the layers' contiguous caches are checked (false: the step runs on
// page pools given apart from the model, and kv0 is left NULL).
dsb_status check_model(const dsb_model* m, const dsb_kv_cache** kv0, bool need_kv = true) {
  if (!m) return fail(DSB_ERR_INVALID_ARG, "model is NULL");
  const dsb_model_shape& s = m->shape;
  if (s.hidden < 256 || s.n_q_heads < 1 || s.n_kv_heads < 1 || s.head_dim < 2 || s.ffn < 256 || s.vocab < 1 ||
      s.n_layers < 1)
    return fail(DSB_ERR_INVALID_ARG, "model shape has a non-positive or too small dimension");
  if (s.n_q_heads % s.n_kv_heads) return fail(DSB_ERR_INVALID_ARG, "n_q_heads %% n_kv_heads != 0");
  if (s.hidden > 8192) return fail(DSB_ERR_UNSUPPORTED, "hidden=%d: the step serves hidden <= 8192", s.hidden);
  if (s.hidden % 256 || s.ffn % 256 || (s.n_q_heads * s.head_dim) % 256)
    return fail(DSB_ERR_UNSUPPORTED, "hidden, ffn and n_q_heads*head_dim must be multiples of 256");
  if (s.head_dim != 64 && s.head_dim != 128) return fail(DSB_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (!(s.rms_eps > 0.0f) || !std::isfinite(s.rms_eps)) return fail(DSB_ERR_INVALID_ARG, "rms_eps must be > 0");
  if (check_rope(&s.rope) != DSB_OK) return DSB_ERR_INVALID_ARG;
  if (!m->embed || !aligned16(m->embed)) return fail(DSB_ERR_INVALID_ARG, "embed is NULL or not 16-byte aligned");
  if (!m->final_norm) return fail(DSB_ERR_INVALID_ARG, "final_norm is NULL");
  if (!m->layers) return fail(DSB_ERR_INVALID_ARG, "layers is NULL");
  const long long qkv_rows = (long long)(s.n_q_heads + 2 * s.n_kv_heads) * s.head_dim;
  for (int l = 0; l < s.n_layers; ++l) {
    const dsb_layer& L = m->layers[l];
    dsb_status st;
    if ((st = check_mat_shape(L.wqkv, qkv_rows, s.hidden, "wqkv", l)) != DSB_OK) return st;
    if ((st = check_mat_shape(L.wo, s.hidden, (long long)s.n_q_heads * s.head_dim, "wo", l)) != DSB_OK) return st;
    if ((st = check_mat_shape(L.wgu, 2LL * s.ffn, s.hidden, "wgu", l)) != DSB_OK) return st;
    if ((st = check_mat_shape(L.wdown, s.hidden, s.ffn, "wdown", l)) != DSB_OK) return st;
    if (!L.attn_norm || !L.ffn_norm) return fail(DSB_ERR_INVALID_ARG, "layer %d norm weights are NULL", l);
    if (!need_kv) continue;
    if ((st = check_kv(&L.kv)) != DSB_OK) return fail(st, "layer %d kv: %s", l, dsb_last_error());
    if (L.kv.n_kv_heads != s.n_kv_heads || L.kv.head_dim != s.head_dim)
      return fail(DSB_ERR_INVALID_ARG, "layer %d kv heads/head_dim do not match the shape", l);
    const dsb_kv_cache& k0 = m->layers[0].kv;
    if (L.kv.full_batch_size != k0.full_batch_size || L.kv.ctx != k0.ctx || L.kv.dtype != k0.dtype)
      return fail(DSB_ERR_INVALID_ARG, "layer %d kv geometry differs from layer 0", l);
  }
  dsb_status st = check_mat_shape(m->head, s.vocab, s.hidden, "head", -1);
  if (st != DSB_OK) return st;
  *kv0 = need_kv ? &m->layers[0].kv : nullptr;
  return DSB_OK;
}

dsb_status check_step_meta(const dsb_model* m, const dsb_kv_cache* kv0, const int32_t* tokens, const int32_t* bi,
                           int n_seq, int tps, const int32_t* seq_lens) {
  dsb_status st = check_batch(kv0, bi, n_seq, tps);
  if (st != DSB_OK) return st;
  if (!tokens || !seq_lens) return fail(DSB_ERR_INVALID_ARG, "token_ids / seq_lens is NULL");
  for (int t = 0; t < n_seq * tps; ++t)
    if (tokens[t] < 0 || tokens[t] >= m->shape.vocab)
      return fail(DSB_ERR_INVALID_ARG, "token_ids[%d]=%d out of [0, vocab=%d)", t, tokens[t], m->shape.vocab);
  for (int s = 0; s < n_seq; ++s)
    if (seq_lens[s] < tps || seq_lens[s] > kv0->ctx)
      return fail(DSB_ERR_INVALID_ARG, "seq_lens[%d]=%d out of [T=%d, ctx=%d]", s, seq_lens[s], tps, kv0->ctx);
  return DSB_OK;
}

// tokens[n_tok] | batch_index[n_seq] | seq_lens[n_seq] | chunk_off[n_seq+1] | pos[n_tok]
std::vector<int32_t> step_words(const int32_t* tokens, const int32_t* bi, int n_seq, int tps, const int32_t* seq_lens,
                                long long* total_chunks) {
  const int n_tok = n_seq * tps;
  std::vector<int32_t> w;
  w.reserve((size_t)2 * n_tok + 3 * n_seq + 1);
  w.insert(w.end(), tokens, tokens + n_tok);
  w.insert(w.end(), bi, bi + n_seq);
  w.insert(w.end(), seq_lens, seq_lens + n_seq);
  long long tot = 0;
  w.push_back(0);
  for (int s = 0; s < n_seq; ++s) {
    tot += (seq_lens[s] + DSB_ATTN_CHUNK - 1) / DSB_ATTN_CHUNK;
    w.push_back((int32_t)tot);
  }
  for (int s = 0; s < n_seq; ++s)
    for (int j = 0; j < tps; ++j) w.push_back(seq_lens[s] - tps + j);
  *total_chunks = tot;
  return w;
}

// n_tok <= DSB_NARROW_MAX: the narrow dp4a kernel; more: the tensor-core
// kernel, with its token operands packed into `pack`.
// Whether the step's matmul of n_tok > 16 token rows runs as narrow launches
// of 16 tokens (the weights read once per 16 tokens) rather than on the
// tensor cores (once per 128): estimated times from this GPU's measurements,
// a 16-token narrow launch about 10 us + 0.234 us per MB of weights, the
// tensor-core kernel about 30 us + 0.65 us per MB per 128 token rows (its
// fixed cost dominates on small matrices: 2304 x 768 at 32 tokens took 30 us
// there, against about 10 us per narrow launch).
bool narrow_chunks_cheaper(int64_t rows, int64_t cols, int n_tok) {
  const double mb = (double)rows * (double)(cols / 32) * 34.0 / 1e6;
  const double narrow = (double)((n_tok + DSB_NARROW_MAX - 1) / DSB_NARROW_MAX) * (10.0 + 0.234 * mb);
  const double tc = 30.0 + (double)((n_tok + 127) / 128) * 0.65 * mb;
  return narrow < tc;
}

cudaError_t run_matmul(const dsb_q8_0_mat& w, const void* xq, int n_tok, float* y, const float* residual, int sms,
                       void* pack, cudaStream_t st) {
  if (n_tok > DSB_NARROW_MAX && !narrow_chunks_cheaper(w.rows, w.cols, n_tok))
    return dsbk::launch_matmul_q8_0_tc(w.blocks, w.rows, w.cols, xq, n_tok, y, residual, pack, st);
  const size_t blk_row = (size_t)(w.cols / 32) * 34;
  for (int t0 = 0; t0 < n_tok; t0 += DSB_NARROW_MAX) {
    const int nt = std::min(DSB_NARROW_MAX, n_tok - t0);
    cudaError_t e = dsbk::launch_matmul_q8_0_narrow(w.blocks, w.rows, w.cols,
                                                    static_cast<const char*>(xq) + (size_t)t0 * blk_row, nt,
                                                    y + (size_t)t0 * w.rows,
                                                    residual ? residual + (size_t)t0 * w.rows : nullptr, nullptr, sms, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Enqueue every kernel of one step; metadata already on the device at meta_dev.
// meta_src: NULL when the metadata already sits at meta_dev; otherwise a
// device-readable copy (mapped pinned host memory) that the first kernel
// copies to meta_dev (n_meta_words words) while it reads the token ids.
// Page pools of a paged step: every layer's pool (host array) and the block
// geometry, staged after the positions in the metadata block.
struct StepPages {
  const dsb_kv_pages* pages = nullptr;
  int max_blocks = 0;
  int max_chunks = 0;  // the most chunks a sequence's attention visits
};

dsb_status enqueue_step(const dsb_model* m, const int32_t* meta_dev, int n_seq, int tps, long long max_items,
                        float* logits, dsb_workspace* ws, int sms, cudaStream_t st, const int32_t* meta_src = nullptr,
                        size_t n_meta_words = 0, const int32_t* meta_words = nullptr,
                        dsbk::EmbedParamNode* embed_node = nullptr, const dsb_step_trace* trace = nullptr,
                        const StepPages* pg = nullptr) {
  const dsb_model_shape& s = m->shape;
  const int n_tok = n_seq * tps;
  const int ctx_cover = pg ? pg->max_chunks * DSB_ATTN_CHUNK : m->layers[0].kv.ctx;
  const StepLayout L = step_layout(s, n_tok, ctx_cover);
  const int32_t* tokens_dev = meta_dev;
  const int32_t* bi_dev = tokens_dev + n_tok;
  const int32_t* sl_dev = bi_dev + n_seq;
  const int32_t* co_dev = sl_dev + n_seq;
  const int32_t* pos_dev = co_dev + n_seq + 1;
  float* h = reinterpret_cast<float*>(ws->dev + L.h);
  float* qkv = reinterpret_cast<float*>(ws->dev + L.qkv);
  float* att = reinterpret_cast<float*>(ws->dev + L.att);
  float* gu = reinterpret_cast<float*>(ws->dev + L.gu);
  void* xq = ws->dev + L.xq;
  float* partials = reinterpret_cast<float*>(ws->dev + L.partials);
  void* pack = ws->dev + L.pack;
  // staged activations for the narrow matmuls (nullptr past DSB_NARROW_MAX tokens)
  void* stg = n_tok <= DSB_NARROW_MAX ? static_cast<void*>(ws->dev + L.staged) : nullptr;
  auto mm = [&](const dsb_q8_0_mat& w, float* y, const float* residual) {
    if (stg) return dsbk::launch_matmul_q8_0_staged(w.blocks, w.rows, w.cols, stg, n_tok, y, residual, sms, st);
    return run_matmul(w, xq, n_tok, y, residual, sms, pack, st);
  };
  const int D = s.head_dim, Hq = s.n_q_heads, Hkv = s.n_kv_heads;
  const long long qkv_stride = (long long)(Hq + 2 * Hkv) * D;
  const int max_chunks = (ctx_cover + DSB_ATTN_CHUNK - 1) / DSB_ATTN_CHUNK;
  const dsbk::MetaView mv{bi_dev, sl_dev, co_dev, pos_dev};
  dsbk::PagedView pv;
  if (pg) {
    pv.block_table = pos_dev + n_tok;
    pv.max_blocks = pg->max_blocks;
    pv.n_blocks = pv.block_table + (size_t)n_seq * pg->max_blocks;
    pv.window = pv.n_blocks + n_seq;
  }
  static thread_local dsbk::RopeFreqs freqs;
  fill_rope_freqs(s.rope, D, &freqs);
  // The first kernel follows the metadata copy; every later kernel may be
  // scheduled while its predecessor finishes (programmatic dependent launch).
  // meta_words: host words passed in the first kernel's parameters (the
  // captured step rewrites them per replay); meta_src: mapped host memory
  // the first kernel reads; neither: the metadata is already at meta_dev.
  cudaError_t e = meta_words ? dsbk::launch_embed_params(m->embed, s.hidden, n_tok, h, meta_words, (int)n_meta_words,
                                                         const_cast<int32_t*>(meta_dev), st, embed_node)
                             : dsbk::launch_embed(m->embed, s.hidden, meta_src ? meta_src : tokens_dev, n_tok, h,
                                                  meta_src, const_cast<int32_t*>(meta_dev), (int)n_meta_words, st);
  // Stage trace (parity checking only): a copy of a stage's result after its
  // kernel, on the same stream; nothing when the pointer is NULL.
  const size_t ntz = (size_t)n_tok;
  auto copy_out = [&](void* dst, const void* src, size_t bytes) {
    if (e == cudaSuccess && dst) e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st);
    return e == cudaSuccess;
  };
  const size_t h_bytes = ntz * s.hidden * 4, xh_bytes = ntz * (s.hidden / 32) * 34;
  if (trace) copy_out(trace->h_embed, h, h_bytes);
  dsbk::set_pdl(true);
  for (int l = 0; l < s.n_layers && e == cudaSuccess; ++l) {
    const dsb_layer& Ly = m->layers[l];
    const dsb_layer_trace* tr = trace && trace->layers ? &trace->layers[l] : nullptr;
    if ((e = dsbk::launch_rmsnorm_quant(h, Ly.attn_norm, n_tok, s.hidden, s.rms_eps, xq, st, stg)) != cudaSuccess)
      break;
    if (tr && !copy_out(tr->x_attn, xq, xh_bytes)) break;
    if ((e = mm(Ly.wqkv, qkv, nullptr)) != cudaSuccess) break;
    if (tr && !copy_out(tr->qkv, qkv, ntz * qkv_stride * 4)) break;
    // this layer's cache: its contiguous cache, or its page pool
    void* kc = pg ? pg->pages[l].k : Ly.kv.k;
    void* vc = pg ? pg->pages[l].v : Ly.kv.v;
    const int kv_dtype = pg ? (int)pg->pages[l].dtype : (int)Ly.kv.dtype;
    const int kv_ctx = pg ? 0 : Ly.kv.ctx;
    const long long kv_rows = pg ? (long long)pg->pages[l].n_pages * Hkv * DSB_KV_PAGE
                                 : (long long)Ly.kv.full_batch_size * Hkv * Ly.kv.ctx;
    if ((e = dsbk::launch_rope_kv_write(qkv, qkv_stride, Hq, Hkv, D, pos_dev, bi_dev, tps, n_tok, kc, vc, kv_dtype,
                                        kv_ctx, freqs, st, Ly.q_norm, Ly.k_norm, s.rms_eps, pv)) != cudaSuccess)
      break;
    if (tr && !copy_out(tr->qkv_rope, qkv, ntz * qkv_stride * 4)) break;
    if ((e = dsbk::launch_attention_decode_multi(qkv, qkv_stride, Hq, kc, vc, kv_dtype, Hkv, kv_ctx, D, kv_rows, mv,
                                                 n_seq, tps, max_items, max_chunks, partials, att, xq, st, pv, stg)) !=
        cudaSuccess)
      break;
    if (tr && !copy_out(tr->att_q8, xq, ntz * ((size_t)Hq * D / 32) * 34)) break;
    if ((e = mm(Ly.wo, h, h)) != cudaSuccess) break;
    if (tr && !copy_out(tr->h_attn, h, h_bytes)) break;
    if ((e = dsbk::launch_rmsnorm_quant(h, Ly.ffn_norm, n_tok, s.hidden, s.rms_eps, xq, st, stg)) != cudaSuccess)
      break;
    if (tr && !copy_out(tr->x_ffn, xq, xh_bytes)) break;
    if ((e = mm(Ly.wgu, gu, nullptr)) != cudaSuccess) break;
    if (tr && !copy_out(tr->gu, gu, ntz * 2 * (size_t)s.ffn * 4)) break;
    if ((e = dsbk::launch_silu_mul_quant(gu, n_tok, s.ffn, xq, st, stg)) != cudaSuccess) break;
    if (tr && !copy_out(tr->act_q8, xq, ntz * ((size_t)s.ffn / 32) * 34)) break;
    if ((e = mm(Ly.wdown, h, h)) != cudaSuccess) break;
    if (tr && !copy_out(tr->h_out, h, h_bytes)) break;
  }
  if (e == cudaSuccess) e = dsbk::launch_rmsnorm_quant(h, m->final_norm, n_tok, s.hidden, s.rms_eps, xq, st, stg);
  if (trace) copy_out(trace->x_final, xq, xh_bytes);
  if (e == cudaSuccess) e = mm(m->head, logits, nullptr);
  dsbk::set_pdl(false);
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "decode step launch");
}

// ctx: the cache length the workspace's attention partials must cover (the
// contiguous caches' ctx; for page pools, 128 x the most chunks a sequence visits).
dsb_status check_step_resources(const dsb_model* m, int n_tok, float* logits, dsb_workspace* ws, int* sms,
                                int ctx = -1) {
  if (!logits || !aligned16(logits)) return fail(DSB_ERR_INVALID_ARG, "logits is NULL or not 16-byte aligned");
  if (!ws) return fail(DSB_ERR_WORKSPACE, "workspace is NULL");
  const StepLayout L = step_layout(m->shape, n_tok, ctx >= 0 ? ctx : m->layers[0].kv.ctx);
  if (L.total > ws->dev_bytes)
    return fail(DSB_ERR_WORKSPACE, "decode step needs %zu workspace bytes, have %zu", L.total, ws->dev_bytes);
  DeviceInfo di;
  dsb_status st = device_info(&di);
  if (st != DSB_OK) return st;
  const dsb_model_shape& s = m->shape;
  const long long mats[4][2] = {{(long long)(s.n_q_heads + 2 * s.n_kv_heads) * s.head_dim, s.hidden},
                                {s.hidden, (long long)s.n_q_heads * s.head_dim},
                                {2LL * s.ffn, s.hidden},
                                {s.hidden, s.ffn}};
  // past 16 tokens a matmul runs on the tensor cores or as 16-token narrow launches
  if (n_tok > DSB_NARROW_MAX && dsbk::matmul_tc_smem_bytes() > (size_t)di.max_smem_optin)
    return fail(DSB_ERR_UNSUPPORTED, "the tensor-core matmul exceeds shared memory");
  for (auto& mm : mats)
    if (dsbk::matmul_smem_bytes(mm[0], mm[1], std::min(n_tok, DSB_NARROW_MAX), di.sms) > (size_t)di.max_smem_optin)
      return fail(DSB_ERR_UNSUPPORTED, "a %lldx%lld matmul exceeds shared memory", mm[0], mm[1]);
  *sms = di.sms;
  return DSB_OK;
}

}  // namespace

struct dsb_step_graph {
  dsb_model_shape shape{};
  dsb_kv_cache kv0{};
  int n_seq = 0, tps = 0;
  dsb_workspace* ws = nullptr;
  int32_t* pinned = nullptr;      // mapped pinned host memory, rewritten between replays
  int32_t* pinned_dev = nullptr;  // its device address
  int32_t* dev_meta = nullptr;
  size_t n_words = 0;
  std::vector<int32_t> last;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaEvent_t done = nullptr;
  bool launched = false;
  // Parameter-block mode (n_words <= kEmbedParamMaxWords): the metadata rides
  // in the first kernel's parameters, rewritten per replay with
  // cudaGraphExecKernelNodeSetParams; the GPU never reads host memory.
  bool param_mode = false;
  cudaGraphNode_t embed_node = nullptr;
  dsbk::EmbedParamNode embed{};
  const void* a_table = nullptr;
  int a_hidden = 0;
  long long a_n_blocks = 0;
  float* a_h = nullptr;
  int32_t* a_meta_dst = nullptr;
  int a_n_words = 0;
  std::vector<int32_t> a_words;  // capacity words: the parameter block
  // A step on page pools: layer 0's pool (for the geometry checks) and the
  // block-table width the graph was captured for.
  bool paged = false;
  dsb_kv_pages pages0{};
  int max_blocks = 0;
};

// The parameters of the graph's embedding node for the current words.
static cudaError_t set_embed_node(dsb_step_graph* g) {
  void* args[7] = {&g->a_table, &g->a_hidden, &g->a_n_blocks, &g->a_h, g->a_words.data(), &g->a_meta_dst,
                   &g->a_n_words};
  cudaKernelNodeParams p{};
  p.func = const_cast<void*>(g->embed.func);
  p.gridDim = dim3(g->embed.grid);
  p.blockDim = dim3(g->embed.block);
  p.sharedMemBytes = 0;
  p.kernelParams = args;
  p.extra = nullptr;
  return cudaGraphExecKernelNodeSetParams(g->exec, g->embed_node, &p);
}

extern "C" {

size_t dsb_step_workspace_bytes(const dsb_model_shape* shape, int max_tokens, int ctx) {
  if (!shape || max_tokens < 1 || max_tokens > DSB_MAX_TOKENS || ctx < 1 || shape->hidden < 1 || shape->ffn < 1 ||
      shape->n_q_heads < 1 || shape->n_kv_heads < 0 || shape->head_dim < 1 || shape->head_dim > 1024)
    return 0;
  return step_layout(*shape, max_tokens, ctx).total;
}

dsb_status dsb_decode_step(const dsb_model* model, const int32_t* token_ids, const int32_t* batch_index, int n_seq,
                           int tokens_per_seq, const int32_t* seq_lens, float* logits, dsb_workspace* ws,
                           void* stream) {
  return dsb_decode_step_trace(model, token_ids, batch_index, n_seq, tokens_per_seq, seq_lens, logits, ws, nullptr,
                               stream);
}

dsb_status dsb_decode_step_trace(const dsb_model* model, const int32_t* token_ids, const int32_t* batch_index,
                                 int n_seq, int tokens_per_seq, const int32_t* seq_lens, float* logits,
                                 dsb_workspace* ws, const dsb_step_trace* trace, void* stream) {
  const dsb_kv_cache* kv0 = nullptr;
  dsb_status st = check_model(model, &kv0);
  if (st != DSB_OK) return st;
  st = check_step_meta(model, kv0, token_ids, batch_index, n_seq, tokens_per_seq, seq_lens);
  if (st != DSB_OK) return st;
  if ((long long)(model->shape.n_q_heads / model->shape.n_kv_heads) * tokens_per_seq > 64)
    return fail(DSB_ERR_UNSUPPORTED, "query rows per kv head (G*T) exceed 64");
  int sms = 0;
  st = check_step_resources(model, n_seq * tokens_per_seq, logits, ws, &sms);
  if (st != DSB_OK) return st;
  long long total = 0;
  const std::vector<int32_t> words = step_words(token_ids, batch_index, n_seq, tokens_per_seq, seq_lens, &total);
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const int32_t* dev = nullptr;
  st = stage(ws, words, cs, &dev);
  if (st != DSB_OK) return st;
  return enqueue_step(model, dev, n_seq, tokens_per_seq, total * model->shape.n_kv_heads, logits, ws, sms, cs,
                      nullptr, 0, nullptr, nullptr, trace);
}

// The metadata words of a step on page pools -- tokens | batch_index (unused:
// zeros) | seq_lens | chunk_off | pos | block_table | n_blocks | window --
// after every check of the call: tokens in range, the block geometry, and no
// two tokens of the step writing one page row.  total: the step's attention
// chunks; max_chunks: the most chunks one sequence visits.
// One page pool per layer, all of the shape's heads and one geometry.
static dsb_status check_pools(const dsb_model_shape& sh, const dsb_kv_pages* pages) {
  if (!pages) return fail(DSB_ERR_INVALID_ARG, "pages is NULL");
  dsb_status st = DSB_OK;
  for (int l = 0; l < sh.n_layers; ++l) {
    if ((st = check_pages(&pages[l])) != DSB_OK) return fail(st, "layer %d pages: %s", l, dsb_last_error());
    if (pages[l].n_kv_heads != sh.n_kv_heads || pages[l].head_dim != sh.head_dim)
      return fail(DSB_ERR_INVALID_ARG, "layer %d page pool heads/head_dim do not match the shape", l);
    if (pages[l].n_pages != pages[0].n_pages || pages[l].dtype != pages[0].dtype)
      return fail(DSB_ERR_INVALID_ARG, "layer %d page pool geometry differs from layer 0", l);
  }
  return DSB_OK;
}

static dsb_status paged_step_words(const dsb_model_shape& sh, const dsb_kv_pages* pages0, const int32_t* token_ids,
                                   int n_seq, int tokens_per_seq, const int32_t* seq_lens, const int32_t* block_table,
                                   int max_blocks, const int32_t* n_blocks, const int32_t* window,
                                   std::vector<int32_t>* out, long long* total_out, int* max_chunks_out) {
  dsb_status st = DSB_OK;
  if ((long long)(sh.n_q_heads / sh.n_kv_heads) * tokens_per_seq > 64)
    return fail(DSB_ERR_UNSUPPORTED, "query rows per kv head (G*T) exceed 64");
  if (!seq_lens || !token_ids) return fail(DSB_ERR_INVALID_ARG, "token_ids / seq_lens is NULL");
  st = check_paged_geometry(pages0, block_table, max_blocks, n_blocks, window, n_seq, tokens_per_seq, seq_lens);
  if (st != DSB_OK) return st;
  const int n_tok = n_seq * tokens_per_seq;
  for (int t = 0; t < n_tok; ++t)
    if (token_ids[t] < 0 || token_ids[t] >= sh.vocab)
      return fail(DSB_ERR_INVALID_ARG, "token_ids[%d]=%d out of [0, vocab=%d)", t, token_ids[t], sh.vocab);
  // every (page, row) the step writes, once: sequences may share pages
  std::vector<long long> rows;
  rows.reserve((size_t)n_tok);
  for (int s = 0; s < n_seq; ++s)
    for (int j = 0; j < tokens_per_seq; ++j) {
      const int p = seq_lens[s] - tokens_per_seq + j;
      int i = p / DSB_KV_PAGE;
      if (window[s] > 0) i %= n_blocks[s];
      rows.push_back((long long)block_table[(size_t)s * max_blocks + i] * DSB_KV_PAGE + p % DSB_KV_PAGE);
    }
  std::sort(rows.begin(), rows.end());
  if (std::adjacent_find(rows.begin(), rows.end()) != rows.end())
    return fail(DSB_ERR_INVALID_ARG, "two tokens of the step write the same page row");
  // tokens | batch_index (unused: zeros) | seq_lens | chunk_off | pos | block_table | n_blocks | window
  std::vector<int32_t>& words = *out;
  words.assign(token_ids, token_ids + n_tok);
  words.insert(words.end(), (size_t)n_seq, 0);
  words.insert(words.end(), seq_lens, seq_lens + n_seq);
  long long total = 0;
  int max_chunks = 1;
  words.push_back(0);
  for (int s = 0; s < n_seq; ++s) {
    const int c0 = paged_first_chunk(seq_lens[s], tokens_per_seq, window[s]);
    const int n = (seq_lens[s] - 1) / DSB_ATTN_CHUNK - c0 + 1;
    max_chunks = std::max(max_chunks, n);
    total += n;
    words.push_back((int32_t)total);
  }
  if (total * sh.n_kv_heads > INT_MAX) return fail(DSB_ERR_INVALID_ARG, "too many attention chunks");
  for (int s = 0; s < n_seq; ++s)
    for (int j = 0; j < tokens_per_seq; ++j) words.push_back(seq_lens[s] - tokens_per_seq + j);
  words.insert(words.end(), block_table, block_table + (size_t)n_seq * max_blocks);
  words.insert(words.end(), n_blocks, n_blocks + n_seq);
  words.insert(words.end(), window, window + n_seq);
  if (words.size() > kMetaWords) return fail(DSB_ERR_UNSUPPORTED, "step metadata with block tables exceeds the staging slot");
  *total_out = total;
  *max_chunks_out = max_chunks;
  return DSB_OK;
}

dsb_status dsb_decode_step_paged(const dsb_model* model, const dsb_kv_pages* pages, const int32_t* token_ids,
                                 int n_seq, int tokens_per_seq, const int32_t* seq_lens, const int32_t* block_table,
                                 int max_blocks, const int32_t* n_blocks, const int32_t* window, float* logits,
                                 dsb_workspace* ws, void* stream) {
  const dsb_kv_cache* unused = nullptr;
  dsb_status st = check_model(model, &unused, false);
  if (st != DSB_OK) return st;
  const dsb_model_shape& sh = model->shape;
  if ((st = check_pools(sh, pages)) != DSB_OK) return st;
  std::vector<int32_t> words;
  long long total = 0;
  int max_chunks = 1;
  st = paged_step_words(sh, &pages[0], token_ids, n_seq, tokens_per_seq, seq_lens, block_table, max_blocks, n_blocks,
                        window, &words, &total, &max_chunks);
  if (st != DSB_OK) return st;
  const int n_tok = n_seq * tokens_per_seq;
  int sms = 0;
  st = check_step_resources(model, n_tok, logits, ws, &sms, max_chunks * DSB_ATTN_CHUNK);
  if (st != DSB_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const int32_t* dev = nullptr;
  st = stage(ws, words, cs, &dev);
  if (st != DSB_OK) return st;
  StepPages pg;
  pg.pages = pages;
  pg.max_blocks = max_blocks;
  pg.max_chunks = max_chunks;
  return enqueue_step(model, dev, n_seq, tokens_per_seq, total * sh.n_kv_heads, logits, ws, sms, cs, nullptr, 0,
                      nullptr, nullptr, nullptr, &pg);
}

// Captures the step into g (n_seq, tps, ws and n_words already set): the
// contiguous caches, or the page pools of pg; ctx_cover: the cache length the
// attention partials cover; max_items: a bound on the attention's work items.
static dsb_status capture_step(dsb_step_graph* g, const dsb_model* model, float* logits, int sms, int ctx_cover,
                               long long max_items, const StepPages* pg) {
  const int n_tok = g->n_seq * g->tps;
  dsb_workspace* ws = g->ws;
  const StepLayout L = step_layout(model->shape, n_tok, ctx_cover);
  g->dev_meta = reinterpret_cast<int32_t*>(ws->dev + L.graph_meta);
  cudaStream_t cs = nullptr;
  // The step's metadata is read by the first kernel straight from mapped
  // pinned host memory (no copy node at the head of the graph).
  cudaError_t e = cudaHostAlloc(reinterpret_cast<void**>(&g->pinned), g->n_words * sizeof(int32_t), cudaHostAllocMapped);
  if (e == cudaSuccess) e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&g->pinned_dev), g->pinned, 0);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&g->done, cudaEventDisableTiming);
  // The legacy default stream cannot be captured, so capture on a private
  // non-blocking stream; work already queued elsewhere is not part of the graph.
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    if (cs) cudaStreamDestroy(cs);
    return cuda_fail(e, "dsb_step_graph_create");
  }
  // Placeholder metadata for the capture; the real values are written before
  // every launch.
  std::memset(g->pinned, 0, g->n_words * sizeof(int32_t));
  g->param_mode = g->n_words <= (size_t)dsbk::kEmbedParamMaxWords;
  std::vector<int32_t> zeros(g->n_words, 0);
  const int32_t* words_arg = g->param_mode ? zeros.data() : nullptr;
  // Warm every launcher's one-time set-up outside the capture.
  dsbk::set_dry_run(true);
  dsb_status dry = enqueue_step(model, g->dev_meta, g->n_seq, g->tps, max_items, logits, ws, sms, cs, g->pinned_dev,
                                g->n_words, words_arg, nullptr, nullptr, pg);
  dsbk::set_dry_run(false);
  if (dry != DSB_OK) {
    cudaStreamDestroy(cs);
    return dry;
  }
  e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  if (e == cudaSuccess) {
    const dsb_status es = enqueue_step(model, g->dev_meta, g->n_seq, g->tps, max_items, logits, ws, sms, cs,
                                       g->pinned_dev, g->n_words, words_arg, &g->embed, nullptr, pg);
    cudaError_t e2 = cudaStreamEndCapture(cs, &g->graph);
    if (es != DSB_OK) {
      if (g->graph) cudaGraphDestroy(g->graph);
      g->graph = nullptr;
      cudaStreamDestroy(cs);
      return es;
    }
    e = e2;
  }
  cudaStreamDestroy(cs);
  if (e == cudaSuccess) e = cudaGraphInstantiate(&g->exec, g->graph, 0);
  if (e == cudaSuccess && g->param_mode) {
    // the embedding kernel is the graph's single root node
    size_t n_roots = 1;
    cudaGraphNode_t root = nullptr;
    e = cudaGraphGetRootNodes(g->graph, &root, &n_roots);
    cudaGraphNodeType type = cudaGraphNodeTypeEmpty;
    if (e == cudaSuccess && n_roots == 1) e = cudaGraphNodeGetType(root, &type);
    if (e == cudaSuccess && (n_roots != 1 || type != cudaGraphNodeTypeKernel)) e = cudaErrorInvalidValue;
    if (e == cudaSuccess) {
      g->embed_node = root;
      g->a_table = model->embed;
      g->a_hidden = model->shape.hidden;
      g->a_n_blocks = g->embed.n_blocks;
      g->a_h = reinterpret_cast<float*>(ws->dev + L.h);
      g->a_meta_dst = g->dev_meta;
      g->a_n_words = (int)g->n_words;
      g->a_words.assign((size_t)g->embed.capacity, 0);
    }
  }
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "step graph capture");
}

// Frees whatever a (possibly half-built) graph holds.
static void free_graph(dsb_step_graph* g) {
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  if (g->done) cudaEventDestroy(g->done);
  if (g->pinned) cudaFreeHost(g->pinned);
  delete g;
}

// Writes the step's metadata words for the next replay and launches it.
static dsb_status launch_words(dsb_step_graph* g, std::vector<int32_t>& words, void* stream) {
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (words.size() != g->n_words) return fail(DSB_ERR_INVALID_ARG, "step metadata of %zu words, the graph holds %zu",
                                              words.size(), g->n_words);
  if (g->param_mode) {
    // the node's parameters are copied when set: no wait for the previous replay
    if (words != g->last) {
      std::copy(words.begin(), words.end(), g->a_words.begin());
      cudaError_t e = set_embed_node(g);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGraphExecKernelNodeSetParams(step)");
      g->last.swap(words);
    }
  } else if (words != g->last) {
    if (g->launched) {  // the previous replay may still be reading the pinned copy
      const auto t0 = std::chrono::steady_clock::now();
      for (;;) {
        cudaError_t q = cudaEventQuery(g->done);
        if (q == cudaSuccess) break;
        if (q != cudaErrorNotReady) return cuda_fail(q, "cudaEventQuery(step graph)");
        if (std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count() > kHostWaitSeconds)
          return fail(DSB_ERR_TIMEOUT, "previous step graph replay still running after %.0f s", kHostWaitSeconds);
        std::this_thread::yield();
      }
    }
    std::memcpy(g->pinned, words.data(), words.size() * sizeof(int32_t));
    g->last.swap(words);
  }
  cudaError_t e = cudaGraphLaunch(g->exec, cs);
  if (e == cudaSuccess) e = cudaEventRecord(g->done, cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGraphLaunch(step)");
  g->launched = true;
  return DSB_OK;
}

dsb_status dsb_step_graph_create(const dsb_model* model, int n_seq, int tokens_per_seq, float* logits,
                                 dsb_workspace* ws, void* stream, dsb_step_graph** out) {
  if (!out) return fail(DSB_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  const dsb_kv_cache* kv0 = nullptr;
  dsb_status st = check_model(model, &kv0);
  if (st != DSB_OK) return st;
  if (n_seq < 1 || n_seq > kv0->full_batch_size || n_seq > DSB_MAX_SEQS || tokens_per_seq < 1 ||
      (long long)n_seq * tokens_per_seq > DSB_MAX_TOKENS)
    return fail(DSB_ERR_INVALID_ARG, "n_seq=%d / tokens_per_seq=%d out of range", n_seq, tokens_per_seq);
  if ((long long)(model->shape.n_q_heads / model->shape.n_kv_heads) * tokens_per_seq > 64)
    return fail(DSB_ERR_UNSUPPORTED, "query rows per kv head (G*T) exceed 64");
  int sms = 0;
  const int n_tok = n_seq * tokens_per_seq;
  st = check_step_resources(model, n_tok, logits, ws, &sms);
  if (st != DSB_OK) return st;
  dsb_step_graph* g = new (std::nothrow) dsb_step_graph();
  if (!g) return fail(DSB_ERR_INVALID_ARG, "out of host memory");
  g->shape = model->shape;
  g->kv0 = *kv0;
  g->n_seq = n_seq;
  g->tps = tokens_per_seq;
  g->ws = ws;
  g->n_words = (size_t)2 * n_tok + 3 * (size_t)n_seq + 1;
  (void)stream;  // the graph is captured on a private stream and replayed on the caller's
  const long long max_items =
      (long long)n_seq * ((kv0->ctx + DSB_ATTN_CHUNK - 1) / DSB_ATTN_CHUNK) * model->shape.n_kv_heads;
  st = capture_step(g, model, logits, sms, kv0->ctx, max_items, nullptr);
  if (st != DSB_OK) {
    free_graph(g);
    return st;
  }
  *out = g;
  return DSB_OK;
}

dsb_status dsb_step_graph_launch(dsb_step_graph* g, const int32_t* token_ids, const int32_t* batch_index,
                                 const int32_t* seq_lens, void* stream) {
  if (!g) return fail(DSB_ERR_INVALID_ARG, "graph is NULL");
  if (g->paged) return fail(DSB_ERR_INVALID_ARG, "a graph on page pools launches with dsb_step_graph_launch_paged");
  dsb_model fake{};
  fake.shape = g->shape;
  dsb_status st = check_step_meta(&fake, &g->kv0, token_ids, batch_index, g->n_seq, g->tps, seq_lens);
  if (st != DSB_OK) return st;
  long long total = 0;
  std::vector<int32_t> words = step_words(token_ids, batch_index, g->n_seq, g->tps, seq_lens, &total);
  return launch_words(g, words, stream);
}

dsb_status dsb_step_graph_create_paged(const dsb_model* model, const dsb_kv_pages* pages, int max_blocks, int n_seq,
                                       int tokens_per_seq, float* logits, dsb_workspace* ws, void* stream,
                                       dsb_step_graph** out) {
  if (!out) return fail(DSB_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  const dsb_kv_cache* unused = nullptr;
  dsb_status st = check_model(model, &unused, false);
  if (st != DSB_OK) return st;
  if ((st = check_pools(model->shape, pages)) != DSB_OK) return st;
  if (n_seq < 1 || n_seq > DSB_MAX_SEQS || tokens_per_seq < 1 || (long long)n_seq * tokens_per_seq > DSB_MAX_TOKENS)
    return fail(DSB_ERR_INVALID_ARG, "n_seq=%d / tokens_per_seq=%d out of range", n_seq, tokens_per_seq);
  if (max_blocks < 1) return fail(DSB_ERR_INVALID_ARG, "max_blocks=%d < 1", max_blocks);
  if ((long long)(model->shape.n_q_heads / model->shape.n_kv_heads) * tokens_per_seq > 64)
    return fail(DSB_ERR_UNSUPPORTED, "query rows per kv head (G*T) exceed 64");
  const int n_tok = n_seq * tokens_per_seq;
  // tokens | batch_index | seq_lens | chunk_off | pos | block_table | n_blocks | window
  const size_t n_words = (size_t)2 * n_tok + 3 * (size_t)n_seq + 1 + (size_t)n_seq * max_blocks + 2 * (size_t)n_seq;
  if (n_words > kMetaWords) return fail(DSB_ERR_UNSUPPORTED, "step metadata with block tables exceeds the staging slot");
  // a sequence visits at most max_blocks + 1 chunks: its blocks, and under a
  // window the partly hidden chunk at the ring's start
  const int max_chunks = max_blocks + 1;
  int sms = 0;
  st = check_step_resources(model, n_tok, logits, ws, &sms, max_chunks * DSB_ATTN_CHUNK);
  if (st != DSB_OK) return st;
  dsb_step_graph* g = new (std::nothrow) dsb_step_graph();
  if (!g) return fail(DSB_ERR_INVALID_ARG, "out of host memory");
  g->shape = model->shape;
  g->n_seq = n_seq;
  g->tps = tokens_per_seq;
  g->ws = ws;
  g->n_words = n_words;
  g->paged = true;
  g->pages0 = pages[0];
  g->max_blocks = max_blocks;
  (void)stream;
  StepPages pg;
  pg.pages = pages;
  pg.max_blocks = max_blocks;
  pg.max_chunks = max_chunks;
  st = capture_step(g, model, logits, sms, max_chunks * DSB_ATTN_CHUNK,
                    (long long)n_seq * max_chunks * model->shape.n_kv_heads, &pg);
  if (st != DSB_OK) {
    free_graph(g);
    return st;
  }
  *out = g;
  return DSB_OK;
}

dsb_status dsb_step_graph_launch_paged(dsb_step_graph* g, const int32_t* token_ids, const int32_t* seq_lens,
                                       const int32_t* block_table, const int32_t* n_blocks, const int32_t* window,
                                       void* stream) {
  if (!g) return fail(DSB_ERR_INVALID_ARG, "graph is NULL");
  if (!g->paged) return fail(DSB_ERR_INVALID_ARG, "a graph on contiguous caches launches with dsb_step_graph_launch");
  std::vector<int32_t> words;
  long long total = 0;
  int max_chunks = 1;
  dsb_status st = paged_step_words(g->shape, &g->pages0, token_ids, g->n_seq, g->tps, seq_lens, block_table,
                                   g->max_blocks, n_blocks, window, &words, &total, &max_chunks);
  if (st != DSB_OK) return st;
  return launch_words(g, words, stream);
}

dsb_status dsb_step_graph_destroy(dsb_step_graph* g) {
  if (!g) return DSB_OK;
  dsb_status st = DSB_OK;
  if (g->launched) {
    const auto t0 = std::chrono::steady_clock::now();
    while (cudaEventQuery(g->done) == cudaErrorNotReady) {
      if (std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count() > kHostWaitSeconds) {
        st = fail(DSB_ERR_TIMEOUT, "step graph still running at destroy");
        break;
      }
      std::this_thread::yield();
    }
  }
  free_graph(g);
  return st;
}

}  // extern "C"

// ===========================================================================
// Attention for callers that cannot allocate (declared in include/dsb.h).
// ===========================================================================
extern "C" dsb_status dsb_attention_decode_multi_noalloc(const float* q, int n_q_heads, const dsb_kv_cache* kv,
                                                         const int32_t* batch_index, int n_seq, int tokens_per_seq,
                                                         const int32_t* seq_lens, float* out, void* stream) {
  dsb_status st = check_kv(kv);
  if (st != DSB_OK) return st;
  if (n_q_heads < 1 || n_q_heads % kv->n_kv_heads)
    return fail(DSB_ERR_INVALID_ARG, "n_q_heads=%d is not a positive multiple of n_kv_heads=%d", n_q_heads,
                kv->n_kv_heads);
  st = check_batch(kv, batch_index, n_seq, tokens_per_seq);
  if (st != DSB_OK) return st;
  if (n_seq > dsbk::kNoAllocMaxSeqs)
    return fail(DSB_ERR_UNSUPPORTED, "n_seq=%d exceeds the no-allocation limit of %d sequences", n_seq,
                dsbk::kNoAllocMaxSeqs);
  if (kv->head_dim != 64 && kv->head_dim != 128)
    return fail(DSB_ERR_UNSUPPORTED, "head_dim=%d: attention serves 64 and 128", kv->head_dim);
  const long long R = (long long)(n_q_heads / kv->n_kv_heads) * tokens_per_seq;
  if (R > 64) return fail(DSB_ERR_UNSUPPORTED, "query rows per kv head (G*T=%lld) exceed 64", R);
  if (!q || !out || !seq_lens) return fail(DSB_ERR_INVALID_ARG, "q / out / seq_lens is NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(DSB_ERR_INVALID_ARG, "q / out not 16-byte aligned");
  for (int s = 0; s < n_seq; ++s)
    if (seq_lens[s] < tokens_per_seq || seq_lens[s] > kv->ctx)
      return fail(DSB_ERR_INVALID_ARG, "seq_lens[%d]=%d out of [T=%d, ctx=%d]", s, seq_lens[s], tokens_per_seq, kv->ctx);
  const int n_tok = n_seq * tokens_per_seq;
  const size_t need = dsbk::attention_partial_bytes(n_tok, n_q_heads, kv->head_dim, kv->ctx);
  if (need > dsbk::kNoAllocScratchBytes - dsbk::kNoAllocTableBytes)
    return fail(DSB_ERR_UNSUPPORTED,
                "attention needs %zu bytes of partials; the no-allocation scratch holds %zu (use "
                "dsb_attention_decode_multi with a workspace)",
                need, dsbk::kNoAllocScratchBytes - dsbk::kNoAllocTableBytes);
  void* scratch = nullptr;
  cudaError_t e = dsbk::noalloc_scratch(&scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-allocation scratch)");
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  long long total = 0;
  e = dsbk::launch_noalloc_table(batch_index, seq_lens, n_seq, scratch, &total, cs);
  if (e != cudaSuccess) return cuda_fail(e, "no-allocation sequence table");
  const int32_t* table = static_cast<const int32_t*>(scratch);
  dsbk::MetaView mv{table, table + n_seq, table + 2 * n_seq, nullptr};
  float* partials = reinterpret_cast<float*>(static_cast<char*>(scratch) + dsbk::kNoAllocTableBytes);
  const int max_chunks = (kv->ctx + DSB_ATTN_CHUNK - 1) / DSB_ATTN_CHUNK;
  e = dsbk::launch_attention_decode_multi(q, (long long)n_q_heads * kv->head_dim, n_q_heads, kv->k, kv->v, kv->dtype,
                                          kv->n_kv_heads, kv->ctx, kv->head_dim,
                                          (long long)kv->full_batch_size * kv->n_kv_heads * kv->ctx, mv, n_seq,
                                          tokens_per_seq, total * kv->n_kv_heads, max_chunks, partials, out, nullptr,
                                          cs);
  return e == cudaSuccess ? DSB_OK : cuda_fail(e, "attention_decode_multi_noalloc launch");
}
