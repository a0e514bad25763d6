// Decode attention for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code running inside an
// allocator hook or a memory-pool callback, a process whose allocator is owned
// by another framework that forbids outside allocations, or a real-time
// serving loop that must not take the allocator's locks.  For them this file
// keeps the attention's scratch -- the split-K partials and the per-call
// sequence table -- in one file-scope device array that exists for as long as
// the library is loaded on a device.  The caller still passes q, the KV
// cache and out; nothing is allocated per call.
//
// Rules of the shared array:
//  * its device address is looked up once per device (cudaGetSymbolAddress,
//    with that device current) on the first call made on that device.  That
//    first call may also load this library's kernels onto the device (lazy
//    module loading, the CUDA default), which the driver backs with device
//    memory: make it outside the no-allocation context, e.g. at start-up;
//  * the address is kept for the life of the process, so a device reset
//    (cudaDeviceReset) after the first call on that device is not supported;
//  * every call on a device uses the same array, so calls whose work overlaps
//    on the GPU (e.g. on two streams at once) race -- serialise them;
//  * nothing in it has to start at zero: each call writes its sequence table
//    and every partial before reading them.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "dsb.h"
#include "dsb_kernels.h"

namespace dsbk {

// The scratch itself: file-scope, one per device that loads the library.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

struct NoAllocTable {
  int32_t n_seq;
  int32_t batch_index[kNoAllocMaxSeqs];
  int32_t seq_lens[kNoAllocMaxSeqs];
  int32_t chunk_off[kNoAllocMaxSeqs + 1];
};

// Writes the by-value sequence table into the start of the array:
// batch_index | seq_lens | chunk_off.
__global__ void noalloc_table_kernel(const __grid_constant__ NoAllocTable tab, int32_t* dst) {
  const int n = tab.n_seq;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    dst[i] = tab.batch_index[i];
    dst[n + i] = tab.seq_lens[i];
  }
  for (int i = threadIdx.x; i <= n; i += blockDim.x) dst[2 * n + i] = tab.chunk_off[i];
}

std::mutex g_mu;
void* g_addr[64];

}  // namespace

cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

// The table is built on this thread's stack (no heap use per call); chunk_off
// is the running count of 128-key chunks.  *total_chunks = chunk_off[n_seq].
cudaError_t launch_noalloc_table(const int32_t* batch_index, const int32_t* seq_lens, int n_seq, void* scratch,
                                 long long* total_chunks, cudaStream_t st) {
  NoAllocTable tab;
  tab.n_seq = n_seq;
  tab.chunk_off[0] = 0;
  for (int i = 0; i < n_seq; ++i) {
    tab.batch_index[i] = batch_index[i];
    tab.seq_lens[i] = seq_lens[i];
    tab.chunk_off[i + 1] = tab.chunk_off[i] + (seq_lens[i] + DSB_ATTN_CHUNK - 1) / DSB_ATTN_CHUNK;
  }
  *total_chunks = tab.chunk_off[n_seq];
  noalloc_table_kernel<<<1, 256, 0, st>>>(tab, static_cast<int32_t*>(scratch));
  return cudaGetLastError();
}

}  // namespace dsbk
