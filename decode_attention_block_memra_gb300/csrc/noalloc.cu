// Decode attention for callers that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: code that runs
// inside a custom allocator or memory pool (where a cudaMalloc could recurse
// into the allocator or break its accounting), plugins and embedded runtimes
// that are given only their input and output buffers, and real-time paths that
// forbid allocation after start-up.  For them this file keeps the split-K
// partials in one fixed array in device global memory, sized at build time,
// instead of a caller-provided workspace.
//
// The array lives as long as the library is loaded on each device that uses
// it (MEMRA_NOALLOC_SCRATCH_BYTES per device).  Every call shares it and it
// keeps the previous call's bytes; nothing in it has to start at zero, since
// the combine pass reads only partials that the split pass of the same call
// wrote.  Two calls whose kernels can overlap on the GPU (different streams,
// no ordering between them) race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "decode_kernel.cuh"

namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[MEMRA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device).  In host code the array's name is only a host-side handle, so
// the kernels must be given this address instead.
int scratch_on_current_device(void **ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MEMRA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MEMRA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MEMRA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return MEMRA_OK;
}

}  // namespace

extern "C" int memra_decode_attn_noalloc(const memra_kv_cache *cache, const void *q, const int32_t *page_table,
                                         int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t max_seq_len,
                                         int32_t batch, int32_t q_len, int32_t n_heads, int32_t n_kv_heads,
                                         int32_t head_dim, float sm_scale, void *out, void *stream) {
  const size_t need = memra_decode_attn_workspace_bytes(batch, q_len, n_heads, head_dim, max_seq_len);
  if (need > MEMRA_NOALLOC_SCRATCH_BYTES) return MEMRA_ERR_WORKSPACE;
  void *scratch = nullptr;
  if (batch > 0) {
    const int st = scratch_on_current_device(&scratch);
    if (st != MEMRA_OK) return st;
  }
  return memra_decode_attn(cache, q, page_table, max_pages_per_seq, seq_lens, max_seq_len, batch, q_len, n_heads,
                           n_kv_heads, head_dim, sm_scale, scratch, MEMRA_NOALLOC_SCRATCH_BYTES, out, stream);
}
