// pa_decode_static_workspace: pa_decode without any device allocation by the caller.
//
// For callers that cannot allocate device memory during a decode step (all free HBM already
// given to the KV-cache pool, plugin enqueue paths that forbid allocation, real-time loops
// that must not take allocator locks).  The Flash-Decode partials go to a scratch array
// compiled into this library instead of a caller-provided workspace; the call then runs the
// ordinary pa_decode path on it.  Nothing here allocates.

#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "pa.h"

namespace {

// Held by every GPU that loads the library, until the process exits.  Shared by all calls on
// a device: calls whose kernels overlap on the GPU race on it.
static __device__ __align__(256) unsigned char g_pa_static_workspace[PA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;

// Device address of this GPU's scratch array.  In host code the array's name is only a
// host-side stand-in, so the address is looked up once per device, with that device current.
int scratch_address(void** out) {
  static std::mutex mu;
  static void* cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pa_static_workspace) != cudaSuccess || !p) return PA_ERR_CUDA;
    cache[dev] = p;
  }
  *out = cache[dev];
  return PA_OK;
}

}  // namespace

extern "C" int pa_decode_static_workspace(const pa_dims* dims, int num_seqs, const void* q,
                                          const void* k_cache, const void* v_cache,
                                          int num_blocks, const int32_t* block_tables,
                                          int max_blocks, const int32_t* context_lens,
                                          int max_context_len, float scale,
                                          int partition_tokens, void* out, void* stream) {
  // 0 when the arguments are invalid; pa_decode then reports the invalid argument itself.
  const size_t need = pa_decode_workspace_size(dims, num_seqs, max_context_len, partition_tokens);
  if (need > PA_STATIC_WORKSPACE_BYTES) return PA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    if (const int rc = scratch_address(&scratch)) return rc;
  }
  return pa_decode(dims, num_seqs, q, k_cache, v_cache, num_blocks, block_tables, max_blocks,
                   context_lens, max_context_len, scale, partition_tokens, scratch,
                   need > 0 ? PA_STATIC_WORKSPACE_BYTES : 0, out, stream);
}
