// C ABI of the paged decode attention library (declared in include/pa.h).
//
// Host side only: argument checks that need no device access, workspace sizing and carving,
// the device status word, and the kernel launches.  Nothing here allocates device memory.

#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "pa.h"
#include "pa_launch.h"

namespace {

// One status word per GPU that loads the library: kernels OR PA_FLAG_* bits into it.
__device__ unsigned int g_pa_status;

constexpr int kMaxDevices = 64;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dims(const pa_dims* d) {
  if (!d) return PA_ERR_NULL;
  if (d->head_dim != 128 || d->block_size != 16) return PA_ERR_SHAPE;
  if (d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->num_kv_heads > pa::kMaxKvHeads) return PA_ERR_SHAPE;
  if (d->num_q_heads % d->num_kv_heads != 0) return PA_ERR_SHAPE;
  const int G = d->num_q_heads / d->num_kv_heads;
  if (G < 1 || G > 8) return PA_ERR_SHAPE;
  return PA_OK;
}

// Validate a partition request: 0 (even split over the warps) or a positive multiple of the
// block size.  Returns it, or a negative PA_ERR_* code.
int check_partition(const pa_dims* d, int num_seqs, int max_context_len, int requested) {
  if (const int rc = check_dims(d)) return rc;
  if (num_seqs < 0 || num_seqs > pa::kMaxDecodeSeqs || max_context_len < 1) return PA_ERR_RANGE;
  if (requested < 0 || requested % d->block_size != 0) return PA_ERR_RANGE;
  return requested;
}

// Partitions of the longest segment: ceil(ceil(max_context_len / 16) / (P / 16)), 1 for P = 0.
long long max_parts_for(const pa_dims* d, int max_context_len, int partition_tokens) {
  if (partition_tokens <= 0) return 1;
  const long long blocks = (max_context_len + d->block_size - 1) / d->block_size;
  const long long chunk = partition_tokens / d->block_size;
  return (blocks + chunk - 1) / chunk;
}

// Partial rows: every piece of a split segment owns a slot of G rows, and slots stay below
// V + (#segments) * max_parts, with V <= min(ceil(J / PA_DECODE_MIN_RANGE), kMaxDecodeWarps)
// the ranges of the even split (J = jobs).  Each row is D partial sums plus a (shift, sum)
// pair.  0 when the rows would not fit in an int.
size_t workspace_bytes_for(const pa_dims* d, int num_seqs, int max_context_len, int partition_tokens) {
  const long long segs = static_cast<long long>(num_seqs) * d->num_kv_heads;
  const long long jobs = segs * ((max_context_len + d->block_size - 1) / d->block_size);
  if (jobs > 0x7fffffffll) return 0;  // positions on the job axis are 32-bit in the kernels
  long long ranges = (jobs + PA_DECODE_MIN_RANGE - 1) / PA_DECODE_MIN_RANGE;
  if (ranges > pa::kMaxDecodeWarps) ranges = pa::kMaxDecodeWarps;
  const long long rows = (ranges + segs * max_parts_for(d, max_context_len, partition_tokens)) *
                         (d->num_q_heads / d->num_kv_heads);
  if (rows > 0x7fffffffll) return 0;
  return static_cast<size_t>(rows) * (static_cast<size_t>(d->head_dim) + 2) * sizeof(float);
}

// Device address of this GPU's status word (looked up once per device).
int status_word(unsigned** out) {
  static std::mutex mu;
  static unsigned* cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pa_status) != cudaSuccess) return PA_ERR_CUDA;
    cache[dev] = static_cast<unsigned*>(p);
  }
  *out = cache[dev];
  return PA_OK;
}

// Checks shared by pa_decode and pa_decode_step, and the decode arguments they launch with
// (the fused-step fields left empty).  PA_OK with num_seqs == 0 means "nothing to do".
int decode_args(const pa_dims* dims, int num_seqs, const void* q, const void* k_cache,
                const void* v_cache, int num_blocks, const int32_t* block_tables, int max_blocks,
                const int32_t* context_lens, int max_context_len, float scale, int partition_tokens,
                void* workspace, size_t workspace_bytes, void* out, pa::DecodeArgs* a) {
  if (const int rc = check_dims(dims)) return rc;
  if (num_seqs < 0 || num_seqs > pa::kMaxDecodeSeqs) return PA_ERR_RANGE;
  if (num_seqs == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PA_ERR_NULL;
  if (num_blocks < 1 || max_blocks < 1 || max_context_len < 1) return PA_ERR_RANGE;
  if (static_cast<long long>(max_context_len) > static_cast<long long>(max_blocks) * dims->block_size)
    return PA_ERR_RANGE;
  if (static_cast<long long>(num_blocks) * dims->num_kv_heads * dims->block_size > (1ll << 31))
    return PA_ERR_RANGE;
  if (!(scale > 0.f) || !std::isfinite(scale)) return PA_ERR_RANGE;
  const int P = check_partition(dims, num_seqs, max_context_len, partition_tokens);
  if (P < 0) return P;
  const size_t need = workspace_bytes_for(dims, num_seqs, max_context_len, P);
  if (need == 0) return PA_ERR_RANGE;
  if (!workspace || workspace_bytes < need) return PA_ERR_WORKSPACE;
  const void* ptrs[] = {q, k_cache, v_cache, block_tables, context_lens, out, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return PA_ERR_ALIGN;
  unsigned* status = nullptr;
  if (const int rc = status_word(&status)) return rc;

  a->q = static_cast<const __nv_bfloat16*>(q);
  a->k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  a->v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  a->block_tables = block_tables;
  a->context_lens = context_lens;
  a->out = static_cast<__nv_bfloat16*>(out);
  // [rows][D] partial sums, then [rows] (max, sum) pairs; rows = need / ((D + 2) * 4).
  float* ws = static_cast<float*>(workspace);
  const size_t rows = need / ((static_cast<size_t>(dims->head_dim) + 2) * sizeof(float));
  a->ws_o = ws;
  a->ws_ml = reinterpret_cast<float2*>(ws + rows * dims->head_dim);
  a->num_seqs = num_seqs;
  a->num_q_heads = dims->num_q_heads;
  a->num_kv_heads = dims->num_kv_heads;
  a->num_blocks = num_blocks;
  a->max_blocks = max_blocks;
  a->max_context_len = max_context_len;
  a->chunk_blocks = P / dims->block_size;
  a->max_parts = static_cast<int>(max_parts_for(dims, max_context_len, P));
  a->num_warps = 0;  // set by the launcher from the grid it picks
  a->scale_log2 = scale * 1.4426950408889634f;
  a->status = status;
  a->k_new = nullptr;
  a->v_new = nullptr;
  a->cos_sin = nullptr;
  a->max_pos = 0;
  a->k_store = nullptr;
  a->v_store = nullptr;
  a->k_scale = nullptr;
  a->v_scale = nullptr;
  return PA_OK;
}

// Device address of a pointer the current GPU can dereference: its own memory, managed
// memory or page-locked host memory.  PA_ERR_MEMORY for anything else.
int device_address(const void* p, const void** out) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();  // clear the (non-sticky) error the failed query recorded
    return PA_ERR_MEMORY;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  switch (attr.type) {
    case cudaMemoryTypeDevice:
      if (attr.device != dev) return PA_ERR_MEMORY;
      *out = attr.devicePointer;
      return *out ? PA_OK : PA_ERR_MEMORY;
    case cudaMemoryTypeManaged:
    case cudaMemoryTypeHost:
      *out = attr.devicePointer;
      return *out ? PA_OK : PA_ERR_MEMORY;
    default:
      return PA_ERR_MEMORY;
  }
}

// pa_rope_kv_store and its E4M3 form (scales non-null).
int rope_store(const pa_dims* dims, int num_tokens, void* q, const void* k, const void* v,
               const int32_t* positions, const float* cos_sin, int max_pos,
               const int64_t* slot_mapping, void* k_cache, void* v_cache, int num_blocks,
               const float* k_scale, const float* v_scale, void* stream) {
  if (const int rc = check_dims(dims)) return rc;
  if (num_tokens < 0) return PA_ERR_RANGE;
  if (num_tokens == 0) return PA_OK;
  if (!q || !k || !v || !positions || !cos_sin || !slot_mapping || !k_cache || !v_cache)
    return PA_ERR_NULL;
  if (max_pos < 1 || num_blocks < 1) return PA_ERR_RANGE;
  const void* ptrs[] = {q, k, v, positions, cos_sin, slot_mapping, k_cache, v_cache};
  for (const void* p : ptrs)
    if (!aligned16(p)) return PA_ERR_ALIGN;
  unsigned* status = nullptr;
  if (const int rc = status_word(&status)) return rc;
  pa::RopeArgs a{};
  a.q = static_cast<__nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.positions = positions;
  a.cos_sin = cos_sin;
  a.slot_mapping = slot_mapping;
  a.k_cache = static_cast<__nv_bfloat16*>(k_cache);
  a.v_cache = static_cast<__nv_bfloat16*>(v_cache);
  a.num_tokens = num_tokens;
  a.num_q_heads = dims->num_q_heads;
  a.num_kv_heads = dims->num_kv_heads;
  a.max_pos = max_pos;
  a.num_blocks = num_blocks;
  a.status = status;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  return pa::launch_rope_kv_store(a, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

// pa_decode_step and its E4M3 form (scales non-null).
int decode_step(const pa_dims* dims, int num_seqs, const void* q, const void* k, const void* v,
                const float* cos_sin, int max_pos, void* k_cache, void* v_cache,
                const float* k_scale, const float* v_scale, int num_blocks,
                const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                int max_context_len, float scale, int partition_tokens, void* workspace,
                size_t workspace_bytes, void* out, unsigned flags, void* stream) {
  // The new token's arguments first (host checks only), then everything pa_decode checks.
  if (const int rc = check_dims(dims)) return rc;
  if (flags & ~PA_STEP_EARLY_METADATA) return PA_ERR_RANGE;
  if (num_seqs < 0 || num_seqs > pa::kMaxDecodeSeqs) return PA_ERR_RANGE;
  if (num_seqs == 0) return PA_OK;
  if (!k || !v || !cos_sin) return PA_ERR_NULL;
  if (max_pos < 1) return PA_ERR_RANGE;
  if (!aligned16(k) || !aligned16(v) || !aligned16(cos_sin)) return PA_ERR_ALIGN;
  pa::DecodeArgs a{};
  const int rc = decode_args(dims, num_seqs, q, k_cache, v_cache, num_blocks, block_tables, max_blocks,
                             context_lens, max_context_len, scale, partition_tokens, workspace,
                             workspace_bytes, out, &a);
  if (rc != PA_OK) return rc;
  a.k_new = static_cast<const __nv_bfloat16*>(k);
  a.v_new = static_cast<const __nv_bfloat16*>(v);
  a.cos_sin = cos_sin;
  a.max_pos = max_pos;
  a.k_store = static_cast<__nv_bfloat16*>(k_cache);
  a.v_store = static_cast<__nv_bfloat16*>(v_cache);
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.early_metadata = (flags & PA_STEP_EARLY_METADATA) ? 1 : 0;
  return pa::launch_decode(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                 : PA_ERR_CUDA;
}

// Host checks of the E4M3 scale arrays (after the shape and count checks their callers share).
int scales_ok(const pa_dims* dims, int num_seqs, const float* k_scale, const float* v_scale) {
  if (const int rc = check_dims(dims)) return rc;
  if (num_seqs < 0 || num_seqs > pa::kMaxDecodeSeqs) return PA_ERR_RANGE;
  if (num_seqs == 0) return PA_OK;
  if (!k_scale || !v_scale) return PA_ERR_NULL;
  if (!aligned16(k_scale) || !aligned16(v_scale)) return PA_ERR_ALIGN;
  return PA_OK;
}

}  // namespace

extern "C" {

int pa_rope_kv_store(const pa_dims* dims, int num_tokens, void* q, const void* k, const void* v,
                     const int32_t* positions, const float* cos_sin, int max_pos,
                     const int64_t* slot_mapping, void* k_cache, void* v_cache, int num_blocks,
                     void* stream) {
  return rope_store(dims, num_tokens, q, k, v, positions, cos_sin, max_pos, slot_mapping, k_cache,
                    v_cache, num_blocks, nullptr, nullptr, stream);
}

int pa_rope_kv_store_fp8(const pa_dims* dims, int num_tokens, void* q, const void* k,
                         const void* v, const int32_t* positions, const float* cos_sin,
                         int max_pos, const int64_t* slot_mapping, void* k_cache, void* v_cache,
                         int num_blocks, const float* k_scale, const float* v_scale, void* stream) {
  if (num_tokens > 0) {
    if (const int rc = check_dims(dims)) return rc;
    if (!k_scale || !v_scale) return PA_ERR_NULL;
    if (!aligned16(k_scale) || !aligned16(v_scale)) return PA_ERR_ALIGN;
  }
  return rope_store(dims, num_tokens, q, k, v, positions, cos_sin, max_pos, slot_mapping, k_cache,
                    v_cache, num_blocks, k_scale, v_scale, stream);
}

int pa_decode_partition_tokens(const pa_dims* dims, int num_seqs, int max_context_len,
                               int partition_tokens) {
  return check_partition(dims, num_seqs, max_context_len, partition_tokens);
}

size_t pa_decode_workspace_size(const pa_dims* dims, int num_seqs, int max_context_len,
                                int partition_tokens) {
  const int P = check_partition(dims, num_seqs, max_context_len, partition_tokens);
  if (P < 0 || num_seqs == 0) return 0;
  return workspace_bytes_for(dims, num_seqs, max_context_len, P);
}

int pa_decode(const pa_dims* dims, int num_seqs, const void* q, const void* k_cache,
              const void* v_cache, int num_blocks, const int32_t* block_tables, int max_blocks,
              const int32_t* context_lens, int max_context_len, float scale,
              int partition_tokens, void* workspace, size_t workspace_bytes, void* out,
              void* stream) {
  pa::DecodeArgs a{};
  const int rc = decode_args(dims, num_seqs, q, k_cache, v_cache, num_blocks, block_tables, max_blocks,
                             context_lens, max_context_len, scale, partition_tokens, workspace,
                             workspace_bytes, out, &a);
  if (rc != PA_OK || num_seqs == 0) return rc;
  return pa::launch_decode(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                 : PA_ERR_CUDA;
}

namespace {

int gather_checksum(const pa_dims* dims, int num_seqs, const void* k_cache, const void* v_cache,
                    int num_blocks, const int32_t* block_tables, int max_blocks,
                    const int32_t* context_lens, int max_context_len, uint32_t* out_xor, bool fp8,
                    void* stream) {
  if (const int rc = check_dims(dims)) return rc;
  if (num_seqs < 0 || num_seqs > pa::kMaxDecodeSeqs) return PA_ERR_RANGE;
  if (num_seqs == 0) return PA_OK;
  if (!k_cache || !v_cache || !block_tables || !context_lens || !out_xor) return PA_ERR_NULL;
  if (num_blocks < 1 || max_blocks < 1 || max_context_len < 1) return PA_ERR_RANGE;
  if (static_cast<long long>(max_context_len) > static_cast<long long>(max_blocks) * dims->block_size)
    return PA_ERR_RANGE;
  if (static_cast<long long>(num_blocks) * dims->num_kv_heads * dims->block_size > (1ll << 31))
    return PA_ERR_RANGE;
  if (static_cast<long long>(num_seqs) * dims->num_kv_heads *
          ((max_context_len + dims->block_size - 1) / dims->block_size) > 0x7fffffffll)
    return PA_ERR_RANGE;
  const void* ptrs[] = {k_cache, v_cache, block_tables, context_lens};
  for (const void* p : ptrs)
    if (!aligned16(p)) return PA_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(out_xor) % 4 != 0) return PA_ERR_ALIGN;
  unsigned* status = nullptr;
  if (const int rc = status_word(&status)) return rc;
  pa::DecodeArgs a{};
  a.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  a.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.num_q_heads = dims->num_q_heads;
  a.num_kv_heads = dims->num_kv_heads;
  a.num_blocks = num_blocks;
  a.max_blocks = max_blocks;
  a.max_context_len = max_context_len;
  a.chunk_blocks = 0;
  a.max_parts = 1;
  a.status = status;
  a.gather_xor = out_xor;
  return pa::launch_gather(a, fp8, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

int pa_gather_checksum(const pa_dims* dims, int num_seqs, const void* k_cache, const void* v_cache,
                       int num_blocks, const int32_t* block_tables, int max_blocks,
                       const int32_t* context_lens, int max_context_len, uint32_t* out_xor,
                       void* stream) {
  return gather_checksum(dims, num_seqs, k_cache, v_cache, num_blocks, block_tables, max_blocks,
                         context_lens, max_context_len, out_xor, false, stream);
}

int pa_gather_checksum_fp8(const pa_dims* dims, int num_seqs, const void* k_cache,
                           const void* v_cache, int num_blocks, const int32_t* block_tables,
                           int max_blocks, const int32_t* context_lens, int max_context_len,
                           uint32_t* out_xor, void* stream) {
  return gather_checksum(dims, num_seqs, k_cache, v_cache, num_blocks, block_tables, max_blocks,
                         context_lens, max_context_len, out_xor, true, stream);
}

int pa_decode_step(const pa_dims* dims, int num_seqs, const void* q, const void* k, const void* v,
                   const float* cos_sin, int max_pos, void* k_cache, void* v_cache, int num_blocks,
                   const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                   int max_context_len, float scale, int partition_tokens, void* workspace,
                   size_t workspace_bytes, void* out, unsigned flags, void* stream) {
  return decode_step(dims, num_seqs, q, k, v, cos_sin, max_pos, k_cache, v_cache, nullptr, nullptr,
                     num_blocks, block_tables, max_blocks, context_lens, max_context_len, scale,
                     partition_tokens, workspace, workspace_bytes, out, flags, stream);
}

int pa_decode_step_fp8(const pa_dims* dims, int num_seqs, const void* q, const void* k,
                       const void* v, const float* cos_sin, int max_pos, void* k_cache,
                       void* v_cache, const float* k_scale, const float* v_scale, int num_blocks,
                       const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                       int max_context_len, float scale, int partition_tokens, void* workspace,
                       size_t workspace_bytes, void* out, unsigned flags, void* stream) {
  if (const int rc = scales_ok(dims, num_seqs, k_scale, v_scale)) return rc;
  return decode_step(dims, num_seqs, q, k, v, cos_sin, max_pos, k_cache, v_cache, k_scale, v_scale,
                     num_blocks, block_tables, max_blocks, context_lens, max_context_len, scale,
                     partition_tokens, workspace, workspace_bytes, out, flags, stream);
}

int pa_decode_fp8(const pa_dims* dims, int num_seqs, const void* q, const void* k_cache,
                  const void* v_cache, const float* k_scale, const float* v_scale, int num_blocks,
                  const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                  int max_context_len, float scale, int partition_tokens, void* workspace,
                  size_t workspace_bytes, void* out, void* stream) {
  if (const int rc = scales_ok(dims, num_seqs, k_scale, v_scale)) return rc;
  pa::DecodeArgs a{};
  const int rc = decode_args(dims, num_seqs, q, k_cache, v_cache, num_blocks, block_tables, max_blocks,
                             context_lens, max_context_len, scale, partition_tokens, workspace,
                             workspace_bytes, out, &a);
  if (rc != PA_OK || num_seqs == 0) return rc;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  return pa::launch_decode(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                 : PA_ERR_CUDA;
}

int pa_prefill(const pa_dims* dims, int num_seqs, int num_tokens, const void* q,
               const int32_t* q_start, int max_query_len, const void* k_cache,
               const void* v_cache, int num_blocks, const int32_t* block_tables, int max_blocks,
               const int32_t* context_lens, int max_context_len, float scale, void* out,
               void* stream) {
  if (const int rc = check_dims(dims)) return rc;
  if (num_seqs < 0 || num_tokens < 0) return PA_ERR_RANGE;
  if (num_seqs == 0 || num_tokens == 0) return PA_OK;
  if (!q || !q_start || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return PA_ERR_NULL;
  if (num_blocks < 1 || max_blocks < 1 || max_context_len < 1 || max_query_len < 1) return PA_ERR_RANGE;
  if (max_query_len > max_context_len) return PA_ERR_RANGE;
  if (static_cast<long long>(max_context_len) > static_cast<long long>(max_blocks) * dims->block_size)
    return PA_ERR_RANGE;
  if (static_cast<long long>(num_blocks) * dims->num_kv_heads * dims->block_size > (1ll << 31))
    return PA_ERR_RANGE;
  if (static_cast<long long>(num_seqs) * dims->num_kv_heads > 65535) return PA_ERR_RANGE;
  if (!(scale > 0.f) || !std::isfinite(scale)) return PA_ERR_RANGE;
  const void* ptrs[] = {q, q_start, k_cache, v_cache, block_tables, context_lens, out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return PA_ERR_ALIGN;
  unsigned* status = nullptr;
  if (const int rc = status_word(&status)) return rc;
  pa::PrefillArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  a.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  a.q_start = q_start;
  a.context_lens = context_lens;
  a.block_tables = block_tables;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.num_seqs = num_seqs;
  a.num_tokens = num_tokens;
  a.num_q_heads = dims->num_q_heads;
  a.num_kv_heads = dims->num_kv_heads;
  a.num_blocks = num_blocks;
  a.max_blocks = max_blocks;
  a.max_query_len = max_query_len;
  a.max_context_len = max_context_len;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status;
  return pa::launch_prefill(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                   : PA_ERR_CUDA;
}

int pa_copy_blocks(const pa_dims* dims, int num_caches, const void* const* src_caches,
                   int64_t src_num_blocks, void* const* dst_caches, int64_t dst_num_blocks,
                   const int64_t* block_pairs, int num_pairs, void* stream) {
  if (const int rc = check_dims(dims)) return rc;
  if (num_pairs < 0) return PA_ERR_RANGE;
  if (num_pairs == 0) return PA_OK;
  if (num_caches < 1 || num_caches > PA_MAX_BLOCK_CACHES) return PA_ERR_RANGE;
  if (src_num_blocks < 1 || dst_num_blocks < 1) return PA_ERR_RANGE;
  if (!src_caches || !dst_caches || !block_pairs) return PA_ERR_NULL;
  for (int c = 0; c < num_caches; ++c) {
    if (!src_caches[c] || !dst_caches[c]) return PA_ERR_NULL;
    if (!aligned16(src_caches[c]) || !aligned16(dst_caches[c])) return PA_ERR_ALIGN;
  }
  if (reinterpret_cast<uintptr_t>(block_pairs) % alignof(int64_t) != 0) return PA_ERR_ALIGN;
  unsigned* status = nullptr;
  if (const int rc = status_word(&status)) return rc;
  pa::BlockCopyArgs a{};
  for (int c = 0; c < num_caches; ++c) {
    const void* s = nullptr;
    const void* d = nullptr;
    if (const int rc = device_address(src_caches[c], &s)) return rc;
    if (const int rc = device_address(dst_caches[c], &d)) return rc;
    a.src[c] = static_cast<const uint4*>(s);
    a.dst[c] = static_cast<uint4*>(const_cast<void*>(d));
  }
  const void* pairs = nullptr;
  if (const int rc = device_address(block_pairs, &pairs)) return rc;
  a.pairs = static_cast<const int64_t*>(pairs);
  a.src_blocks = src_num_blocks;
  a.dst_blocks = dst_num_blocks;
  a.num_pairs = num_pairs;
  a.num_caches = num_caches;
  a.tiles_per_block = dims->num_kv_heads;
  a.status = status;
  return pa::launch_copy_blocks(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                     : PA_ERR_CUDA;
}

int pa_stage_copy(void* dst, const void* src, size_t bytes, void* stream) {
  if (bytes == 0) return PA_OK;
  if (!dst || !src) return PA_ERR_NULL;
  if (!aligned16(dst) || !aligned16(src) || bytes % 16 != 0) return PA_ERR_ALIGN;
  const void* d = nullptr;
  const void* s = nullptr;
  if (const int rc = device_address(dst, &d)) return rc;
  if (const int rc = device_address(src, &s)) return rc;
  return pa::launch_stage_copy(const_cast<void*>(d), s, static_cast<long long>(bytes / 16),
                               static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

int pa_get_device_status(void* stream, uint32_t* flags) {
  unsigned* status = nullptr;
  if (const int rc = status_word(&status)) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned host = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaMemcpy(&host, status, sizeof host, cudaMemcpyDeviceToHost) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaMemset(status, 0, sizeof host) != cudaSuccess) return PA_ERR_CUDA;
  if (flags) *flags = host;
  if (host & PA_FLAG_TIMEOUT) return PA_ERR_TIMEOUT;
  if (host) return PA_ERR_DEVICE_OOB;
  return PA_OK;
}

int pa_selftest_wait_timeout(uint32_t limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return PA_ERR_RANGE;
  unsigned* status = nullptr;
  if (const int rc = status_word(&status)) return rc;
  return pa::launch_wait_selftest(status, static_cast<uint64_t>(limit_us) * 1000ull,
                                  static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_NULL: return "PA_ERR_NULL: a required pointer is NULL";
    case PA_ERR_SHAPE: return "PA_ERR_SHAPE: unsupported head_dim, block_size or head counts";
    case PA_ERR_RANGE: return "PA_ERR_RANGE: a count or length is out of range";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing or too small";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: a CUDA runtime call failed";
    case PA_ERR_DEVICE_OOB: return "PA_ERR_DEVICE_OOB: a kernel met an out-of-range value";
    case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT: a kernel gave up a bounded wait";
    case PA_ERR_ALIGN: return "PA_ERR_ALIGN: a pointer is not 16-byte aligned";
    case PA_ERR_MEMORY: return "PA_ERR_MEMORY: a pointer is not memory this GPU can address";
    default: return "unknown pa status";
  }
}

}  // extern "C"
