// Internal host interface between the C ABI (pa_api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pa.h"

// Decode kernel shape: warps per CTA and shared-memory stages per warp.
#ifndef PA_DECODE_WARPS
#define PA_DECODE_WARPS 8
#endif
#ifndef PA_DECODE_STAGES
#define PA_DECODE_STAGES 2
#endif
// Shortest range of the even split, in blocks.
#ifndef PA_DECODE_MIN_RANGE
#define PA_DECODE_MIN_RANGE 2
#endif

namespace pa {

// Decode limits: sequences per call (their block-count prefix lives in shared memory) and
// warps of the persistent grid (bounds the partial slots the workspace must hold).
constexpr int kMaxDecodeSeqs = 8192;
constexpr int kMaxDecodeWarps = 2048;
// KV heads per layer (the decode kernel packs the KV head index into 16 bits of a job word).
constexpr int kMaxKvHeads = 4096;

struct RopeArgs {
  __nv_bfloat16* q;                 // [T][Hq][128], rotated in place
  const __nv_bfloat16* k;           // [T][Hkv][128]
  const __nv_bfloat16* v;           // [T][Hkv][128]
  const int32_t* positions;         // [T]
  const float* cos_sin;             // [max_pos][128]
  const int64_t* slot_mapping;      // [T]
  __nv_bfloat16* k_cache;           // [num_blocks][Hkv][16][128]
  __nv_bfloat16* v_cache;
  int num_tokens, num_q_heads, num_kv_heads, max_pos, num_blocks;
  unsigned* status;                 // device status word
  // E4M3 caches (k_scale == nullptr for bf16): the caches hold one-byte codes.
  const float* k_scale;             // [Hkv]
  const float* v_scale;             // [Hkv]
};

struct DecodeArgs {
  const __nv_bfloat16* q;           // [S][Hq][128]
  const __nv_bfloat16* k_cache;     // [num_blocks][Hkv][16][128]
  const __nv_bfloat16* v_cache;
  const int32_t* block_tables;      // [S][max_blocks]
  const int32_t* context_lens;      // [S]
  __nv_bfloat16* out;               // [S][Hq][128]
  float* ws_o;                      // [slots][G][128]  partial sum_t p_t V_t of each piece
  float2* ws_ml;                    // [slots][G]       partial (max, sum p), log2 domain
  int num_seqs, num_q_heads, num_kv_heads, num_blocks, max_blocks, max_context_len;
  int chunk_blocks;                 // 0, or P / 16: no piece spans a P-token partition boundary
  int max_parts;                    // partitions of the longest segment (1 without partitions)
  int num_warps;                    // warps of the partition kernel's grid (set at launch)
  float scale_log2;                 // softmax scale * log2(e)
  unsigned* status;
  // Fused step only (k_new == nullptr for plain decode): q above is NOT yet rotated, and
  // each sequence's new token -- position context_len - 1, the last slot of its context --
  // is rotated and stored by the kernel that reads that slot's block.
  const __nv_bfloat16* k_new;       // [S][Hkv][128]
  const __nv_bfloat16* v_new;       // [S][Hkv][128]
  const float* cos_sin;             // [max_pos][128]
  int max_pos;
  __nv_bfloat16* k_store;           // the caches again, writable: destination of the new token
  __nv_bfloat16* v_store;
  // E4M3 caches (k_scale == nullptr for bf16): the caches hold one-byte codes, element =
  // code * scale of its KV head.
  const float* k_scale;             // [Hkv]
  const float* v_scale;             // [Hkv]
  // Lengths and block table are read before the preceding kernel on the stream has finished
  // (the caller's promise that it writes neither).
  int early_metadata;
  // Gather checksum only: [S][Hkv] words that each (sequence, KV head)'s tile words are XORed
  // into.
  uint32_t* gather_xor;
};

// Whole-block copies between pools (copy-on-write, swap out / in).  Pool pointers are device
// addresses (of device memory or of page-locked host memory).
struct BlockCopyArgs {
  const uint4* src[PA_MAX_BLOCK_CACHES];
  uint4* dst[PA_MAX_BLOCK_CACHES];
  const int64_t* pairs;             // [num_pairs][2] (from, to)
  long long src_blocks, dst_blocks;
  int num_pairs, num_caches;
  int tiles_per_block;              // Hkv: 4 KiB (block, KV head) tiles per block of one cache
  unsigned* status;
};

// Paged (chunked) prefill: q [num_tokens][Hq][128], sequence s owns rows
// q_start[s] .. q_start[s+1] - 1, query i of s at position context_lens[s] - n_s + i.
struct PrefillArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_cache;     // [num_blocks][Hkv][16][128]
  const __nv_bfloat16* v_cache;
  const int32_t* q_start;           // [S + 1]
  const int32_t* context_lens;      // [S]
  const int32_t* block_tables;      // [S][max_blocks]
  __nv_bfloat16* out;               // [num_tokens][Hq][128]
  int num_seqs, num_tokens, num_q_heads, num_kv_heads, num_blocks, max_blocks;
  int max_query_len, max_context_len;
  float scale_log2;
  unsigned* status;
};

// TMA tensor map of a paged cache viewed as [num_blocks * Hkv * 16][128], 128-byte swizzle;
// encoded once per (address, rows, type, box).  bf16: a 3-D view (64 columns, rows, 2 halves of
// 64 columns) whose box is 64 x 16 x box_halves (both halves of a tile: 4 KiB as two 2 KiB
// halves; or one half); E4M3: boxes of 128 x 16 bytes.
bool cache_tensor_map(const void* cache, long long rows, bool fp8, CUtensorMap* out, int box_halves = 2);

cudaError_t launch_rope_kv_store(const RopeArgs& a, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_copy_blocks(const BlockCopyArgs& a, cudaStream_t stream);
// n16 16-byte words from src to dst (device or page-locked host addresses the GPU can access)
cudaError_t launch_stage_copy(void* dst, const void* src, long long n16, cudaStream_t stream);
cudaError_t launch_wait_selftest(unsigned* status, uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
// The decode kernel's gather of K/V tiles alone (no attention, no merge): pa_gather_checksum,
// over bf16 or E4M3 (fp8) caches.
cudaError_t launch_gather(const DecodeArgs& a, bool fp8, cudaStream_t stream);

}  // namespace pa
