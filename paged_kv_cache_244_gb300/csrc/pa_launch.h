// Internal host interface between the C ABI (pa_api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace pa {

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
};

struct DecodeArgs {
  const __nv_bfloat16* q;           // [S][Hq][128]
  const __nv_bfloat16* k_cache;     // [num_blocks][Hkv][16][128]
  const __nv_bfloat16* v_cache;
  const int32_t* block_tables;      // [S][max_blocks]
  const int32_t* context_lens;      // [S]
  __nv_bfloat16* out;               // [S][Hq][128]
  float* ws_o;                      // [S][Hq][max_parts][128]   partial sum_t p_t V_t
  float2* ws_ml;                    // [S][Hq][max_parts]        partial (max, sum p) log2 domain
  int num_seqs, num_q_heads, num_kv_heads, num_blocks, max_blocks, max_context_len;
  int partition_tokens, max_parts;
  float scale_log2;                 // softmax scale * log2(e)
  unsigned* status;
};

cudaError_t launch_rope_kv_store(const RopeArgs& a, cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

}  // namespace pa
