/*
 * pa.h -- paged GQA decode attention and the fused RoPE + KV-cache store, as a C ABI.
 *
 * Library: paged_kv_cache_244_gb300/libpa_gb300.so (CUDA, sm_103a).  Plain C: no CUDA,
 * C++ or framework types appear here.  Streams are passed as `void*` and are CUDA stream
 * handles (cudaStream_t); NULL means the legacy default stream.
 *
 * The operations follow these passages (page title, section):
 *   [PV]  "Pico-vLLM：从零手写的工业级LLM推理引擎实现"
 *         §1 模型实现层: RoPE computed with rotate_half in place; GQA, where groups of query
 *            heads share one KV head.
 *         §2 Kernel层: the PagedAttention prefill and decode kernels (new tokens attend over
 *            their cached context) and the fused RoPE + KV cache store.
 *         §H200上的详细对比: Flash Decode, i.e. the context split into partitions whose
 *            partial softmax results are merged.
 *   [NV]  "nano-vllm：vLLM 极简实现与大模型推理流程解析"
 *         §学习要点: FP8 / INT4 quantisation cuts memory with almost no loss of accuracy.
 *   [15x] "从零实现15倍加速：一个纯PyTorch LLM推理引擎的技术剖析"
 *         §未来展望: INT8 / FP16 quantisation to save memory and bandwidth.
 *   [ME]  "从零实现 LLM 推理引擎：深挖 vLLM 的六大核心优化"
 *         §3.1 Paged KV Cache: the cache is made of fixed blocks of 16 tokens, and each
 *            sequence has a block_table mapping logical block index -> physical block id.
 *         §3.2 Continuous Batching: append_slot gives every running sequence one new slot
 *            per decode step.
 *         §3.3 Chunked Prefill: a long prompt is prefilled a chunk at a time, each chunk
 *            continuing from the tokens already prefilled.
 *         §3.4 Prefix Caching: blocks shared between sequences are reference counted and
 *            copied before a write (copy-on-write), so the block a new token goes to is
 *            never shared.
 *         §3.5 CPU Swap: swap_out moves a preempted sequence's KV blocks to CPU memory and
 *            swap_in restores them into newly allocated GPU blocks.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Element types: q, k, v, caches and out are bf16 (16-bit, passed as void*).  cos_sin is
 *    fp32.  All arithmetic inside is fp32 with fp32 accumulation.
 *  - Layouts are dense row-major, with no strides:
 *      q            [num_tokens or num_seqs][num_q_heads][head_dim]
 *      k, v         [num_tokens][num_kv_heads][head_dim]
 *      k_cache,
 *      v_cache      [num_blocks][num_kv_heads][block_size][head_dim]   ("HND" blocks)
 *      cos_sin      [max_pos][head_dim] fp32: row p = cos(p*w_0..w_{D/2-1}) | sin(...)
 *      block_tables [num_seqs][max_blocks] int32 physical block ids
 *      out          [num_seqs][num_q_heads][head_dim]
 *    With block_size 16 and head_dim 128 each (block, KV head) tile is 4 KiB contiguous.
 *  - Slot of a token: physical_block * block_size + offset_in_block.
 *  - Supported shape: head_dim == 128, block_size == 16, num_kv_heads <= 4096,
 *    num_q_heads a multiple of num_kv_heads with group size num_q_heads / num_kv_heads in
 *    [1, 8].  Anything else returns PA_ERR_SHAPE.
 *  - Memory: every pointer is device memory owned by the caller (cudaMalloc, PyTorch, ...)
 *    and must be 16-byte aligned (PA_ERR_ALIGN otherwise).  The library allocates nothing.
 *    Its only global state is one 32-bit device status word per GPU, and the fixed scratch
 *    array of pa_decode_static_workspace (PA_STATIC_WORKSPACE_BYTES per GPU).
 *  - Host-side caches: per GPU, the library looks up the device addresses of its globals (the
 *    status word, the static scratch) and sets its kernels' shared-memory attributes once, and
 *    keeps the TMA descriptors it encodes for each cache pointer; all live for the process.  A
 *    cudaDeviceReset (or anything else that destroys the device's primary context) makes them
 *    stale: do not call the library on a device after resetting it.
 *  - Asynchrony: calls enqueue work on `stream` and return at once.  Arguments the host can
 *    check are checked before anything is enqueued; on error nothing is launched.
 *  - Values only the device can see (block ids, positions, slots, per-sequence lengths) are
 *    checked by the kernels: an out-of-range one is skipped (never dereferenced) and a flag
 *    is raised in the device status word; read it with pa_get_device_status().
 *  - Kernels launch with programmatic dependent launch: they wait for the previous kernel
 *    on the stream before reading any input, so ordinary stream order holds.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_dims {
  int32_t num_q_heads;   /* Hq, e.g. 12 */
  int32_t num_kv_heads;  /* Hkv, e.g. 2; GQA group G = Hq / Hkv */
  int32_t head_dim;      /* D, must be 128 */
  int32_t block_size;    /* tokens per cache block, must be 16 */
} pa_dims;

/* Return codes (negative = error, nothing was enqueued unless noted). */
enum {
  PA_OK = 0,
  PA_ERR_NULL = -1,        /* a required pointer is NULL */
  PA_ERR_SHAPE = -2,       /* unsupported head_dim / block_size / head counts */
  PA_ERR_RANGE = -3,       /* a count or length is out of range */
  PA_ERR_WORKSPACE = -4,   /* workspace missing or smaller than pa_decode_workspace_size */
  PA_ERR_CUDA = -5,        /* a CUDA runtime call failed (the launch itself, or a query) */
  PA_ERR_DEVICE_OOB = -6,  /* pa_get_device_status: a kernel met an out-of-range value */
  PA_ERR_TIMEOUT = -7,     /* pa_get_device_status: a kernel gave up a bounded wait */
  PA_ERR_ALIGN = -8,       /* a pointer is not 16-byte aligned */
  PA_ERR_MEMORY = -9       /* a pointer is not memory the device can address (pageable host
                              memory, or another GPU's memory) */
};

/* Flags of the device status word (bitwise OR of everything seen since the last read). */
#define PA_FLAG_BLOCK_ID_OOB    0x1u  /* block_tables entry outside [0, num_blocks) */
#define PA_FLAG_CONTEXT_LEN_OOB 0x2u  /* context_lens[s] outside [0, max_context_len] */
#define PA_FLAG_SLOT_OOB        0x4u  /* slot_mapping[t] >= num_blocks * block_size */
#define PA_FLAG_POSITION_OOB    0x8u  /* positions[t] outside [0, max_pos) */
#define PA_FLAG_TIMEOUT         0x10u /* a copy into shared memory did not land in time */

/*
 * pa_rope_kv_store -- fused RoPE + KV-cache store for `num_tokens` new tokens
 * ([PV] §1 and §2: RoPE with rotate_half, fused with the KV cache store; [ME] §3.1/§3.2:
 * the token's K and V go to the slot append_slot gave it).
 *
 * For each token t with p = positions[t], (c_i, s_i) = cos_sin[p][i], cos_sin[p][D/2 + i]:
 *   every query head  q[t][h]:  q'[i] = q[i] c_i - q[i+D/2] s_i,  q'[i+D/2] = q[i+D/2] c_i + q[i] s_i
 *                               written back into q (IN PLACE), rounded to bf16 (RNE);
 *   every KV head g:            k_cache[slot][g] = rotate(k[t][g]) (same formula, bf16 RNE),
 *                               v_cache[slot][g] = v[t][g] (bit copy),
 *   where slot = slot_mapping[t] (block = slot / block_size, offset = slot % block_size).
 * A negative slot means "padding token": q is rotated, nothing is stored.
 * Device-side errors: p outside [0, max_pos) -> token skipped entirely (q left unrotated),
 * PA_FLAG_POSITION_OOB; slot >= num_blocks * block_size -> store skipped, PA_FLAG_SLOT_OOB.
 *
 *   dims          shape (see conventions)
 *   num_tokens    T >= 0 (0 is a no-op)
 *   q             [T][Hq][D] bf16, read and overwritten
 *   k, v          [T][Hkv][D] bf16, read only
 *   positions     [T] int32
 *   cos_sin       [max_pos][D] fp32, read only
 *   max_pos       rows of cos_sin, >= 1
 *   slot_mapping  [T] int64
 *   k_cache, v_cache  [num_blocks][Hkv][block_size][D] bf16, written at the slots only
 *   num_blocks    >= 1
 *   stream        CUDA stream
 * Returns PA_OK or a PA_ERR_* code (nothing launched on error).
 */
int pa_rope_kv_store(const pa_dims* dims, int num_tokens, void* q, const void* k, const void* v,
                     const int32_t* positions, const float* cos_sin, int max_pos,
                     const int64_t* slot_mapping, void* k_cache, void* v_cache, int num_blocks,
                     void* stream);

/*
 * pa_decode_partition_tokens -- validate a partition request for pa_decode (Flash Decode,
 * [PV] §H200上的详细对比).  pa_decode lays the (sequence, KV head, block) jobs of the batch
 * on one axis and cuts it into equal contiguous ranges, one per warp of its persistent grid
 * (every warp gets the same number of blocks +-1).  A sequence's blocks for one KV head are
 * computed in pieces: a piece ends at a range boundary, at the end of the sequence and, when
 * `partition_tokens` P > 0, at every P-token partition boundary, so that each P-token
 * partition yields its own partial softmax result (one piece, or more when range boundaries
 * fall inside it).  The pieces of a split sequence are then reduced by a second kernel
 * (log-sum-exp merge, in axis order).  P changes how the partial results are grouped, not how
 * the work is spread over the GPU.  Returns the request (0 or a positive multiple of
 * block_size) or a negative PA_ERR_* code (PA_ERR_RANGE also for num_seqs > 8192 or
 * max_context_len < 1).
 */
int pa_decode_partition_tokens(const pa_dims* dims, int num_seqs, int max_context_len,
                               int partition_tokens);

/*
 * pa_decode_workspace_size -- bytes of device workspace pa_decode needs for these
 * arguments: (R + num_seqs * Hkv * M) * (Hq / Hkv) * (D + 2) * 4, where R = min(2048,
 * ceil(J / 2)) bounds the ranges, J = num_seqs * Hkv * ceil(max_context_len / 16), and M = 1
 * for partition_tokens == 0, else ceil(ceil(max_context_len / 16) / (partition_tokens / 16)).
 * Returns 0 for invalid arguments (pa_decode then reports the error).
 */
size_t pa_decode_workspace_size(const pa_dims* dims, int num_seqs, int max_context_len,
                                int partition_tokens);

/*
 * pa_decode -- single-token paged GQA decode attention ([PV] §2: PagedAttention decode
 * kernel; [ME] §3.1: block tables; [PV] §1: GQA; [PV] §H200上的详细对比: Flash Decode).
 *
 * For each sequence s with n = context_lens[s] (the new token, already stored, included)
 * and each query head h, with g = h / (Hq / Hkv) and, for t < n,
 *   K_t = k_cache[block_tables[s][t / 16]][g][t % 16],  V_t likewise,
 *   out[s][h] = sum_t softmax_t(scale * q[s][h] . K_t) V_t      (bf16 RNE of the fp32 result)
 * Table entries past ceil(n / 16) and cache slots past n are never read.  n == 0 gives an
 * all-zero output row.  The work is split as pa_decode_partition_tokens describes; pieces
 * of a split sequence give partial (max, sum, weighted V) that a second kernel merges, and
 * the result is the same softmax up to fp32 rounding order.
 * Device-side errors: a block id outside [0, num_blocks) -> that block is skipped,
 * PA_FLAG_BLOCK_ID_OOB; n outside [0, max_context_len] -> clamped, PA_FLAG_CONTEXT_LEN_OOB.
 *
 *   num_seqs          0 <= S <= 8192 (0 is a no-op)
 *   q                 [S][Hq][D] bf16 (already rotated), read only
 *   k_cache, v_cache  [num_blocks][Hkv][16][D] bf16, read only
 *   block_tables      [S][max_blocks] int32
 *   context_lens      [S] int32 (device copy)
 *   max_context_len   host-side upper bound of context_lens, 1 <= it <= max_blocks * 16
 *   scale             softmax scale, finite and > 0 (1/sqrt(D) for standard attention)
 *   partition_tokens  0 (even split over the grid) or a positive multiple of 16
 *   workspace         device memory of >= pa_decode_workspace_size(...) bytes, 16-byte
 *                     aligned; its contents need no initialisation.  Two calls whose kernels
 *                     overlap on the GPU must not share a workspace.
 *   out               [S][Hq][D] bf16, written
 * Returns PA_OK or a PA_ERR_* code (nothing launched on error).  Launches one kernel, plus
 * one merge kernel.
 */
int pa_decode(const pa_dims* dims, int num_seqs, const void* q, const void* k_cache,
              const void* v_cache, int num_blocks, const int32_t* block_tables, int max_blocks,
              const int32_t* context_lens, int max_context_len, float scale,
              int partition_tokens, void* workspace, size_t workspace_bytes, void* out,
              void* stream);

/*
 * pa_decode_step -- one decode step of a layer in one launch: the RoPE + KV-cache store of
 * each sequence's new token fused into pa_decode ([PV] §2: RoPE fused with the KV cache
 * store, and the PagedAttention decode kernel; [ME] §3.2: the new token takes the next slot
 * of its sequence, which is the last slot of its context).
 *
 * The result equals pa_rope_kv_store followed by pa_decode with, for every sequence s with
 * n = context_lens[s] >= 1 (n counts the new token):
 *   positions[s]    = n - 1,
 *   slot_mapping[s] = block_tables[s][(n - 1) / 16] * 16 + (n - 1) % 16,
 * except that q is NOT modified: the kernel rotates its own copy of q in registers.  So:
 *   k_cache[slot][g] = rotate(k[s][g]) and v_cache[slot][g] = v[s][g], bit for bit what
 *   pa_rope_kv_store writes; out = pa_decode over the updated caches with the rotated q.
 * The block reached through block_tables[s][(n - 1) / 16] is read and written by this
 * sequence only: it must not appear in another sequence's table within its context (the
 * block of a sequence's newest token is never shared -- a shared block is copied before it
 * is written, [ME] §3.4 copy-on-write).  Within that block, the slots before n - 1 are read
 * and slot n - 1 is written by the same warp, in that order.
 * Sequences with n == 0 store nothing and get a zero output row.
 * Device-side errors: as pa_decode; and n - 1 >= max_pos -> that sequence's token is treated
 * as pa_rope_kv_store treats it (q used unrotated, nothing stored), PA_FLAG_POSITION_OOB.
 *
 *   q                 [S][Hq][D] bf16, NOT yet rotated, read only
 *   k, v              [S][Hkv][D] bf16, the new token's key and value, read only
 *   cos_sin, max_pos  as for pa_rope_kv_store
 *   k_cache, v_cache  [num_blocks][Hkv][16][D] bf16, read, and written at the new slots
 *   flags             0 or PA_STEP_EARLY_METADATA (below); other bits -> PA_ERR_RANGE
 *   everything else   as for pa_decode (same workspace size: pa_decode_workspace_size)
 * Returns PA_OK or a PA_ERR_* code (nothing launched on error).  Launches one kernel, plus
 * one merge kernel.
 */
int pa_decode_step(const pa_dims* dims, int num_seqs, const void* q, const void* k, const void* v,
                   const float* cos_sin, int max_pos, void* k_cache, void* v_cache, int num_blocks,
                   const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                   int max_context_len, float scale, int partition_tokens, void* workspace,
                   size_t workspace_bytes, void* out, unsigned flags, void* stream);

/*
 * PA_STEP_EARLY_METADATA -- flag of pa_decode_step / pa_decode_step_fp8.  The caller promises
 * that no kernel which can still be running when the call is made on `stream` writes
 * context_lens or block_tables: they were written earlier (by the host, a copy, or kernels
 * that have completed).  The decode kernel then starts while the preceding kernel on the
 * stream is still finishing (programmatic dependent launch): it reads the lengths, builds its
 * block-count prefix and resolves its first jobs through the block table, and waits for that
 * kernel before its first copy into shared memory (q, k, v, cos_sin, cache tiles) and before
 * any write.  The decode entry points (pa_decode*) let the next launch on the stream start
 * only once they no longer need the preceding work, so a step may follow another step with
 * this flag; a step right after a kernel that rewrites the tables must not set it.  A
 * multi-layer decode step whose layers follow one another on one stream is the intended use:
 * layer l + 1 resolves its work while layer l finishes.  Breaking the promise gives stale
 * lengths or block ids, never out-of-range accesses (both are still checked).
 */
#define PA_STEP_EARLY_METADATA 0x1u

/*
 * pa_prefill -- paged (chunked) prefill attention ([PV] §2: the PagedAttention prefill kernel;
 * [ME] §3.3 Chunked Prefill: a prompt is prefilled in chunks, each continuing from the tokens
 * already in the cache; [ME] §3.4: a prefix found in the cache is not recomputed).
 *
 * Sequence s brings n_s = q_start[s+1] - q_start[s] new query tokens, rows q_start[s] ..
 * q_start[s+1] - 1 of q and out, whose K and V are already stored in the paged cache (e.g. by
 * pa_rope_kv_store with positions context_lens[s] - n_s + i).  context_lens[s] counts every
 * cached token of s including the new ones.  Query i of s sits at position
 * p = context_lens[s] - n_s + i and, for each query head h (KV head g = h / (Hq / Hkv)):
 *   out[q_start[s] + i][h] = sum_{t <= p} softmax_t(scale * q . K_t) V_t   (bf16 RNE)
 * with K_t, V_t reached through block_tables[s][t / 16] as in pa_decode.  A full prefill is
 * context_lens[s] = n_s; one new token per sequence is pa_decode's result.
 * Device-side errors: a sequence with q_start[s] < 0, n_s < 0, q_start[s+1] > num_tokens,
 * n_s > max_query_len, context_lens[s] < n_s or > max_context_len is skipped (its rows are not
 * written), PA_FLAG_CONTEXT_LEN_OOB; a block id outside [0, num_blocks) -> that block is
 * skipped, PA_FLAG_BLOCK_ID_OOB.
 *
 *   num_seqs          S >= 0, S * Hkv <= 65535 (0 is a no-op)
 *   num_tokens        T = rows of q and out (0 is a no-op)
 *   q                 [T][Hq][D] bf16 (rotated), read only
 *   q_start           [S + 1] int32, device, non-decreasing, q_start[0] = 0
 *   max_query_len     host bound of every n_s, 1 <= it <= max_context_len
 *   k_cache, v_cache  [num_blocks][Hkv][16][D] bf16, read only
 *   block_tables      [S][max_blocks] int32
 *   context_lens      [S] int32
 *   max_context_len   host bound of context_lens, 1 <= it <= max_blocks * 16
 *   scale             softmax scale, finite and > 0
 *   out               [T][Hq][D] bf16, written at the rows of valid sequences
 * Returns PA_OK or a PA_ERR_* code (nothing launched on error).  Launches one kernel.
 */
int pa_prefill(const pa_dims* dims, int num_seqs, int num_tokens, const void* q,
               const int32_t* q_start, int max_query_len, const void* k_cache,
               const void* v_cache, int num_blocks, const int32_t* block_tables, int max_blocks,
               const int32_t* context_lens, int max_context_len, float scale, void* out,
               void* stream);

/*
 * FP8 (E4M3) KV cache -- the same three operations over caches of one-byte codes
 * ([NV] §学习要点 and [15x] §未来展望: low-precision quantisation of the cache to cut its
 * memory and bandwidth; the pages fix no format, the reading below is this library's).
 *
 *  - Format: OCP E4M3 ("E4M3FN"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent 0
 *    holds subnormals m/8 * 2^-6; 0x7F / 0xFF are NaN; no infinities, largest finite 448.
 *  - Layout: k_cache, v_cache are [num_blocks][Hkv][block_size][head_dim] uint8, the bf16
 *    layout with one byte per element (each (block, KV head) tile is 2 KiB).
 *  - Scales: k_scale, v_scale are [Hkv] fp32 device arrays, one per KV head, positive and
 *    finite (not checked).  Element value = code * scale of its KV head.
 *  - Storing x (a bf16 value: the rotated k, or v): code = E4M3(fp32(x) * fp32(1 / scale)),
 *    each product and the reciprocal rounded to nearest in fp32, the code rounded to nearest
 *    even, magnitudes beyond 448 (and infinities) saturating to +-448, NaN giving NaN.
 *  - Reading: codes widen exactly; attention runs on f16 copies of q (exact for bf16 values
 *    of magnitude below 65504) and P, with fp32 accumulation; results as the bf16 calls.
 */

/*
 * pa_rope_kv_store_fp8 -- pa_rope_kv_store into E4M3 caches: q rotated in place (bf16, as
 * pa_rope_kv_store), the rotated k (rounded to bf16 first) and v stored as E4M3 codes with
 * the KV head's scales.  Arguments, checks and errors as pa_rope_kv_store, plus k_scale,
 * v_scale ([Hkv] fp32, device, 16-byte aligned; PA_ERR_NULL / PA_ERR_ALIGN otherwise).
 */
int pa_rope_kv_store_fp8(const pa_dims* dims, int num_tokens, void* q, const void* k,
                         const void* v, const int32_t* positions, const float* cos_sin,
                         int max_pos, const int64_t* slot_mapping, void* k_cache, void* v_cache,
                         int num_blocks, const float* k_scale, const float* v_scale, void* stream);

/*
 * pa_decode_fp8 -- pa_decode over E4M3 caches:
 *   out[s][h] = sum_t softmax_t(scale * q[s][h] . K_t) V_t,  K_t = code * k_scale[g], V_t = code * v_scale[g].
 * Arguments, workspace (same size: pa_decode_workspace_size), checks and errors as pa_decode,
 * plus k_scale, v_scale as for pa_rope_kv_store_fp8.  Launches one kernel plus the merge.
 */
int pa_decode_fp8(const pa_dims* dims, int num_seqs, const void* q, const void* k_cache,
                  const void* v_cache, const float* k_scale, const float* v_scale, int num_blocks,
                  const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                  int max_context_len, float scale, int partition_tokens, void* workspace,
                  size_t workspace_bytes, void* out, void* stream);

/*
 * pa_decode_step_fp8 -- pa_decode_step over E4M3 caches: equals pa_rope_kv_store_fp8 (position
 * context_lens[s] - 1, that position's slot) followed by pa_decode_fp8, with q left unchanged.
 * Arguments as pa_decode_step plus k_scale, v_scale (flags included).
 */
int pa_decode_step_fp8(const pa_dims* dims, int num_seqs, const void* q, const void* k,
                       const void* v, const float* cos_sin, int max_pos, void* k_cache,
                       void* v_cache, const float* k_scale, const float* v_scale, int num_blocks,
                       const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                       int max_context_len, float scale, int partition_tokens, void* workspace,
                       size_t workspace_bytes, void* out, unsigned flags, void* stream);

/* Most caches one pa_copy_blocks call can name (K and V of up to 128 layers). */
#define PA_MAX_BLOCK_CACHES 256

/*
 * pa_copy_blocks -- copy whole KV-cache blocks between two block pools, for every cache of a
 * model in one launch: copy-on-write inside one pool ([ME] §3.4: a block shared by several
 * sequences is replaced, before it is written, by a freshly allocated block that must hold
 * the same contents) and swap out / swap in between the GPU pool and a pool in CPU memory
 * ([ME] §3.5).
 *
 * For each pair i, (from, to) = (block_pairs[2i], block_pairs[2i + 1]), and each cache c:
 *   dst_caches[c][to] = src_caches[c][from]   (the whole block: every KV head, slot and dim,
 *                                              bit for bit)
 * Pairs are copied concurrently: the destination blocks must be distinct and none may be the
 * source of another pair (true of copy-on-write and of swaps); otherwise the result is
 * unspecified.
 * Device-side errors: a pair naming a block outside its pool is skipped (nothing of it is
 * read or written), PA_FLAG_BLOCK_ID_OOB.
 *
 *   dims            shape; one block of one cache is num_kv_heads * block_size * head_dim
 *                   bf16 (block_size 16, head_dim 128: num_kv_heads tiles of 4 KiB)
 *   num_caches      1 .. PA_MAX_BLOCK_CACHES (e.g. 2 * layers: K and V of every layer)
 *   src_caches      HOST array of num_caches pool pointers, each [src_num_blocks][Hkv][16][D]
 *   src_num_blocks  >= 1
 *   dst_caches      HOST array of num_caches pool pointers, each [dst_num_blocks][Hkv][16][D]
 *                   (the same pointers as src_caches for copy-on-write inside one pool)
 *   dst_num_blocks  >= 1
 *   block_pairs     [num_pairs][2] int64, in memory the device can read
 *   num_pairs       >= 0 (0 is a no-op)
 * Every pool pointer, and block_pairs, may be this GPU's memory or page-locked host memory
 * (cudaHostAlloc, cudaHostRegister, PyTorch pin_memory), which the kernel reads and writes
 * in place over the CPU-GPU link.  Anything else (pageable host memory, another GPU's
 * memory) returns PA_ERR_MEMORY.  Pool pointers must be 16-byte aligned.
 * Returns PA_OK or a PA_ERR_* code (nothing launched on error).  Launches one kernel.
 */
int pa_copy_blocks(const pa_dims* dims, int num_caches, const void* const* src_caches,
                   int64_t src_num_blocks, void* const* dst_caches, int64_t dst_num_blocks,
                   const int64_t* block_pairs, int num_pairs, void* stream);

/*
 * pa_stage_copy -- copy `bytes` from src to dst in one kernel, either side in this GPU's
 * memory or in page-locked host memory (cudaHostAlloc, cudaHostRegister, PyTorch pin_memory),
 * which the kernel reads or writes in place over the CPU-GPU link.  For staging a decode
 * step's packed inputs (new-token q, k, v, block tables, lengths) before the step's calls and
 * reading its outputs after them: for a few hundred KiB, one kernel's loads are all in flight
 * at once, where a copy-engine transfer costs several microseconds of set-up.  Plumbing around
 * the pages' method, not part of it.
 *
 *   dst, src  16-byte aligned; the two ranges must not overlap
 *   bytes     a multiple of 16 (0 is a no-op)
 * Like every call it waits for the previous kernel on the stream before reading.  Pageable
 * host memory or another GPU's memory returns PA_ERR_MEMORY.  Returns PA_OK, PA_ERR_NULL,
 * PA_ERR_ALIGN, PA_ERR_MEMORY or PA_ERR_CUDA (nothing launched on error).  Launches one kernel.
 */
int pa_stage_copy(void* dst, const void* src, size_t bytes, void* stream);

/*
 * pa_set_timing_jitter -- test hook for the pipelined kernels' barriers: from the next launch
 * on, every role of the pa_prefill kernel (softmax warps, TMA warps, MMA warp) sleeps a
 * pseudo-random time below max_ns (the same for the whole warp, a function of seed, the CTA,
 * the role and the step) at each step of its pipeline loop, so that tests can drive the
 * barriers through orders of arrival that undisturbed runs rarely take.  Results must not
 * change: the arithmetic does not depend on timing.  max_ns = 0 turns it off (the default).
 * Applies to the calling thread's current GPU; set it only while none of this library's
 * kernels runs there.  No counterpart in the source pages: race detection support.
 * Returns PA_OK, PA_ERR_RANGE (max_ns > 1,000,000) or PA_ERR_CUDA.
 */
int pa_set_timing_jitter(uint32_t max_ns, uint32_t seed);

/*
 * pa_get_device_status -- synchronise `stream`, then read and clear the calling thread's
 * current GPU's status word.  *flags receives the PA_FLAG_* bits raised since the last
 * read (may be NULL).  Returns PA_OK when no flag was set, PA_ERR_TIMEOUT when the timeout
 * flag was set, PA_ERR_DEVICE_OOB when any other flag was set, PA_ERR_CUDA on a CUDA error.
 */
int pa_get_device_status(void* stream, uint32_t* flags);

/*
 * pa_selftest_wait_timeout -- exercise the bounded wait that guards every copy into shared
 * memory.  Launches one warp that waits on an mbarrier nothing ever arrives on, for
 * `limit_us` microseconds (1 .. 1,000,000); the wait gives up and raises PA_FLAG_TIMEOUT in
 * the device status word, which pa_get_device_status() then reports as PA_ERR_TIMEOUT.  The
 * GPU stays usable: nothing traps, faults or spins without limit.  (The decode kernel uses the
 * same wait with a 1 s limit.)  No counterpart in the source pages: failure detection support.
 * Returns PA_OK once launched, PA_ERR_RANGE for a bad limit, PA_ERR_CUDA on a launch error.
 */
int pa_selftest_wait_timeout(uint32_t limit_us, void* stream);

/*
 * pa_gather_checksum -- the gather half of pa_decode alone: every (block, KV head) tile of K
 * and V that pa_decode would read is brought into shared memory through the block tables, by
 * the same kernel shape (persistent grid, even split of the jobs, lookahead over the block
 * table, one TMA box per tile, the same stage ring), and folded into a checksum instead of
 * attention; nothing is merged.  No counterpart in the source pages: it measures the floor
 * that the decode's access pattern sets on this GPU, and checks cache contents after block
 * copies or swaps.
 *
 * For each sequence s with n = min(context_lens[s], max_context_len) and each KV head g,
 *   out_xor[s * Hkv + g] ^= XOR over t < n of the 64 32-bit words of k_cache row
 *   [block_tables[s][t / 16]][g][t % 16] and of the same v_cache row,
 * each word as stored (bf16 pairs).  XOR is order-free, so the result does not depend on how
 * the work is split.  Table entries past ceil(n / 16) are never read.
 *
 *   k_cache, v_cache  [num_blocks][Hkv][16][128] bf16, read only
 *   block_tables, context_lens, max_context_len, num_blocks, max_blocks  as for pa_decode
 *   out_xor           [S][Hkv] uint32, device memory, 4-byte aligned; XORed into (zero-fill it
 *                     first for the plain checksum)
 * Device-side errors as for pa_decode.  Returns PA_OK or a PA_ERR_* code (nothing launched on
 * error).  Launches one kernel.
 */
int pa_gather_checksum(const pa_dims* dims, int num_seqs, const void* k_cache, const void* v_cache,
                       int num_blocks, const int32_t* block_tables, int max_blocks,
                       const int32_t* context_lens, int max_context_len, uint32_t* out_xor,
                       void* stream);

/*
 * pa_gather_checksum_fp8 -- pa_gather_checksum over E4M3 caches ([num_blocks][Hkv][16][128]
 * one-byte codes, the layout of pa_decode_fp8): the gather half of pa_decode_fp8 alone, by the
 * same kernel shape.  Each row is 128 bytes = 32 32-bit words of codes as stored; otherwise as
 * pa_gather_checksum (no scales are read).
 */
int pa_gather_checksum_fp8(const pa_dims* dims, int num_seqs, const void* k_cache,
                           const void* v_cache, int num_blocks, const int32_t* block_tables,
                           int max_blocks, const int32_t* context_lens, int max_context_len,
                           uint32_t* out_xor, void* stream);

/* Human-readable name of a PA_* return code (static storage, never NULL). */
const char* pa_status_string(int status);

/*
 * pa_decode_static_workspace -- pa_decode for callers that cannot allocate device memory.
 *
 * No counterpart in the source pages: this entry point exists for callers that may not call
 * cudaMalloc or any allocator while a decode step runs -- for example an engine that has
 * already handed all free HBM to its KV-cache pool, a plugin whose enqueue function is not
 * allowed to allocate, or a real-time loop that must not take the allocator's locks.  It
 * takes the same arguments as pa_decode minus the workspace, and uses instead a scratch
 * array of PA_STATIC_WORKSPACE_BYTES that lives in the library itself (a file-scope
 * __device__ array): every GPU that loads the library holds that much device memory until
 * the process exits.  Neither this call nor anything it calls allocates.
 *
 *  - Limit: when pa_decode_workspace_size() for these arguments exceeds
 *    PA_STATIC_WORKSPACE_BYTES the call returns PA_ERR_WORKSPACE and launches nothing
 *    (use a larger partition_tokens, fewer sequences, or pa_decode with your own workspace).
 *  - The scratch needs no clearing: each call writes every partial it later reads.
 *  - All calls on a GPU share the one array and it keeps the last call's contents: two calls
 *    whose kernels overlap on that GPU (different streams, no ordering between them) race on
 *    it and give wrong results.  Order such calls on one stream or with events.
 *  - The first call on each device looks up the array's device address (once per device,
 *    with that device current); make that first call before any stream capture.
 * Returns PA_OK or a PA_ERR_* code, with the same meaning as for pa_decode.
 */
#define PA_STATIC_WORKSPACE_BYTES ((size_t)8 << 20)
int pa_decode_static_workspace(const pa_dims* dims, int num_seqs, const void* q,
                               const void* k_cache, const void* v_cache, int num_blocks,
                               const int32_t* block_tables, int max_blocks,
                               const int32_t* context_lens, int max_context_len, float scale,
                               int partition_tokens, void* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
