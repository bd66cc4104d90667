// Paged (chunked) prefill attention for sm_103a on the tcgen05 tensor cores.
//
// "Pico-vLLM：从零手写的工业级LLM推理引擎实现", §2 Kernel层 (PagedAttention prefill kernel, after
// the FlashAttention work); "从零实现 LLM 推理引擎：深挖 vLLM 的六大核心优化", §3.1 (16-token blocks,
// block tables) and §3.3 Chunked Prefill (a prompt prefilled in chunks, each continuing from
// the tokens already in the cache).
//
// Sequence s brings n_s = q_start[s+1] - q_start[s] new query tokens whose K and V are already
// in the paged cache; context_lens[s] counts every cached token including them.  Query i sits
// at position p_i = context_lens[s] - n_s + i and attends causally to cached tokens 0..p_i.
//
// CTA = (sequence, KV head g, tile of Tq = floor(128 / G) query tokens).  Its 128 matrix rows
// are the (query, head) pairs of the GQA group, row r = i G + h for query i and head g G + h,
// so every K/V tile brought in serves all G heads and the tensor core sees M = 128 rows.  Keys
// come 64 at a time (four blocks) through a 3-stage ring of shared memory filled by TMA.  Per
// stage j:
//   S_j (128 x 64, fp32, TMEM) = Q K_j^T   8 tcgen05.mma, M = 128, N = 64, K = 16 each
//   softmax (one thread per row): S_j read with tcgen05.ld, causal mask, a lazy row shift in
//   the log2 domain (it moves only when the row maximum passes it by more than 8, so P <= 2^8
//   and O is rarely rescaled), P_j = bf16(2^(scale_log2 s - shift)) written to a shared-memory
//   P buffer (128 rows x 64 keys), the fp32 values added to the row sum (exponent arguments and
//   sums two at a time, packed f32x2)
//   O (128 x 128, fp32, TMEM) += P_j V_j   4 tcgen05.mma (one per key block), M = N = 128, K = 16
// Tensor memory (256 columns): Q as bf16 pairs in columns 0-63 (the A operand of S, read from
// tensor memory: with N = 64 an A read from shared memory at every MMA would crowd shared
// memory), S in 64-127, O in 128-255.  An MMA takes a fixed minimum time whatever its N up to
// 64, so S runs 64 keys wide.
//
// Warps 0-3 load Q and run the softmax (warp w owns TMEM lanes 32w..32w+31); warps 4, 6 and 7
// issue the TMA loads, one box kind each (K columns 0-63, K columns 64-127, V), lanes 0-3 the
// stage's four blocks (their lanes read 32 block ids at a time, a window ahead); warp 5 runs
// the MMA loop, one elected lane issuing.  The softmax frees the S columns as soon as it has
// loaded S_j, and the MMA warp then issues S_{j+1} at once, so the tensor core computes the
// next scores (and P_{j-1} V_{j-1}) while the softmax works on stage j.  K and V of a stage have
// barriers of their own: K_j is dead once S_j is done and its slot refills for stage j + 3
// then, while V_j waits for P_j V_j -- a K refill does not wait for the softmax of its stage.
// Shared memory is ~113 KB (three 32 KiB stages, the 16 KiB P buffer, the barriers last), so
// two CTAs share an SM.
//
// K, V and P use the 128-byte swizzle (16-byte chunk c of a 128-byte row r at c ^ (r % 8),
// 8-row atoms of 1024 bytes).  A stage holds K half 0 of the four blocks (rows 0-63, 8 KiB), K
// half 1 (8 KiB), then V of blocks 0-3 (4 KiB each, as two 2 KiB halves of 16 rows).  Keys
// past the context in the context's last block may hold anything: their scores are masked and
// their V rows zeroed in shared memory before P V.  A block id out of range is not loaded: its
// keys are masked and its P V step skipped.  Every wait is bounded; a timeout raises
// PA_FLAG_TIMEOUT and the CTA drains its copies and MMAs before it exits.  Tiles are scheduled
// latest first over the whole grid: the last tiles of a sequence see the most keys.

#include <mutex>

#include <cuda.h>

#include "pa_device.cuh"
#include "pa_launch.h"
#include "umma_desc.h"

namespace pa {
namespace {

constexpr int kPfRows = 128;                        // MMA rows: (query, head) pairs per CTA
constexpr int kPfKB = 4;                            // key blocks per stage
constexpr int kPfKeys = kPfKB * kBlockSize;         // 64 keys per stage
constexpr int kPfStages = 3;
constexpr int kPfHalf = kBlockSize * 128;           // 16 rows x 64 bf16: 2 KiB
constexpr int kPfKHalfBytes = kPfKB * kPfHalf;      // one K half of the stage's blocks: 8 KiB
constexpr int kPfVOff = 2 * kPfKHalfBytes;          // V tiles after the two K halves
constexpr int kPfStageBytes = kPfVOff + kPfKB * kTileBytes;   // 32 KiB
constexpr int kPfPBytes = kPfRows * kPfKeys * 2;    // P: 128 rows x 64 bf16 keys, 16 KiB
constexpr int kPfPOff = kPfStages * kPfStageBytes;  // after the stages
constexpr int kPfHdrOff = kPfPOff + kPfPBytes;      // then the header
constexpr int kPfHeader = 256;                      // mbarriers, present masks, TMEM address
// Two CTAs per SM: 2 x (this + 1 KiB reserved per CTA) fits the SM's 228 KiB exactly.  The
// stages start on the first 1024-byte boundary; the header sits in the padding before them
// when that is at least kPfHeader bytes, else after the P buffer.  For any 16-byte aligned
// start (padding 0..1008) the layout ends within kPfSmem: 1008 + kPfHdrOff in the first case,
// 255 + kPfHdrOff + kPfHeader in the second.
constexpr int kPfSmem = kPfHdrOff + kPfHeader + 768;
static_assert(2 * (kPfSmem + 1024) <= 228 * 1024, "two CTAs per SM");
static_assert(1008 + kPfHdrOff <= kPfSmem && kPfHeader - 1 + kPfHdrOff + kPfHeader <= kPfSmem, "layout");
constexpr int kPfThreads = 256;                     // 4 softmax warps, TMA warps 4, 6, 7, MMA warp 5
constexpr uint32_t kPfTmemCols = 256;
constexpr uint32_t kPfQCol = 0;                     // Q: 64 columns of bf16 pairs
constexpr uint32_t kPfSCol = 64;                    // S: columns 64-127
constexpr uint32_t kPfOCol = 128;                   // O: columns 128-255

// header layout (byte offsets from the header's start)
constexpr int kBarKFull = 0;                        // [3] K TMA -> MMA (S)
constexpr int kBarVFull = 24;                       // [3] V TMA -> MMA (P V), softmax (V rows zeroed)
constexpr int kBarKEmpty = 48;                      // [3] MMA (S done) -> K TMA
constexpr int kBarVEmpty = 72;                      // [3] MMA (P V done) -> V TMA, softmax (P buffer, O)
constexpr int kBarSFull = 96;                       // MMA (S done) -> softmax
constexpr int kBarSFree = 104;                      // softmax (S loaded) -> MMA, 128 arrivals
constexpr int kBarPFull = 112;                      // [2] softmax (P written) -> MMA, 128 arrivals
constexpr int kBarDone = 128;                       // MMA thread: its last MMAs finished
constexpr int kBarQReady = 136;                     // softmax (Q in TMEM) -> MMA, 128 arrivals
constexpr int kPresent = 144;                       // [6] int, stage j at j % 6: bit i = block i loaded (MMA warp)
constexpr int kPresentSlots = 2 * kPfStages;        // a refill (stage j + 3) never overwrites stage j's
constexpr int kTmemSlot = kPresent + 4 * kPresentSlots;
static_assert(kTmemSlot + 4 <= kPfHeader, "header");

// Timing jitter, a test hook (pa_set_timing_jitter): {max_ns, seed}; max_ns 0 = off.  When on,
// each role sleeps a pseudo-random time below max_ns at each step of its pipeline loop, the same
// for the whole warp, so that tests can drive the barriers through orders of arrival that
// undisturbed runs rarely take.
__constant__ uint32_t c_pf_jitter[2];

__device__ __forceinline__ void pf_jitter(uint32_t role, uint32_t j) {
  const uint32_t max_ns = c_pf_jitter[0];
  if (max_ns == 0) return;
  uint32_t x = c_pf_jitter[1] ^ (blockIdx.x * 0x9E3779B1u) ^ (blockIdx.y * 0x85EBCA77u) ^
               (role * 0xC2B2AE3Du) ^ (j * 0x27D4EB2Fu);
  x ^= x >> 16;
  x *= 0x7FEB352Du;
  x ^= x >> 15;
  x *= 0x846CA68Bu;
  x ^= x >> 16;
  __nanosleep(x % max_ns);
}

__global__ void __launch_bounds__(kPfThreads, 2)
prefill_kernel(const __grid_constant__ CUtensorMap tm_kh, const __grid_constant__ CUtensorMap tm_v,
               const PrefillArgs a) {
  extern __shared__ unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Hkv = a.num_kv_heads;
  const int G = a.num_q_heads / Hkv;
  const int Tq = kPfRows / G;                       // query tokens per CTA
  // CTAs start in the order of their linear index (x fastest).  Consecutive indices take the
  // same query tile of every (sequence, KV head) pair, latest tile first, so the CTAs with the
  // most keys start first across the whole grid and the last wave holds the cheapest ones.
  const unsigned long long pairs = gridDim.y;  // sequences x KV heads
  const unsigned long long lin = static_cast<unsigned long long>(blockIdx.y) * gridDim.x + blockIdx.x;
  const int sg = static_cast<int>(lin % pairs);
  const int tile = static_cast<int>(gridDim.x) - 1 - static_cast<int>(lin / pairs);
  const int s = sg / Hkv;
  const int g = sg - s * Hkv;
  pdl_wait_prior_grid();
  pdl_allow_next_grid();

  // ---- the tile's queries and keys (uniform over the CTA) --------------------------------
  const int q0 = a.q_start[s];
  const int n = a.q_start[s + 1] - q0;
  const int ctx = a.context_lens[s];
  if (q0 < 0 || n < 0 || q0 + n > a.num_tokens || n > a.max_query_len || ctx < n ||
      ctx > a.max_context_len) {
    if (threadIdx.x == 0 && tile == 0 && g == 0) raise_flag(a.status, PA_FLAG_CONTEXT_LEN_OOB);
    return;
  }
  const int i0 = tile * Tq;
  if (i0 >= n) return;
  const int rows_q = min(Tq, n - i0);               // real queries of the tile
  const int pos0 = ctx - n + i0;                    // position of the tile's first query
  const int nblocks = (pos0 + rows_q - 1) / kBlockSize + 1;
  const int nst = (nblocks + kPfKB - 1) / kPfKB;    // stages of kPfKB key blocks

  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t stages = (raw + 1023u) & ~1023u;
  const uint32_t pad = stages - raw;                // 0 when the start is 1 KiB aligned
  const uint32_t hdr = pad >= static_cast<uint32_t>(kPfHeader) ? stages - kPfHeader : stages + kPfHdrOff;
  unsigned char* const hdr_gen = smem_raw + (hdr - raw);
  volatile int* present = reinterpret_cast<volatile int*>(hdr_gen + kPresent);

  // The first global reads of each role go out before the set-up below, so their latency
  // overlaps it: the softmax threads' Q rows, the TMA warp's first two windows of block ids.
  const int32_t* bt_row = a.block_tables + static_cast<size_t>(s) * a.max_blocks;
  auto load_ids = [&](int w) { const int b = 32 * w + lane; return b < nblocks ? bt_row[b] : -1; };
  int ids = -1, ids_next = -1;
  uint4 qpre[16];
  const bool producer = warp == 4 || warp >= 6;
  const int kind = warp == 4 ? 0 : warp - 5;        // producers: K cols 0-63, K cols 64-127, V
  if (producer || warp < 4) {
    ids = load_ids(0);
    ids_next = load_ids(1);
  }
  if (warp < 4) {
    // row r = query i, head g G + h: 128 bf16 (zero past the queries)
    const int r = threadIdx.x, i = r / G, h = r - (r / G) * G;
    const uint4* src = reinterpret_cast<const uint4*>(
        a.q + (static_cast<size_t>(q0 + i0 + (i < rows_q ? i : 0)) * a.num_q_heads + g * G + h) * kHeadDim);
#pragma unroll
    for (int c = 0; c < 16; ++c) qpre[c] = i < rows_q ? src[c] : make_uint4(0u, 0u, 0u, 0u);
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kPfStages; ++i) {
      mbar_init(hdr + kBarKFull + 8 * i, 1);
      mbar_init(hdr + kBarVFull + 8 * i, 1);
      mbar_init(hdr + kBarKEmpty + 8 * i, 1);
      mbar_init(hdr + kBarVEmpty + 8 * i, 1);
    }
    mbar_init(hdr + kBarSFull, 1);
    mbar_init(hdr + kBarSFree, 128);
    mbar_init(hdr + kBarPFull, 128);
    mbar_init(hdr + kBarPFull + 8, 128);
    mbar_init(hdr + kBarDone, 1);
    mbar_init(hdr + kBarQReady, 128);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(hdr + kTmemSlot, kPfTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(hdr_gen + kTmemSlot);

  if (producer) {
    // ---- TMA producers: stage j holds key blocks 4j .. 4j + 3 -------------------------------
    // Three warps share a stage's 12 boxes, one kind each (lanes 0-3: the four blocks): a warp's
    // TMA instruction issues its lanes' boxes one after another, so one warp issuing all 12
    // leaves the stage latency-bound; with three, the SM's fill rate is the limit.  The K warps
    // refill a slot once S of its last stage is done, the V warp once P V is.  The first K warp
    // announces the K bytes and the stage's present mask, the V warp the V bytes (the other K
    // warp's boxes may land first: the phase cannot complete before that arrival).
    // Lane k holds the id of block 32 w + k of the current window w (-1 past the tile's
    // blocks); the next window's ids are loaded when the current one starts.
    if (lane == 0) {
      prefetch_tensor_map(&tm_kh);
      prefetch_tensor_map(&tm_v);
    }
    const uint32_t full = hdr + (kind < 2 ? kBarKFull : kBarVFull);
    const uint32_t empty = hdr + (kind < 2 ? kBarKEmpty : kBarVEmpty);
    int issued = 0;
    bool failed = false;
    for (int j = 0; j < nst; ++j) {
      pf_jitter(8 + kind, j);
      const int st = j % kPfStages;
      const int k = (kPfKB * j) & 31;               // lane holding block 4j
      if (j > 0 && k == 0) {
        ids = ids_next;
        ids_next = load_ids((kPfKB * j) / 32 + 1);
      }
      bool ok = true;
      if (lane == 0 && j >= kPfStages) ok = mbar_wait_bounded(empty + 8 * st, ((j / kPfStages) - 1) & 1);
      if (!__shfl_sync(kFullMask, ok, 0)) {
        failed = true;
        break;
      }
      const int bi = lane & (kPfKB - 1);
      const int blk = __shfl_sync(kFullMask, ids, k + bi);
      const int b = kPfKB * j + bi;
      const bool here = b < nblocks && blk >= 0 && blk < a.num_blocks;
      const int mask = static_cast<int>(__ballot_sync(kFullMask, here) & ((1u << kPfKB) - 1));
      const uint32_t bar = full + 8 * st;
      if (kind != 1 && lane == 0) {
        if (kind == 0) present[j % kPresentSlots] = mask;
        // K: both halves of each block; V: the whole tile
        if (mask) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(__popc(mask)) * kTileBytes);
        else mbar_arrive(bar);
      }
      if (kind == 0 && lane < kPfKB && b < nblocks && !here) raise_flag(a.status, PA_FLAG_BLOCK_ID_OOB);
      if (lane < kPfKB && here) {
        const int y = (blk * Hkv + g) * kBlockSize;
        const uint32_t dst = stages + st * kPfStageBytes;
        if (kind < 2)
          tma_load_3d(dst + kind * kPfKHalfBytes + bi * kPfHalf, &tm_kh, 0, y, kind, bar);   // K cols 64 kind + 0..63
        else
          tma_load_3d(dst + kPfVOff + bi * kTileBytes, &tm_v, 0, y, 0, bar);                  // V, both halves
      }
      issued = j + 1;
    }
    if (lane == 0) {
      if (failed) raise_flag(a.status, PA_FLAG_TIMEOUT);
      // Copies still in flight can only be those of this warp's last kPfStages fills: let them
      // land (immediate in a normal run, where the MMAs consumed every stage) before the CTA exits.
      for (int j = max(0, issued - kPfStages); j < issued; ++j)
        mbar_wait_bounded(full + 8 * (j % kPfStages), (j / kPfStages) & 1, 10000000ull);
    }
  } else if (warp == 5) {
    // ---- MMA issuer: the whole warp runs the loop, one elected lane issues ----------------------
    const uint32_t id_s = umma_idesc_bf16(kPfRows, kPfKeys, false, false);
    const uint32_t id_pv = umma_idesc_bf16(kPfRows, kHeadDim, false, true);
    // descriptors of stage 0; a stage, a k step or a block moves the start address field by
    // (byte offset) / 16, which never carries out of its 14 bits (shared memory < 256 KiB)
    const uint64_t k_desc0 = umma_smem_desc(stages, 16, 1024);
    const uint64_t p_desc = umma_smem_desc(stages + kPfPOff, 16, 1024);   // P: 128-byte rows
    const uint64_t v_desc0 = umma_smem_desc(stages + kPfVOff, kPfHalf, 1024);
    bool o_started = false;
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(kFullMask, mbar_wait_bounded(bar, parity));
    };
    // S_j = Q K_j^T into the S columns, once K_j has landed and the softmax has loaded S_{j-1};
    // its completion frees K_j's slot as well.  Returns the stage's present mask (-1: timeout),
    // read while the slot cannot be refilled.
    auto issue_s = [&](int j) -> int {
      const int st = j % kPfStages;
      if (!wait_all(hdr + kBarKFull + 8 * st, (j / kPfStages) & 1)) return -1;
      if (j > 0 && !wait_all(hdr + kBarSFree, (j - 1) & 1)) return -1;
      tc_fence_after();
      const int mask = present[j % kPresentSlots];
      const uint64_t kd = k_desc0 + static_cast<uint64_t>((st * kPfStageBytes) >> 4);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16_tmem_a(tmem + kPfSCol, tmem + kPfQCol + 8 * kk,
                           kd + static_cast<uint64_t>(((kk >> 2) * kPfKHalfBytes + (kk & 3) * 32) >> 4), id_s,
                           kk > 0);
        umma_commit(hdr + kBarSFull);
        umma_commit(hdr + kBarKEmpty + 8 * st);
      }
      __syncwarp();
      return mask;
    };
    bool failed = !wait_all(hdr + kBarQReady, 0);
    int mask_cur = 0;
    if (!failed) {
      tc_fence_after();
      mask_cur = issue_s(0);
      failed = mask_cur < 0;
    }
    for (int j = 0; j < nst && !failed; ++j) {
      pf_jitter(16, j);
      int mask_next = 0;
      if (j + 1 < nst) {
        mask_next = issue_s(j + 1);
        if (mask_next < 0) {
          failed = true;
          break;
        }
      }
      // P_j: two barriers alternate, so the softmax of stage j + 1 (which may run while this
      // warp still waits here) arrives on the other one
      const int st = j % kPfStages;
      if (!wait_all(hdr + kBarPFull + 8 * (j & 1), (j >> 1) & 1) ||
          !wait_all(hdr + kBarVFull + 8 * st, (j / kPfStages) & 1)) {
        failed = true;
        break;
      }
      tc_fence_after();
      const uint64_t vd = v_desc0 + static_cast<uint64_t>((st * kPfStageBytes) >> 4);
      if (elect_one()) {
        bool acc = o_started;                       // the first P V of the tile overwrites O
#pragma unroll
        for (int i = 0; i < kPfKB; ++i) {
          if (!(mask_cur & (1 << i))) continue;
          umma_bf16(tmem + kPfOCol, p_desc + static_cast<uint64_t>((32 * i) >> 4),
                    vd + static_cast<uint64_t>((i * kTileBytes) >> 4), id_pv, acc);
          acc = true;
        }
        // P V of stage j done: the V warp may refill the stage, the softmax may write P_{j+1}
        // and rescale O
        umma_commit(hdr + kBarVEmpty + 8 * st);
      }
      __syncwarp();
      o_started = o_started || mask_cur != 0;
      mask_cur = mask_next;
    }
    if (lane == 0) {
      if (failed) raise_flag(a.status, PA_FLAG_TIMEOUT);
      // Every MMA issued has finished before the CTA frees TMEM and exits.
      umma_commit(hdr + kBarDone);
      mbar_wait_bounded(hdr + kBarDone, 0);
    }
    __syncwarp();
  } else {
    // ---- Q into TMEM, then the softmax: thread = row r of the tile ------------------------------
    const int r = threadIdx.x;                      // 0..127 = TMEM lane
    const int i = r / G, h = r - (r / G) * G;
    const int p_r = pos0 + i;                       // rows past the tile's queries are never stored
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    {
      // Q row r (loaded before the set-up) = 64 columns of bf16 pairs
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t qv[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = qpre[8 * half + c];
          qv[4 * c] = v.x;
          qv[4 * c + 1] = v.y;
          qv[4 * c + 2] = v.z;
          qv[4 * c + 3] = v.w;
        }
        tmem_st32(trow + kPfQCol + 32 * half, qv);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(hdr + kBarQReady);
    }
    const float sl = a.scale_log2;
    // the context's last block, if partial: its V rows valid_last..15 are zeroed before P V
    const int last_blk = (ctx - 1) / kBlockSize;
    const int valid_last = ctx - kBlockSize * last_blk;
    float m = -INFINITY, l = 0.f;
    bool failed = false;
    const uint32_t sbuf = trow + kPfSCol;
    for (int j = 0; j < nst; ++j) {
      pf_jitter(warp, j);
      const int st = j % kPfStages;
      // The stage's present mask, from the same block ids the TMA warps test (lane k holds block
      // 32 w + k of window w).  Not from K_j's barrier: once S_j is done the slot refills for
      // stage j + 3, and a late look at that barrier could find it two phases on.
      const int kw = (kPfKB * j) & 31;
      if (j > 0 && kw == 0) {
        ids = ids_next;
        ids_next = load_ids((kPfKB * j) / 32 + 1);
      }
      const int blk = __shfl_sync(kFullMask, ids, kw + (lane & (kPfKB - 1)));
      const int bq = kPfKB * j + (lane & (kPfKB - 1));
      const int mask = static_cast<int>(
          __ballot_sync(kFullMask, bq < nblocks && blk >= 0 && blk < a.num_blocks) & ((1u << kPfKB) - 1));
      // tcgen05.ld / st are warp-collective: a warp goes on only if all its lanes saw the phase
      if (!__all_sync(kFullMask, mbar_wait_bounded(hdr + kBarSFull, j & 1))) {
        failed = true;
        break;
      }
      tc_fence_after();
      float sc[kPfKeys];
      {
        uint32_t sv[32];
        tmem_ld32(sbuf, sv);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) sc[c] = __uint_as_float(sv[c]);
        tmem_ld32(sbuf + 32, sv);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) sc[32 + c] = __uint_as_float(sv[c]);
      }
      // S_j is in registers: the MMA warp may compute S_{j+1} over it
      tc_fence_before();
      mbar_arrive(hdr + kBarSFree);
      // Scores stay unscaled until the exponent (scale > 0, so the row maxima are the same).
      // Causal mask and missing blocks -> -inf, only on a stage that reaches past the tile's
      // first query or lacks a block; the others lie wholly before every query of the tile.
      if (mask != (1 << kPfKB) - 1 || kPfKeys * (j + 1) - 1 > pos0) {
        const int lim = p_r - kPfKeys * j;          // keys c <= lim are causal for this row
#pragma unroll
        for (int c = 0; c < kPfKeys; ++c)
          if (!((mask >> (c / kBlockSize)) & 1) || c > lim) sc[c] = -INFINITY;
      }
      // row maximum by three-input max: 64 -> 22 -> 8 -> 3 -> 1
      float m1[22], m2[8];
#pragma unroll
      for (int c = 0; c < 21; ++c) m1[c] = fmax3(sc[3 * c], sc[3 * c + 1], sc[3 * c + 2]);
      m1[21] = sc[63];
#pragma unroll
      for (int c = 0; c < 7; ++c) m2[c] = fmax3(m1[3 * c], m1[3 * c + 1], m1[3 * c + 2]);
      m2[7] = m1[21];
      const float mrow = fmax3(fmax3(m2[0], m2[1], m2[2]), fmax3(m2[3], m2[4], m2[5]), fmaxf(m2[6], m2[7]));
      // Shift m in the log2 domain (scale * log2(e) applied): it moves to the row maximum only
      // when that exceeds it by more than 8, so P stays at most 2^8 and O is rescaled rarely.
      const float bs = mrow * sl;
      const float mn = bs > m + 8.f ? bs : m;
      const float sh = mn == -INFINITY ? 0.f : mn;  // a row with no key yet keeps the shift 0
      const float alpha = (mn == m || m == -INFINITY) ? 1.f : ex2_ftz(m - sh);
      m = mn;
      // P = 2^(scale_log2 s - shift) with the exponent argument formed two at a time (packed
      // fp32 FMA), rounded to bf16 (the MMA operand).  The row sum adds the fp32 values, two at
      // a time; it differs from the sum of the rounded values by the rounding errors of P, about
      // 2^-9 of each term and of random sign.
      uint32_t pw[kPfKeys / 2];
      uint64_t psum[4] = {0ull, 0ull, 0ull, 0ull};
      const uint64_t sl2 = pack_f32x2(sl, sl), nsh2 = pack_f32x2(-sh, -sh);
#pragma unroll
      for (int k = 0; k < kPfKeys / 2; ++k) {
        const uint64_t x = fma_f32x2(pack_f32x2(sc[2 * k], sc[2 * k + 1]), sl2, nsh2);
        float x0, x1;
        unpack_f32x2(x, x0, x1);
        const float p0 = ex2_ftz(x0), p1 = ex2_ftz(x1);
        pw[k] = pack_bf16x2(p0, p1);
        psum[k & 3] = add_f32x2(psum[k & 3], pack_f32x2(p0, p1));
      }
      float ps;
      {
        const uint64_t t = add_f32x2(add_f32x2(psum[0], psum[1]), add_f32x2(psum[2], psum[3]));
        float t0, t1;
        unpack_f32x2(t, t0, t1);
        ps = t0 + t1;
      }
      l = fmaf(l, alpha, ps);
      // P V of stage j - 1 must be done before P_j overwrites the P buffer it reads and before O
      // is rescaled.  It completes use (j - 1) / kPfStages of its stage's V-empty barrier; the
      // next completion needs P_{j+2}, so the parity is unambiguous.
      pf_jitter(4 + warp, j);
      if (j > 0) {
        const int pj = j - 1;
        if (!__all_sync(kFullMask, mbar_wait_bounded(hdr + kBarVEmpty + 8 * (pj % kPfStages),
                                                     (pj / kPfStages) & 1))) {
          failed = true;
          break;
        }
        tc_fence_after();
      }
      // O *= alpha (warp-collective TMEM access)
      if (j > 0 && __any_sync(kFullMask, alpha != 1.f)) {
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t ov[32];
          tmem_ld32(trow + kPfOCol + 32 * q4, ov);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
          tmem_st32(trow + kPfOCol + 32 * q4, ov);
        }
        tmem_wait_st();
      }
      // P row r: 64 keys = 8 chunks of 16 bytes, chunk c at c ^ (r % 8)
      {
        unsigned char* prow = smem_raw + (stages - raw) + kPfPOff + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(prow + ((c ^ (r & 7)) << 4)) =
              make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
      }
      // Keys past the context in its last block: zero their V rows (both 64-column halves),
      // once V_j has landed.
      const int vb = last_blk - kPfKB * j;
      if (valid_last < kBlockSize && vb >= 0 && vb < kPfKB && ((mask >> vb) & 1)) {
        if (!__all_sync(kFullMask, mbar_wait_bounded(hdr + kBarVFull + 8 * st, (j / kPfStages) & 1))) {
          failed = true;
          break;
        }
        const int chunks = (kBlockSize - valid_last) * 16;
        unsigned char* vt = smem_raw + (stages - raw) + st * kPfStageBytes + kPfVOff + vb * kTileBytes;
        for (int x = r; x < chunks; x += 128) {
          const int row = valid_last + (x >> 4), half = (x >> 3) & 1, ch = x & 7;
          *reinterpret_cast<uint4*>(vt + half * kPfHalf + row * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();                     // P and zeroed V rows before the tensor core reads them
      tc_fence_before();
      mbar_arrive(hdr + kBarPFull + 8 * (j & 1));
    }
    if (failed) {
      if (lane == 0) raise_flag(a.status, PA_FLAG_TIMEOUT);
    } else if (__all_sync(kFullMask, mbar_wait_bounded(hdr + kBarDone, 0))) {
      // ---- out = O / l for the tile's real rows (kBarDone: the MMA thread's last P V) ---------
      tc_fence_after();
      // a row whose every key was skipped (all its blocks out of range) has l = 0 and an O
      // never written: it stores zeros
      const bool any = l > 0.f;
      const float inv = any ? 1.f / l : 0.f;
      const bool store = i < rows_q;
      uint4* dst = reinterpret_cast<uint4*>(
          a.out + (static_cast<size_t>(q0 + i0 + (store ? i : 0)) * a.num_q_heads + g * G + h) * kHeadDim);
#pragma unroll 1
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t ov[32];
        tmem_ld32(trow + kPfOCol + 32 * q4, ov);
        tmem_wait_ld();
        if (store) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = any ? __uint_as_float(ov[8 * k + e]) : 0.f;
            dst[4 * q4 + k] = make_uint4(pack_bf16x2(f[0] * inv, f[1] * inv), pack_bf16x2(f[2] * inv, f[3] * inv),
                                         pack_bf16x2(f[4] * inv, f[5] * inv), pack_bf16x2(f[6] * inv, f[7] * inv));
          }
        }
      }
    } else if (lane == 0) {
      raise_flag(a.status, PA_FLAG_TIMEOUT);
    }
  }
  // every TMEM access and MMA of the CTA is complete: free the columns
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kPfTmemCols);
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  const int G = a.num_q_heads / a.num_kv_heads;
  if (G < 1 || G > kPfRows) return cudaErrorInvalidValue;
  const int Tq = kPfRows / G;
  const long long rows = static_cast<long long>(a.num_blocks) * a.num_kv_heads * kBlockSize;
  CUtensorMap tm_kh, tm_v;
  if (!cache_tensor_map(a.k_cache, rows, false, &tm_kh, 1) || !cache_tensor_map(a.v_cache, rows, false, &tm_v, 2))
    return cudaErrorInvalidValue;
  {  // opt in to the shared-memory size once per device
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
      err = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
      if (err != cudaSuccess) return err;
      // the whole 228 KiB as shared memory: two CTAs per SM need all of it
      err = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
      if (err != cudaSuccess) return err;
      done[dev] = true;
    }
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((a.max_query_len + Tq - 1) / Tq),
                     static_cast<unsigned>(a.num_seqs * a.num_kv_heads));
  cfg.blockDim = dim3(static_cast<unsigned>(kPfThreads));
  cfg.dynamicSmemBytes = kPfSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_kernel, tm_kh, tm_v, a);
}

}  // namespace pa

extern "C" int pa_set_timing_jitter(uint32_t max_ns, uint32_t seed) {
  if (max_ns > 1000000u) return PA_ERR_RANGE;
  const uint32_t v[2] = {max_ns, seed};
  return cudaMemcpyToSymbol(pa::c_pf_jitter, v, sizeof v) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
