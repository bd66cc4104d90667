// Single-token paged GQA decode attention for sm_103a, with Flash-Decode splitting.
//
// "Pico-vLLM：从零手写的工业级LLM推理引擎实现": §2 Kernel层 (PagedAttention decode kernel),
// §1 模型实现层 (GQA), §H200上的详细对比 (Flash Decode); "从零实现 LLM 推理引擎：深挖 vLLM 的
// 六大核心优化", §3.1 Paged KV Cache (16-token blocks reached through a block table).
//
// Work.  Segment i = s * Hkv + g is the block list of sequence s for KV head g: n_s =
// ceil(len_s / 16) blocks, starting at X_i = Hkv * N_s + g * n_s on one flattened axis of
// T = Hkv * N_S block jobs (N_s = sum of n over the sequences before s).  The axis is cut into
// V equal contiguous ranges ("virtual warps"): V = min(#warps, ceil(T / 2)) so that every warp of
// the persistent grid gets the same number of blocks +-1, or ranges of a fixed C = P / 16 blocks
// when the caller asks for P-token partitions.  A range cut by segment boundaries gives
// pieces; piece (v, i) covers the part of segment i inside range v and owns partial slot v + i.
// A warp serves all G <= 8 query heads of a segment's KV head, so each (block, KV head) tile of
// K and V is read from HBM exactly once.
//
// Each warp is its own producer and consumer over a ring of shared-memory stages that runs
// straight through piece boundaries.  The CTA's stages are shared out evenly among its warps that
// have work, so that with fewer ranges than warps each busy warp keeps more tiles in flight:
//   lookahead  the lanes of the warp resolve 32 jobs at a time -- segment (binary search over
//              the CTA's shared prefix of block counts), block id from the block table, valid
//              tokens, first / last / whole-segment flags -- one window ahead of use;
//   producer   per job, lane 0 writes a small descriptor and issues two TMA tensor loads (the
//              K tile and the V tile, each one box landing as two 64-column halves, 128-byte
//              swizzle) on the stage's mbarrier, plus on a piece's first block a bulk copy of
//              the q rows;
//   consumer   waits on the stage (bounded), on a first block loads q^T fragments from the
//              stage and resets the softmax state, computes S^T = K q^T (16 tokens x 8 head
//              columns) with 8 m16n8k16 bf16 MMAs in two accumulator chains (A = K via
//              ldmatrix), updates the online softmax in the log2 domain (scale * log2(e) folded
//              into one FMA per exponent; a head's shift moves only when its maximum passes it
//              by more than 8), rounds P to bf16 and transposes it with movmatrix into the B
//              operand, and accumulates O^T += V^T P^T (128 dims x 8 heads, fp32) with 8 MMAs
//              (A = V via transposing ldmatrix); on a piece's last block it writes bf16 `out`
//              (the piece is the whole segment) or the partial (sum p V, (shift, l)) to slot
//              v + i.
// decode_merge_kernel combines the pieces of split segments:
//   M = max_p m_p,  out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p  (m_p: each piece's
//   softmax shift, which serves as its maximum would).
// Ranges are dealt to the CTAs round-robin (range v to warp v / grid of CTA v % grid).
//
// Shared memory per stage: [K cols 0-63 | K cols 64-127 | V cols 0-63 | V cols 64-127 | q rows],
// the four tile halves 16 rows x 128 B each, swizzled so that 16-byte chunk c of row r sits at
// chunk c ^ (r % 8); the ldmatrix row addresses apply the same XOR, so all eight rows of a
// matrix hit distinct banks.
//
// Variants (template <kStep, kFp8, kGather, kOnce>):
//   kStep  the fused decode step ("Pico-vLLM" §2: RoPE fused with the KV cache store): the warp
//          whose job holds a sequence's new token (position len - 1) stages the token's k, v and
//          cos/sin row with the tiles, rotates k, writes both rows into the staged tiles before
//          the MMAs and into the cache slot; each piece rotates its q fragments in registers.
//   kFp8   E4M3 caches with one scale per KV head: 2 KiB tiles, one 128-byte box each, CTAs of
//          12 warps with 2 stages; the byte tiles are read by ldmatrix as 16-bit pairs and widened exactly to
//          f16 with cvt.f16x2.e4m3x2, the q.K k index permuted alike in both operands; f16 MMAs,
//          the K scale folded into the softmax scale, the V scale into the output.
//   kGather the tile gather alone (pa_gather_checksum): an XOR of the tile words instead of the
//          attention, no merge -- the floor of this kernel's access pattern.
//   kOnce  launched for calls with early metadata (a layer of a chain): the K/V tiles load with
//          an evict-first L2 policy, so that what the next layers read again stays in L2.

#include <cmath>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {
namespace {

constexpr int kWarps = PA_DECODE_WARPS;     // warps per CTA, bf16 caches
constexpr int kStages = PA_DECODE_STAGES;
constexpr int kHalfBytes = kBlockSize * 128;                // 16 rows x 64 bf16
constexpr int kQBytes = 8 * kHeadDim * 2;                   // q rows of up to 8 heads

// Per CTA in shared memory: the block-count prefix N_s (S + 1 ints), then per sequence the
// valid rows of its last block (1..16; one byte each).
__host__ __device__ inline int prefix_bytes(int num_seqs) {
  return (((num_seqs + 1) * 4 + 15) & ~15) + ((num_seqs + 15) & ~15);
}

// Shared-memory layout of one kernel variant.  kStep fuses the new token's RoPE + store; kFp8
// reads E4M3 caches, whose (block, KV head) tiles are 2 KiB instead of 4 KiB: there the CTA
// runs 12 warps of 2 stages, since its per-job work (widening the codes) is heavier and more
// independent warps hide it better than deeper rings (measured: 12 x 2 beat 8 x 4 and 8 x 3).  Header: the mbarriers (8 bytes each), the int4 job descriptors on a 16-byte boundary,
// the prefix of block counts.  Stage: [K tile | V tile | q rows | (kStep) the new token's
// cos/sin row (fp32), k row and v row (bf16)], a multiple of 1024 bytes so that every tile
// stays on the 1024-byte boundary its 128-byte swizzle needs.
template <bool kStep, bool kFp8>
struct Layout {
  static constexpr int kTile = kFp8 ? kTileBytes / 2 : kTileBytes;
  static constexpr int kWarpsN = kFp8 ? 12 : kWarps;
  static constexpr int kStagesN = kFp8 ? 2 : kStages;
  static constexpr int kQOff = 2 * kTile;
  static constexpr int kCosSinOff = kQOff + kQBytes;
  static constexpr int kNewKOff = kCosSinOff + kHeadDim * 4;
  static constexpr int kNewVOff = kNewKOff + kHeadDim * 2;
  static constexpr int kStage = kStep ? kNewVOff + kHeadDim * 2 : kQOff + kQBytes;
  static constexpr int kDescOff = (kWarpsN * kStagesN * 8 + 15) & ~15;
  static constexpr int kPrefixOff = kDescOff + kWarpsN * kStagesN * 16;
  static_assert(kStage % 1024 == 0 && kTile % 1024 == 0, "tiles on 1024-byte boundaries");
  static_assert(kDescOff % 16 == 0 && kPrefixOff % 16 == 0, "descriptor alignment");
  __host__ __device__ static int smem(int num_seqs) {
    return kPrefixOff + prefix_bytes(num_seqs) + 1024 + kWarpsN * kStagesN * kStage;  // + pad
  }
};

// Job flags (low bits of a descriptor's flag word; valid tokens sit at bits 8-12, the KV head
// at bits 16-31).
constexpr uint32_t kFirst = 1u, kLast = 2u, kWhole = 4u, kHasData = 8u;
constexpr uint32_t kNew = 16u;   // fused step: the block holding the segment's new token
constexpr uint32_t kRope = 32u;  // fused step: the sequence's position has a cos/sin row
constexpr uint32_t kGap = 64u;   // the piece starts at a range boundary that is also a partition
                                 // boundary inside the segment: the slot before it is a gap
constexpr int kMinRangeBlocks = PA_DECODE_MIN_RANGE;


// Flattened-axis ranges: V = min(num_warps, ceil(T / kMinRangeBlocks)) equal ranges, range
// v = [floor(v T / V), floor((v+1) T / V)), none shorter than kMinRangeBlocks blocks unless T
// is, so that a small batch is not cut into one-block pieces that the merge must then gather.
// With V <= #warps of the grid, every warp has at most one range.
struct Ranges {
  long long T;
  int V;
  __device__ __forceinline__ long long begin(int v) const { return (static_cast<long long>(v) * T) / V; }
  __device__ __forceinline__ int owner(long long x) const {
    return static_cast<int>(((x + 1) * V - 1) / T);
  }
};

__device__ __forceinline__ Ranges make_ranges(long long T, const DecodeArgs& a) {
  Ranges r;
  r.T = T;
  r.V = static_cast<int>(min(static_cast<long long>(a.num_warps), (T + kMinRangeBlocks - 1) / kMinRangeBlocks));
  return r;
}

// Partial slot of the piece of segment `seg` in range v and P-token partition `part` (0
// without partitions; max_parts = partitions of the longest segment, 1 without).  Along the
// job axis consecutive pieces differ in range, partition or segment, and each such step
// raises the slot by at least one, so slots are distinct and below V + (#segments) * max_parts.
// Within one segment a step raises it by exactly one, except where a range boundary is also a
// partition boundary: there it skips one slot, which the warp whose range starts there marks
// empty (shift -inf, sum 0).  So a segment's pieces, with those gaps, fill the slots from
// v_first + seg * max_parts to v_last + seg * max_parts + (its last partition), in axis order.
__device__ __forceinline__ long long piece_slot(int v, int seg, int part, int max_parts) {
  return static_cast<long long>(v) + static_cast<long long>(seg) * max_parts + part;
}

__device__ __forceinline__ int clamp_len(int len, int max_len) {
  return len < 0 ? 0 : (len > max_len ? max_len : len);
}

template <bool kStep, bool kFp8, bool kGather = false, bool kOnce = false>
__global__ void __launch_bounds__(Layout<kStep, kFp8>::kWarpsN * 32, 1)
decode_partition_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
  using L = Layout<kStep, kFp8>;
  constexpr int kWarps = L::kWarpsN;           // warps of this variant's CTA
  constexpr int kPool = kWarps * L::kStagesN;  // stages of the CTA
  constexpr int kStageB = L::kStage;
  static_assert(kPool <= kWarps * 32, "one initialising thread per stage");
  extern __shared__ unsigned char smem_raw[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t raw = smem_addr(smem_raw);
  int* prefix = reinterpret_cast<int*>(smem_raw + L::kPrefixOff);  // N_s, s = 0..S
  unsigned char* last_rows = smem_raw + L::kPrefixOff + (((a.num_seqs + 1) * 4 + 15) & ~15);
  // 128-byte swizzled TMA destinations must sit on 1024-byte boundaries.
  const uint32_t tile_base = (raw + L::kPrefixOff + prefix_bytes(a.num_seqs) + 1023u) & ~1023u;
  if (tid < kPool) {
    mbar_init(raw + 8 * tid, 1);
    fence_mbar_init();
  }
  if (tid == 0) {
    prefetch_tensor_map(&tm_k);
    prefetch_tensor_map(&tm_v);
  }

  // With early metadata the lengths and block table are read, and the work resolved, before
  // the preceding kernel has finished; the first copy into shared memory and every write
  // wait for it (below, before the pipeline's first fill).
  const bool early = a.early_metadata != 0;
  if (!early) pdl_wait_prior_grid();
  pdl_allow_next_grid();

  const int S = a.num_seqs;
  const int Hkv = a.num_kv_heads;
  const int G = a.num_q_heads / Hkv;

  // ---- CTA prologue: exclusive prefix N_s of per-sequence block counts in shared memory ----
  {
    __shared__ int warp_sums[kWarps];
    const int per = (S + kWarps * 32 - 1) / (kWarps * 32);
    const int lo = min(S, tid * per), hi = min(S, lo + per);
    int sum = 0;
    for (int s = lo; s < hi; ++s) {
      const int len = a.context_lens[s];
      if ((len < 0 || len > a.max_context_len) && blockIdx.x == 0)
        raise_flag(a.status, PA_FLAG_CONTEXT_LEN_OOB);
      sum += (clamp_len(len, a.max_context_len) + kBlockSize - 1) / kBlockSize;
    }
    int incl = sum;
#pragma unroll
    for (int x = 1; x < 32; x <<= 1) {
      const int y = __shfl_up_sync(kFullMask, incl, x);
      if (lane >= x) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    int run = incl - sum;
    for (int w = 0; w < warp; ++w) run += warp_sums[w];
    for (int s = lo; s < hi; ++s) {
      prefix[s] = run;
      const int len = clamp_len(a.context_lens[s], a.max_context_len);
      run += (len + kBlockSize - 1) / kBlockSize;
      last_rows[s] = static_cast<unsigned char>(((len - 1) & (kBlockSize - 1)) + 1);  // unused if len == 0
    }
    if (tid == kWarps * 32 - 1) {
      int total = 0;
      for (int w = 0; w < kWarps; ++w) total += warp_sums[w];
      prefix[S] = total;
    }
    __syncthreads();
  }
  const long long T = static_cast<long long>(Hkv) * prefix[S];
  const Ranges R = make_ranges(T, a);
  // Stage pool: the CTA's kPool stages are shared out among its warps that have a range.  Range
  // v goes to warp v / grid of CTA v % grid, so these are warps 0 .. active - 1 (the others have
  // no work); with fewer ranges than warps (fixed-size partitions over a few long sequences)
  // each of them runs a deeper pipeline.
  const int active = R.V > static_cast<int>(blockIdx.x)
                         ? min(kWarps, (R.V - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                                           static_cast<int>(gridDim.x))
                         : 1;
  const int n_st = kPool / active;  // this warp's stages, used in ring order
  const uint32_t bars = raw + warp * n_st * 8;
  int4* descs = reinterpret_cast<int4*>(smem_raw + L::kDescOff) + warp * n_st;
  const uint32_t tiles = tile_base + warp * n_st * kStageB;
  const int gq = lane >> 2;  // fragment row group
  const int cq = lane & 3;   // fragment column pair
  const int mi = lane >> 3;  // ldmatrix: matrix this lane addresses
  const int r = lane & 7;    // ldmatrix: row of that matrix

  // ---------------------------------------------------------------- lookahead windows --
  // Window = up to 32 consecutive jobs of one range; lane j resolves job j.  Fields per lane:
  // physical block id, segment, flags | valid << 8 | KV head << 16, partial slot.  The block
  // id is left as loaded -- nothing here waits for the block-table load, so the two windows
  // resolved up front have their loads in flight together; the producer uses it.
  struct Window {
    int v;                // range
    long long x;          // first position
    int n;                // jobs in the window (0: none left)
    int blk, seg, fl, slot;
    int pos;              // fused step: position of the sequence's new token
  };
  // This warp's range (at most one): its bounds, found once.
  const int my_v = static_cast<int>(blockIdx.x) + warp * static_cast<int>(gridDim.x);
  const long long x0 = my_v < R.V ? R.begin(my_v) : 0;
  const long long x1 = my_v < R.V ? R.begin(my_v + 1) : 0;
  auto resolve = [&](Window& W) {
    W.blk = -1;
    W.seg = W.fl = W.slot = W.pos = 0;
    if (W.n == 0 || lane >= W.n) return;
    const long long p = W.x + lane;
    // largest s with Hkv * N_s <= p (N_0 = 0 <= p < Hkv * N_S = T)
    int lo = 0, hi = S;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (static_cast<long long>(Hkv) * prefix[mid] <= p) lo = mid;
      else hi = mid;
    }
    const int s = lo;
    const int ns = prefix[s + 1] - prefix[s];
    const int off = static_cast<int>(p - static_cast<long long>(Hkv) * prefix[s]);  // < Hkv * ns
    const int g = off / ns;
    const int j = off - g * ns;
    const long long Xi = static_cast<long long>(Hkv) * prefix[s] + static_cast<long long>(g) * ns;
    W.blk = a.block_tables[static_cast<size_t>(s) * a.max_blocks + j];
    W.seg = s * Hkv + g;
    const int tail = last_rows[s];
    const int len = (ns - 1) * kBlockSize + tail;
    const int valid = j == ns - 1 ? tail : kBlockSize;
    // Pieces end at range, segment and (P-token partitions) partition boundaries.
    const int chunk = a.chunk_blocks;
    const int part = chunk ? j / chunk : 0;
    const bool p_first = chunk && j == part * chunk;
    const bool p_last = chunk && j == part * chunk + chunk - 1;
    uint32_t flags = ((p == x0 || j == 0 || p_first) ? kFirst : 0u) |
                     ((p == x1 - 1 || j == ns - 1 || p_last) ? kLast : 0u) |
                     ((Xi >= x0 && Xi + ns <= x1 && (chunk == 0 || ns <= chunk)) ? kWhole : 0u) |
                     ((p == x0 && j > 0 && p_first) ? kGap : 0u);
    if (kStep) {
      W.pos = len - 1;
      if (j == ns - 1) flags |= kNew;
      if (W.pos < a.max_pos) flags |= kRope;  // len >= 1 here, so pos >= 0
    }
    W.fl = static_cast<int>(flags | (static_cast<uint32_t>(valid) << 8) | (static_cast<uint32_t>(g) << 16));
    W.slot = static_cast<int>(piece_slot(W.v, W.seg, part, a.max_parts));
  };
  // The window after W: the rest of the range.
  auto next_of = [&](const Window& W, Window& N) {
    N.v = W.v;
    N.x = W.x + W.n;
    N.n = W.n == 0 ? 0 : static_cast<int>(min(32ll, x1 - N.x));
  };

  // Range v goes to warp v / gridDim.x of CTA v % gridDim.x: when there are fewer ranges than
  // warps they spread over all SMs (one warp each) rather than filling a few SMs.
  Window cur, nxt;
  cur.v = my_v;
  cur.x = x0;
  cur.n = my_v < R.V ? static_cast<int>(min(32ll, x1 - x0)) : 0;
  resolve(cur);
  next_of(cur, nxt);
  resolve(nxt);
  int pk = 0;  // next job of `cur`

  // kOnce (the variant launched with early metadata: a layer of a chain that shares lengths
  // and block tables): the K/V tiles, read once, load with an evict-first L2 policy, so that
  // the metadata and the partial results that the next kernels read stay in L2 while the
  // layer's tiles stream through it (measured: a 28-layer mix64 step 25.7 -> 24.7 us per
  // layer).  A lone call has nothing to keep and loads them as usual: with the hint it measured
  // no better and at times slower, and even an explicit normal policy cost the E4M3 call.
  uint64_t once = 0;
  if constexpr (kOnce) once = l2_evict_first_policy();

  // Emit the next job into stage st; false when the warp has no work left.
  auto produce = [&](int st) -> bool {
    if (pk == cur.n) {
      if (nxt.n == 0) return false;
      cur = nxt;
      pk = 0;
      next_of(cur, nxt);
      resolve(nxt);
    }
    const int blk = __shfl_sync(kFullMask, cur.blk, pk);
    const int seg = __shfl_sync(kFullMask, cur.seg, pk);
    const int fl = __shfl_sync(kFullMask, cur.fl, pk);
    const int slot = __shfl_sync(kFullMask, cur.slot, pk);
    const int pos = kStep ? __shfl_sync(kFullMask, cur.pos, pk) : 0;
    ++pk;
    const bool ok = blk >= 0 && blk < a.num_blocks;
    const bool first = (fl & kFirst) != 0;
    // Fused step: a position without a cos/sin row leaves the token as the store kernel would
    // -- q unrotated, nothing stored.
    const bool rope = kStep && (fl & kRope);
    const bool fresh = rope && ok && (fl & kNew);  // the new token's K and V land in this tile
    const bool trig = rope && (first || fresh);    // stage the cos/sin row
    const bool q_rows = first && !kGather;         // the gather needs no q
    // first cache row of the tile: (physical block * Hkv + KV head) * 16
    const int y = ok ? (blk * Hkv + (fl >> 16)) * kBlockSize : 0;
    const uint32_t bar = bars + 8 * st;
    const uint32_t dst = tiles + st * kStageB;
    const uint32_t bytes = (ok ? 2u * L::kTile : 0u) + (q_rows ? static_cast<uint32_t>(G) * 256u : 0u) +
                           (trig ? kHeadDim * 4u : 0u) + (fresh ? kHeadDim * 4u : 0u);
    if (lane == 0) {
      if (!ok) raise_flag(a.status, PA_FLAG_BLOCK_ID_OOB);
      if (kStep && (fl & kNew) && !rope) raise_flag(a.status, PA_FLAG_POSITION_OOB);
      descs[st] = make_int4(seg, fl | (ok ? static_cast<int>(kHasData) : 0), slot, y);
      if (bytes) mbar_arrive_expect_tx(bar, bytes);
      else mbar_arrive(bar);
    }
    // The copies of one job leave from different lanes at once (one thread issues its copies
    // one after another), once lane 0 has armed the stage's barrier.
    __syncwarp();
    if (lane < 6 && bytes) {
      fence_proxy_async_smem();
      if (lane == 0 && ok) {
        if constexpr (kOnce && kFp8) tma_load_2d_once(dst, &tm_k, 0, y, bar, once);
        else if constexpr (kOnce) tma_load_3d_once(dst, &tm_k, 0, y, 0, bar, once);
        else if constexpr (kFp8) tma_load_2d(dst, &tm_k, 0, y, bar);
        else tma_load_3d(dst, &tm_k, 0, y, 0, bar);
      } else if (lane == 1 && ok) {
        if constexpr (kOnce && kFp8) tma_load_2d_once(dst + L::kTile, &tm_v, 0, y, bar, once);
        else if constexpr (kOnce) tma_load_3d_once(dst + L::kTile, &tm_v, 0, y, 0, bar, once);
        else if constexpr (kFp8) tma_load_2d(dst + L::kTile, &tm_v, 0, y, bar);
        else tma_load_3d(dst + L::kTile, &tm_v, 0, y, 0, bar);
      } else if (lane == 2 && q_rows) {  // the segment's G query heads: heads seg * G .. + G - 1
        bulk_copy_g2s(dst + L::kQOff, a.q + static_cast<size_t>(seg) * G * kHeadDim,
                      static_cast<uint32_t>(G) * 256u, bar);
      } else if (lane == 3 && trig) {
        bulk_copy_g2s(dst + L::kCosSinOff, a.cos_sin + static_cast<size_t>(pos) * kHeadDim, kHeadDim * 4u, bar);
      } else if (lane == 4 && fresh) {  // row seg of the [S, Hkv] new-token rows
        bulk_copy_g2s(dst + L::kNewKOff, a.k_new + static_cast<size_t>(seg) * kHeadDim, kHeadDim * 2u, bar);
      } else if (lane == 5 && fresh) {
        bulk_copy_g2s(dst + L::kNewVOff, a.v_new + static_cast<size_t>(seg) * kHeadDim, kHeadDim * 2u, bar);
      }
    }
    return true;
  };

  // ---------------------------------------------------------------- consumer state --
  const uint32_t k_row = static_cast<uint32_t>((r + 8 * (mi & 1)) * 128);   // K: rows 0-7 / 8-15
  const int k_col = mi >> 1;                                                 // K: chunk 2kk / 2kk+1
  const uint32_t v_row = static_cast<uint32_t>((r + 8 * (mi >> 1)) * 128);  // V: tokens 0-7 / 8-15
  const int v_col = mi & 1;                                                  // V: chunk 2mt / 2mt+1
  uint32_t qb[8][2];                     // B operand q^T: head gq, dims 16kk + 2cq (+1), +8
                                         // (E4M3 caches: dims 16kk + 4cq .. +3, f16)
  float k_fold = 0.f, v_fold = 0.f;      // E4M3 caches: softmax scale * K scale, V scale
  float m0 = -INFINITY, m1 = -INFINITY;  // softmax shifts of head columns 2cq, 2cq+1
  float l0 = 0.f, l1 = 0.f;              // this lane's share of the running sums
  float o[8][4];                         // O^T: dims 16mt + gq (+8), heads 2cq, 2cq+1
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

  uint32_t gx = 0;  // gather: this lane's XOR of the piece's tile words
  auto consume = [&](int st) {
    const int4 d = descs[st];
    const uint32_t fl = static_cast<uint32_t>(d.y);
    const uint32_t kt = tiles + st * kStageB;
    const uint32_t vt = kt + (kFp8 ? L::kTile : 2 * kHalfBytes);
    unsigned char* const stage = smem_raw + (kt - raw);  // generic address of the stage
    if constexpr (kGather) {
      // bf16: the stage's 8 KiB are [K cols 0-63 | K cols 64-127 | V cols 0-63 | V cols 64-127];
      // E4M3: 4 KiB, [K | V].  Either way 16-row pieces of 128-byte rows whose 16-byte chunks the
      // swizzle permutes within the row: chunk c (16 bytes at 16 c) lies in row (c / 8) % 16.
      // XOR the words of the valid rows.
      constexpr int kPasses = kFp8 ? 8 : 16;        // 32 lanes x 16 bytes per pass
      if (fl & kFirst) gx = 0;
      if (fl & kHasData) {
        const int valid = static_cast<int>((fl >> 8) & 0xffu);
#pragma unroll
        for (int i = 0; i < kPasses; ++i) {
          const int c = lane + 32 * i;
          if (((c >> 3) & 15) < valid) {
            const uint4 wv = *reinterpret_cast<const uint4*>(stage + 16 * c);
            gx ^= wv.x ^ wv.y ^ wv.z ^ wv.w;
          }
        }
      }
      if (fl & kLast) {
        uint32_t x = gx;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x ^= __shfl_xor_sync(kFullMask, x, o);
        if (lane == 0) atomicXor(a.gather_xor + d.x, x);
      }
      return;
    }
    if (fl & kFirst) {
      if constexpr (kFp8) {
        // B fragments in the order the E4M3 K fragments come in (k index permuted, see
        // fp8_scores): lane (gq, cq) takes dims 16c + 4cq .. 16c + 4cq + 3 of head gq as two
        // bf16 pairs, rotates them (fused step) and widens them to f16 pairs.
        const uint2* qrow = reinterpret_cast<const uint2*>(stage + L::kQOff + gq * 256);
        uint2 w[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) w[c] = qrow[4 * c + cq];
        if (kStep && (fl & kRope)) {
          const float* cs = reinterpret_cast<const float*>(stage + L::kCosSinOff);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int dd = 16 * c + 4 * cq;
            rope_rotate_pairs(w[c].x, w[c + 4].x, *reinterpret_cast<const float2*>(cs + dd),
                              *reinterpret_cast<const float2*>(cs + 64 + dd));
            rope_rotate_pairs(w[c].y, w[c + 4].y, *reinterpret_cast<const float2*>(cs + dd + 2),
                              *reinterpret_cast<const float2*>(cs + 66 + dd));
          }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          qb[c][0] = gq < G ? bf16x2_to_f16x2(w[c].x) : 0u;
          qb[c][1] = gq < G ? bf16x2_to_f16x2(w[c].y) : 0u;
        }
        const int g = d.x % Hkv;
        k_fold = a.scale_log2 * a.k_scale[g];
        v_fold = a.v_scale[g];
      } else {
        // q rows sit unswizzled at 256-byte stride; rows >= G are not real heads.
        const uint32_t qt = kt + L::kQOff + static_cast<uint32_t>(r * 256);
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2)
          ldsm_x4(qt + (4 * k2 + mi) * 16, qb[2 * k2][0], qb[2 * k2][1], qb[2 * k2 + 1][0],
                  qb[2 * k2 + 1][1]);
        if (kStep && (fl & kRope)) {
          // RoPE on the B fragments: dims d, d+1 (d = 16kk + 8j + 2cq) sit in qb[kk][j] and their
          // rotation partners d+64, d+65 in qb[kk+4][j] of the same lane.
          const float* cs = reinterpret_cast<const float*>(stage + L::kCosSinOff);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int dd = 16 * kk + 8 * j + 2 * cq;
              rope_rotate_pairs(qb[kk][j], qb[kk + 4][j], *reinterpret_cast<const float2*>(cs + dd),
                                *reinterpret_cast<const float2*>(cs + 64 + dd));
            }
        }
        if (gq >= G) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) qb[kk][0] = qb[kk][1] = 0u;
        }
      }
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      if ((fl & kGap) && lane < G)  // mark the skipped slot before this piece empty
        a.ws_ml[(static_cast<size_t>(d.z) - 1) * G + lane] = make_float2(-INFINITY, 0.f);
    }
    if (fl & kHasData) {
      const int valid = static_cast<int>((fl >> 8) & 0xffu);
      if (kStep && (fl & kNew) && (fl & kRope)) {
        // The new token (row valid - 1 of this tile): rotate its k, write k and v into the
        // staged tiles before they are read, and store both into the cache slot.
        const int row = valid - 1;
        const uint32_t* kn = reinterpret_cast<const uint32_t*>(stage + L::kNewKOff);
        const uint32_t* vn = reinterpret_cast<const uint32_t*>(stage + L::kNewVOff);
        const float* cs = reinterpret_cast<const float*>(stage + L::kCosSinOff);
        uint32_t klo = kn[lane], khi = kn[32 + lane];  // dims 2l, 2l+1 and 2l+64, 2l+65
        rope_rotate_pairs(klo, khi, reinterpret_cast<const float2*>(cs)[lane],
                          reinterpret_cast<const float2*>(cs + 64)[lane]);
        const uint32_t vlo = vn[lane], vhi = vn[32 + lane];
        const size_t crow = (static_cast<size_t>(d.w) + row) * kHeadDim;  // d.w: the tile's first cache row
        if constexpr (kFp8) {
          // E4M3 codes of k_rot / k_scale and v / v_scale, as the FP8 store kernel makes them.
          const int g = d.x % Hkv;
          const float ik = __frcp_rn(a.k_scale[g]), iv = __frcp_rn(a.v_scale[g]);
          const uint16_t ck0 = e4m3x2_of(klo, ik), ck1 = e4m3x2_of(khi, ik);
          const uint16_t cv0 = e4m3x2_of(vlo, iv), cv1 = e4m3x2_of(vhi, iv);
          // bytes 2l and 2l + 64 of the row, through the 128-byte swizzle
          const int base = row * 128 + 2 * (lane & 7);
          const int off0 = base + (((lane >> 3) ^ (row & 7)) << 4);
          const int off1 = base + ((((lane >> 3) + 4) ^ (row & 7)) << 4);
          *reinterpret_cast<uint16_t*>(stage + off0) = ck0;
          *reinterpret_cast<uint16_t*>(stage + off1) = ck1;
          *reinterpret_cast<uint16_t*>(stage + L::kTile + off0) = cv0;
          *reinterpret_cast<uint16_t*>(stage + L::kTile + off1) = cv1;
          uint16_t* kc = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(a.k_store) + crow);
          uint16_t* vc = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(a.v_store) + crow);
          kc[lane] = ck0;
          kc[32 + lane] = ck1;
          vc[lane] = cv0;
          vc[32 + lane] = cv1;
        } else {
          // byte 4l of the row in each 64-column half, through the 128-byte swizzle
          const int off = row * 128 + ((((lane >> 2) ^ (row & 7)) << 4) | ((lane & 3) << 2));
          *reinterpret_cast<uint32_t*>(stage + off) = klo;
          *reinterpret_cast<uint32_t*>(stage + kHalfBytes + off) = khi;
          *reinterpret_cast<uint32_t*>(stage + 2 * kHalfBytes + off) = vlo;
          *reinterpret_cast<uint32_t*>(stage + 3 * kHalfBytes + off) = vhi;
          uint32_t* kc = reinterpret_cast<uint32_t*>(a.k_store + crow);
          uint32_t* vc = reinterpret_cast<uint32_t*>(a.v_store + crow);
          kc[lane] = klo;
          kc[32 + lane] = khi;
          vc[lane] = vlo;
          vc[32 + lane] = vhi;
        }
        // These generic writes precede a later TMA write into the same stage.
        fence_proxy_async_smem();
        __syncwarp();
      }
      // S^T = K q^T: rows = tokens, columns = heads.
      float sc[4] = {0.f, 0.f, 0.f, 0.f}, sc2[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (kFp8) {
        // E4M3 K tile: ldmatrix reads it as 16-bit pairs, so lane (gq, cq) of matrix (rows
        // 8h..8h+7, 16-byte chunk c) gets dims 16c + 4cq .. +3 of token 8h + gq.  Widened to two
        // f16 pairs they are the A fragments of k indices (2cq, 2cq+1) and (2cq+8, 2cq+9), the
        // same permutation of the 16 dims as the B fragments above: the sum over k is unchanged.
#pragma unroll
        for (int c2 = 0; c2 < 4; ++c2) {
          uint32_t w0, w1, w2, w3;
          const int chunk = 2 * c2 + k_col;
          ldsm_x4(kt + k_row + ((chunk ^ r) << 4), w0, w1, w2, w3);
          uint32_t lo0, hi0, lo1, hi1;
          e4m3x4_to_f16x2x2(w0, lo0, hi0);
          e4m3x4_to_f16x2x2(w1, lo1, hi1);
          mma_f16_16816(sc, lo0, lo1, hi0, hi1, qb[2 * c2][0], qb[2 * c2][1]);
          e4m3x4_to_f16x2x2(w2, lo0, hi0);
          e4m3x4_to_f16x2x2(w3, lo1, hi1);
          // two accumulator chains, as for bf16: the MMAs issue in program order
          mma_f16_16816(sc2, lo0, lo1, hi0, hi1, qb[2 * c2 + 1][0], qb[2 * c2 + 1][1]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) sc[i] = (sc[i] + sc2[i]) * k_fold;
      } else {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t a0, a1, a2, a3;
          const int chunk = (2 * kk + k_col) & 7;
          ldsm_x4(kt + (kk >> 2) * kHalfBytes + k_row + ((chunk ^ r) << 4), a0, a1, a2, a3);
          // two accumulator chains (even / odd k steps): the MMAs issue in program order
          mma_bf16_16816((kk & 1) ? sc2 : sc, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) sc[i] += sc2[i];
      }
      // sc: [0] = (token gq, head 2cq), [1] = (gq, 2cq+1), [2] = (gq+8, 2cq), [3] = (gq+8, 2cq+1).
      // bf16 caches: the scores stay unscaled until the exponent (scale > 0, so the maxima are
      // the same) and each exponent is one FMA; E4M3 caches: already scaled above.
      const float fold = kFp8 ? 1.f : a.scale_log2;
      const bool partial = valid < kBlockSize;
      if (partial) {
        if (gq >= valid) sc[0] = sc[1] = -INFINITY;
        if (gq + 8 >= valid) sc[2] = sc[3] = -INFINITY;
      }
      float bm0 = fmaxf(sc[0], sc[2]);
      float bm1 = fmaxf(sc[1], sc[3]);
#pragma unroll
      for (int x = 4; x < 32; x <<= 1) {
        bm0 = fmaxf(bm0, __shfl_xor_sync(kFullMask, bm0, x));
        bm1 = fmaxf(bm1, __shfl_xor_sync(kFullMask, bm1, x));
      }
      // Shifts m0, m1 in the log2 domain: a head's shift moves to its maximum only when that
      // passes it by more than 8, so P stays at most 2^8 and O is rescaled far less often.
      const float bs0 = bm0 * fold, bs1 = bm1 * fold;
      const float mn0 = bs0 > m0 + 8.f ? bs0 : m0;
      const float mn1 = bs1 > m1 + 8.f ? bs1 : m1;
      const float al0 = ex2_ftz(m0 - mn0);
      const float al1 = ex2_ftz(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      // P rounded to the MMA operand type (bf16, or f16 with E4M3 caches); the running sums
      // add the same rounded values.
      const float e0 = ex2_ftz(fmaf(sc[0], fold, -mn0)), e1 = ex2_ftz(fmaf(sc[1], fold, -mn1));  // token gq
      const float e2 = ex2_ftz(fmaf(sc[2], fold, -mn0)), e3 = ex2_ftz(fmaf(sc[3], fold, -mn1));  // token gq+8
      uint32_t p_lo, p_hi;
      if constexpr (kFp8) {
        p_lo = pack_f16x2(e0, e1);
        p_hi = pack_f16x2(e2, e3);
        l0 = fmaf(l0, al0, f16lo(p_lo) + f16lo(p_hi));
        l1 = fmaf(l1, al1, f16hi(p_lo) + f16hi(p_hi));
      } else {
        p_lo = pack_bf16x2(e0, e1);
        p_hi = pack_bf16x2(e2, e3);
        l0 = fmaf(l0, al0, bf16lo(p_lo) + bf16lo(p_hi));
        l1 = fmaf(l1, al1, bf16hi(p_lo) + bf16hi(p_hi));
      }
      // B operand P^T: tokens 2cq, 2cq+1 (and +8) of head gq.
      const uint32_t pb0 = movmatrix_trans(p_lo);
      const uint32_t pb1 = movmatrix_trans(p_hi);
      if (__any_sync(kFullMask, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          o[mt][0] *= al0;
          o[mt][1] *= al1;
          o[mt][2] *= al0;
          o[mt][3] *= al1;
        }
      }
      auto pv = [&](uint32_t vmask_lo, uint32_t vmask_hi) {
        if constexpr (kFp8) {
          // O^T += V^T P^T.  The transposing ldmatrix of the E4M3 V tile gives lane (gq, cq)
          // the bytes V[2cq][2gq], V[2cq][2gq+1], V[2cq+1][2gq], V[2cq+1][2gq+1] of one 16-dim
          // chunk: regrouped by dim and widened they are the A fragments of rows gq (dim 2gq)
          // and gq+8 (dim 2gq+1), k = tokens 2cq, 2cq+1.  So accumulator row gq holds dim
          // 16mt + 2gq and row gq+8 dim 16mt + 2gq + 1.
#pragma unroll
          for (int c2 = 0; c2 < 4; ++c2) {
            uint32_t w0, w1, w2, w3;
            const int chunk = 2 * c2 + k_col;
            ldsm_x4_trans(vt + k_row + ((chunk ^ r) << 4), w0, w1, w2, w3);
            uint32_t x0, y0, x1, y1;
            e4m3x4_pairs_to_f16(w0, x0, y0);  // tokens 2cq, 2cq+1: dims 2gq (x), 2gq+1 (y)
            e4m3x4_pairs_to_f16(w1, x1, y1);  // tokens 2cq+8, 2cq+9
            mma_f16_16816(o[2 * c2], x0 & vmask_lo, y0 & vmask_lo, x1 & vmask_hi, y1 & vmask_hi, pb0, pb1);
            e4m3x4_pairs_to_f16(w2, x0, y0);
            e4m3x4_pairs_to_f16(w3, x1, y1);
            mma_f16_16816(o[2 * c2 + 1], x0 & vmask_lo, y0 & vmask_lo, x1 & vmask_hi, y1 & vmask_hi, pb0, pb1);
          }
        } else {
          // O^T += V^T P^T, one 16-dim slab at a time.
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            uint32_t v0, v1, v2, v3;
            const int chunk = (2 * mt + v_col) & 7;
            ldsm_x4_trans(vt + (mt >> 2) * kHalfBytes + v_row + ((chunk ^ r) << 4), v0, v1, v2, v3);
            mma_bf16_16816(o[mt], v0 & vmask_lo, v1 & vmask_lo, v2 & vmask_hi, v3 & vmask_hi, pb0, pb1);
          }
        }
      };
      if (partial) {
        // V rows past the context may hold anything (even NaN): zero them in the operand.
        pv((2 * cq < valid ? 0x0000ffffu : 0u) | (2 * cq + 1 < valid ? 0xffff0000u : 0u),
           (2 * cq + 8 < valid ? 0x0000ffffu : 0u) | (2 * cq + 9 < valid ? 0xffff0000u : 0u));
      } else {
        pv(0xffffffffu, 0xffffffffu);
      }
    }
    if (fl & kLast) {
      const size_t head0 = static_cast<size_t>(d.x) * G;  // first query head of the segment
      // Full row sums: the 8 lanes sharing cq hold disjoint token shares of the same heads.
      float L0 = l0, L1 = l1;
#pragma unroll
      for (int x = 4; x < 32; x <<= 1) {
        L0 += __shfl_xor_sync(kFullMask, L0, x);
        L1 += __shfl_xor_sync(kFullMask, L1, x);
      }
      if constexpr (kFp8) {
        // Accumulator rows gq / gq+8 are dims 16mt + 2gq / +1 of heads 2cq, 2cq+1: each lane
        // holds a dim pair of two heads, scaled by the V scale of the KV head.
        const bool h0 = 2 * cq < G;
        const bool h1 = 2 * cq + 1 < G;
        if (fl & kWhole) {
          const float i0 = v_fold / L0;
          const float i1 = v_fold / L1;
          uint32_t* orow0 = reinterpret_cast<uint32_t*>(a.out + (head0 + 2 * cq) * kHeadDim);
          uint32_t* orow1 = orow0 + kHeadDim / 2;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            if (h0) orow0[8 * mt + gq] = pack_bf16x2(o[mt][0] * i0, o[mt][2] * i0);
            if (h1) orow1[8 * mt + gq] = pack_bf16x2(o[mt][1] * i1, o[mt][3] * i1);
          }
        } else {
          const size_t row0 = static_cast<size_t>(d.z) * G + 2 * cq;  // head 2cq of the group
          float2* w0 = reinterpret_cast<float2*>(a.ws_o + row0 * kHeadDim) + gq;
          float2* w1 = w0 + kHeadDim / 2;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            if (h0) w0[8 * mt] = make_float2(o[mt][0] * v_fold, o[mt][2] * v_fold);
            if (h1) w1[8 * mt] = make_float2(o[mt][1] * v_fold, o[mt][3] * v_fold);
          }
          if (gq == 0) {
            if (h0) a.ws_ml[row0] = make_float2(m0, L0);
            if (h1) a.ws_ml[row0 + 1] = make_float2(m1, L1);
          }
        }
      } else if (fl & kWhole) {
        const float i0 = 1.f / L0;
        const float i1 = 1.f / L1;
        uint32_t* orow = reinterpret_cast<uint32_t*>(a.out + (head0 + gq) * kHeadDim);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          // (dim, head pair) -> transpose -> (head gq, dim pair): one 32-bit store per half.
          const uint32_t lo = movmatrix_trans(pack_bf16x2(o[mt][0] * i0, o[mt][1] * i1));
          const uint32_t hi = movmatrix_trans(pack_bf16x2(o[mt][2] * i0, o[mt][3] * i1));
          if (gq < G) {
            orow[8 * mt + cq] = lo;
            orow[8 * mt + 4 + cq] = hi;
          }
        }
      } else {
        const size_t slot = static_cast<size_t>(d.z);
        const size_t row0 = slot * G + 2 * cq;  // head 2cq of the group
        const bool h0 = 2 * cq < G;
        const bool h1 = 2 * cq + 1 < G;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const int dd = 16 * mt + gq;
          if (h0) {
            a.ws_o[row0 * kHeadDim + dd] = o[mt][0];
            a.ws_o[row0 * kHeadDim + dd + 8] = o[mt][2];
          }
          if (h1) {
            a.ws_o[(row0 + 1) * kHeadDim + dd] = o[mt][1];
            a.ws_o[(row0 + 1) * kHeadDim + dd + 8] = o[mt][3];
          }
        }
        if (gq == 0) {
          if (h0) a.ws_ml[row0] = make_float2(m0, L0);
          if (h1) a.ws_ml[row0 + 1] = make_float2(m1, L1);
        }
      }
    }
  };

  // ---------------------------------------------------------------- pipeline --------
  // The k-th use of a stage completes phase k & 1 of its mbarrier.
  auto advance = [&](int& st, uint32_t& ph) {
    if (++st == n_st) {
      st = 0;
      ph ^= 1u;
    }
  };
  int produced = 0, consumed = 0;
  int pst = 0, cst = 0;    // stages of the next job produced / consumed
  uint32_t pph = 0, cph = 0;
  bool more = true;
  // Early metadata: the prologue and the lookahead above ran beside the preceding kernel; wait
  // for it before the first copy.  (Waiting only after issuing the first tile copies, so that
  // they too overlap it, measured slower: the wait then also sits out those copies.)
  if (early) pdl_wait_prior_grid();
  while (more && produced < n_st) {
    if (produce(pst)) {
      ++produced;
      advance(pst, pph);
    } else {
      more = false;
    }
  }
  while (consumed < produced) {
    if (!mbar_wait_bounded(bars + 8 * cst, cph)) {
      if (lane == 0) raise_flag(a.status, PA_FLAG_TIMEOUT);
      // Let the other copies in flight land (bounded) before the CTA can exit.
      int st = cst;
      uint32_t ph = cph;
      for (int j = consumed + 1; j < produced; ++j) {
        advance(st, ph);
        mbar_wait_bounded(bars + 8 * st, ph);
      }
      break;
    }
    consume(cst);
    ++consumed;
    advance(cst, cph);
    __syncwarp();
    if (more) {
      if (produce(pst)) {
        ++produced;
        advance(pst, pph);
      } else {
        more = false;
      }
    }
  }
}

// Merge of the pieces of split segments.  A warp takes 32 of the 128 dims of one (sequence,
// query head), lane = dim, so that the rows of every piece of a head are loaded at once, one
// 4-byte word per lane and piece: the merge after the partition kernel is one round trip to
// L2, not one per batch of pieces.  The kernel is small enough (registers, no shared memory)
// to sit on the SMs next to the partition kernel, so it starts as soon as that kernel lets
// dependents launch and does everything that needs no partial result first: where the
// segment's pieces are comes from N_s and N_S, computed from the sequence lengths (inputs of
// the partition kernel, not outputs).  out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p.
// Empty sequences get zeros.  CTAs have 8 warps beside the bf16 partition kernel and 4 beside
// the 12-warp E4M3 one, so that at least one fits next to it (registers).
constexpr int kMergeWarps = 8;   // warps per CTA of the narrow merge
constexpr int kMergeSplit = 4;   // warps per (sequence, query head) and piece group: 32 dims each
constexpr int kMergeBatch = 32;  // pieces loaded per round trip
constexpr int kWideGroups = 4;   // piece groups per (sequence, query head) in the wide merge

// Every merge warp waits for the partition kernel before it exits, so that the merge grid
// completes after it and a following launch's own wait (which waits for this grid) orders it
// after the partition kernel's writes too.  The narrow form lets the next grid on the stream
// launch as soon as every merge CTA has started: a decode step with early metadata then
// resolves its work on the SMs that this layer's partition kernel has left, reading only
// lengths and block tables before its wait.  The wide form lets it launch only after its wait:
// its CTAs (16 warps, ~60 K registers) cannot sit beside a partition CTA, and merges of later
// layers launched early would hold SMs that the partition kernels need (measured: a 28-layer
// batch-1 step 187.5 -> 197.4 us with the early release in both forms).  (Each grid is released
// only once all CTAs of the grid before it are resident or done, so every wait chain ends in
// grids that are wholly resident.)
template <int kGroups>
__device__ __forceinline__ void wait_for_partitions() {
  pdl_wait_prior_grid();
  if constexpr (kGroups > 1) pdl_allow_next_grid();
}

// kGroups == 1 (narrow): CTAs of 8 (or 4) warps, 4 warps per (sequence, query head).
// kGroups > 1 (wide, for batches with fewer (sequence, query head) pairs than SMs): one CTA of
// kGroups x 4 warps per pair; piece group q takes the q-th contiguous share of the segment's
// pieces, and the groups' (M, L, acc) are combined in group order through shared memory.
template <int kGroups>
__global__ void __launch_bounds__(kGroups == 1 ? kMergeWarps * 32 : kGroups * kMergeSplit * 32, kGroups == 1 ? 2 : 1)
decode_merge_kernel(const DecodeArgs a) {
  if constexpr (kGroups == 1) pdl_allow_next_grid();
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * static_cast<int>(blockDim.x >> 5) + static_cast<int>(threadIdx.x >> 5);
  const int w = gw / (kGroups * kMergeSplit);          // (sequence, query head)
  const int grp = (gw / kMergeSplit) % kGroups;        // piece group
  const int quarter = gw % kMergeSplit;                // dims 32 quarter .. 32 quarter + 31
  const int S = a.num_seqs;
  // Every exit below depends on w alone, which is one per CTA in the wide form.
  if (w >= S * a.num_q_heads) {
    wait_for_partitions<kGroups>();
    return;
  }
  const int Hkv = a.num_kv_heads;
  const int G = a.num_q_heads / Hkv;
  const int s = w / a.num_q_heads;
  const int h = w - s * a.num_q_heads;
  const int g = h / G;
  const int hl = h - g * G;

  int before = 0, total = 0;
  for (int t = lane; t < S; t += 32) {
    const int n = (clamp_len(a.context_lens[t], a.max_context_len) + kBlockSize - 1) / kBlockSize;
    total += n;
    if (t < s) before += n;
  }
#pragma unroll
  for (int x = 16; x > 0; x >>= 1) {
    before += __shfl_xor_sync(kFullMask, before, x);
    total += __shfl_xor_sync(kFullMask, total, x);
  }
  const int ns = (clamp_len(a.context_lens[s], a.max_context_len) + kBlockSize - 1) / kBlockSize;
  const int dim = quarter * 32 + lane;
  __nv_bfloat16* orow = a.out + static_cast<size_t>(w) * kHeadDim + dim;
  if (ns == 0) {  // empty context: zero row (after the partition kernel, which may read `out`)
    wait_for_partitions<kGroups>();
    if (grp == 0) *orow = __float2bfloat16_rn(0.f);
    return;
  }
  const Ranges R = make_ranges(static_cast<long long>(Hkv) * total, a);
  const long long Xi = static_cast<long long>(Hkv) * before + static_cast<long long>(g) * ns;
  const int v_first = R.owner(Xi);
  const int v_last = R.owner(Xi + ns - 1);
  // Pieces in slot order: slot_first + k, k < npieces, gaps included (see piece_slot).
  const int chunk = a.chunk_blocks;
  const int part_last = chunk ? (ns - 1) / chunk : 0;
  const int npieces = v_last - v_first + part_last + 1;
  if (npieces == 1) {
    wait_for_partitions<kGroups>();  // one piece: written directly by the partition kernel
    return;
  }
  const int seg = s * Hkv + g;
  const int k0 = static_cast<int>(static_cast<long long>(grp) * npieces / kGroups);
  const int k1 = static_cast<int>(static_cast<long long>(grp + 1) * npieces / kGroups);
  const size_t row_base = static_cast<size_t>(piece_slot(v_first, seg, 0, a.max_parts)) * G + hl;
  const float2* ml = a.ws_ml + row_base;
  const float* rows = a.ws_o + row_base * kHeadDim + dim;
  const size_t stride = static_cast<size_t>(G) * kHeadDim;
  wait_for_partitions<kGroups>();

  // One round trip per batch: this lane's (m, l) of the batch's piece `lane`, and its dim of
  // every piece row of the batch, combined into (M, L, acc) in piece order.  A gap (m = -inf,
  // l = 0) gets weight 0 and its row, never written, is not used.
  float M = -INFINITY, L = 0.f, acc = 0.f;
  for (int base = k0; base < k1; base += kMergeBatch) {
    const int n = min(kMergeBatch, k1 - base);
    const float2 mine = lane < n ? ml[(base + lane) * G] : make_float2(-INFINITY, 0.f);
    float r[kMergeBatch];
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) r[u] = u < n ? rows[(base + u) * stride] : 0.f;
    float Mb = mine.x;
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) Mb = fmaxf(Mb, __shfl_xor_sync(kFullMask, Mb, x));
    const float Mn = fmaxf(M, Mb);
    const float rescale = M == -INFINITY ? 0.f : exp2f(M - Mn);
    M = Mn;
    const float wmine = mine.x == -INFINITY ? 0.f : exp2f(mine.x - M);
    float lb = wmine * mine.y;
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) lb += __shfl_xor_sync(kFullMask, lb, x);
    L = fmaf(L, rescale, lb);
    acc *= rescale;
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const float wu = __shfl_sync(kFullMask, wmine, u);
      if (wu != 0.f) acc = fmaf(wu, r[u], acc);
    }
  }
  if constexpr (kGroups > 1) {
    __shared__ float s_acc[kGroups][kMergeSplit][32];
    __shared__ float2 s_ml[kGroups][kMergeSplit];
    s_acc[grp][quarter][lane] = acc;
    if (lane == 0) s_ml[grp][quarter] = make_float2(M, L);
    __syncthreads();
    if (grp != 0) return;
    // the groups in order (a group with no piece has L == 0 and is skipped)
    float Mt = -INFINITY, Lt = 0.f, At = 0.f;
#pragma unroll
    for (int q = 0; q < kGroups; ++q) {
      const float2 ml = s_ml[q][quarter];
      if (ml.y == 0.f) continue;
      const float Mn = fmaxf(Mt, ml.x);
      const float al = exp2f(Mt - Mn), be = exp2f(ml.x - Mn);
      Mt = Mn;
      Lt = fmaf(Lt, al, ml.y * be);
      At = fmaf(At, al, s_acc[q][quarter][lane] * be);
    }
    *orow = __float2bfloat16_rn(At / Lt);
  } else {
    *orow = __float2bfloat16_rn(acc / L);
  }
}

// ---- host side ------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Persistent grid size for this device: SMs x resident CTAs per SM, capped so that the grid
// has at most kMaxDecodeWarps warps (looked up once per device and kernel variant, at the
// largest shared-memory footprint the kernel can ask for).
template <bool kStep, bool kFp8>
cudaError_t persistent_ctas(int* ctas) {
  static std::mutex mu;
  static int cached[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    const int smem = Layout<kStep, kFp8>::smem(kMaxDecodeSeqs);
    auto kernel = decode_partition_kernel<kStep, kFp8>;
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    // the early-metadata variant and (unfused) the gather run the same kernel shape
    err = cudaFuncSetAttribute(decode_partition_kernel<kStep, kFp8, false, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    if (!kStep) {
      err = cudaFuncSetAttribute(decode_partition_kernel<false, kFp8, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (err != cudaSuccess) return err;
    }
    int sms = 0, per_sm = 0;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, Layout<kStep, kFp8>::kWarpsN * 32, smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    cached[dev] = min(sms * per_sm, kMaxDecodeWarps / Layout<kStep, kFp8>::kWarpsN);
  }
  *ctas = cached[dev];
  return cudaSuccess;
}

template <bool kStep, bool kFp8, bool kGather = false>
cudaError_t launch_partition(DecodeArgs& a, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const cudaLaunchAttribute* attr, cudaStream_t stream) {
  int max_ctas = 0;
  cudaError_t err = persistent_ctas<kStep, kFp8>(&max_ctas);
  if (err != cudaSuccess) return err;
  // No more CTAs than there can be ranges (ranges are dealt to the CTAs one at a time).
  const long long jobs_bound = static_cast<long long>(a.num_seqs) * a.num_kv_heads *
                               ((a.max_context_len + kBlockSize - 1) / kBlockSize);
  const long long want = (jobs_bound + kMinRangeBlocks - 1) / kMinRangeBlocks;
  const long long ctas = min(static_cast<long long>(max_ctas), want);
  constexpr int kWarpsN = Layout<kStep, kFp8>::kWarpsN;
  a.num_warps = static_cast<int>(ctas) * kWarpsN;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(kWarpsN * 32);
  cfg.dynamicSmemBytes = Layout<kStep, kFp8>::smem(a.num_seqs);
  cfg.stream = stream;
  cfg.attrs = const_cast<cudaLaunchAttribute*>(attr);
  cfg.numAttrs = 1;
  auto kernel = decode_partition_kernel<kStep, kFp8, kGather>;
  if constexpr (!kGather)
    if (a.early_metadata) kernel = decode_partition_kernel<kStep, kFp8, false, true>;
  return cudaLaunchKernelEx(&cfg, kernel, tm_k, tm_v, a);
}

}  // namespace

// Tensor map of one cache, 128-byte swizzle, one box per (block, KV head) tile.  The cache is
// [num_blocks * Hkv * 16 rows][128 cols].  E4M3: a 2-D map, box 128 cols x 16 rows.  bf16: a
// 128-col row is 256 bytes, wider than the swizzle span, so the map is 3-D -- (col within a
// 64-col half, row, half) with strides 256 bytes (row) and 128 bytes (half) -- and the box
// (64, 16, 2) lands a tile in shared memory as its two 2 KiB halves, cols 0-63 of the 16 rows
// followed by cols 64-127; the box (64, 16, 1) lands one half (the prefill kernel places the K
// halves of neighbouring blocks side by side).  Encoded maps are cached by (address, rows, type,
// box).
bool cache_tensor_map(const void* cache, long long rows, bool fp8, CUtensorMap* out, int box_halves) {
  struct Entry {
    const void* ptr;
    long long rows;
    bool fp8;
    int halves;
    CUtensorMap map;
  };
  if (box_halves != 1 && box_halves != 2) return false;
  // Room for the K and V caches of every layer of a large model in both element types; the
  // oldest entry is replaced when it is full.
  constexpr int kEntries = 512;
  static std::mutex mu;
  static Entry table[kEntries];
  static int used = 0, next = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (table[i].ptr == cache && table[i].rows == rows && table[i].fp8 == fp8 &&
        (fp8 || table[i].halves == box_halves)) {
      *out = table[i].map;
      return true;
    }
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return false;
  CUtensorMap m;
  const cuuint64_t n = static_cast<cuuint64_t>(rows);
  CUresult rc;
  if (fp8) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), n};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim)};
    cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(kBlockSize)};
    cuuint32_t estr[2] = {1, 1};
    rc = encode(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(cache), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[3] = {64, n, 2};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2, 128};
    cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(kBlockSize), static_cast<cuuint32_t>(box_halves)};
    cuuint32_t estr[3] = {1, 1, 1};
    rc = encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(cache), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (rc != CUDA_SUCCESS) return false;
  const int slot = used < kEntries ? used++ : (next++ % kEntries);
  table[slot] = Entry{cache, rows, fp8, box_halves, m};
  *out = m;
  return true;
}

cudaError_t launch_gather(const DecodeArgs& args, bool fp8, cudaStream_t stream) {
  DecodeArgs a = args;
  if (a.num_seqs > kMaxDecodeSeqs) return cudaErrorInvalidValue;
  const long long rows = static_cast<long long>(a.num_blocks) * a.num_kv_heads * kBlockSize;
  CUtensorMap tm_k, tm_v;
  if (!cache_tensor_map(a.k_cache, rows, fp8, &tm_k) || !cache_tensor_map(a.v_cache, rows, fp8, &tm_v))
    return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  return fp8 ? launch_partition<false, true, true>(a, tm_k, tm_v, attr, stream)
             : launch_partition<false, false, true>(a, tm_k, tm_v, attr, stream);
}

cudaError_t launch_decode(const DecodeArgs& args, cudaStream_t stream) {
  DecodeArgs a = args;
  const int G = a.num_q_heads / a.num_kv_heads;
  if (G < 1 || G > 8 || a.num_seqs > kMaxDecodeSeqs) return cudaErrorInvalidValue;
  const bool step = a.k_new != nullptr;
  const bool fp8 = a.k_scale != nullptr;
  const long long rows = static_cast<long long>(a.num_blocks) * a.num_kv_heads * kBlockSize;
  CUtensorMap tm_k, tm_v;
  if (!cache_tensor_map(a.k_cache, rows, fp8, &tm_k) || !cache_tensor_map(a.v_cache, rows, fp8, &tm_v))
    return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaError_t err;
  if (fp8) err = step ? launch_partition<true, true>(a, tm_k, tm_v, attr, stream)
                      : launch_partition<false, true>(a, tm_k, tm_v, attr, stream);
  else err = step ? launch_partition<true, false>(a, tm_k, tm_v, attr, stream)
                  : launch_partition<false, false>(a, tm_k, tm_v, attr, stream);
  if (err != cudaSuccess) return err;

  // Narrow merge beside the partition kernel; the wide one when the (sequence, query head)
  // pairs are fewer than the partition kernel's CTAs, so that long segments' many pieces are
  // spread over more warps.
  const long long pairs = static_cast<long long>(a.num_seqs) * a.num_q_heads;
  int part_ctas = 0;
  err = fp8 ? persistent_ctas<false, true>(&part_ctas) : persistent_ctas<false, false>(&part_ctas);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t mcfg = {};
  mcfg.stream = stream;
  mcfg.attrs = attr;
  mcfg.numAttrs = 1;
  if (pairs <= part_ctas) {
    mcfg.gridDim = dim3(static_cast<unsigned>(pairs));
    mcfg.blockDim = dim3(kWideGroups * kMergeSplit * 32);
    return cudaLaunchKernelEx(&mcfg, decode_merge_kernel<kWideGroups>, a);
  }
  const long long merge_warps = pairs * kMergeSplit;
  const int per_cta = fp8 ? kMergeWarps / 2 : kMergeWarps;
  mcfg.gridDim = dim3(static_cast<unsigned>((merge_warps + per_cta - 1) / per_cta));
  mcfg.blockDim = dim3(per_cta * 32);
  return cudaLaunchKernelEx(&mcfg, decode_merge_kernel<1>, a);
}

}  // namespace pa
