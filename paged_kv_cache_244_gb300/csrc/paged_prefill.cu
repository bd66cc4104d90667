// Paged (chunked) prefill attention for sm_103a.
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
// CTA = (sequence, KV head g, tile of 16 query tokens), one warp per query head of the group
// (G <= 8 warps), so every K/V tile brought in is used by all G heads.  Each warp holds its
// 16 x 128 Q tile as MMA A fragments and walks the key blocks 0 .. p_last / 16:
//   S (16 x 64) = Q K^T      64 mma.sync m16n8k16 (bf16 -> fp32), B = K via ldmatrix
//   online softmax           per row, in the log2 domain, the scale folded into one FMA per
//                            exponent; a row's shift moves only when its maximum passes it by
//                            more than 8 (P <= 2^8, few O rescales); causal mask t > p_i only on
//                            the stages that reach the tile's diagonal; V rows past the context
//                            zeroed in the operand (they may hold anything), in the context's
//                            last block only
//   O (16 x 128) += P V      64 MMAs; P is the S accumulators rounded to bf16 (the C layout of
//                            two n8 tiles is the A layout of one k16 step), B = V via
//                            transposing ldmatrix
// Keys come 64 at a time (4 blocks) through a 2-stage ring, so the softmax bookkeeping and the
// handshakes are paid once per 128 MMAs: the warp whose release of stage j is the last of the
// G (a shared-memory count) issues at once the TMA tensor loads of stage j + 2 (one box per K
// tile and per V tile, landing as two 64-column halves, 128-byte swizzle), so no warp waits
// for the others.  Measured against 3 stages of 48 keys, 2 of 64 are 1-2% faster; 4 of 32
// were slower.  All waits are bounded.
// Tiles are scheduled latest first over the whole grid: the last tiles of a sequence see the
// most keys.

#include <mutex>

#include <cuda.h>

#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {
namespace {

constexpr int kQTile = 16;                          // query tokens per CTA
constexpr int kKB = 4;                              // key blocks (16 tokens each) per stage
constexpr int kPfStages = 2;
constexpr int kPfMaxWarps = 8;                      // G <= 8
constexpr int kPfHalf = kBlockSize * 128;           // 16 rows x 64 bf16
constexpr int kPfBlockBytes = 2 * kTileBytes;       // K tile + V tile of one key block
constexpr int kPfStageBytes = kKB * kPfBlockBytes;  // 32 KiB
constexpr int kPfQBytes = kQTile * kHeadDim * 2;    // one warp's Q tile: 4 KiB
// header: per stage a full mbarrier, a block-present mask and a release count; then the
// 1024-aligned stages and the Q tiles
constexpr int kPfHeader = 1024;
constexpr int kPfSmem = kPfHeader + kPfStages * kPfStageBytes + kPfMaxWarps * kPfQBytes + 1024;

__global__ void __maxnreg__(168)  // two CTAs of up to 6 warps per SM; 8 warps still fit one
prefill_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               const PrefillArgs a) {
  extern __shared__ unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Hkv = a.num_kv_heads;
  const int G = a.num_q_heads / Hkv;
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
  const int i0 = tile * kQTile;
  if (i0 >= n) return;
  const int rows = min(kQTile, n - i0);
  const int pos0 = ctx - n + i0;                    // position of the tile's first query
  const int nblocks = (pos0 + rows - 1) / kBlockSize + 1;
  const int nst = (nblocks + kKB - 1) / kKB;        // stages of kKB key blocks

  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t full = raw;                        // kPfStages x 8 bytes
  int* present = reinterpret_cast<int*>(smem_raw + 8 * kPfStages);   // bit i: block i loaded
  // per stage: releases so far, G a round; the release that completes a round refills it
  unsigned* released = reinterpret_cast<unsigned*>(smem_raw + 12 * kPfStages);
  const uint32_t stages = (raw + kPfHeader + 1023u) & ~1023u;
  const uint32_t qtiles = stages + kPfStages * kPfStageBytes;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kPfStages; ++i) {
      mbar_init(full + 8 * i, 1);
      released[i] = 0u;
    }
    fence_mbar_init();
    prefetch_tensor_map(&tm_k);
    prefetch_tensor_map(&tm_v);
  }
  __syncthreads();

  // Bring key blocks kKB j .. kKB j + kKB - 1 into stage j % kPfStages (one thread).
  const int32_t* bt_row = a.block_tables + static_cast<size_t>(s) * a.max_blocks;
  auto issue = [&](int j) {
    const int st = j % kPfStages;
    int blk[kKB];
    int mask = 0;
#pragma unroll
    for (int i = 0; i < kKB; ++i) {
      const int b = kKB * j + i;
      blk[i] = b < nblocks ? bt_row[b] : -1;
      if (b < nblocks && blk[i] >= 0 && blk[i] < a.num_blocks) mask |= 1 << i;
      else if (b < nblocks) raise_flag(a.status, PA_FLAG_BLOCK_ID_OOB);
    }
    present[st] = mask;
    const uint32_t bar = full + 8 * st;
    const uint32_t dst = stages + st * kPfStageBytes;
    fence_proxy_async_smem();
    if (mask) {
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(__popc(mask)) * kPfBlockBytes);
#pragma unroll
      for (int i = 0; i < kKB; ++i) {
        if (!(mask & (1 << i))) continue;
        const int y = (blk[i] * Hkv + g) * kBlockSize;
        const uint32_t d = dst + i * kPfBlockBytes;
        tma_load_3d(d, &tm_k, 0, y, 0, bar);              // both 64-col halves of the K tile
        tma_load_3d(d + 2 * kPfHalf, &tm_v, 0, y, 0, bar);
      }
    } else {
      mbar_arrive(bar);
    }
  };
  if (threadIdx.x == 0)
    for (int j = 0; j < min(kPfStages, nst); ++j) issue(j);

  // ---- this warp's Q tile (query head g * G + warp) as A fragments ------------------------
  const int h = g * G + warp;
  const int gq = lane >> 2, cq = lane & 3;          // fragment row group / column pair
  const int mi = lane >> 3, r = lane & 7;           // ldmatrix: matrix / row this lane addresses
  const uint32_t qs = qtiles + warp * kPfQBytes;
  {
    // row = query i0 + row (zero past the tile), 16 chunks of 16 bytes, chunk c at c ^ (row % 8)
    unsigned char* qgen = smem_raw + (qs - raw);
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int idx = it * 32 + lane;
      const int row = idx >> 4, c = idx & 15;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (row < rows)
        v = reinterpret_cast<const uint4*>(a.q + (static_cast<size_t>(q0 + i0 + row) * a.num_q_heads + h) *
                                                     kHeadDim)[c];
      *reinterpret_cast<uint4*>(qgen + row * 256 + ((c ^ (row & 7)) << 4)) = v;
    }
  }
  __syncwarp();
  uint32_t qa[8][4];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const int row = r + 8 * (mi & 1);
    const int c = 2 * kk + (mi >> 1);
    ldsm_x4(qs + row * 256 + ((c ^ r) << 4), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
  }

  float o[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows gq, gq + 8
  const int p0 = pos0 + gq, p1 = pos0 + gq + 8;               // their positions
  bool failed = false;
  int seen = 0;                                               // stages this warp waited for

  for (int j = 0; j < nst; ++j) {
    const int st = j % kPfStages;
    if (!mbar_wait_bounded(full + 8 * st, (j / kPfStages) & 1)) {
      failed = true;
      break;
    }
    seen = j + 1;
    const int mask = present[st];
    const uint32_t stage = stages + st * kPfStageBytes;
    // S = Q K^T for the stage's 16 kKB keys: n8 tile 2i (+1) = keys 0-7 (8-15) of block i.
    // k steps outside, blocks inside: 2 kKB independent accumulator chains between two MMAs
    // of one chain (the MMAs issue in program order).
    float sc[2 * kKB][4];
#pragma unroll
    for (int nt = 0; nt < 2 * kKB; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
    const int key = r + 8 * (mi >> 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int chunk = (2 * kk + (mi & 1)) & 7;
      const uint32_t ko = (kk >> 2) * kPfHalf + key * 128 + ((chunk ^ r) << 4);
#pragma unroll
      for (int i = 0; i < kKB; ++i) {
        if (!(mask & (1 << i))) continue;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(stage + i * kPfBlockBytes + ko, b0, b1, b2, b3);
        mma_bf16_16816(sc[2 * i], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
        mma_bf16_16816(sc[2 * i + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
      }
    }
    // Scores stay unscaled until the exponent (scale > 0, so the row maxima are the same).
    // Causal mask and missing blocks -> -inf, only on a stage that reaches past the tile's first
    // query or lacks a block; the others lie wholly before every query of the tile.
    // sc[nt]: [0] (row gq, key 8nt+2cq), [1] (gq, +1), [2] (gq+8, 8nt+2cq), [3] (gq+8, +1)
    if (mask != (1 << kKB) - 1 || kKB * kBlockSize * (j + 1) - 1 > pos0) {
      const int tbase = kKB * kBlockSize * j + 2 * cq;
#pragma unroll
      for (int nt = 0; nt < 2 * kKB; ++nt) {
        const bool here = (mask >> (nt >> 1)) & 1;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = tbase + 8 * nt + e;
          if (!(here && t <= p0)) sc[nt][e] = -INFINITY;
          if (!(here && t <= p1)) sc[nt][2 + e] = -INFINITY;
        }
      }
    }
    float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2 * kKB; ++nt) {
      bm0 = fmaxf(bm0, fmaxf(sc[nt][0], sc[nt][1]));
      bm1 = fmaxf(bm1, fmaxf(sc[nt][2], sc[nt][3]));
    }
#pragma unroll
    for (int x = 1; x < 4; x <<= 1) {
      bm0 = fmaxf(bm0, __shfl_xor_sync(kFullMask, bm0, x));
      bm1 = fmaxf(bm1, __shfl_xor_sync(kFullMask, bm1, x));
    }
    // Shifts m0, m1 in the log2 domain (scale * log2(e) applied): a row's shift moves to its
    // maximum only when that exceeds it by more than 8, so P stays at most 2^8 and O is rescaled
    // far less often.
    const float bs0 = bm0 * a.scale_log2, bs1 = bm1 * a.scale_log2;
    const float mn0 = bs0 > m0 + 8.f ? bs0 : m0, mn1 = bs1 > m1 + 8.f ? bs1 : m1;
    // a row with no key yet keeps the shift 0 (only rows past the tile can stay that way)
    const float sh0 = mn0 == -INFINITY ? 0.f : mn0;
    const float sh1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = ex2_ftz(m0 - sh0), al1 = ex2_ftz(m1 - sh1);
    m0 = mn0;
    m1 = mn1;
    // P = 2^(scale_log2 * s - shift), one FMA and one exp2 per score, rounded to bf16 (the MMA
    // operand) as A fragments of one k16 step per block; the running sums add the same
    // rounded values
    const float sl = a.scale_log2;
    uint32_t pa[kKB][4];
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int i = 0; i < kKB; ++i) {
      pa[i][0] = pack_bf16x2(ex2_ftz(fmaf(sc[2 * i][0], sl, -sh0)), ex2_ftz(fmaf(sc[2 * i][1], sl, -sh0)));
      pa[i][1] = pack_bf16x2(ex2_ftz(fmaf(sc[2 * i][2], sl, -sh1)), ex2_ftz(fmaf(sc[2 * i][3], sl, -sh1)));
      pa[i][2] = pack_bf16x2(ex2_ftz(fmaf(sc[2 * i + 1][0], sl, -sh0)), ex2_ftz(fmaf(sc[2 * i + 1][1], sl, -sh0)));
      pa[i][3] = pack_bf16x2(ex2_ftz(fmaf(sc[2 * i + 1][2], sl, -sh1)), ex2_ftz(fmaf(sc[2 * i + 1][3], sl, -sh1)));
      ps0 += bf16lo(pa[i][0]) + bf16hi(pa[i][0]) + bf16lo(pa[i][2]) + bf16hi(pa[i][2]);
      ps1 += bf16lo(pa[i][1]) + bf16hi(pa[i][1]) + bf16lo(pa[i][3]) + bf16hi(pa[i][3]);
    }
    l0 = fmaf(l0, al0, ps0);
    l1 = fmaf(l1, al1, ps1);
    if (__any_sync(kFullMask, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        o[nt][0] *= al0;
        o[nt][1] *= al0;
        o[nt][2] *= al1;
        o[nt][3] *= al1;
      }
    }
    // O += P V, block by block; two n8 dim tiles per transposing ldmatrix
    auto pv = [&](int i, uint32_t vm_lo, uint32_t vm_hi) {
      const uint32_t vt = stage + i * kPfBlockBytes + 2 * kPfHalf;
#pragma unroll
      for (int d2 = 0; d2 < 8; ++d2) {
        uint32_t v0, v1, v2, v3;
        const int key = r + 8 * (mi & 1);
        const int chunk = (2 * d2 + (mi >> 1)) & 7;
        ldsm_x4_trans(vt + (d2 >> 2) * kPfHalf + key * 128 + ((chunk ^ r) << 4), v0, v1, v2, v3);
        mma_bf16_16816(o[2 * d2], pa[i][0], pa[i][1], pa[i][2], pa[i][3], v0 & vm_lo, v1 & vm_hi);
        mma_bf16_16816(o[2 * d2 + 1], pa[i][0], pa[i][1], pa[i][2], pa[i][3], v2 & vm_lo, v3 & vm_hi);
      }
    };
#pragma unroll
    for (int i = 0; i < kKB; ++i) {
      if (!(mask & (1 << i))) continue;
      const int valid = ctx - kBlockSize * (kKB * j + i);
      if (valid >= kBlockSize) {
        pv(i, 0xffffffffu, 0xffffffffu);
      } else {
        // keys past the context may hold anything (even NaN): zero their V rows in the operand
        pv(i, (2 * cq < valid ? 0x0000ffffu : 0u) | (2 * cq + 1 < valid ? 0xffff0000u : 0u),
           (2 * cq + 8 < valid ? 0x0000ffffu : 0u) | (2 * cq + 9 < valid ? 0xffff0000u : 0u));
      }
    }
    // Release the stage.  The warp whose release is the G-th of this round refills it at once,
    // so no warp waits for the others here.
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();  // this warp's reads of the stage before the refill's writes
      const unsigned before = atomicAdd(&released[st], 1u);
      if ((before + 1u) % static_cast<unsigned>(G) == 0u && j + kPfStages < nst) {
        __threadfence_block();
        issue(j + kPfStages);
      }
    }
    __syncwarp();
  }
  if (failed && lane == 0) {
    raise_flag(a.status, PA_FLAG_TIMEOUT);
    // Only stages seen .. seen + kPfStages - 1 can have copies in flight (a stage is refilled
    // after every warp released its previous round, and this warp released none from `seen`
    // on): let them land (bounded; a stage never refilled gives up after 10 ms) before the
    // CTA can exit.
    for (int j = seen; j < min(nst, seen + kPfStages); ++j)
      mbar_wait_bounded(full + 8 * (j % kPfStages), (j / kPfStages) & 1, 10000000ull);
  }
  if (failed) return;

  // ---- out = O / l for the tile's real rows -----------------------------------------------
  float L0 = l0, L1 = l1;
#pragma unroll
  for (int x = 1; x < 4; x <<= 1) {
    L0 += __shfl_xor_sync(kFullMask, L0, x);
    L1 += __shfl_xor_sync(kFullMask, L1, x);
  }
  const float i0f = 1.f / L0, i1f = 1.f / L1;
  uint32_t* out0 = reinterpret_cast<uint32_t*>(
      a.out + (static_cast<size_t>(q0 + i0 + gq) * a.num_q_heads + h) * kHeadDim);
  uint32_t* out1 = reinterpret_cast<uint32_t*>(
      a.out + (static_cast<size_t>(q0 + i0 + gq + 8) * a.num_q_heads + h) * kHeadDim);
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    if (gq < rows) out0[4 * nt + cq] = pack_bf16x2(o[nt][0] * i0f, o[nt][1] * i0f);
    if (gq + 8 < rows) out1[4 * nt + cq] = pack_bf16x2(o[nt][2] * i1f, o[nt][3] * i1f);
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  const int G = a.num_q_heads / a.num_kv_heads;
  if (G < 1 || G > kPfMaxWarps) return cudaErrorInvalidValue;
  const long long rows = static_cast<long long>(a.num_blocks) * a.num_kv_heads * kBlockSize;
  CUtensorMap tm_k, tm_v;
  if (!cache_tensor_map(a.k_cache, rows, false, &tm_k) || !cache_tensor_map(a.v_cache, rows, false, &tm_v))
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
      done[dev] = true;
    }
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((a.max_query_len + kQTile - 1) / kQTile),
                     static_cast<unsigned>(a.num_seqs * a.num_kv_heads));
  cfg.blockDim = dim3(static_cast<unsigned>(G * 32));
  cfg.dynamicSmemBytes = kPfSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_kernel, tm_k, tm_v, a);
}

}  // namespace pa
