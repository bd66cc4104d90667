// Single-token paged GQA decode attention for sm_103a, with Flash-Decode partitions.
//
// "Pico-vLLM：从零手写的工业级LLM推理引擎实现": §2 Kernel层 (PagedAttention decode kernel),
// §1 模型实现层 (GQA), §H200上的详细对比 (Flash Decode); "从零实现 LLM 推理引擎：深挖 vLLM 的
// 六大核心优化", §3.1 Paged KV Cache (16-token blocks reached through a block table).
//
// Work unit = (partition, sequence, KV head), one warp each; a CTA holds kWarps units.  The
// warp serves all G query heads of its KV head, so each (block, KV head) tile of K and V is
// read from HBM exactly once.  Per block the warp:
//   1. has the 4 KiB K tile and 4 KiB V tile in shared memory, brought by two bulk async
//      copies (cp.async.bulk, completion on an mbarrier) issued kStages blocks ahead, the
//      physical id coming from the block table;
//   2. computes the 16 x G scores in fp32 (lane l owns dims 4l..4l+3 for every head, then a
//      butterfly that halves the live values each step turns 32 partial sums per score into
//      G/2 finished scores per lane: lane l ends with token l/2, heads (l&1)*G/2 + i);
//   3. updates the online softmax (running max m, running sum l, rescale factor
//      exp2(m_old - m_new)) in the log2 domain, scale * log2(e) folded into q;
//   4. accumulates p * V into 4 dims x G heads per lane.
// A unit whose sequence fits in one partition writes bf16 `out`; otherwise it writes its
// partial (sum p V, (m, l)) to the workspace and decode_merge_kernel combines partitions:
//   M = max_p m_p,  out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p.

#include <cmath>
#include <mutex>

#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {
namespace {

constexpr int kWarps = 4;
constexpr int kStages = 3;
constexpr int kStageBytes = 2 * kTileBytes;              // K tile + V tile
constexpr int kSmemBytes = kWarps * kStages * kStageBytes + kWarps * kStages * 8;

template <int GP>
__global__ void __launch_bounds__(kWarps * 32) decode_partition_kernel(const DecodeArgs a) {
  constexpr int HPL = GP / 2;       // heads per lane after the butterfly
  constexpr int NV = 16 * GP;       // partial scores per block (token-major: t * GP + h)
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  unsigned char* tiles = smem + warp * kStages * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWarps * kStages * kStageBytes) + warp * kStages;
  if (lane == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(smem_addr(&bars[st]), 1);
    fence_mbar_init();
  }
  __syncwarp();
  pdl_wait_prior_grid();
  pdl_allow_next_grid();

  const int units_per_part = a.num_seqs * a.num_kv_heads;
  const int unit = blockIdx.x * kWarps + warp;
  if (unit >= units_per_part * a.max_parts) return;
  const int part = unit / units_per_part;
  const int rem = unit - part * units_per_part;
  const int s = rem / a.num_kv_heads;
  const int g = rem - s * a.num_kv_heads;
  const int G = a.num_q_heads / a.num_kv_heads;
  const int P = a.partition_tokens;

  int ctx = a.context_lens[s];
  if (ctx < 0 || ctx > a.max_context_len) {
    if (lane == 0 && part == 0 && g == 0) raise_flag(a.status, PA_FLAG_CONTEXT_LEN_OOB);
    ctx = ctx < 0 ? 0 : a.max_context_len;
  }
  const int t0 = part * P;
  const size_t head0 = static_cast<size_t>(s) * a.num_q_heads + static_cast<size_t>(g) * G;
  if (t0 >= ctx) {
    if (part == 0) {  // empty context: zero rows
      for (int h = 0; h < G; ++h)
        reinterpret_cast<uint2*>(a.out + (head0 + h) * kHeadDim)[lane] = make_uint2(0u, 0u);
    }
    return;
  }
  const int t1 = min(ctx, t0 + P);
  const int j0 = t0 / kBlockSize;
  const int nblk = (t1 + kBlockSize - 1) / kBlockSize - j0;
  const int nparts = (ctx + P - 1) / P;

  // q for every head of the group: lane owns dims 4*lane .. 4*lane+3, pre-scaled.
  float qr[GP][4];
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    uint2 w = make_uint2(0u, 0u);
    if (h < G) w = reinterpret_cast<const uint2*>(a.q + (head0 + h) * kHeadDim)[lane];
    qr[h][0] = bf16lo(w.x) * a.scale_log2;
    qr[h][1] = bf16hi(w.x) * a.scale_log2;
    qr[h][2] = bf16lo(w.y) * a.scale_log2;
    qr[h][3] = bf16hi(w.y) * a.scale_log2;
  }

  const int32_t* bt = a.block_tables + static_cast<size_t>(s) * a.max_blocks;
  int blk_chunk = -1;           // block ids of the 32-block chunk the producer is in
  uint32_t issued = 0;          // bit st: a copy is in flight into stage st
  uint32_t parity = 0;          // bit st: phase parity to wait for on stage st

  // Whole warp calls; lane 0 issues the two copies of block (j0 + jj) into stage st.
  auto issue = [&](int jj, int st) {
    if ((jj & 31) == 0) {
      const int j = j0 + jj + lane;
      blk_chunk = (jj + lane < nblk) ? bt[j] : -1;
    }
    const int blk = __shfl_sync(kFullMask, blk_chunk, jj & 31);
    if (blk < 0 || blk >= a.num_blocks) {
      if (lane == 0) raise_flag(a.status, PA_FLAG_BLOCK_ID_OOB);
      issued &= ~(1u << st);
      return;
    }
    issued |= 1u << st;
    if (lane == 0) {
      const uint32_t bar = smem_addr(&bars[st]);
      const size_t tile = (static_cast<size_t>(blk) * a.num_kv_heads + g) * (kBlockSize * kHeadDim);
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, kStageBytes);
      bulk_copy_g2s(smem_addr(tiles + st * kStageBytes), a.k_cache + tile, kTileBytes, bar);
      bulk_copy_g2s(smem_addr(tiles + st * kStageBytes + kTileBytes), a.v_cache + tile, kTileBytes, bar);
    }
  };

#pragma unroll
  for (int st = 0; st < kStages; ++st)
    if (st < nblk) issue(st, st);

  float m[HPL], l[HPL];
#pragma unroll
  for (int i = 0; i < HPL; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
  }
  float acc[GP][4];
#pragma unroll
  for (int h = 0; h < GP; ++h)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[h][i] = 0.f;

  for (int jj = 0; jj < nblk; ++jj) {
    const int st = jj % kStages;
    if (issued & (1u << st)) {
      if (!mbar_wait_bounded(smem_addr(&bars[st]), (parity >> st) & 1u)) {
        if (lane == 0) raise_flag(a.status, PA_FLAG_TIMEOUT);
        // Let the other copies in flight land (bounded) before the CTA can exit.
        for (int o = 0; o < kStages; ++o)
          if (o != st && (issued & (1u << o))) mbar_wait_bounded(smem_addr(&bars[o]), (parity >> o) & 1u);
        return;
      }
      parity ^= 1u << st;
      const int valid = min(kBlockSize, t1 - (j0 + jj) * kBlockSize);
      const uint2* K2 = reinterpret_cast<const uint2*>(tiles + st * kStageBytes);
      const uint2* V2 = reinterpret_cast<const uint2*>(tiles + st * kStageBytes + kTileBytes);

      // Scores: partial dot products over this lane's 4 dims.
      float vals[NV];
#pragma unroll
      for (int t = 0; t < kBlockSize; ++t) {
        const uint2 w = K2[t * 32 + lane];
        const float k0 = bf16lo(w.x), k1 = bf16hi(w.x), k2 = bf16lo(w.y), k3 = bf16hi(w.y);
#pragma unroll
        for (int h = 0; h < GP; ++h)
          vals[t * GP + h] = fmaf(qr[h][3], k3, fmaf(qr[h][2], k2, fmaf(qr[h][1], k1, qr[h][0] * k0)));
      }
      // Butterfly: at each step a lane keeps the half of its live values selected by its
      // lane bit and adds its partner's copy of that half.
#pragma unroll
      for (int step = 0; step < 5; ++step) {
        const int msk = 16 >> step;
        const int half = (NV >> step) / 2;
        const bool upper = (lane & msk) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
          const float send = upper ? vals[i] : vals[i + half];
          const float keep = upper ? vals[i + half] : vals[i];
          vals[i] = keep + __shfl_xor_sync(kFullMask, send, msk);
        }
      }
      // lane holds token lane/2, heads (lane&1)*HPL + i.
      const bool tok_ok = (lane >> 1) < valid;
      float p[HPL], alpha[HPL];
#pragma unroll
      for (int i = 0; i < HPL; ++i) {
        const float sc = tok_ok ? vals[i] : -INFINITY;
        float bm = sc;
        bm = fmaxf(bm, __shfl_xor_sync(kFullMask, bm, 2));
        bm = fmaxf(bm, __shfl_xor_sync(kFullMask, bm, 4));
        bm = fmaxf(bm, __shfl_xor_sync(kFullMask, bm, 8));
        bm = fmaxf(bm, __shfl_xor_sync(kFullMask, bm, 16));
        const float mn = fmaxf(m[i], bm);
        alpha[i] = exp2f(m[i] - mn);
        m[i] = mn;
        p[i] = tok_ok ? exp2f(sc - mn) : 0.f;
        l[i] = l[i] * alpha[i] + p[i];
      }
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        const float ah = __shfl_sync(kFullMask, alpha[h % HPL], h / HPL);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[h][i] *= ah;
      }
#pragma unroll
      for (int t = 0; t < kBlockSize; ++t) {
        if (t < valid) {
          const uint2 w = V2[t * 32 + lane];
          const float v0 = bf16lo(w.x), v1 = bf16hi(w.x), v2 = bf16lo(w.y), v3 = bf16hi(w.y);
#pragma unroll
          for (int h = 0; h < GP; ++h) {
            const float pt = __shfl_sync(kFullMask, p[h % HPL], 2 * t + h / HPL);
            acc[h][0] = fmaf(pt, v0, acc[h][0]);
            acc[h][1] = fmaf(pt, v1, acc[h][1]);
            acc[h][2] = fmaf(pt, v2, acc[h][2]);
            acc[h][3] = fmaf(pt, v3, acc[h][3]);
          }
        }
      }
    }
    __syncwarp();
    if (jj + kStages < nblk) issue(jj + kStages, st);
  }

  // Row sums: lanes of equal parity hold the same heads' per-token sums.
#pragma unroll
  for (int i = 0; i < HPL; ++i) {
    l[i] += __shfl_xor_sync(kFullMask, l[i], 2);
    l[i] += __shfl_xor_sync(kFullMask, l[i], 4);
    l[i] += __shfl_xor_sync(kFullMask, l[i], 8);
    l[i] += __shfl_xor_sync(kFullMask, l[i], 16);
  }
  if (nparts == 1) {
#pragma unroll
    for (int h = 0; h < GP; ++h) {
      if (h < G) {
        const float inv = 1.f / __shfl_sync(kFullMask, l[h % HPL], h / HPL);
        const uint2 o = make_uint2(pack_bf16x2(acc[h][0] * inv, acc[h][1] * inv),
                                   pack_bf16x2(acc[h][2] * inv, acc[h][3] * inv));
        reinterpret_cast<uint2*>(a.out + (head0 + h) * kHeadDim)[lane] = o;
      }
    }
  } else {
#pragma unroll
    for (int h = 0; h < GP; ++h) {
      if (h < G) {
        const size_t row = (head0 + h) * a.max_parts + part;
        reinterpret_cast<float4*>(a.ws_o + row * kHeadDim)[lane] =
            make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
        if (lane == h / HPL) a.ws_ml[row] = make_float2(m[h % HPL], l[h % HPL]);
      }
    }
  }
}

// Merge of the partitions of one (sequence, query head) per warp.
constexpr int kMergeWarps = 4;

__global__ void __launch_bounds__(kMergeWarps * 32) decode_merge_kernel(const DecodeArgs a) {
  pdl_wait_prior_grid();
  const int lane = threadIdx.x & 31;
  const int w = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  if (w >= a.num_seqs * a.num_q_heads) return;
  const int s = w / a.num_q_heads;
  int ctx = a.context_lens[s];
  ctx = ctx < 0 ? 0 : (ctx > a.max_context_len ? a.max_context_len : ctx);
  const int nparts = (ctx + a.partition_tokens - 1) / a.partition_tokens;
  if (nparts <= 1) return;  // written directly by the partition kernel
  const size_t row0 = static_cast<size_t>(w) * a.max_parts;
  const float2* ml = a.ws_ml + row0;
  float M = -INFINITY;
  for (int p = lane; p < nparts; p += 32) M = fmaxf(M, ml[p].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, o));
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int pb = 0; pb < nparts; pb += 32) {
    float wmine = 0.f;
    if (pb + lane < nparts) {
      const float2 v = ml[pb + lane];
      wmine = exp2f(v.x - M);
      L = fmaf(wmine, v.y, L);
    }
    const int n = min(32, nparts - pb);
    for (int k = 0; k < n; ++k) {
      const float wk = __shfl_sync(kFullMask, wmine, k);
      const float4 o = reinterpret_cast<const float4*>(a.ws_o + (row0 + pb + k) * kHeadDim)[lane];
      acc.x = fmaf(wk, o.x, acc.x);
      acc.y = fmaf(wk, o.y, acc.y);
      acc.z = fmaf(wk, o.z, acc.z);
      acc.w = fmaf(wk, o.w, acc.w);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(kFullMask, L, o);
  const float inv = 1.f / L;
  reinterpret_cast<uint2*>(a.out + static_cast<size_t>(w) * kHeadDim)[lane] =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
}

template <int GP>
cudaError_t launch_partition(const DecodeArgs& a, cudaStream_t stream) {
  static std::mutex mu;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
      err = cudaFuncSetAttribute(decode_partition_kernel<GP>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (err != cudaSuccess) return err;
      configured[dev] = true;
    }
  }
  const long long units = static_cast<long long>(a.num_seqs) * a.num_kv_heads * a.max_parts;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((units + kWarps - 1) / kWarps));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_partition_kernel<GP>, a);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  const int G = a.num_q_heads / a.num_kv_heads;
  cudaError_t err;
  switch ((G + 1) & ~1) {
    case 2: err = launch_partition<2>(a, stream); break;
    case 4: err = launch_partition<4>(a, stream); break;
    case 6: err = launch_partition<6>(a, stream); break;
    case 8: err = launch_partition<8>(a, stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (err != cudaSuccess || a.max_parts <= 1) return err;
  const long long warps = static_cast<long long>(a.num_seqs) * a.num_q_heads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((warps + kMergeWarps - 1) / kMergeWarps));
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel, a);
}

}  // namespace pa
