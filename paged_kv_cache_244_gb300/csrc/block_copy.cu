// Whole-block copies between KV-cache block pools, for every cache of a model in one launch:
// copy-on-write inside one pool and swap out / swap in between the GPU pool and a CPU pool.
//
// "从零实现 LLM 推理引擎：深挖 vLLM 的六大核心优化", §3.4 Prefix Caching / Copy-on-Write (a
// shared block is replaced, before it is written, by a fresh block with the same contents) and
// §3.5 CPU Swap (swap_out moves a sequence's blocks to CPU memory, swap_in restores them into
// newly allocated GPU blocks).
//
// A block of one cache is Hkv contiguous (block, KV head) tiles of 4 KiB.  Work unit = one
// 4 KiB tile of one (pair, cache): a warp loads it with eight 16-byte loads per lane (512
// contiguous bytes per instruction), all in flight together, then stores it.  Units of the
// same pair are consecutive, so the tiles of one block are copied by neighbouring warps.  A
// persistent grid strides over the units.  Pools in page-locked host memory are read and
// written in place by the same loads and stores, over the CPU-GPU link: there is no staging
// copy and no per-block memcpy.

#include <mutex>

#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {
namespace {

constexpr int kCopyWarps = 8;
constexpr int kTileVec = kTileBytes / 16;   // uint4 per tile: 256
constexpr int kPerLane = kTileVec / 32;     // 8

__global__ void __launch_bounds__(kCopyWarps * 32) copy_blocks_kernel(const __grid_constant__ BlockCopyArgs a) {
  pdl_wait_prior_grid();
  pdl_allow_next_grid();
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * kCopyWarps;
  const long long per_pair = static_cast<long long>(a.num_caches) * a.tiles_per_block;
  const long long units = per_pair * a.num_pairs;
  for (long long u = static_cast<long long>(blockIdx.x) * kCopyWarps + (threadIdx.x >> 5); u < units;
       u += warps) {
    const long long i = u / per_pair;
    const int rem = static_cast<int>(u - i * per_pair);
    const int c = rem / a.tiles_per_block;
    const int tile = rem - c * a.tiles_per_block;
    const long long from = a.pairs[2 * i];
    const long long to = a.pairs[2 * i + 1];
    if (from < 0 || from >= a.src_blocks || to < 0 || to >= a.dst_blocks) {
      if (lane == 0 && rem == 0) raise_flag(a.status, PA_FLAG_BLOCK_ID_OOB);
      continue;
    }
    const uint4* src = a.src[c] + (from * a.tiles_per_block + tile) * kTileVec + lane;
    uint4* dst = a.dst[c] + (to * a.tiles_per_block + tile) * kTileVec + lane;
    uint4 v[kPerLane];
#pragma unroll
    for (int k = 0; k < kPerLane; ++k) v[k] = src[32 * k];
#pragma unroll
    for (int k = 0; k < kPerLane; ++k) dst[32 * k] = v[k];
  }
}

// pa_stage_copy: n 16-byte words from src to dst, either of them in this GPU's memory or in
// page-locked host memory (read and written in place over the CPU-GPU link).  Each thread
// issues its kStageVec loads before its stores, so every word of a few hundred KiB is in flight
// at once: one round trip over the link, where a copy-engine transfer of the same bytes costs
// several microseconds of set-up.
constexpr int kStageThreads = 256;
constexpr int kStageVec = 2;

__global__ void __launch_bounds__(kStageThreads) stage_copy_kernel(uint4* dst, const uint4* src, long long n) {
  pdl_wait_prior_grid();
  pdl_allow_next_grid();
  const long long stride = static_cast<long long>(gridDim.x) * kStageThreads;
  for (long long base = static_cast<long long>(blockIdx.x) * kStageThreads + threadIdx.x; base < n;
       base += stride * kStageVec) {
    uint4 v[kStageVec];
#pragma unroll
    for (int k = 0; k < kStageVec; ++k) {
      const long long i = base + k * stride;
      if (i < n) v[k] = src[i];
    }
#pragma unroll
    for (int k = 0; k < kStageVec; ++k) {
      const long long i = base + k * stride;
      if (i < n) dst[i] = v[k];
    }
  }
}

int sm_count(int* out) {
  static std::mutex mu;
  static int sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::lock_guard<std::mutex> lock(mu);
  if (!sms[dev] && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  *out = sms[dev];
  return 0;
}

}  // namespace

cudaError_t launch_stage_copy(void* dst, const void* src, long long n16, cudaStream_t stream) {
  if (n16 <= 0) return cudaSuccess;
  int n_sms = 0;
  if (sm_count(&n_sms) != 0) return cudaErrorInvalidDevice;
  const long long per_cta = static_cast<long long>(kStageThreads) * kStageVec;
  const long long ctas = min(static_cast<long long>(n_sms) * 8, (n16 + per_cta - 1) / per_cta);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(kStageThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stage_copy_kernel, static_cast<uint4*>(dst), static_cast<const uint4*>(src), n16);
}

cudaError_t launch_copy_blocks(const BlockCopyArgs& a, cudaStream_t stream) {
  static std::mutex mu;
  static int sms[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int n_sms = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!sms[dev]) {
      err = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
      if (err != cudaSuccess) return err;
    }
    n_sms = sms[dev];
  }
  const long long units = static_cast<long long>(a.num_pairs) * a.num_caches * a.tiles_per_block;
  // Enough resident warps to keep ~16 MB in flight, never more CTAs than units need.
  const long long ctas = min(static_cast<long long>(n_sms) * 8, (units + kCopyWarps - 1) / kCopyWarps);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(kCopyWarps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, copy_blocks_kernel, a);
}

}  // namespace pa
