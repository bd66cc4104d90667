// Fused RoPE + KV-cache store for sm_103a.
//
// "Pico-vLLM：从零手写的工业级LLM推理引擎实现", §1 模型实现层 (RoPE with rotate_half, in
// place) and §2 Kernel层 (fused RoPE + KV cache store); "从零实现 LLM 推理引擎：深挖 vLLM 的
// 六大核心优化", §3.1 (16-token blocks) and §3.2 (append_slot: one new slot per sequence).
//
// One warp per (token, head).  Warps for query heads rotate q in place; warps for KV heads
// rotate k into its cache slot and copy v next to it.  Lane l owns the rotation pairs
// (2l, 2l+64) and (2l+1, 2l+65): two 32-bit loads of bf16 pairs, two float2 loads of the
// cos/sin row, two 32-bit stores, so each head vector moves as one 256-byte line.
// With E4M3 caches (kFp8) the rotated k and the raw v are stored as the E4M3 codes of
// x * (1 / scale of the KV head), both in fp32 with round to nearest, coded round to nearest
// even with saturation; two one-byte codes per lane and pair.
// Launch-bound (a few KiB per token): no shared memory, no staging.

#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {
namespace {

constexpr int kRopeWarps = 8;

template <bool kFp8>
__global__ void __launch_bounds__(kRopeWarps * 32) rope_kv_store_kernel(const RopeArgs a) {
  pdl_wait_prior_grid();
  pdl_allow_next_grid();
  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * kRopeWarps + (threadIdx.x >> 5);
  const int heads = a.num_q_heads + a.num_kv_heads;
  if (warp >= a.num_tokens * heads) return;
  const int t = warp / heads;
  const int h = warp - t * heads;

  const int pos = a.positions[t];
  if (pos < 0 || pos >= a.max_pos) {
    if (lane == 0) raise_flag(a.status, PA_FLAG_POSITION_OOB);
    return;
  }
  const uint32_t* src;
  uint32_t* dst;
  uint16_t* dst8 = nullptr;  // E4M3 K cache row
  float inv_k = 0.f;
  if (h < a.num_q_heads) {
    dst = reinterpret_cast<uint32_t*>(a.q + (static_cast<size_t>(t) * a.num_q_heads + h) * kHeadDim);
    src = dst;
  } else {
    const int g = h - a.num_q_heads;
    const int64_t slot = a.slot_mapping[t];
    if (slot < 0) return;  // padding token: nothing to store
    if (slot >= static_cast<int64_t>(a.num_blocks) * kBlockSize) {
      if (lane == 0) raise_flag(a.status, PA_FLAG_SLOT_OOB);
      return;
    }
    const int64_t blk = slot / kBlockSize;
    const int off = static_cast<int>(slot - blk * kBlockSize);
    const size_t in_off = (static_cast<size_t>(t) * a.num_kv_heads + g) * kHeadDim;
    const size_t cache_off = ((static_cast<size_t>(blk) * a.num_kv_heads + g) * kBlockSize + off) * kHeadDim;
    src = reinterpret_cast<const uint32_t*>(a.k + in_off);
    dst = reinterpret_cast<uint32_t*>(a.k_cache + cache_off);
    if constexpr (kFp8) {
      uint8_t* kc8 = reinterpret_cast<uint8_t*>(a.k_cache) + cache_off;
      uint16_t* vc8 = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(a.v_cache) + cache_off);
      const uint32_t* vin = reinterpret_cast<const uint32_t*>(a.v + in_off);
      const float inv_v = __frcp_rn(a.v_scale[g]);
      vc8[lane] = e4m3x2_of(vin[lane], inv_v);             // dims 2l, 2l+1
      vc8[32 + lane] = e4m3x2_of(vin[32 + lane], inv_v);   // dims 2l+64, 2l+65
      dst8 = reinterpret_cast<uint16_t*>(kc8);
      inv_k = __frcp_rn(a.k_scale[g]);
    } else {
      reinterpret_cast<uint2*>(a.v_cache + cache_off)[lane] =
          reinterpret_cast<const uint2*>(a.v + in_off)[lane];
    }
  }
  const float* row = a.cos_sin + static_cast<size_t>(pos) * kHeadDim;
  const float2 c = reinterpret_cast<const float2*>(row)[lane];        // cos of pairs 2l, 2l+1
  const float2 s = reinterpret_cast<const float2*>(row + 64)[lane];   // sin of pairs 2l, 2l+1
  uint32_t lo = src[lane];        // x[2l], x[2l+1]
  uint32_t hi = src[32 + lane];   // x[2l+64], x[2l+65]
  rope_rotate_pairs(lo, hi, c, s);
  if (kFp8 && dst8) {
    dst8[lane] = e4m3x2_of(lo, inv_k);
    dst8[32 + lane] = e4m3x2_of(hi, inv_k);
  } else {
    dst[lane] = lo;
    dst[32 + lane] = hi;
  }
}

// Self-test of the bounded wait every kernel here uses on its shared-memory copies: one warp
// initialises an mbarrier that nothing will ever arrive on and waits on it with the given
// limit.  The wait must give up and raise PA_FLAG_TIMEOUT; nothing faults and nothing hangs.
__global__ void wait_selftest_kernel(unsigned* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const bool done = mbar_wait_bounded(b, 0u, limit_ns);
  if (!done && threadIdx.x == 0) raise_flag(status, PA_FLAG_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned* status, uint64_t limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_rope_kv_store(const RopeArgs& a, cudaStream_t stream) {
  const long long warps = static_cast<long long>(a.num_tokens) * (a.num_q_heads + a.num_kv_heads);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((warps + kRopeWarps - 1) / kRopeWarps));
  cfg.blockDim = dim3(kRopeWarps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.k_scale) return cudaLaunchKernelEx(&cfg, rope_kv_store_kernel<true>, a);
  return cudaLaunchKernelEx(&cfg, rope_kv_store_kernel<false>, a);
}

}  // namespace pa
