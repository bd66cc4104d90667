// Fused RoPE + KV-cache store for sm_103a.
//
// "Pico-vLLM：从零手写的工业级LLM推理引擎实现", §1 模型实现层 (RoPE with rotate_half, in
// place) and §2 Kernel层 (fused RoPE + KV cache store); "从零实现 LLM 推理引擎：深挖 vLLM 的
// 六大核心优化", §3.1 (16-token blocks) and §3.2 (append_slot: one new slot per sequence).
//
// One warp per token.  It reads the token's position and cos/sin row once, then moves the
// token's Hq query vectors (rotated in place), Hkv key vectors (rotated into the cache slot) and
// Hkv value vectors (copied next to them) four at a time: lanes 8v .. 8v+7 take vector v of a
// pass, lane 8v + j the dims 8j .. 8j+7 and their rotation partners 64+8j .. 64+8j+7 as two
// 16-byte words.  A group of passes is loaded before any of it is stored (below).  With E4M3
// caches (kFp8) the rotated k and the raw v are stored as the E4M3 codes of
// x * (1 / scale of the KV head), both in fp32 with round to nearest, coded round to nearest
// even with saturation.

#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {
namespace {

constexpr int kRopeWarps = 8;   // tokens per CTA
// Passes of four vectors loaded before any is stored.  Few tokens: 4, so that all of a
// token's loads are in flight at once (its latency is the call's).  Many tokens: 2 and at most
// 64 registers, so that 4 CTAs fit per SM and more warps hide the memory latency (measured on
// 32,768 tokens: 6.7 TB/s against 6.3 TB/s).
constexpr int kRopeManyTokens = 2048;

// Rotate the 8 dims of lo (8j .. 8j+7) with their partners in hi (64+8j .. 64+8j+7).
__device__ __forceinline__ void rotate8(uint4& lo, uint4& hi, const float4& c0, const float4& c1,
                                        const float4& s0, const float4& s1) {
  rope_rotate_pairs(lo.x, hi.x, make_float2(c0.x, c0.y), make_float2(s0.x, s0.y));
  rope_rotate_pairs(lo.y, hi.y, make_float2(c0.z, c0.w), make_float2(s0.z, s0.w));
  rope_rotate_pairs(lo.z, hi.z, make_float2(c1.x, c1.y), make_float2(s1.x, s1.y));
  rope_rotate_pairs(lo.w, hi.w, make_float2(c1.z, c1.w), make_float2(s1.z, s1.w));
}

// E4M3 codes of 8 bf16 values times inv, element 0 in the lowest byte.
__device__ __forceinline__ uint2 e4m3x8_of(const uint4& x, float inv) {
  const uint32_t a = e4m3x2_of(x.x, inv) | (static_cast<uint32_t>(e4m3x2_of(x.y, inv)) << 16);
  const uint32_t b = e4m3x2_of(x.z, inv) | (static_cast<uint32_t>(e4m3x2_of(x.w, inv)) << 16);
  return make_uint2(a, b);
}

template <bool kFp8, int kRopeGroup>
__global__ void __launch_bounds__(kRopeWarps * 32, kRopeGroup == 2 ? 4 : 1) rope_kv_store_kernel(const RopeArgs a) {
  pdl_wait_prior_grid();
  pdl_allow_next_grid();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRopeWarps + static_cast<int>(threadIdx.x >> 5);
  if (t >= a.num_tokens) return;
  const int j = lane & 7;     // dims 8j .. 8j+7 and 64+8j .. 64+8j+7
  const int sub = lane >> 3;  // vector of the pass
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads;
  const int all = Hq + 2 * Hkv;  // q heads, then k heads, then v heads
  uint4 lo[kRopeGroup], hi[kRopeGroup];
  auto load_group = [&](int base) {
#pragma unroll
    for (int p = 0; p < kRopeGroup; ++p) {
      const int i = base + 4 * p + sub;
      lo[p] = hi[p] = make_uint4(0u, 0u, 0u, 0u);
      if (i >= all) continue;
      const __nv_bfloat16* src;
      if (i < Hq) src = a.q + (static_cast<size_t>(t) * Hq + i) * kHeadDim;
      else if (i < Hq + Hkv) src = a.k + (static_cast<size_t>(t) * Hkv + (i - Hq)) * kHeadDim;
      else src = a.v + (static_cast<size_t>(t) * Hkv + (i - Hq - Hkv)) * kHeadDim;
      lo[p] = reinterpret_cast<const uint4*>(src)[j];
      hi[p] = reinterpret_cast<const uint4*>(src)[8 + j];
    }
  };
  // The position, the slot and the first group of vectors are independent loads: issue them
  // all before anything waits on the position.
  const int pos = a.positions[t];
  const int64_t slot = a.slot_mapping[t];
  load_group(0);
  if (pos < 0 || pos >= a.max_pos) {  // the token is left as it is: q unrotated, nothing stored
    if (lane == 0) raise_flag(a.status, PA_FLAG_POSITION_OOB);
    return;
  }
  bool store = slot >= 0;  // a negative slot is a padding token: q is rotated, nothing stored
  if (store && slot >= static_cast<int64_t>(a.num_blocks) * kBlockSize) {
    if (lane == 0) raise_flag(a.status, PA_FLAG_SLOT_OOB);
    store = false;
  }
  const int64_t blk = store ? slot / kBlockSize : 0;
  const int off = store ? static_cast<int>(slot - blk * kBlockSize) : 0;
  const float4* row = reinterpret_cast<const float4*>(a.cos_sin + static_cast<size_t>(pos) * kHeadDim);
  const float4 c0 = row[2 * j], c1 = row[2 * j + 1];            // cos of dims 8j .. 8j+7
  const float4 s0 = row[16 + 2 * j], s1 = row[16 + 2 * j + 1];  // sin of the same

  const int items = store ? all : Hq;
  for (int base = 0; base < items; base += 4 * kRopeGroup) {
    if (base) load_group(base);
#pragma unroll
    for (int p = 0; p < kRopeGroup; ++p) {
      const int i = base + 4 * p + sub;
      if (i >= items) continue;
      if (i < Hq + Hkv) rotate8(lo[p], hi[p], c0, c1, s0, s1);  // q and k rotate; v does not
      if (i < Hq) {
        uint4* dst = reinterpret_cast<uint4*>(a.q + (static_cast<size_t>(t) * Hq + i) * kHeadDim);
        dst[j] = lo[p];
        dst[8 + j] = hi[p];
        continue;
      }
      const bool is_k = i < Hq + Hkv;
      const int g = is_k ? i - Hq : i - Hq - Hkv;
      const size_t cache_row = (static_cast<size_t>(blk) * Hkv + g) * kBlockSize + off;  // in rows of 128
      if constexpr (kFp8) {
        const float inv = __frcp_rn(is_k ? a.k_scale[g] : a.v_scale[g]);
        uint2* dst = reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(is_k ? a.k_cache : a.v_cache) +
                                              cache_row * kHeadDim);
        dst[j] = e4m3x8_of(lo[p], inv);
        dst[8 + j] = e4m3x8_of(hi[p], inv);
      } else {
        uint4* dst = reinterpret_cast<uint4*>((is_k ? a.k_cache : a.v_cache) + cache_row * kHeadDim);
        dst[j] = lo[p];
        dst[8 + j] = hi[p];
      }
    }
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((static_cast<long long>(a.num_tokens) + kRopeWarps - 1) / kRopeWarps));
  cfg.blockDim = dim3(kRopeWarps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool many = a.num_tokens > kRopeManyTokens;
  if (a.k_scale)
    return many ? cudaLaunchKernelEx(&cfg, rope_kv_store_kernel<true, 2>, a)
                : cudaLaunchKernelEx(&cfg, rope_kv_store_kernel<true, 4>, a);
  return many ? cudaLaunchKernelEx(&cfg, rope_kv_store_kernel<false, 2>, a)
              : cudaLaunchKernelEx(&cfg, rope_kv_store_kernel<false, 4>, a);
}

}  // namespace pa
