// Device helpers shared by the sm_103a kernels: inline PTX for mbarriers, bulk copies into
// shared memory, programmatic dependent launch, tcgen05 tensor-core and tensor-memory
// operations, the bounded wait and the status flags.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa.h"

namespace pa {

constexpr int kHeadDim = 128;
constexpr int kBlockSize = 16;
constexpr int kTileBytes = kBlockSize * kHeadDim * 2;  // one (block, KV head) tile: 4 KiB
constexpr unsigned kFullMask = 0xffffffffu;
// A wait on a copy into shared memory gives up after this long (ns of %globaltimer) and
// raises PA_FLAG_TIMEOUT instead of hanging the GPU.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ void raise_flag(unsigned* status, unsigned flag) {
  atomicOr(status, flag);
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- programmatic dependent launch --------------------------------------------------
// Block until the grid this one depends on has completed and its writes are visible.
__device__ __forceinline__ void pdl_wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allow the next grid on the stream to be scheduled (it still waits for our completion).
__device__ __forceinline__ void pdl_allow_next_grid() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}


// ---- mbarrier ------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once and announce `bytes` of incoming asynchronous copies on this phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Arrive once with no byte count: completes the phase when nothing else is pending.
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for phase `parity` of the barrier to complete, for at most limit_ns of %globaltimer.
// Returns false on timeout (the caller raises PA_FLAG_TIMEOUT and stops using the stage).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0u && global_ns() - t0 > limit_ns) return false;
  }
}

// ---- bulk asynchronous copy global -> shared (no tensor map) -------------------------
// `bytes` must be a multiple of 16 and both addresses 16-byte aligned.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst_smem, const void* src_gmem,
                                              uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst_smem), "l"(src_gmem), "r"(bytes), "r"(bar)
      : "memory");
}

// Order this thread's earlier generic-proxy accesses to shared memory before later
// async-proxy (bulk copy) writes to it.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- TMA tiled load (tensor map), global -> shared -----------------------------------
// 2-D tile at element coordinates (x, y); x * 2 bytes must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(uint32_t dst_smem, const void* tensor_map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst_smem), "l"(reinterpret_cast<uint64_t>(tensor_map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 3-D tile at element coordinates (x, y, z); x * element size must be a multiple of 16 bytes.
// An L2 policy for data read exactly once (the K/V tiles of a decode step): its lines are the
// first to be evicted, so that what later kernels read again (lengths, block tables, partial
// results) stays in L2 while tens of MB stream through it.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  return policy;
}

__device__ __forceinline__ void tma_load_2d_once(uint32_t dst_smem, const void* tensor_map, int x, int y,
                                                 uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(dst_smem), "l"(reinterpret_cast<uint64_t>(tensor_map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_once(uint32_t dst_smem, const void* tensor_map, int x, int y,
                                                 int z, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;"
      ::"r"(dst_smem), "l"(reinterpret_cast<uint64_t>(tensor_map)), "r"(x), "r"(y), "r"(z), "r"(bar),
        "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst_smem, const void* tensor_map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst_smem), "l"(reinterpret_cast<uint64_t>(tensor_map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensor_map(const void* tensor_map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tensor_map)) : "memory");
}

// ---- warp-level tensor-core helpers ----------------------------------------------------
// Four 8x8 b16 matrices from shared memory; lanes 8i..8i+7 give the row addresses of matrix i,
// register i of lane l receives row l/4, columns 2(l%4), 2(l%4)+1 of matrix i.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// Same, each matrix transposed on the way into registers.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// Transpose an 8x8 b16 matrix held one packed pair per lane (row l/4, cols 2(l%4), +1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// D = A (16x16 bf16, row) * B (16x8 bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Same shape with f16 operands (the E4M3 cache path: E4M3 widens exactly to f16).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- tcgen05: 5th-generation tensor core, accumulators in tensor memory (TMEM) ----------
// TMEM addresses: lane (row) in bits 31..16, column in bits 15..0.  A warp may access the 32
// lanes 32 (warp % 4) .. 32 (warp % 4) + 31.

// Allocate `cols` columns (a power of two >= 32) for this CTA; the base address is written to
// shared memory at `slot`.  Warp-collective; one warp allocates and later frees.
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(cols)
               : "memory");
}
// This CTA allocates no more: other CTAs on the SM may allocate without waiting for it.
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}
// Order tcgen05 operations across a thread synchronisation (barrier, mbarrier, __syncthreads):
// `before` in the thread whose tcgen05 work precedes the sync, `after` in the one that follows.
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D (TMEM) = A (shared, descriptor a) * B (shared, descriptor b) (+ D if accumulate), one
// instruction of kind::f16 described by idesc (bf16 operands, fp32 accumulator).  Issued by one
// thread; runs asynchronously.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}
// Same with A read from tensor memory (row r of A in lane r, bf16 pairs along the columns, K = 16
// elements in 8 columns starting at a_tmem).
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                 bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}
// True in exactly one lane of the (converged) warp.  Work issued under it keeps the warp's
// values uniform, so descriptors stay in uniform registers.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}
// Arrive once on the mbarrier when every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
#define PA_R32(v)                                                                                    \
  "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),     \
      "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),         \
      "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),       \
      "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),       \
      "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
#define PA_W32(v)                                                                                    \
  "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),  \
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),  \
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), \
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
#define PA_OPS32                                                                                     \
  "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, "  \
  "%21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}"
// 32 consecutive 32-bit columns of this thread's lane (warp-collective); complete after
// tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 " PA_OPS32 ", [%32];" : PA_R32(v) : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
               "%10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, "
               "%27, %28, %29, %30, %31, %32};" ::"r"(taddr), PA_W32(v)
               : "memory");
}
#undef PA_R32
#undef PA_W32
#undef PA_OPS32
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---- bf16 ------------------------------------------------------------------------------
// Widen a packed pair of bf16 (low half = element 0) to two floats: bf16 is the top half
// of an fp32 bit pattern.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 2^x on the special-function unit (ex2.approx, subnormal results flushed to zero).  The
// softmax exponents are <= 8 and their results are rounded to bf16 or f16 right after.
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction (a NaN operand is ignored, as by fmaxf)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// ---- packed fp32 pairs (Blackwell f32x2 arithmetic: two lanes' worth per instruction) ------
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
// a * b + c elementwise, each rounded to nearest
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Round two floats to bf16 (nearest even) and pack them, a in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---- f16 and E4M3 (FP8) -----------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float f16lo(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
}
__device__ __forceinline__ float f16hi(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}
// bf16 pair -> f16 pair, round to nearest (exact for bf16 values inside the f16 range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) { return pack_f16x2(bf16lo(w), bf16hi(w)); }

// Two E4M3 codes (low byte = element 0) -> f16 pair, exact (NaN stays NaN).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t x) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(x));
  return r;
}
// Four codes b0..b3 -> f16 pairs (b0, b1) and (b2, b3).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = e4m3x2_to_f16x2(static_cast<uint16_t>(w & 0xffffu));
  hi = e4m3x2_to_f16x2(static_cast<uint16_t>(w >> 16));
}
// Four codes b0..b3 -> f16 pairs (b0, b2) and (b1, b3).
__device__ __forceinline__ void e4m3x4_pairs_to_f16(uint32_t w, uint32_t& even, uint32_t& odd) {
  uint32_t p;
  asm("prmt.b32 %0, %1, 0, 0x3120;" : "=r"(p) : "r"(w));  // bytes b0 b2 b1 b3
  e4m3x4_to_f16x2x2(p, even, odd);
}
// E4M3 codes of a bf16 pair times `inv` (fp32, round to nearest), round to nearest even,
// saturating to +-448; low byte = element 0.
__device__ __forceinline__ uint16_t e4m3x2_of(uint32_t bf16_pair, float inv) {
  const float lo = __fmul_rn(bf16lo(bf16_pair), inv);
  const float hi = __fmul_rn(bf16hi(bf16_pair), inv);
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// a b - c d in fp32 with the rounding error of c d recovered by an FMA (the compensated
// difference of products: w = c d rounded, e = w - c d exactly, result (a b - w) + e).  Within
// about two fp32 ulps of the exact value even when a b and c d nearly cancel, where the plain
// fma(a, b, -c d) can be off by many bf16 ulps of the (tiny) result.
__device__ __forceinline__ float diff_of_products(float a, float b, float c, float d) {
  const float w = __fmul_rn(c, d);
  const float e = __fmaf_rn(-c, d, w);
  const float f = __fmaf_rn(a, b, -w);
  return __fadd_rn(f, e);
}

// rotate_half RoPE of two adjacent rotation pairs: lo holds x[i], x[i+1], hi holds x[i+64],
// x[i+65] (bf16), c and s the cos and sin of angles i and i+1.  In fp32 (compensated, above),
// rounded to bf16 RNE:
//   x'[i] = x[i] c - x[i+64] s,   x'[i+64] = x[i+64] c + x[i] s.
// Every kernel that rotates goes through this one function, so they all agree bit for bit.
__device__ __forceinline__ void rope_rotate_pairs(uint32_t& lo, uint32_t& hi, float2 c, float2 s) {
  const float x0 = bf16lo(lo), x1 = bf16hi(lo), y0 = bf16lo(hi), y1 = bf16hi(hi);
  const float r0 = diff_of_products(x0, c.x, y0, s.x);
  const float r1 = diff_of_products(x1, c.y, y1, s.y);
  const float r2 = diff_of_products(y0, c.x, -x0, s.x);
  const float r3 = diff_of_products(y1, c.y, -x1, s.y);
  lo = pack_bf16x2(r0, r1);
  hi = pack_bf16x2(r2, r3);
}

}  // namespace pa
