// Operand descriptors of the sm_100-family tensor core instruction tcgen05.mma, as plain
// functions usable from host and device code, so that every field can be checked on the CPU.
//
// Bit layouts from the public PTX ISA (tcgen05 "Matrix Descriptors"):
//
// Shared-memory matrix descriptor (64 bits)
//   [ 0,14)  matrix start address in shared memory >> 4
//   [16,30)  leading-dimension byte offset >> 4
//   [32,46)  stride-dimension byte offset >> 4
//   [46,48)  fixed value 1 (descriptor version of the sm_100 family)
//   [49,52)  matrix base offset (0: the swizzle pattern starts on a 1024-byte boundary)
//   [52]     leading-dimension offset mode (0: relative byte offset)
//   [61,64)  swizzle mode: 0 none, 1 128-byte with 32-byte atoms, 2 128-byte, 4 64-byte, 6 32-byte
//   other bits 0
//
// Instruction descriptor of kind::f16 (32 bits)
//   [ 0, 2)  sparsity selector, [2] sparsity, [3] saturate      (all 0 here)
//   [ 4, 6)  accumulator format: 0 f16, 1 f32
//   [ 7,10)  A format: 0 f16, 1 bf16
//   [10,13)  B format: 0 f16, 1 bf16
//   [13]     negate A, [14] negate B                             (0 here)
//   [15]     A major: 0 K-major, 1 M-major
//   [16]     B major: 0 K-major, 1 N-major
//   [17,23)  N >> 3
//   [24,29)  M >> 4
//   [30,32)  maximum shift (weight-stationary only; 0 here)
//
// With the 128-byte swizzle, a K-major operand is stored as rows of 128 bytes (64 bf16 of K),
// eight rows forming a 1024-byte atom whose 16-byte chunks are permuted within each row (chunk
// c of row r at c ^ (r % 8)), the atoms of successive 8-row groups (M or N) `stride` bytes
// apart; an MN-major operand as rows of 128 bytes along M or N (64 elements), one row per K
// index, eight K rows per atom, the atoms of successive 8-row groups along K `stride` bytes apart
// and those of successive 64-element groups along M / N `leading` bytes apart.
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define PA_HOST_DEVICE __host__ __device__
#else
#define PA_HOST_DEVICE
#endif

namespace pa {

constexpr uint32_t kUmmaSwizzle128B = 2u;

PA_HOST_DEVICE inline uint64_t umma_smem_desc(uint32_t smem_addr, uint32_t leading_bytes,
                                              uint32_t stride_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3fffu);
  d |= static_cast<uint64_t>((leading_bytes >> 4) & 0x3fffu) << 16;
  d |= static_cast<uint64_t>((stride_bytes >> 4) & 0x3fffu) << 32;
  d |= 1ull << 46;
  d |= static_cast<uint64_t>(kUmmaSwizzle128B) << 61;
  return d;
}

// bf16 x bf16 -> f32, M x N tile; *_mn_major: the operand is stored with M (or N) contiguous.
PA_HOST_DEVICE inline uint32_t umma_idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((static_cast<uint32_t>(N) >> 3) << 17) |
         ((static_cast<uint32_t>(M) >> 4) << 24);
}

}  // namespace pa
