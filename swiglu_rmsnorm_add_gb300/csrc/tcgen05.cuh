// Blackwell tensor-core (tcgen05) building blocks: tensor-memory allocation, the
// shared-memory matrix descriptor, the instruction descriptor of a 16-bit MMA
// with fp32 accumulation, the MMA itself (issued by one thread), its completion
// on an mbarrier, and loads of the accumulator back into registers.
//
// Each wrapper is one PTX instruction of the tcgen05 family as the PTX ISA
// defines it for sm_100-class GPUs (sm_103a here); the field layouts below are
// the ISA's.
#pragma once

#include <stdint.h>

#include "tma.cuh"

namespace sra {
namespace tc {

// ------------------------------------------------------------------ tensor memory
// Tensor memory is 128 lanes x 512 columns of 32 bits per SM. A CTA allocates a
// power-of-two number of columns (>= 32) with one warp; the address (lane 0,
// first column) lands in shared memory. Lane l of a 128-row accumulator holds
// row l; column c holds its c-th 32-bit value.
__device__ __forceinline__ void alloc(uint32_t* dst, uint32_t ncols) {  // whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void relinquish() {  // whole warp: this CTA allocates no more
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Orders tcgen05 operations across a thread synchronisation (barrier, mbarrier wait).
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// ------------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor for a K-major operand tile stored as the 128-byte
// swizzle of a TMA copy: rows of 64 16-bit elements (128 bytes), row r at r * 128,
// its 16-byte chunk c at (c ^ (r % 8)) * 16, 8-row groups 1024 bytes apart. The
// tile starts on a 1024-byte boundary; the k-th 16-element slice of K starts 32 k
// bytes further (the swizzle is applied to the address, so the offset is plain).
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4 (not used by a swizzled K-major tile; 1)
//   bits 32-45  stride-dimension byte offset >> 4 (1024 bytes between 8-row groups)
//   bits 46-47  descriptor version (1)
//   bits 49-51  base offset (0: the swizzle pattern starts at the tile)
//   bits 61-63  layout: 2 = 128-byte swizzle
__device__ __forceinline__ uint64_t sdesc_sw128(const void* tile, int k_bytes) {
    const uint32_t a = smem_u32(tile) + static_cast<uint32_t>(k_bytes);
    uint64_t d = static_cast<uint64_t>((a >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>((1024u >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor of kind::f16: D fp32, A and B both bf16 (or both fp16),
// both K-major, M x N.
//   bits  4-5   D format (1 = f32)
//   bits  7-9   A format (0 = f16, 1 = bf16)
//   bits 10-12  B format (0 = f16, 1 = bf16)
//   bits 15/16  A / B transposed (0 = K-major)
//   bits 17-22  N >> 3
//   bits 24-28  M >> 4
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, int M, int N) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------------------------ MMA
// D[tmem] (+)= A[smem] * B[smem]^T, one instruction of K = 16; `accumulate` 0
// overwrites D. Issued by one thread; completes asynchronously.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The mbarrier completes one arrival once every tcgen05 operation this thread
// issued before has completed (its shared-memory operands may then be reused).
__device__ __forceinline__ void commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// ------------------------------------------------------------------ accumulator loads
// 32 lanes x 16 columns: lane t of the warp gets row (lane base + t), columns
// [col, col + 16) of the address. A warp may read only its own quarter of the
// lanes: lanes 32 (warp % 4) ... + 31. Completes at wait_ld().
__device__ __forceinline__ void ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace tc
}  // namespace sra
