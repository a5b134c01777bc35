// Tensor-memory-access (TMA) tile copies and the shared-memory barriers they complete on.
//
// A tile is described on the host by a tensor map (cuTensorMapEncodeTiled, reached through
// the runtime's driver entry point, so the library links no driver library) and copied by
// one thread with cp.async.bulk.tensor; the copy engine reports its bytes to an mbarrier,
// which the consuming threads poll by phase parity. Every poll loop is bounded: after about
// a second without completion the waiter counts a timeout in a device-wide counter
// (sra_wait_timeouts() adds up those counters) and goes on, so a copy that never lands cannot hang the GPU.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sra {

// Timeouts seen by this translation unit's bounded waits since the library was loaded, on
// the current device (each unit that includes this header has its own counter and reads it
// back through a host accessor of its own).
static __device__ unsigned int g_wait_timeouts;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Makes barrier initialisation visible to the copy engine (the async proxy).
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// One arrival that also announces `bytes` of copies completing on this barrier's phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// One plain arrival (no byte count).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; bounded (about 2^31 SM clocks).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > (1LL << 31)) {
            atomicAdd(&g_wait_timeouts, 1u);
            return false;
        }
    }
    return true;
}

// Orders this thread's earlier shared-memory accesses before later copy-engine writes.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Copy the box at element coordinates (c0, c1) of a 2-D tensor map into shared memory.
// c0 * element size must be a multiple of 16 bytes; dst 1024-byte aligned for 128-byte swizzle.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}
// Distributed shared memory: the shared::cluster address of `local` (a shared variable of this
// CTA) in the CTA of the cluster with the given rank, and 4- / 16-byte accesses through it.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local_addr, uint32_t rank) {
    uint32_t r;
    asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
    return dsmem_addr(smem_u32(local), rank);
}
__device__ __forceinline__ float4 dsmem_ld_f4(uint32_t addr) {
    float4 v;
    // (not volatile: the loads follow the barrier that made the data visible, and the
    // compiler may then issue all of a thread's loads before their first use)
    asm("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ void dsmem_st_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Hint the L2 to fetch the box at (c0, c1) of a 2-D tensor map (no data moves to the SM, and no
// barrier completes). A prefetch has no semantic effect, so it may run before a dependency wait on
// data the previous kernel is still writing: the L2 is the point of coherence. c0 as for a load.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void tma_load_1d(void* dst, const CUtensorMap* map, int c0, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.1d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2}], [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(smem_u32(bar))
        : "memory");
}

// Copy the box at element coordinates (c0, c1, c2, c3) of a 4-D tensor map into shared memory.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
        : "memory");
}

// Host: encode a tensor map of 16-bit elements of rank 1-4: dims[i] elements along dimension i
// (0 innermost), strides[i] bytes between consecutive indices of dimension i + 1, box[i] elements
// per copy. 128-byte swizzle or none. Returns false when the driver rejects the description.
bool encode_tmap_16_nd(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                       const uint32_t* box, bool bf16, bool swizzle128);

// Host: encode a tensor map of 16-bit elements. rank 1: {dim0}, box {box0}; rank 2: {dim0, dim1}
// with row stride `stride1` bytes, box {box0, box1}. Returns false (nothing encoded) when the
// driver entry point is missing or the driver rejects the description.
bool encode_tmap_16(CUtensorMap* map, const void* base, int rank, uint64_t dim0, uint64_t dim1, uint64_t stride1,
                    uint32_t box0, uint32_t box1, bool bf16, bool swizzle128);

}  // namespace sra
