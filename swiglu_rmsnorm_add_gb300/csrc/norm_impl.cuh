// RMSNorm and residual-add + RMSNorm kernels (one template family, ADD selects
// the fused residual update).
//
// RMSNorm as the pages state it (koas-w.github.io "preformanceimprovement"
// section 3; m.lsln.cn/news/61269 section 2.3; agent.csdn.net
// "使用Triton实现RMSNorm算子"): out = x * rsqrt(mean(x^2) + eps) * w, widened to
// fp32, one rounding on the store. The fused add (same "preformanceimprovement"
// page, section 4) first stores x <- round(x + res) in place and normalises the
// rounded sum, reading each row once and writing it twice.
//
// Per-shape variants, all with 16-byte vector accesses when the layout allows
// and a predicated scalar tail (never a power-of-two padded width):
//   warp_rows  one warp per row, the row held in registers (short rows)
//   cta_row    one CTA per row, the row held in registers (long rows)
//   cta_smem   one CTA per row staged in shared memory (rows past the registers)
//   two_pass   one CTA per row, statistics pass then a re-reading scale pass (any D)
//   cta_pair   a 2-CTA cluster per row: each CTA holds half the row in registers
//              and the two partial sums of squares meet through distributed
//              shared memory (wide rows when rows alone cannot fill the SMs evenly)
// The register variants stage w once per CTA in shared memory with cp.async
// (no registers held, no software wait), so the registers hold only the row.
// Every variant keeps a row's elements with one thread across both passes, so
// in-place use (out == x) is safe and no inter-thread hazard exists on the row.
// Each translation unit instantiates one ADD value only (norm_rms.cu: false,
// norm_add.cu: true), so no kernel is registered from two modules.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace sra {
namespace norm {

namespace cg = cooperative_groups;

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Copy w[e0, e1) (elements) to ws[0, e1 - e0) with every thread of the CTA:
// 16-byte asynchronous copies for whole vectors, plain loads for the rest.
// e0 is a multiple of VEC.
template <typename T, int VEC>
__device__ __forceinline__ void stage_weights(const T* __restrict__ w, T* ws, int64_t e0, int64_t e1) {
    if constexpr (VEC * sizeof(T) == 16) {
        const int64_t nv = (e1 - e0) / VEC;
        for (int64_t i = threadIdx.x; i < nv; i += blockDim.x) cp_async16(ws + i * VEC, w + e0 + i * VEC);
        for (int64_t j = e0 + nv * VEC + threadIdx.x; j < e1; j += blockDim.x) ws[j - e0] = w[j];
        cp_async_wait_all();
    } else {
        for (int64_t j = e0 + threadIdx.x; j < e1; j += blockDim.x) ws[j - e0] = w[j];
    }
    __syncthreads();
}

// How the row's sum of squares is reduced.
enum Reduce { RED_WARP = 0, RED_CTA = 1, RED_PAIR = 2 };

// One row, held in registers. The caller's group (a warp, a CTA or a CTA of a
// pair) covers accesses [a0, a1) of the row: thread tid owns
// idx = a0 + v * threads + tid for v < NV. `tail_owner` marks the group that
// also owns the D % VEC trailing elements. ws holds w from element a0 * VEC on.
template <typename T, int VEC, int NV, bool ADD, int RED>
__device__ __forceinline__ void row_in_registers(const NormArgs& a, int64_t r, int tid, int threads, int64_t a0,
                                                 int64_t a1, bool tail_owner, const T* ws, float* scratch,
                                                 float* pair_slot, int parity) {
    using V = Vec<T, VEC>;
    using R = typename V::Raw;
    const int64_t nvec = a.D / VEC;
    const int tail = tail_owner ? static_cast<int>(a.D - nvec * VEC) : 0;
    T* xr = static_cast<T*>(a.x) + r * a.xs;
    T* orow = static_cast<T*>(a.out) + r * a.os;

    R xv[NV];
    float xt = 0.0f;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int64_t idx = a0 + static_cast<int64_t>(v) * threads + tid;
        if (idx < a1) xv[v] = V::load(xr + idx * VEC);
    }
    if (tid < tail) xt = to_f32(xr[nvec * VEC + tid]);

    float ss = 0.0f;
    if constexpr (ADD) {
        const T* rr = static_cast<const T*>(a.res) + r * a.rs;
        R rv[NV];
        float rt = 0.0f;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int64_t idx = a0 + static_cast<int64_t>(v) * threads + tid;
            if (idx < a1) rv[v] = V::load(rr + idx * VEC);
        }
        if (tid < tail) rt = to_f32(rr[nvec * VEC + tid]);
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int64_t idx = a0 + static_cast<int64_t>(v) * threads + tid;
            if (idx < a1) {
                float xf[VEC], rf[VEC];
                V::unpack(xv[v], xf);
                V::unpack(rv[v], rf);
#pragma unroll
                for (int i = 0; i < VEC; ++i) xf[i] += rf[i];
                xv[v] = V::pack(xf);  // the rounded sum
                V::store(xr + idx * VEC, xv[v]);
                V::unpack(xv[v], xf);
#pragma unroll
                for (int i = 0; i < VEC; ++i) ss = fmaf(xf[i], xf[i], ss);
            }
        }
        if (tid < tail) {
            const T s = from_f32<T>(xt + rt);
            xr[nvec * VEC + tid] = s;
            xt = to_f32(s);
            ss = fmaf(xt, xt, ss);
        }
    } else {
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int64_t idx = a0 + static_cast<int64_t>(v) * threads + tid;
            if (idx < a1) {
                float xf[VEC];
                V::unpack(xv[v], xf);
#pragma unroll
                for (int i = 0; i < VEC; ++i) ss = fmaf(xf[i], xf[i], ss);
            }
        }
        if (tid < tail) ss = fmaf(xt, xt, ss);
    }

    if constexpr (RED == RED_WARP) {
        ss = warp_sum(ss);
    } else if constexpr (RED == RED_CTA) {
        ss = block_sum(ss, scratch);
    } else {
        // Pair: each CTA's partial goes to its own slot (double-buffered by row
        // parity), the cluster barrier publishes both, each CTA adds the peer's.
        const float part = block_sum(ss, scratch);
        cg::cluster_group cl = cg::this_cluster();
        if (threadIdx.x == 0) pair_slot[parity] = part;
        cl.sync();
        const float peer = *cl.map_shared_rank(pair_slot + parity, static_cast<int>(cl.block_rank()) ^ 1);
        ss = part + peer;  // the same sum on both CTAs (addition commutes exactly)
    }
    const float rinv = rsqrtf(ss / static_cast<float>(a.D) + a.eps);

#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int64_t idx = a0 + static_cast<int64_t>(v) * threads + tid;
        if (idx < a1) {
            float xf[VEC], wf[VEC];
            V::unpack(xv[v], xf);
            V::unpack(V::load(ws + (idx - a0) * VEC), wf);
#pragma unroll
            for (int i = 0; i < VEC; ++i) xf[i] = xf[i] * rinv * wf[i];
            V::store(orow + idx * VEC, V::pack(xf));
        }
    }
    if (tid < tail) {
        const int64_t j = nvec * VEC + tid;
        orow[j] = from_f32<T>(xt * rinv * to_f32(ws[j - a0 * VEC]));
    }
}

template <typename T, int VEC, int NV, bool ADD>
__global__ void __launch_bounds__(256) warp_rows_kernel(NormArgs a) {
    extern __shared__ __align__(16) unsigned char dyn_smem[];
    T* ws = reinterpret_cast<T*>(dyn_smem);
    pdl_enter();
    stage_weights<T, VEC>(static_cast<const T*>(a.w), ws, 0, a.D);
    const int warps_per_cta = blockDim.x >> 5;
    const int64_t step = static_cast<int64_t>(gridDim.x) * warps_per_cta;
    const int lane = threadIdx.x & 31;
    const int64_t nvec = a.D / VEC;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * warps_per_cta + (threadIdx.x >> 5); r < a.rows;
         r += step) {
        row_in_registers<T, VEC, NV, ADD, RED_WARP>(a, r, lane, 32, 0, nvec, true, ws, nullptr, nullptr, 0);
    }
}

// Largest CTA the register-resident CTA variants are compiled for, per NV.
template <int NV> constexpr int cta_row_max_threads() { return NV >= 8 ? 256 : (NV >= 4 ? 512 : 1024); }

template <typename T, int VEC, int NV, bool ADD>
__global__ void __launch_bounds__(cta_row_max_threads<NV>()) cta_row_kernel(NormArgs a) {
    __shared__ float scratch[33];
    extern __shared__ __align__(16) unsigned char dyn_smem[];
    T* ws = reinterpret_cast<T*>(dyn_smem);
    pdl_enter();
    stage_weights<T, VEC>(static_cast<const T*>(a.w), ws, 0, a.D);
    const int64_t nvec = a.D / VEC;
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        row_in_registers<T, VEC, NV, ADD, RED_CTA>(a, r, threadIdx.x, blockDim.x, 0, nvec, true, ws, scratch,
                                                   nullptr, 0);
    }
}

template <typename T, int VEC, int NV, bool ADD>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(cta_row_max_threads<NV>()) cta_pair_kernel(NormArgs a) {
    __shared__ float scratch[33];
    __shared__ float pair_slot[2];
    extern __shared__ __align__(16) unsigned char dyn_smem[];
    T* ws = reinterpret_cast<T*>(dyn_smem);
    pdl_enter();
    cg::cluster_group cl = cg::this_cluster();
    const int rank = static_cast<int>(cl.block_rank());
    const int64_t nvec = a.D / VEC;
    const int64_t half = norm_pair_half(nvec);
    const int64_t a0 = rank == 0 ? 0 : half;
    const int64_t a1 = rank == 0 ? half : nvec;
    stage_weights<T, VEC>(static_cast<const T*>(a.w), ws, a0 * VEC, rank == 0 ? half * VEC : a.D);
    const int64_t pairs = gridDim.x / 2;
    int parity = 0;
    for (int64_t r = blockIdx.x / 2; r < a.rows; r += pairs) {
        row_in_registers<T, VEC, NV, ADD, RED_PAIR>(a, r, threadIdx.x, blockDim.x, a0, a1, rank == 1, ws, scratch,
                                                    pair_slot, parity);
        parity ^= 1;
    }
    // No CTA may exit while its peer can still read its pair_slot.
    cl.sync();
}

// Row staged in shared memory (STAGED) or re-read from global memory (two-pass).
template <typename T, int VEC, bool ADD, bool STAGED>
__global__ void __launch_bounds__(1024) cta_wide_kernel(NormArgs a) {
    using V = Vec<T, VEC>;
    using R = typename V::Raw;
    extern __shared__ __align__(16) unsigned char dyn_smem[];
    __shared__ float scratch[33];
    T* row_s = reinterpret_cast<T*>(dyn_smem);
    pdl_enter();
    const int tid = threadIdx.x, threads = blockDim.x;
    const int64_t nvec = a.D / VEC;
    const int tail = static_cast<int>(a.D - nvec * VEC);
    const T* w = static_cast<const T*>(a.w);

    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        T* xr = static_cast<T*>(a.x) + r * a.xs;
        const T* rr = static_cast<const T*>(a.res) + r * a.rs;
        T* orow = static_cast<T*>(a.out) + r * a.os;
        float ss = 0.0f;
        for (int64_t idx = tid; idx < nvec; idx += threads) {
            R xv = V::load(xr + idx * VEC);
            float xf[VEC];
            V::unpack(xv, xf);
            if constexpr (ADD) {
                float rf[VEC];
                V::unpack(V::load(rr + idx * VEC), rf);
#pragma unroll
                for (int i = 0; i < VEC; ++i) xf[i] += rf[i];
                xv = V::pack(xf);
                V::store(xr + idx * VEC, xv);
                V::unpack(xv, xf);
            }
            if constexpr (STAGED) V::store(row_s + idx * VEC, xv);
#pragma unroll
            for (int i = 0; i < VEC; ++i) ss = fmaf(xf[i], xf[i], ss);
        }
        float xt = 0.0f;
        if (tid < tail) {
            const int64_t j = nvec * VEC + tid;
            xt = to_f32(xr[j]);
            if constexpr (ADD) {
                const T s = from_f32<T>(xt + to_f32(rr[j]));
                xr[j] = s;
                xt = to_f32(s);
            }
            ss = fmaf(xt, xt, ss);
        }
        ss = block_sum(ss, scratch);
        const float rinv = rsqrtf(ss / static_cast<float>(a.D) + a.eps);
        for (int64_t idx = tid; idx < nvec; idx += threads) {
            float xf[VEC], wf[VEC];
            if constexpr (STAGED) {
                V::unpack(V::load(row_s + idx * VEC), xf);
            } else {
                V::unpack(V::load(xr + idx * VEC), xf);  // this thread's own element(s)
            }
            V::unpack(V::load(w + idx * VEC), wf);
#pragma unroll
            for (int i = 0; i < VEC; ++i) xf[i] = xf[i] * rinv * wf[i];
            V::store(orow + idx * VEC, V::pack(xf));
        }
        if (tid < tail) {
            const int64_t j = nvec * VEC + tid;
            orow[j] = from_f32<T>(xt * rinv * to_f32(w[j]));
        }
    }
}

template <typename KArgs>
cudaError_t smem_opt_in(void (*kernel)(KArgs), size_t smem) {
    if (smem <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
}

template <typename KArgs>
cudaError_t launch_persistent(void (*kernel)(KArgs), const NormArgs& a, const NormPlan& p, size_t smem,
                              cudaStream_t s) {
    const cudaError_t e = smem_opt_in(kernel, smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(persistent_grid(kernel, p.threads, smem, p.num_sms, p.grid)), block(p.threads);
    return launch_kernel(kernel, grid, block, smem, s, p.pdl, a);
}

template <typename KArgs>
cudaError_t launch_pair(void (*kernel)(KArgs), const NormArgs& a, const NormPlan& p, size_t smem,
                        cudaStream_t s) {
    const cudaError_t e = smem_opt_in(kernel, smem);
    if (e != cudaSuccess) return e;
    // Whole pairs only, at most the CTAs resident at once.
    unsigned g = persistent_grid(kernel, p.threads, smem, p.num_sms, p.grid);
    g &= ~1u;
    if (g < 2) g = 2;
    return launch_kernel(kernel, dim3(g), dim3(p.threads), smem, s, p.pdl, a);
}

template <typename T, int VEC, bool ADD>
cudaError_t launch_vec(const NormArgs& a, const NormPlan& p, cudaStream_t s) {
    switch (p.variant) {
        case NORM_WARP_ROWS:
            switch (p.nv) {
                case 1: return launch_persistent(warp_rows_kernel<T, VEC, 1, ADD>, a, p, p.smem, s);
                case 2: return launch_persistent(warp_rows_kernel<T, VEC, 2, ADD>, a, p, p.smem, s);
                case 3: return launch_persistent(warp_rows_kernel<T, VEC, 3, ADD>, a, p, p.smem, s);
                case 4: return launch_persistent(warp_rows_kernel<T, VEC, 4, ADD>, a, p, p.smem, s);
                case 6: return launch_persistent(warp_rows_kernel<T, VEC, 6, ADD>, a, p, p.smem, s);
                case 8: return launch_persistent(warp_rows_kernel<T, VEC, 8, ADD>, a, p, p.smem, s);
                default: return cudaErrorInvalidValue;
            }
        case NORM_CTA_ROW:
            switch (p.nv) {
                case 1: return launch_persistent(cta_row_kernel<T, VEC, 1, ADD>, a, p, p.smem, s);
                case 2: return launch_persistent(cta_row_kernel<T, VEC, 2, ADD>, a, p, p.smem, s);
                case 4: return launch_persistent(cta_row_kernel<T, VEC, 4, ADD>, a, p, p.smem, s);
                case 8: return launch_persistent(cta_row_kernel<T, VEC, 8, ADD>, a, p, p.smem, s);
                default: return cudaErrorInvalidValue;
            }
        case NORM_CTA_PAIR:
            switch (p.nv) {
                case 2: return launch_pair(cta_pair_kernel<T, VEC, 2, ADD>, a, p, p.smem, s);
                case 4: return launch_pair(cta_pair_kernel<T, VEC, 4, ADD>, a, p, p.smem, s);
                case 8: return launch_pair(cta_pair_kernel<T, VEC, 8, ADD>, a, p, p.smem, s);
                default: return cudaErrorInvalidValue;
            }
        case NORM_CTA_SMEM:
            return launch_persistent(cta_wide_kernel<T, VEC, ADD, true>, a, p, p.smem, s);
        case NORM_TWO_PASS:
            return launch_persistent(cta_wide_kernel<T, VEC, ADD, false>, a, p, 0, s);
        default:
            return cudaErrorInvalidValue;
    }
}

template <typename T, bool ADD>
cudaError_t launch_typed(const NormArgs& a, const NormPlan& p, cudaStream_t s) {
    if (p.vec == vec16<T>()) return launch_vec<T, vec16<T>(), ADD>(a, p, s);
    if (p.vec == 1) return launch_vec<T, 1, ADD>(a, p, s);
    return cudaErrorInvalidValue;
}

template <bool ADD>
cudaError_t launch(const NormArgs& a, const NormPlan& p, int dtype, cudaStream_t s) {
    switch (dtype) {
        case DT_F32: return launch_typed<float, ADD>(a, p, s);
        case DT_F16: return launch_typed<__half, ADD>(a, p, s);
        case DT_BF16: return launch_typed<__nv_bfloat16, ADD>(a, p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace norm
}  // namespace sra
