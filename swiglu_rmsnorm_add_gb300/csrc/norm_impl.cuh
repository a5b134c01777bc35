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
// Every variant keeps a row's elements with one thread across both passes, so
// in-place use (out == x) is safe and no inter-thread hazard exists on the row.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace sra {
namespace norm {

// Row pointers for a row index.
template <typename T>
struct Row {
    T* x;
    const T* res;
    T* out;
};

template <typename T>
__device__ __forceinline__ Row<T> row_ptrs(const NormArgs& a, int64_t r) {
    Row<T> p;
    p.x = static_cast<T*>(a.x) + r * a.xs;
    p.res = static_cast<const T*>(a.res) + r * a.rs;
    p.out = static_cast<T*>(a.out) + r * a.os;
    return p;
}

// Register-resident row: THREADS threads own accesses idx = v * THREADS + tid,
// v < NV. GROUP_IS_WARP selects a shuffle-only reduction.
template <typename T, int VEC, int NV, bool ADD, bool GROUP_IS_WARP>
__device__ __forceinline__ void row_in_registers(const NormArgs& a, int64_t r, int tid, int threads,
                                                 float* scratch) {
    using V = Vec<T, VEC>;
    using R = typename V::Raw;
    const int64_t nvec = a.D / VEC;
    const int tail = static_cast<int>(a.D - nvec * VEC);
    const T* w = static_cast<const T*>(a.w);
    Row<T> p = row_ptrs<T>(a, r);

    R xv[NV];
    R wv[NV];
    float xt = 0.0f, wt = 0.0f;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int64_t idx = static_cast<int64_t>(v) * threads + tid;
        if (idx < nvec) xv[v] = V::load(p.x + idx * VEC);
    }
    if (tid < tail) xt = to_f32(p.x[nvec * VEC + tid]);

    float ss = 0.0f;
    if constexpr (ADD) {
        R rv[NV];
        float rt = 0.0f;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int64_t idx = static_cast<int64_t>(v) * threads + tid;
            if (idx < nvec) rv[v] = V::load(p.res + idx * VEC);
        }
        if (tid < tail) rt = to_f32(p.res[nvec * VEC + tid]);
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int64_t idx = static_cast<int64_t>(v) * threads + tid;
            if (idx < nvec) {
                float xf[VEC], rf[VEC];
                V::unpack(xv[v], xf);
                V::unpack(rv[v], rf);
#pragma unroll
                for (int i = 0; i < VEC; ++i) xf[i] += rf[i];
                xv[v] = V::pack(xf);          // the rounded sum
                V::store(p.x + idx * VEC, xv[v]);
                V::unpack(xv[v], xf);
#pragma unroll
                for (int i = 0; i < VEC; ++i) ss = fmaf(xf[i], xf[i], ss);
            }
        }
        if (tid < tail) {
            const T s = from_f32<T>(xt + rt);
            p.x[nvec * VEC + tid] = s;
            xt = to_f32(s);
            ss = fmaf(xt, xt, ss);
        }
    } else {
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int64_t idx = static_cast<int64_t>(v) * threads + tid;
            if (idx < nvec) {
                float xf[VEC];
                V::unpack(xv[v], xf);
#pragma unroll
                for (int i = 0; i < VEC; ++i) ss = fmaf(xf[i], xf[i], ss);
            }
        }
        if (tid < tail) ss = fmaf(xt, xt, ss);
    }

    // Weights: issued before the reduction so their latency hides behind it.
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int64_t idx = static_cast<int64_t>(v) * threads + tid;
        if (idx < nvec) wv[v] = V::load(w + idx * VEC);
    }
    if (tid < tail) wt = to_f32(w[nvec * VEC + tid]);

    if constexpr (GROUP_IS_WARP) {
        ss = warp_sum(ss);
    } else {
        ss = block_sum(ss, scratch);
    }
    const float rinv = rsqrtf(ss / static_cast<float>(a.D) + a.eps);

#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int64_t idx = static_cast<int64_t>(v) * threads + tid;
        if (idx < nvec) {
            float xf[VEC], wf[VEC];
            V::unpack(xv[v], xf);
            V::unpack(wv[v], wf);
#pragma unroll
            for (int i = 0; i < VEC; ++i) xf[i] = xf[i] * rinv * wf[i];
            V::store(p.out + idx * VEC, V::pack(xf));
        }
    }
    if (tid < tail) p.out[nvec * VEC + tid] = from_f32<T>(xt * rinv * wt);
}

template <typename T, int VEC, int NV, bool ADD>
__global__ void __launch_bounds__(256) warp_rows_kernel(NormArgs a) {
    const int warps_per_cta = blockDim.x >> 5;
    const int64_t step = static_cast<int64_t>(gridDim.x) * warps_per_cta;
    const int lane = threadIdx.x & 31;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * warps_per_cta + (threadIdx.x >> 5); r < a.rows;
         r += step) {
        row_in_registers<T, VEC, NV, ADD, true>(a, r, lane, 32, nullptr);
    }
}

// Largest CTA the register-resident CTA variant is compiled for, per NV.
template <int NV> constexpr int cta_row_max_threads() { return NV >= 8 ? 256 : (NV >= 4 ? 512 : 1024); }

template <typename T, int VEC, int NV, bool ADD>
__global__ void __launch_bounds__(cta_row_max_threads<NV>()) cta_row_kernel(NormArgs a) {
    __shared__ float scratch[33];
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        row_in_registers<T, VEC, NV, ADD, false>(a, r, threadIdx.x, blockDim.x, scratch);
    }
}

// Row staged in shared memory (STAGED) or re-read from global memory (two-pass).
template <typename T, int VEC, bool ADD, bool STAGED>
__global__ void __launch_bounds__(1024) cta_wide_kernel(NormArgs a) {
    using V = Vec<T, VEC>;
    using R = typename V::Raw;
    extern __shared__ __align__(16) unsigned char dyn_smem[];
    __shared__ float scratch[33];
    T* row_s = reinterpret_cast<T*>(dyn_smem);
    const int tid = threadIdx.x, threads = blockDim.x;
    const int64_t nvec = a.D / VEC;
    const int tail = static_cast<int>(a.D - nvec * VEC);
    const T* w = static_cast<const T*>(a.w);

    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        Row<T> p = row_ptrs<T>(a, r);
        float ss = 0.0f;
        for (int64_t idx = tid; idx < nvec; idx += threads) {
            R xr = V::load(p.x + idx * VEC);
            float xf[VEC];
            V::unpack(xr, xf);
            if constexpr (ADD) {
                float rf[VEC];
                V::unpack(V::load(p.res + idx * VEC), rf);
#pragma unroll
                for (int i = 0; i < VEC; ++i) xf[i] += rf[i];
                xr = V::pack(xf);
                V::store(p.x + idx * VEC, xr);
                V::unpack(xr, xf);
            }
            if constexpr (STAGED) V::store(row_s + idx * VEC, xr);
#pragma unroll
            for (int i = 0; i < VEC; ++i) ss = fmaf(xf[i], xf[i], ss);
        }
        float xt = 0.0f;
        if (tid < tail) {
            const int64_t j = nvec * VEC + tid;
            xt = to_f32(p.x[j]);
            if constexpr (ADD) {
                const T s = from_f32<T>(xt + to_f32(p.res[j]));
                p.x[j] = s;
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
                V::unpack(V::load(p.x + idx * VEC), xf);  // this thread's own element(s)
            }
            V::unpack(V::load(w + idx * VEC), wf);
#pragma unroll
            for (int i = 0; i < VEC; ++i) xf[i] = xf[i] * rinv * wf[i];
            V::store(p.out + idx * VEC, V::pack(xf));
        }
        if (tid < tail) {
            const int64_t j = nvec * VEC + tid;
            p.out[j] = from_f32<T>(xt * rinv * to_f32(w[j]));
        }
    }
}

template <typename T, int VEC, bool ADD>
cudaError_t launch_vec(const NormArgs& a, const NormPlan& p, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(p.grid)), block(p.threads);
    switch (p.variant) {
        case NORM_WARP_ROWS:
            switch (p.nv) {
                case 1: warp_rows_kernel<T, VEC, 1, ADD><<<grid, block, 0, s>>>(a); break;
                case 2: warp_rows_kernel<T, VEC, 2, ADD><<<grid, block, 0, s>>>(a); break;
                case 4: warp_rows_kernel<T, VEC, 4, ADD><<<grid, block, 0, s>>>(a); break;
                case 8: warp_rows_kernel<T, VEC, 8, ADD><<<grid, block, 0, s>>>(a); break;
                default: return cudaErrorInvalidValue;
            }
            break;
        case NORM_CTA_ROW:
            switch (p.nv) {
                case 1: cta_row_kernel<T, VEC, 1, ADD><<<grid, block, 0, s>>>(a); break;
                case 2: cta_row_kernel<T, VEC, 2, ADD><<<grid, block, 0, s>>>(a); break;
                case 4: cta_row_kernel<T, VEC, 4, ADD><<<grid, block, 0, s>>>(a); break;
                case 8: cta_row_kernel<T, VEC, 8, ADD><<<grid, block, 0, s>>>(a); break;
                default: return cudaErrorInvalidValue;
            }
            break;
        case NORM_CTA_SMEM:
            cta_wide_kernel<T, VEC, ADD, true><<<grid, block, p.smem, s>>>(a);
            break;
        case NORM_TWO_PASS:
            cta_wide_kernel<T, VEC, ADD, false><<<grid, block, 0, s>>>(a);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
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

template <typename T, bool ADD>
cudaError_t smem_prepare_typed(int vec, size_t bytes) {
    if (vec == vec16<T>())
        return cudaFuncSetAttribute(cta_wide_kernel<T, vec16<T>(), ADD, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (vec == 1)
        return cudaFuncSetAttribute(cta_wide_kernel<T, 1, ADD, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    return cudaErrorInvalidValue;
}

template <bool ADD>
cudaError_t smem_prepare(int dtype, int vec, size_t bytes) {
    switch (dtype) {
        case DT_F32: return smem_prepare_typed<float, ADD>(vec, bytes);
        case DT_F16: return smem_prepare_typed<__half, ADD>(vec, bytes);
        case DT_BF16: return smem_prepare_typed<__nv_bfloat16, ADD>(vec, bytes);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace norm
}  // namespace sra
