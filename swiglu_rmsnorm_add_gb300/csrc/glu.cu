// Gated linear units over a fused gate_up tensor: SwiGLU silu(g) * u and
// ReGLU relu(g) * u.
//
// koas-w.github.io "preformanceimprovement", section 2: gate and up are loaded
// together, the activation and the product happen in registers and the output
// is written once (one memory pass instead of three). mer.dev "AsyncT vllm
// 适配加速笔记（一）", section 3.3: ReGLU as a single relu_and_mul kernel.
// gate = columns [0, I) of a row, up = columns [I, 2I).
//
// Layout: a 2-D grid. Thread (x) owns one VEC-wide column group j of every row
// it visits; CTA rows (y) stride over the T rows, two rows in flight per
// thread. No index division anywhere; all accesses 16 bytes when the row
// widths, strides and base pointers allow.
//
// SiLU: g * sigma(g) with sigma from one ex2 and one reciprocal (fast
// intrinsics, relative error ~1e-6, far inside half an output ulp of bf16 or
// fp16). For g < 0 sigma(g) = e^g / (1 + e^g) is used, so the exponential
// never overflows; |g| > ~87 underflows e^-|g| to zero, where the true SiLU
// magnitude is below 2^-119.
#include "common.cuh"
#include "internal.h"

namespace sra {
namespace glu {

template <int ACT>
__device__ __forceinline__ float act(float g) {
    if constexpr (ACT == 0) {
        const float e = __expf(-fabsf(g));            // e^-|g| in (0, 1]
        const float r = __fdividef(1.0f, 1.0f + e);   // sigma(|g|); denominator in [1, 2]
        const float sig = g >= 0.0f ? r : e * r;      // sigma(g)
        return g * sig;
    } else {
        return fmaxf(g, 0.0f);
    }
}

template <typename T, int VEC, int ACT>
__device__ __forceinline__ typename Vec<T, VEC>::Raw combine(const typename Vec<T, VEC>::Raw& gr,
                                                             const typename Vec<T, VEC>::Raw& ur) {
    using V = Vec<T, VEC>;
    float g[VEC], u[VEC];
    V::unpack(gr, g);
    V::unpack(ur, u);
#pragma unroll
    for (int i = 0; i < VEC; ++i) g[i] = act<ACT>(g[i]) * u[i];
    return V::pack(g);
}

template <typename T, int VEC, int ACT>
__global__ void __launch_bounds__(256) cols_rows_kernel(GluArgs a) {
    using V = Vec<T, VEC>;
    using R = typename V::Raw;
    const int64_t nv = a.I / VEC;
    const int64_t jv = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (jv >= nv) return;
    const T* __restrict__ gcol = static_cast<const T*>(a.gate_up) + jv * VEC;
    T* __restrict__ ocol = static_cast<T*>(a.out) + jv * VEC;
    const int64_t step = gridDim.y;
    int64_t t = blockIdx.y;
    // Two rows per iteration: four independent 16-byte loads in flight per thread.
    for (; t + step < a.T; t += 2 * step) {
        const T* g0 = gcol + t * a.is;
        const T* g1 = gcol + (t + step) * a.is;
        const R ga = V::load_stream(g0), ua = V::load_stream(g0 + a.I);
        const R gb = V::load_stream(g1), ub = V::load_stream(g1 + a.I);
        V::store_stream(ocol + t * a.os, combine<T, VEC, ACT>(ga, ua));
        V::store_stream(ocol + (t + step) * a.os, combine<T, VEC, ACT>(gb, ub));
    }
    if (t < a.T) {
        const T* g0 = gcol + t * a.is;
        const R ga = V::load_stream(g0), ua = V::load_stream(g0 + a.I);
        V::store_stream(ocol + t * a.os, combine<T, VEC, ACT>(ga, ua));
    }
}

template <typename T, int ACT>
cudaError_t launch_act(const GluArgs& a, const GluPlan& p, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(p.grid_x), static_cast<unsigned>(p.grid_y)), block(p.threads);
    constexpr int V16 = vec16<T>();
    if (p.vec == V16) {
        cols_rows_kernel<T, V16, ACT><<<grid, block, 0, s>>>(a);
    } else if (p.vec == V16 / 2) {
        cols_rows_kernel<T, V16 / 2, ACT><<<grid, block, 0, s>>>(a);
    } else if (p.vec == V16 / 4) {
        cols_rows_kernel<T, V16 / 4, ACT><<<grid, block, 0, s>>>(a);
    } else if (p.vec == 1) {
        cols_rows_kernel<T, 1, ACT><<<grid, block, 0, s>>>(a);
    } else {
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const GluArgs& a, const GluPlan& p, int act_kind, cudaStream_t s) {
    return act_kind == 0 ? launch_act<T, 0>(a, p, s) : launch_act<T, 1>(a, p, s);
}

}  // namespace glu

cudaError_t launch_glu(const GluArgs& a, const GluPlan& p, int act, int dtype, cudaStream_t s) {
    if (p.variant != GLU_COLS_ROWS) return cudaErrorInvalidValue;
    switch (dtype) {
        case DT_F32: return glu::launch_typed<float>(a, p, act, s);
        case DT_F16: return glu::launch_typed<__half>(a, p, act, s);
        case DT_BF16: return glu::launch_typed<__nv_bfloat16>(a, p, act, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sra
