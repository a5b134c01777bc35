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
// it visits; CTA rows (y) stride over the T rows. The loop is software-
// pipelined: the loads of the next pair of rows are issued before the current
// pair is computed and stored, so four 16-byte loads per thread stay in flight
// while the activation runs. No index division anywhere; all accesses 16 bytes
// when the row widths, strides and base pointers allow.
//
// SiLU: g / (1 + e^-g) with one ex2 and one reciprocal (fast intrinsics,
// relative error ~1e-6, far inside half an output ulp of bf16 or fp16); gates
// below -64 take the scaled form of glu_mul (common.cuh), which stays accurate
// down to the smallest outputs the formats hold.
#include "common.cuh"
#include "internal.h"

namespace sra {
namespace glu {

template <typename T, int VEC, int ACT>
__device__ __forceinline__ typename Vec<T, VEC>::Raw combine(const typename Vec<T, VEC>::Raw& gr,
                                                             const typename Vec<T, VEC>::Raw& ur) {
    using V = Vec<T, VEC>;
    float g[VEC], u[VEC];
    V::unpack(gr, g);
    V::unpack(ur, u);
#pragma unroll
    for (int i = 0; i < VEC; ++i) g[i] = glu_mul_fast<ACT>(g[i], u[i]);
    return V::pack(g);
}

// Output vector t of this thread through glu_mul one element at a time, re-read
// from memory (the rare vectors needs_careful finds; kept scalar and rolled so the
// common path keeps its registers).
template <typename T, int VEC, int ACT>
__device__ __forceinline__ void careful_vec(const T* g, T* o, int64_t I) {
#pragma unroll 1
    for (int i = 0; i < VEC; ++i) o[i] = from_f32<T>(glu_mul<ACT>(to_f32(g[i]), to_f32(g[i + I])));
}

// Store the result of row t's vector: the fast form, or careful_vec.
template <typename T, int VEC, int ACT>
__device__ __forceinline__ void emit(const typename Vec<T, VEC>::Raw& gr, const typename Vec<T, VEC>::Raw& ur,
                                     const T* g, T* o, int64_t I) {
    using V = Vec<T, VEC>;
    if (ACT == 0 && __builtin_expect(needs_careful<T, VEC>(gr), 0)) {
        careful_vec<T, VEC, ACT>(g, o, I);
    } else {
        V::store_stream(o, combine<T, VEC, ACT>(gr, ur));
    }
}

// MINB: the CTAs of 256 threads each SM should hold (the launch bound): 5 caps the
// kernel at 48 registers a thread (variant cols_rows, the default), 1 lets the
// compiler take the registers it wants (variant cols_rows_regs, for A/B).
template <typename T, int VEC, int ACT, int MINB>
__global__ void __launch_bounds__(256, MINB) cols_rows_kernel(GluArgs a) {
    using V = Vec<T, VEC>;
    using R = typename V::Raw;
    const int64_t nv = a.I / VEC;
    if (threadIdx.x == 0) {
        // this CTA's column segment of its first two rows, gate and up
        const int64_t j0 = static_cast<int64_t>(blockIdx.x) * blockDim.x;
        const int64_t cols = (nv - j0 < blockDim.x ? nv - j0 : blockDim.x) * VEC;
        for (int64_t t = blockIdx.y; t < a.T && t < blockIdx.y + 2 * static_cast<int64_t>(gridDim.y);
             t += gridDim.y) {
            const T* g = static_cast<const T*>(a.gate_up) + t * a.is + j0 * VEC;
            prefetch_l2(g, cols * static_cast<int64_t>(sizeof(T)));
            prefetch_l2(g + a.I, cols * static_cast<int64_t>(sizeof(T)));
        }
    }
    pdl_enter();
    const int64_t jv = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (jv >= nv) return;
    const T* __restrict__ gcol = static_cast<const T*>(a.gate_up) + jv * VEC;
    T* __restrict__ ocol = static_cast<T*>(a.out) + jv * VEC;
    const int64_t step = gridDim.y;
    int64_t t = blockIdx.y;
    if (t >= a.T) return;
    // current pair (t, t + step); the second row may not exist
    bool have1 = t + step < a.T;
    R ga = V::load_stream(gcol + t * a.is), ua = V::load_stream(gcol + t * a.is + a.I);
    R gb = ga, ub = ua;
    if (have1) {
        gb = V::load_stream(gcol + (t + step) * a.is);
        ub = V::load_stream(gcol + (t + step) * a.is + a.I);
    }
    while (true) {
        const int64_t tn = t + 2 * step;
        const bool next0 = tn < a.T, next1 = tn + step < a.T;
        R gc = ga, uc = ua, gd = gb, ud = ub;
        if (next0) {
            gc = V::load_stream(gcol + tn * a.is);
            uc = V::load_stream(gcol + tn * a.is + a.I);
        }
        if (next1) {
            gd = V::load_stream(gcol + (tn + step) * a.is);
            ud = V::load_stream(gcol + (tn + step) * a.is + a.I);
        }
        emit<T, VEC, ACT>(ga, ua, gcol + t * a.is, ocol + t * a.os, a.I);
        if (have1) emit<T, VEC, ACT>(gb, ub, gcol + (t + step) * a.is, ocol + (t + step) * a.os, a.I);
        if (!next0) break;
        ga = gc, ua = uc, gb = gd, ub = ud;
        have1 = next1;
        t = tn;
    }
}

template <typename T, int VEC, int ACT>
cudaError_t launch_vec(const GluArgs& a, const GluPlan& p, cudaStream_t s) {
    auto kernel = p.variant == GLU_COLS_ROWS_REGS ? cols_rows_kernel<T, VEC, ACT, 1> : cols_rows_kernel<T, VEC, ACT, 5>;
    // Rows are strided over grid_y; size it so that grid_x * grid_y CTAs are all
    // resident at once (one wave, every CTA with the same number of rows +- 1).
    const int64_t resident = static_cast<int64_t>(resident_ctas_per_sm(kernel, p.threads, 0)) * p.num_sms;
    int64_t gy = resident / (p.grid_x > 0 ? p.grid_x : 1);
    if (gy < 1) gy = 1;
    if (gy > a.T) gy = a.T;
    if (gy > 65535) gy = 65535;
    const dim3 grid(static_cast<unsigned>(p.grid_x), static_cast<unsigned>(gy)), block(p.threads);
    return launch_kernel(kernel, grid, block, 0, s, p.pdl, 1, a);
}

template <typename T, int ACT>
cudaError_t launch_act(const GluArgs& a, const GluPlan& p, cudaStream_t s) {
    constexpr int V16 = vec16<T>();
    if (p.vec == V16) return launch_vec<T, V16, ACT>(a, p, s);
    if (p.vec == V16 / 2) return launch_vec<T, V16 / 2, ACT>(a, p, s);
    if (p.vec == V16 / 4) return launch_vec<T, V16 / 4, ACT>(a, p, s);
    if (p.vec == 1) return launch_vec<T, 1, ACT>(a, p, s);
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_typed(const GluArgs& a, const GluPlan& p, int act_kind, cudaStream_t s) {
    return act_kind == 0 ? launch_act<T, 0>(a, p, s) : launch_act<T, 1>(a, p, s);
}

}  // namespace glu

cudaError_t launch_glu(const GluArgs& a, const GluPlan& p, int act, int dtype, cudaStream_t s) {
    if (p.variant != GLU_COLS_ROWS && p.variant != GLU_COLS_ROWS_REGS) return cudaErrorInvalidValue;
    switch (dtype) {
        case DT_F32: return glu::launch_typed<float>(a, p, act, s);
        case DT_F16: return glu::launch_typed<__half>(a, p, act, s);
        case DT_BF16: return glu::launch_typed<__nv_bfloat16>(a, p, act, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sra
