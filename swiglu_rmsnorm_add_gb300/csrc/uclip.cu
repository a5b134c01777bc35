// UClip / DyHT: out = clamp(alpha * x, lo, hi) * gamma over rows of D channels.
//
// mer.dev "AsyncT vllm 适配加速笔记（一）": section 0 replaces every RMSNorm of the
// model (pre-norm, Q/K norm, final norm, post-attention norm) by
// DyHT(x) = y * clamp(a x, -1, 1); section 3.3 writes it as one kernel with a
// scalar or per-channel alpha and gamma and free clip bounds, and notes that the
// Q/K norms read narrow 3-D [N, H, D] views of the fused QKV projection, whose
// middle (head) stride a single row stride cannot express.
//
// No reduction: every element is independent. Layout: a 2-D grid of 2-D CTAs.
// threadIdx.x owns one VEC-wide column group of every row the thread visits, so
// its alpha / gamma values are loaded once; threadIdx.y and blockIdx.y stride
// over the N * H rows, which are decoded to (n, h) once and then stepped
// without division (RowWalk). alpha / gamma being per-channel or scalar is a
// template choice, so a scalar costs one register. Four rows per thread are loaded before any is computed, so
// four 16-byte loads are in flight per thread. An element is read and written
// by the same thread only, so out == x (in place) is safe.
//
// Arithmetic: fp32 a * x, the clamp (a NaN product becomes the lower bound, as
// in the page's fminf(fmaxf(..)) form), then * g, one RNE to the dtype.
#include "common.cuh"
#include "internal.h"

namespace sra {
namespace uclip {

constexpr int kRowsInFlight = 4;

// fmaxf returns its other operand when one is NaN, so a NaN product takes the
// lower bound, as the page's kernel (fmaxf, then fminf) has it.
__device__ __forceinline__ float clip(float v, float lo, float hi) { return fminf(fmaxf(v, lo), hi); }

// VEC consecutive fp32 parameters starting at p + col (per channel), or p[0] repeated.
template <int VEC, bool PER_CHANNEL>
__device__ __forceinline__ void load_params(const float* p, int64_t col, float (&f)[VEC]) {
    if constexpr (!PER_CHANNEL) {
        const float v = p[0];
#pragma unroll
        for (int i = 0; i < VEC; ++i) f[i] = v;
    } else {
        constexpr int W = VEC >= 4 ? 4 : VEC;
        using P = Vec<float, W>;
#pragma unroll
        for (int i = 0; i < VEC; i += W) {
            float g[W];
            P::unpack(P::load(p + col + i), g);
#pragma unroll
            for (int j = 0; j < W; ++j) f[i + j] = g[j];
        }
    }
}

// Element offsets of consecutive rows r, r + step, r + 2 step, ... of an
// [N, H, D] view, advanced without division: h counts heads within a token.
struct RowWalk {
    int64_t xoff, ooff;    // offsets of the current row in x and out
    int64_t xstep, ostep;  // offset change for step = dn tokens + dh heads
    int64_t xwrap, owrap;  // extra change when h wraps past H: one token on, H heads back
    int h, dh, H;          // H < 2^31 (checked on the host)
    __device__ __forceinline__ void advance() {
        xoff += xstep, ooff += ostep, h += dh;
        if (h >= H) h -= H, xoff += xwrap, ooff += owrap;
    }
};

template <typename T, int VEC, bool APC, bool GPC>
__global__ void __launch_bounds__(256) rows_kernel(UclipArgs a) {
    using V = Vec<T, VEC>;
    using R = typename V::Raw;
    const int64_t nv = a.D / VEC;
    const int64_t cv = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // column group
    const int64_t rows = a.N * a.H;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * blockDim.y + threadIdx.y;
    const int64_t step = static_cast<int64_t>(gridDim.y) * blockDim.y;
    const bool active = cv < nv && r0 < rows;
    const T* __restrict__ xcol = static_cast<const T*>(a.x) + cv * VEC;
    RowWalk w;
    {
        const int64_t H = a.H > 0 ? a.H : 1;  // the host never launches with no rows
        const int64_t n = r0 / H, dn = step / H;
        w.h = static_cast<int>(r0 - n * H), w.dh = static_cast<int>(step - dn * H), w.H = static_cast<int>(H);
        w.xoff = n * a.xn + w.h * a.xh, w.ooff = n * a.on + w.h * a.oh;
        w.xstep = dn * a.xn + w.dh * a.xh, w.ostep = dn * a.on + w.dh * a.oh;
        w.xwrap = a.xn - H * a.xh, w.owrap = a.on - H * a.oh;
    }
    if (active && ((cv * VEC * static_cast<int64_t>(sizeof(T))) & 127) == 0) {
        // this thread's first batch of rows into L2, one prefetch per 128-byte line
        RowWalk p = w;
        for (int k = 0; k < kRowsInFlight && r0 + k * step < rows; ++k) {
            asm volatile("prefetch.global.L2 [%0];" ::"l"(xcol + p.xoff) : "memory");
            p.advance();
        }
    }
    pdl_enter();
    if (!active) return;

    float al[VEC], ga[VEC];
    load_params<VEC, APC>(a.alpha, cv * VEC, al);
    load_params<VEC, GPC>(a.gamma, cv * VEC, ga);
    T* ocol = static_cast<T*>(a.out) + cv * VEC;
    const float lo = a.lo, hi = a.hi;

    for (int64_t r = r0; r < rows; r += kRowsInFlight * step) {
        R raw[kRowsInFlight];
        int64_t oo[kRowsInFlight];
#pragma unroll
        for (int k = 0; k < kRowsInFlight; ++k) {
            oo[k] = w.ooff;
            if (r + k * step < rows) raw[k] = V::load(xcol + w.xoff);
            w.advance();
        }
#pragma unroll
        for (int k = 0; k < kRowsInFlight; ++k) {
            if (r + k * step >= rows) break;
            float f[VEC];
            V::unpack(raw[k], f);
#pragma unroll
            for (int i = 0; i < VEC; ++i) f[i] = clip(al[i] * f[i], lo, hi) * ga[i];
            V::store(ocol + oo[k], V::pack(f));
        }
    }
}

template <typename T, int VEC, bool APC, bool GPC>
cudaError_t launch_flags(const UclipArgs& a, const UclipPlan& p, cudaStream_t s) {
    auto kernel = rows_kernel<T, VEC, APC, GPC>;
    const int threads = p.bx * p.by;
    // every CTA resident at once: grid_y from the exact kernel's occupancy
    const int64_t resident = static_cast<int64_t>(resident_ctas_per_sm(kernel, threads, 0)) * p.num_sms;
    int64_t gy = resident / (p.grid_x > 0 ? p.grid_x : 1);
    gy = gy < 1 ? 1 : gy;
    gy = gy > p.grid_y ? p.grid_y : gy;
    gy = gy > 65535 ? 65535 : gy;
    const dim3 grid(static_cast<unsigned>(p.grid_x), static_cast<unsigned>(gy)), block(p.bx, p.by);
    return launch_kernel(kernel, grid, block, 0, s, p.pdl, 1, a);
}

template <typename T, int VEC>
cudaError_t launch_vec(const UclipArgs& a, const UclipPlan& p, cudaStream_t s) {
    if (a.alpha_pc) return a.gamma_pc ? launch_flags<T, VEC, true, true>(a, p, s) : launch_flags<T, VEC, true, false>(a, p, s);
    return a.gamma_pc ? launch_flags<T, VEC, false, true>(a, p, s) : launch_flags<T, VEC, false, false>(a, p, s);
}

template <typename T>
cudaError_t launch_typed(const UclipArgs& a, const UclipPlan& p, cudaStream_t s) {
    constexpr int V16 = vec16<T>();
    if (p.vec == V16) return launch_vec<T, V16>(a, p, s);
    if (p.vec == V16 / 2) return launch_vec<T, V16 / 2>(a, p, s);
    if (p.vec == V16 / 4) return launch_vec<T, V16 / 4>(a, p, s);
    if (p.vec == 1) return launch_vec<T, 1>(a, p, s);
    return cudaErrorInvalidValue;
}

}  // namespace uclip

cudaError_t launch_uclip(const UclipArgs& a, const UclipPlan& p, int dtype, cudaStream_t s) {
    switch (dtype) {
        case DT_F32: return uclip::launch_typed<float>(a, p, s);
        case DT_F16: return uclip::launch_typed<__half>(a, p, s);
        case DT_BF16: return uclip::launch_typed<__nv_bfloat16>(a, p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sra
