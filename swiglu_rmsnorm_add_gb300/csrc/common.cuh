// Device helpers shared by the kernels: element formats, vector accesses,
// reductions. Internal to the library (not part of the C ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <unordered_map>
#include <utility>

namespace sra {

// Resident CTAs per SM of `kernel` at `threads` threads and `smem` bytes of
// dynamic shared memory (occupancy of the exact function launched), cached per
// (kernel, threads, smem). Persistent grids are sized from it so that every CTA
// is resident at once and no partial second wave forms.
template <typename... KArgs>
inline int resident_ctas_per_sm(void (*kernel)(KArgs...), int threads, size_t smem) {
    static std::mutex mu;
    static std::unordered_map<uint64_t, int> cache;
    const uint64_t key = (reinterpret_cast<uint64_t>(reinterpret_cast<void*>(kernel)) << 20) ^
                         (static_cast<uint64_t>(threads) << 40) ^ static_cast<uint64_t>(smem);
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess) {
        cudaGetLastError();
        n = 1;
    }
    if (n < 1) n = 1;
    std::lock_guard<std::mutex> g(mu);
    cache[key] = n;
    return n;
}

// A persistent grid: `needed` CTAs, capped at what is resident at once.
template <typename... KArgs>
inline unsigned persistent_grid(void (*kernel)(KArgs...), int threads, size_t smem, int num_sms, int64_t needed) {
    const int64_t cap = static_cast<int64_t>(resident_ctas_per_sm(kernel, threads, smem)) * num_sms;
    int64_t g = needed < cap ? needed : cap;
    if (g < 1) g = 1;
    if (g > 0x7fffffff) g = 0x7fffffff;
    return static_cast<unsigned>(g);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch (sm_90 and later). Every kernel calls
// pdl_enter() before its first global-memory access: it waits until the grid
// that precedes it in the stream has completed and its writes are visible,
// then allows the next grid in the stream to be scheduled. When a kernel was
// launched without programmatic stream serialization both instructions are
// no-ops, so the kernels are correct either way.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Hint the L2 to fetch the 128-byte lines of [p, p + bytes), spread over `n`
// cooperating threads (this one is number `i`): plain prefetch instructions, no
// bulk-copy engine involved. Same semantics as prefetch_l2 below.
__device__ __forceinline__ void prefetch_lines(const void* p, int64_t bytes, int i, int n) {
    const char* c = static_cast<const char*>(p);
    const int64_t first = -static_cast<int64_t>(reinterpret_cast<uintptr_t>(p) & 127u);  // line-aligned start
    for (int64_t off = first + static_cast<int64_t>(i) * 128; off < bytes; off += static_cast<int64_t>(n) * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(c + off) : "memory");
}

// Hint the L2 to fetch [p, p + bytes) (p 16-byte aligned, bytes a multiple of 16;
// anything else is ignored). Issued before pdl_enter() for a CTA's own input
// rows: with programmatic dependent launch the CTA runs while the previous
// kernel drains, so the first DRAM round trip overlaps that tail. The L2 is the
// point of coherence and a prefetch has no semantic effect, so data the
// previous kernel is still writing is read correctly after the wait.
__device__ __forceinline__ void prefetch_l2(const void* p, int64_t bytes) {
    if (bytes < 16 || (reinterpret_cast<uintptr_t>(p) & 15u) != 0) return;
    bytes &= ~static_cast<int64_t>(15);
    const char* c = static_cast<const char*>(p);
    constexpr int64_t kMax = int64_t(1) << 20;  // one instruction per MiB
    for (int64_t off = 0; off < bytes; off += kMax) {
        const int64_t n = bytes - off < kMax ? bytes - off : kMax;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c + off), "r"(static_cast<unsigned>(n))
                     : "memory");
    }
}

// Launch `kernel` on `stream`, with programmatic stream serialization when
// `pdl` is set (the kernel may then be scheduled while the previous kernel in
// the stream finishes; pdl_enter() orders its memory accesses after it).
// `cluster` > 1 launches thread-block clusters of that many CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, bool pdl, int cluster, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// Element formats: widen to fp32, narrow with round-to-nearest-even.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Round an fp32 value to T and back (the value a T store would hold).
template <typename T> __device__ __forceinline__ float round_trip(float v) {
    return to_f32(from_f32<T>(v));
}

// ---------------------------------------------------------------------------
// Vector accesses of VEC elements (VEC * sizeof(T) in {2, 4, 8, 16} bytes).
// ---------------------------------------------------------------------------
template <int BYTES> struct RawOf;
template <> struct RawOf<16> { using type = uint4; };
template <> struct RawOf<8> { using type = uint2; };
template <> struct RawOf<4> { using type = unsigned int; };
template <> struct RawOf<2> { using type = unsigned short; };

// 32-bit words of a raw vector.
__device__ __forceinline__ uint32_t word(const uint4& r, int i) {
    return i == 0 ? r.x : (i == 1 ? r.y : (i == 2 ? r.z : r.w));
}
__device__ __forceinline__ uint32_t word(const uint2& r, int i) { return i == 0 ? r.x : r.y; }
__device__ __forceinline__ uint32_t word(const unsigned int& r, int) { return r; }
__device__ __forceinline__ void set_word(uint4& r, int i, uint32_t v) {
    if (i == 0) r.x = v; else if (i == 1) r.y = v; else if (i == 2) r.z = v; else r.w = v;
}
__device__ __forceinline__ void set_word(uint2& r, int i, uint32_t v) { if (i == 0) r.x = v; else r.y = v; }
__device__ __forceinline__ void set_word(unsigned int& r, int, uint32_t v) { r = v; }

// Per-format conversion of packed words (4 bytes) and 16-bit patterns.
template <typename T> struct Elem;
template <> struct Elem<float> {
    __device__ __forceinline__ static void unpack_word(uint32_t w, float* f) { f[0] = __uint_as_float(w); }
    __device__ __forceinline__ static uint32_t pack_word(const float* f) { return __float_as_uint(f[0]); }
    __device__ __forceinline__ static float from_bits16(unsigned short) { return 0.0f; }  // unused
    __device__ __forceinline__ static unsigned short to_bits16(float) { return 0; }      // unused
};
template <> struct Elem<__nv_bfloat16> {
    __device__ __forceinline__ static void unpack_word(uint32_t w, float* f) {
        f[0] = __uint_as_float(w << 16);
        f[1] = __uint_as_float(w & 0xffff0000u);
    }
    __device__ __forceinline__ static uint32_t pack_word(const float* f) {
        __nv_bfloat162 h = __floats2bfloat162_rn(f[0], f[1]);  // RNE, .x = low half
        uint32_t w;
        memcpy(&w, &h, 4);
        return w;
    }
    __device__ __forceinline__ static float from_bits16(unsigned short b) {
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
    __device__ __forceinline__ static unsigned short to_bits16(float f) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(f));
    }
};
template <> struct Elem<__half> {
    __device__ __forceinline__ static void unpack_word(uint32_t w, float* f) {
        __half2 h;
        memcpy(&h, &w, 4);
        const float2 v = __half22float2(h);
        f[0] = v.x;
        f[1] = v.y;
    }
    __device__ __forceinline__ static uint32_t pack_word(const float* f) {
        __half2 h = __floats2half2_rn(f[0], f[1]);
        uint32_t w;
        memcpy(&w, &h, 4);
        return w;
    }
    __device__ __forceinline__ static float from_bits16(unsigned short b) {
        return __half2float(__ushort_as_half(b));
    }
    __device__ __forceinline__ static unsigned short to_bits16(float f) {
        return __half_as_ushort(__float2half_rn(f));
    }
};

template <typename T, int VEC>
struct Vec {
    static constexpr int BYTES = VEC * int(sizeof(T));
    using Raw = typename RawOf<BYTES>::type;

    // Plain load (cached in L1 / L2).
    __device__ __forceinline__ static Raw load(const T* p) { return *reinterpret_cast<const Raw*>(p); }
    // Read-only streaming load: each byte is read once; evict first.
    __device__ __forceinline__ static Raw load_stream(const T* p) {
        return ldcs(reinterpret_cast<const Raw*>(p));
    }
    __device__ __forceinline__ static void store(T* p, Raw r) { *reinterpret_cast<Raw*>(p) = r; }
    __device__ __forceinline__ static void store_stream(T* p, Raw r) {
        stcs(reinterpret_cast<Raw*>(p), r);
    }

    __device__ __forceinline__ static void unpack(const Raw& r, float (&f)[VEC]) {
        if constexpr (BYTES == 2) {
            f[0] = Elem<T>::from_bits16(r);
        } else {
            constexpr int W = BYTES / 4, PER = 4 / int(sizeof(T));
#pragma unroll
            for (int i = 0; i < W; ++i) Elem<T>::unpack_word(word(r, i), f + i * PER);
        }
    }
    __device__ __forceinline__ static Raw pack(const float (&f)[VEC]) {
        Raw r;
        if constexpr (BYTES == 2) {
            r = Elem<T>::to_bits16(f[0]);
        } else {
            constexpr int W = BYTES / 4, PER = 4 / int(sizeof(T));
#pragma unroll
            for (int i = 0; i < W; ++i) set_word(r, i, Elem<T>::pack_word(f + i * PER));
        }
        return r;
    }

  private:
    __device__ __forceinline__ static uint4 ldcs(const uint4* p) { return __ldcs(p); }
    __device__ __forceinline__ static uint2 ldcs(const uint2* p) { return __ldcs(p); }
    __device__ __forceinline__ static unsigned int ldcs(const unsigned int* p) { return __ldcs(p); }
    __device__ __forceinline__ static unsigned short ldcs(const unsigned short* p) { return __ldcs(p); }
    __device__ __forceinline__ static void stcs(uint4* p, uint4 v) { __stcs(p, v); }
    __device__ __forceinline__ static void stcs(uint2* p, uint2 v) { __stcs(p, v); }
    __device__ __forceinline__ static void stcs(unsigned int* p, unsigned int v) { __stcs(p, v); }
    __device__ __forceinline__ static void stcs(unsigned short* p, unsigned short v) { __stcs(p, v); }
};

// Elements per 16-byte access.
template <typename T> __host__ __device__ constexpr int vec16() { return 16 / int(sizeof(T)); }

// ---------------------------------------------------------------------------
// Gated linear units: act(g) * u in fp32, act = SiLU (ACT 0) or ReLU (ACT 1).
//
// SiLU as g / (1 + e^-g) with one ex2 and one fast reciprocal; the fast
// reciprocal returns 0 once its divisor passes 2^126 (g below -87.3), and the
// true value there is still a normal number of bf16 and fp32 (silu(-88) is about
// -5e-37). So gates below -64 take another form: there e^g < 2^-92, so 1 + e^g
// rounds to 1 in fp32 and silu(g) * u = g * u * e^g to far below an fp32 ulp.
// e^g itself leaves fp32's normal range below -87.3, so it is applied as four
// equal factors e^(g/4) (g/4 is exact), the operand u scaled down first: every
// intermediate is a normal fp32 number whenever the result is one, and the
// result is within a few fp32 ulps of the exact product (expf is CUDA's accurate
// exponential). A NaN gate stays NaN; -inf gives NaN, as g / (1 + e^-g) does.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float silu_mul_far(float g, float u) {
    const float e = expf(0.25f * g);
    return (((u * e) * g) * e) * e * e;
}

constexpr float kSiluFar = -64.0f;  // gates below take silu_mul_far

// act(g) * u in the fast form: g / (1 + e^-g) (one ex2, one fast reciprocal),
// times u. Exact to a few fp32 ulps for gates at or above kSiluFar, except that
// for a gate below 2^-64 in size g * sigma can be an fp32 subnormal whose lost
// digits a large u would scale back into view; glu_mul covers both cases.
template <int ACT>
__device__ __forceinline__ float glu_mul_fast(float g, float u) {
    if constexpr (ACT == 0) {
        return __fdividef(g, 1.0f + __expf(-g)) * u;
    } else {
        return fmaxf(g, 0.0f) * u;
    }
}

// act(g) * u for every gate. Below kSiluFar: silu_mul_far. Otherwise sigma(g) =
// 1 / (1 + e^-g) first and then g * u * sigma in the order that keeps the
// partial product normal: g * u first for |g| < 1 (no overflow there: |g u| <
// |u|), g * sigma first otherwise (at least 64 e^-64 in size, and g * u could
// overflow where the result does not).
template <int ACT>
__device__ __forceinline__ float glu_mul(float g, float u) {
    if constexpr (ACT == 0) {
        if (g < kSiluFar) return silu_mul_far(g, u);
        const float sig = __fdividef(1.0f, 1.0f + __expf(-g));
        return fabsf(g) < 1.0f ? (g * u) * sig : (g * sig) * u;
    } else {
        return fmaxf(g, 0.0f) * u;
    }
}

// Whether a raw vector of gates needs glu_mul's careful forms (never on the
// configured inputs): a gate below -64 — a negative value's bit pattern grows with
// its magnitude, so that is an unsigned compare of each element's bits with those
// of -64 (negative NaNs compare above it too; glu_mul keeps them NaN) — or, in
// fp32, a nonzero gate below 2^-64 in size, whose g * sigma could be subnormal.
// In bf16 and fp16 the smallest gate, halved, is still an fp32 number with 15 or
// more significant bits, so only the far-negative test applies there.
template <typename T> struct FarBits;
template <> struct FarBits<__nv_bfloat16> { static constexpr uint32_t v = 0xC280u; };
template <> struct FarBits<__half> { static constexpr uint32_t v = 0xD400u; };
template <> struct FarBits<float> { static constexpr uint32_t v = 0xC2800000u; };

template <typename T, int VEC>
__device__ __forceinline__ bool needs_careful(const typename Vec<T, VEC>::Raw& gr) {
    constexpr int BYTES = VEC * int(sizeof(T));
    if constexpr (BYTES == 2) {
        return static_cast<uint32_t>(gr) > FarBits<T>::v;
    } else {
        uint32_t hit = 0;
#pragma unroll
        for (int i = 0; i < BYTES / 4; ++i) {
            const uint32_t w = word(gr, i);
            if constexpr (sizeof(T) == 4) {
                const uint32_t m = w & 0x7fffffffu;
                hit |= (w > FarBits<T>::v || (m != 0u && m < 0x1f800000u)) ? 1u : 0u;  // 2^-64
            } else {
                hit |= __vcmpgtu2(w, FarBits<T>::v * 0x10001u);
            }
        }
        return hit != 0;
    }
}

// ---------------------------------------------------------------------------
// Reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Sum over the whole CTA; every thread gets the total. `scratch` holds >= 33 floats
// of shared memory. blockDim.x must be a multiple of 32.
__device__ __forceinline__ float block_sum(float v, float* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    v = warp_sum(v);
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float s = lane < nwarps ? scratch[lane] : 0.0f;
        s = warp_sum(s);
        if (lane == 0) scratch[32] = s;
    }
    __syncthreads();
    float total = scratch[32];
    __syncthreads();  // scratch may be reused by the next row
    return total;
}

// Double-precision sum over a warp / a CTA (for the rare rows whose fp32 sum of
// squares leaves fp32's range). `scratch` holds >= 33 doubles of shared memory.
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ double block_sum_d(double v, double* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    v = warp_sum_d(v);
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    if (warp == 0) {
        double s = lane < nwarps ? scratch[lane] : 0.0;
        s = warp_sum_d(s);
        if (lane == 0) scratch[32] = s;
    }
    __syncthreads();
    const double total = scratch[32];
    __syncthreads();
    return total;
}

// ---------------------------------------------------------------------------
// RMSNorm scale outside fp32's comfortable range.
//
// The sum of squares is accumulated in fp32. It overflows for rows with
// elements of about 1.8e19 and up (bf16 and fp32 hold up to 3.4e38), and once
// sum / D + eps falls below 2^-64, squares in fp32's subnormal range have lost
// digits that then matter. Rows in either case (never the configured inputs)
// are summed again in double, and the factor 1 / sqrt(mean + eps) is split
// into a power of two `pre` and an fp32 `rinv`: out = ((x * pre) * rinv) * w,
// every factor finite and normal (the factor itself can exceed fp32's range,
// up to about 2^155 for rows of fp32 subnormals with eps = 0). A NaN sum stays
// on the ordinary path (every output is NaN either way).
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool ss_in_range(float ss, int64_t D, float eps) {
    return !(ss > 3.40282347e38f) && !(ss / static_cast<float>(D) + eps < 0x1p-64f);
}

struct WideScale {
    float pre, rinv;
};

__device__ __forceinline__ WideScale wide_scale(double sd, int64_t D, float eps) {
    const double rd = 1.0 / sqrt(sd / static_cast<double>(D) + static_cast<double>(eps));
    if (rd > 0x1p64) return {0x1p64f, static_cast<float>(rd * 0x1p-64)};
    if (rd < 0x1p-64) return {0x1p-64f, static_cast<float>(rd * 0x1p64)};
    return {1.0f, static_cast<float>(rd)};
}

}  // namespace sra
