// Fused RoPE (neox halves, or interleaved GPT-J pairs) + paged KV-cache store.
//
// koas-w.github.io "preformanceimprovement", section 1: Q, K, V, cos and sin
// are read once; Q and K are rotated in registers; Q is written back in place;
// K_rot and V go straight into the paged cache through slot_mapping, with no
// temporary tensors. GQA is handled inside the kernel (each KV head is written
// once per token; kv_head = head / (n_head / n_kv_head) is the read-side map).
// Cache layout [2, num_blocks, block_size, n_kv_head, head_dim] (mer.dev
// "AsyncT vllm 适配加速笔记（一）", section 1.1).
//
// Work decomposition: a token's work is U = (n_head + 2 * n_kv_head) * (h / P)
// tasks of P rotation pairs each (h = head_dim / 2; P = 16 bytes of elements, or
// 1). Task u of a token is fixed per thread (thread u of the CTA), so a thread
// decodes its head and offset once; CTAs stride over tokens. A second kernel
// gives each thread two tasks of a token (token_cta2_kernel below). With Qwen2.5-1.5B
// shapes (12 Q + 2 K + 2 V heads, head_dim 128, bf16) a token is exactly 128
// tasks: one 128-thread CTA per token, every access 16 bytes, a warp's
// accesses to one head row fully coalesced.
//
// The rotation y = x_lo * c - x_hi * s (and x_hi * c + x_lo * s) is evaluated
// with Kahan's fma-based difference of products, so its fp32 error is a few
// ulps of the RESULT even under cancellation; one RNE to the dtype follows.
#include "common.cuh"
#include "internal.h"

namespace sra {
namespace rope {

// a * b - c * d, accurate to a few ulps of the result (W. Kahan).
__device__ __forceinline__ float diff_of_products(float a, float b, float c, float d) {
    const float w = c * d;
    const float e = fmaf(-c, d, w);  // w - c * d, exactly
    const float f = fmaf(a, b, -w);
    return f + e;
}

// The per-channel parameters of the dimensions a task's lo[j] / hi[j] hold:
// neox lo = i0 + j, hi = h + i0 + j; interleaved lo = 2 (i0 + j), hi = lo + 1.
template <int P, bool IL>
__device__ __forceinline__ void load_pair_params(const float* p, int i0, int h, float (&lo)[P], float (&hi)[P]) {
    constexpr int CW = P >= 4 ? 4 : 1;
    using C = Vec<float, CW>;
    if constexpr (IL && P >= 2) {
#pragma unroll
        for (int j = 0; j < 2 * P; j += CW) {
            float f[CW];
            C::unpack(C::load(p + 2 * i0 + j), f);
#pragma unroll
            for (int q = 0; q < CW; ++q) {
                if ((j + q) % 2 == 0) lo[(j + q) / 2] = f[q];
                else hi[(j + q) / 2] = f[q];
            }
        }
    } else {
        const float* plo = IL ? p + 2 * i0 : p + i0;
        const float* phi = IL ? p + 2 * i0 + 1 : p + h + i0;
#pragma unroll
        for (int j = 0; j < P; j += CW) {
            float fl[CW], fh[CW];
            C::unpack(C::load(plo + j), fl);
            C::unpack(C::load(phi + j), fh);
#pragma unroll
            for (int q = 0; q < CW; ++q) lo[j + q] = fl[q], hi[j + q] = fh[q];
        }
    }
}

// clamp(a x, lo, hi) * g in fp32; a NaN product takes the lower bound (fmaxf
// returns its non-NaN operand), as in the separate UClip kernel.
__device__ __forceinline__ float uclip1(float x, float a, float g, float lo, float hi) {
    return fminf(fmaxf(a * x, lo), hi) * g;
}

// One Q or K task: unpack the two accesses (r0, r1) into the pair halves, UClip
// them first if NORM, rotate by (c, s) and store both accesses at dst.
template <typename T, int P, bool IL, bool NORM>
__device__ __forceinline__ void rotate_store(const RopeArgs& a, typename Vec<T, P>::Raw r0,
                                             typename Vec<T, P>::Raw r1, bool is_q, int i0, int h, int o0, int o1,
                                             const float* crow, const float* srow, T* dst) {
    using V = Vec<T, P>;
    constexpr int CW = P >= 4 ? 4 : 1;
    using C = Vec<float, CW>;
    float c[P], s[P];
#pragma unroll
    for (int j = 0; j < P; j += CW) {
        float cf[CW], sf[CW];
        C::unpack(C::load(crow + j), cf);
        C::unpack(C::load(srow + j), sf);
#pragma unroll
        for (int q = 0; q < CW; ++q) {
            c[j + q] = cf[q];
            s[j + q] = sf[q];
        }
    }
    float lo[P], hi[P];
    if constexpr (IL && P >= 2) {
        float f0[P], f1[P];
        V::unpack(r0, f0);
        V::unpack(r1, f1);
#pragma unroll
        for (int j = 0; j < P / 2; ++j) {
            lo[j] = f0[2 * j], hi[j] = f0[2 * j + 1];
            lo[P / 2 + j] = f1[2 * j], hi[P / 2 + j] = f1[2 * j + 1];
        }
    } else {  // neox, or interleaved with one pair: (r0, r1) is (lo, hi)
        V::unpack(r0, lo);
        V::unpack(r1, hi);
    }
    if constexpr (NORM) {
        // parameters from L1: 4P floats per task, the same for every token
        float alo[P], ahi[P], glo[P], ghi[P];
        load_pair_params<P, IL>(is_q ? a.qa : a.ka, i0, h, alo, ahi);
        load_pair_params<P, IL>(is_q ? a.qg : a.kg, i0, h, glo, ghi);
#pragma unroll
        for (int j = 0; j < P; ++j) {
            lo[j] = round_trip<T>(uclip1(lo[j], alo[j], glo[j], a.clip_lo, a.clip_hi));
            hi[j] = round_trip<T>(uclip1(hi[j], ahi[j], ghi[j], a.clip_lo, a.clip_hi));
        }
    }
    float ylo[P], yhi[P];
#pragma unroll
    for (int j = 0; j < P; ++j) {
        ylo[j] = diff_of_products(lo[j], c[j], hi[j], s[j]);
        yhi[j] = diff_of_products(hi[j], c[j], -lo[j], s[j]);
    }
    if constexpr (IL && P >= 2) {
        float f0[P], f1[P];
#pragma unroll
        for (int j = 0; j < P / 2; ++j) {
            f0[2 * j] = ylo[j], f0[2 * j + 1] = yhi[j];
            f1[2 * j] = ylo[P / 2 + j], f1[2 * j + 1] = yhi[P / 2 + j];
        }
        V::store(dst + o0, V::pack(f0));
        V::store(dst + o1, V::pack(f1));
    } else {
        V::store(dst + o0, V::pack(ylo));
        V::store(dst + o1, V::pack(yhi));
    }
}

// P rotation pairs per task, two P-element accesses per task in both styles.
// STYLE 0 (neox): the pairs (i, i + h); the accesses are [i0, i0 + P) and
// [h + i0, h + i0 + P). STYLE 1 (interleaved, GPT-J): the pairs (2i, 2i + 1);
// the accesses are the 2P contiguous elements [2 i0, 2 i0 + 2P), split in two.
//
// NORM: Q and K heads first go through UClip clamp(a x, lo, hi) * g with
// per-channel parameters (mer.dev "AsyncT vllm 适配加速笔记（一）", section 3.3: the
// Q/K norms of the fused QKV output), rounded to T as the separate norm kernel
// would store them, then rotated. A token with a bad position is left as is.
template <typename T, int P, int STYLE, bool NORM>
__global__ void __launch_bounds__(1024) token_cta_kernel(RopeArgs a) {
    constexpr bool IL = STYLE == 1;
    using V = Vec<T, P>;
    using R = typename V::Raw;
    constexpr int CW = P >= 4 ? 4 : 1;  // cos / sin floats per access
    using C = Vec<float, CW>;
    static_assert(P == 1 || P % 2 == 0, "interleaved pairs split evenly over two accesses");
    if (threadIdx.x == 0 && blockIdx.x < a.T) {
        const int64_t t = blockIdx.x, es = static_cast<int64_t>(sizeof(T));
        prefetch_l2(static_cast<const T*>(a.q) + t * a.qs, static_cast<int64_t>(a.n_head) * a.head_dim * es);
        prefetch_l2(static_cast<const T*>(a.k) + t * a.ks, static_cast<int64_t>(a.n_kv) * a.head_dim * es);
        prefetch_l2(static_cast<const T*>(a.v) + t * a.vs, static_cast<int64_t>(a.n_kv) * a.head_dim * es);
    }
    // The CTA's first token's position, read before the dependency wait (relaxed: the previous
    // kernel may still be writing it). It warms that token's cos / sin rows and, after the wait,
    // says which rows to load together with the position's own read; the position read after
    // the wait decides, and a different one (never, unless the previous kernel wrote it) loads
    // its rows again.
    int64_t p_pre = -1;
    if (blockIdx.x < a.T) asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(p_pre) : "l"(a.pos + blockIdx.x));
    if (threadIdx.x == blockDim.x - 1 && p_pre >= 0 && p_pre < a.max_pos) {
        const int64_t half = a.head_dim >> 1;
        prefetch_l2(a.cos + p_pre * half, half * 4);
        prefetch_l2(a.sin + p_pre * half, half * 4);
    }
    pdl_enter();

    const int h = a.head_dim >> 1;
    const int per_head = h / P;
    const int n_units = a.n_head + 2 * a.n_kv;
    const int U = n_units * per_head;
    const int64_t capacity = a.num_blocks * static_cast<int64_t>(a.block_size);

    for (int u = threadIdx.x; u < U; u += blockDim.x) {
        const int unit = u / per_head;
        const int i0 = (u - unit * per_head) * P;
        // 0: Q head, 1: K head, 2: V head
        const int kind = unit < a.n_head ? 0 : (unit < a.n_head + a.n_kv ? 1 : 2);
        const int head = kind == 0 ? unit : (kind == 1 ? unit - a.n_head : unit - a.n_head - a.n_kv);

        for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
            const int64_t p = a.pos[t];
            int64_t slot = -1;
            if (kind != 0 || u == 0) slot = a.slot[t];
            // element offsets of the task's two accesses
            const int o0 = IL ? 2 * i0 : i0;
            const int o1 = IL ? 2 * i0 + P : h + i0;
            // the task's row and (from the early position) its cos / sin, requested with the
            // position and the slot: none of these loads waits for them
            const T* src = kind == 0   ? static_cast<const T*>(a.q) + t * a.qs + static_cast<int64_t>(head) * a.head_dim
                           : kind == 1 ? static_cast<const T*>(a.k) + t * a.ks + static_cast<int64_t>(head) * a.head_dim
                                       : static_cast<const T*>(a.v) + t * a.vs + static_cast<int64_t>(head) * a.head_dim;
            const R r0 = V::load(src + o0);
            const R r1 = V::load(src + o1);
            // (not with the UClip parameters: their registers and these would not fit together)
            const int64_t ps = !NORM && t == blockIdx.x && p_pre >= 0 && p_pre < a.max_pos ? p_pre : -1;
            float c[P], s[P];
            auto load_cs = [&](int64_t pp) {
                const float* crow = a.cos + pp * h + i0;
                const float* srow = a.sin + pp * h + i0;
#pragma unroll
                for (int j = 0; j < P; j += CW) {
                    float cf[CW], sf[CW];
                    C::unpack(C::load(crow + j), cf);
                    C::unpack(C::load(srow + j), sf);
#pragma unroll
                    for (int q = 0; q < CW; ++q) {
                        c[j + q] = cf[q];
                        s[j + q] = sf[q];
                    }
                }
            };
            if (kind != 2 && ps >= 0) load_cs(ps);

            const bool pos_ok = p >= 0 && p < a.max_pos;
            const bool slot_in_range = slot < capacity;
            if (u == 0 && a.err != nullptr) {
                const int bad = (pos_ok ? 0 : 1) + ((slot >= 0 && !slot_in_range) ? 1 : 0);
                if (bad) atomicAdd(a.err, bad);
            }
            if (!pos_ok) continue;                       // q[t] unchanged, nothing cached
            if (kind != 0 && (slot < 0 || !slot_in_range)) continue;  // padding / bad slot

            T* dst;
            if (kind == 0) {
                dst = static_cast<T*>(a.q) + t * a.qs + static_cast<int64_t>(head) * a.head_dim;
            } else {
                const int64_t blk = slot / a.block_size;
                const int64_t off = slot - blk * a.block_size;
                const int plane = kind == 1 ? 0 : 1;
                dst = static_cast<T*>(a.cache) +
                      (((plane * a.num_blocks + blk) * a.block_size + off) * a.n_kv + head) *
                          static_cast<int64_t>(a.head_dim);
            }
            if (kind == 2) {  // V: bit copy
                V::store(dst + o0, r0);
                V::store(dst + o1, r1);
                continue;
            }
            if (!NORM && p != ps) load_cs(p);
            float lo[P], hi[P];
            if constexpr (IL && P >= 2) {
                float f0[P], f1[P];
                V::unpack(r0, f0);
                V::unpack(r1, f1);
#pragma unroll
                for (int j = 0; j < P / 2; ++j) {
                    lo[j] = f0[2 * j], hi[j] = f0[2 * j + 1];
                    lo[P / 2 + j] = f1[2 * j], hi[P / 2 + j] = f1[2 * j + 1];
                }
            } else {  // neox, or interleaved with one pair: (r0, r1) is (lo, hi)
                V::unpack(r0, lo);
                V::unpack(r1, hi);
            }
            if constexpr (NORM) {
                // parameters from L1: 4P floats per task, the same for every token
                float alo[P], ahi[P], glo[P], ghi[P];
                load_pair_params<P, IL>(kind == 0 ? a.qa : a.ka, i0, h, alo, ahi);
                load_pair_params<P, IL>(kind == 0 ? a.qg : a.kg, i0, h, glo, ghi);
#pragma unroll
                for (int j = 0; j < P; ++j) {
                    lo[j] = round_trip<T>(uclip1(lo[j], alo[j], glo[j], a.clip_lo, a.clip_hi));
                    hi[j] = round_trip<T>(uclip1(hi[j], ahi[j], ghi[j], a.clip_lo, a.clip_hi));
                }
                load_cs(p);
            }
            float ylo[P], yhi[P];
#pragma unroll
            for (int j = 0; j < P; ++j) {
                ylo[j] = diff_of_products(lo[j], c[j], hi[j], s[j]);
                yhi[j] = diff_of_products(hi[j], c[j], -lo[j], s[j]);
            }
            if constexpr (IL && P >= 2) {
                float f0[P], f1[P];
#pragma unroll
                for (int j = 0; j < P / 2; ++j) {
                    f0[2 * j] = ylo[j], f0[2 * j + 1] = yhi[j];
                    f1[2 * j] = ylo[P / 2 + j], f1[2 * j + 1] = yhi[P / 2 + j];
                }
                V::store(dst + o0, V::pack(f0));
                V::store(dst + o1, V::pack(f1));
            } else {
                V::store(dst + o0, V::pack(ylo));
                V::store(dst + o1, V::pack(yhi));
            }
        }
    }
}

// Two tasks per thread: thread u0 of a token owns the tasks u0 and u0 + U / 2
// (U tasks per token). U / 2 is a whole number of heads' tasks (the planner
// checks that n_head + 2 n_kv_head is even), so both tasks have the same pair
// offset i0 and read the same cos / sin chunk (the second read hits L1). Both
// tasks' row loads are issued before the first rotation. A token then takes
// U / 2 threads at no more than 64 registers each (the one-task kernel: U
// threads at 52), so about twice as many tokens are resident per SM
// (Qwen2.5-1.5B bf16: 64 threads per token; T = 2048 in one wave on 152 SMs,
// where the one-task kernel needs two rounds). Results are those of
// token_cta_kernel: the same arithmetic per element.
template <typename T, int P, int STYLE, bool NORM>
__global__ void __launch_bounds__(512, 2) token_cta2_kernel(RopeArgs a) {
    constexpr bool IL = STYLE == 1;
    using V = Vec<T, P>;
    using R = typename V::Raw;
    constexpr int CW = P >= 4 ? 4 : 1;  // cos / sin floats per access
    using C = Vec<float, CW>;
    static_assert(P == 1 || P % 2 == 0, "interleaved pairs split evenly over two accesses");
    if (threadIdx.x == 0 && blockIdx.x < a.T) {
        const int64_t t = blockIdx.x, es = static_cast<int64_t>(sizeof(T));
        prefetch_l2(static_cast<const T*>(a.q) + t * a.qs, static_cast<int64_t>(a.n_head) * a.head_dim * es);
        prefetch_l2(static_cast<const T*>(a.k) + t * a.ks, static_cast<int64_t>(a.n_kv) * a.head_dim * es);
        prefetch_l2(static_cast<const T*>(a.v) + t * a.vs, static_cast<int64_t>(a.n_kv) * a.head_dim * es);
    }
    if (threadIdx.x == blockDim.x - 1 && blockIdx.x < a.T) {
        // first token's cos / sin rows, steered by a relaxed read of its position (a hint only)
        int64_t p;
        asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(p) : "l"(a.pos + blockIdx.x));
        if (p >= 0 && p < a.max_pos) {
            const int64_t half = a.head_dim >> 1;
            prefetch_l2(a.cos + p * half, half * 4);
            prefetch_l2(a.sin + p * half, half * 4);
        }
    }
    pdl_enter();

    const int h = a.head_dim >> 1;
    const int per_head = h / P;
    const int n_units = a.n_head + 2 * a.n_kv;
    const int Uh = (n_units >> 1) * per_head;  // half of a token's tasks
    const int64_t capacity = a.num_blocks * static_cast<int64_t>(a.block_size);

    for (int u0 = threadIdx.x; u0 < Uh; u0 += blockDim.x) {
        const int i0 = (u0 % per_head) * P;
        // task k (k = 0, 1) is head unit unit0 + k * n_units / 2; 0: Q head, 1: K head, 2: V head
        int kind[2], head[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int unit = u0 / per_head + k * (n_units >> 1);
            kind[k] = unit < a.n_head ? 0 : (unit < a.n_head + a.n_kv ? 1 : 2);
            head[k] = kind[k] == 0 ? unit : (kind[k] == 1 ? unit - a.n_head : unit - a.n_head - a.n_kv);
        }
        const bool need_slot = u0 == 0 || kind[0] != 0 || kind[1] != 0;
        const int o0 = IL ? 2 * i0 : i0;
        const int o1 = IL ? 2 * i0 + P : h + i0;

        for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
            const int64_t p = a.pos[t];
            const bool pos_ok = p >= 0 && p < a.max_pos;
            int64_t slot = -1;
            if (need_slot) slot = a.slot[t];
            const bool slot_in_range = slot < capacity;

            if (u0 == 0 && a.err != nullptr) {
                const int bad = (pos_ok ? 0 : 1) + ((slot >= 0 && !slot_in_range) ? 1 : 0);
                if (bad) atomicAdd(a.err, bad);
            }
            if (!pos_ok) continue;                                  // q[t] unchanged, nothing cached
            const bool slot_ok = slot >= 0 && slot_in_range;       // else padding / bad slot: K, V skipped

            // a task's row: its Q head in place, or its slot's row of the K / V plane
            auto row_of = [&](int k) -> T* {
                if (kind[k] == 0)
                    return static_cast<T*>(a.q) + t * a.qs + static_cast<int64_t>(head[k]) * a.head_dim;
                const int64_t blk = slot / a.block_size;
                const int64_t off = slot - blk * a.block_size;
                const int plane = kind[k] == 1 ? 0 : 1;
                return static_cast<T*>(a.cache) +
                       (((plane * a.num_blocks + blk) * a.block_size + off) * a.n_kv + head[k]) *
                           static_cast<int64_t>(a.head_dim);
            };
            R r0[2], r1[2];
            bool live[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                live[k] = kind[k] == 0 || slot_ok;
                if (live[k]) {
                    const int64_t hoff = static_cast<int64_t>(head[k]) * a.head_dim;
                    const T* src = kind[k] == 0   ? row_of(k)
                                   : kind[k] == 1 ? static_cast<const T*>(a.k) + t * a.ks + hoff
                                                  : static_cast<const T*>(a.v) + t * a.vs + hoff;
                    r0[k] = V::load(src + o0);
                    r1[k] = V::load(src + o1);
                }
            }
            const float* crow = a.cos + p * h + i0;
            const float* srow = a.sin + p * h + i0;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if (!live[k]) continue;
                T* dst = row_of(k);
                if (kind[k] == 2) {  // V: bit copy
                    V::store(dst + o0, r0[k]);
                    V::store(dst + o1, r1[k]);
                } else {
                    rotate_store<T, P, IL, NORM>(a, r0[k], r1[k], kind[k] == 0, i0, h, o0, o1, crow, srow, dst);
                }
            }
        }
    }
}

template <typename T, bool NORM>
void (*pick(const RopePlan& p))(RopeArgs) {
    constexpr int V = vec16<T>();
    const bool two = p.variant == ROPE_TOKEN_CTA2;
    if (p.style == 0) {
        if (p.pairs == 1) return two ? token_cta2_kernel<T, 1, 0, NORM> : token_cta_kernel<T, 1, 0, NORM>;
        if (p.pairs == V) return two ? token_cta2_kernel<T, V, 0, NORM> : token_cta_kernel<T, V, 0, NORM>;
    } else {
        if (p.pairs == 1) return two ? token_cta2_kernel<T, 1, 1, NORM> : token_cta_kernel<T, 1, 1, NORM>;
        if (p.pairs == V) return two ? token_cta2_kernel<T, V, 1, NORM> : token_cta_kernel<T, V, 1, NORM>;
    }
    return nullptr;
}

template <typename T>
cudaError_t launch_typed(const RopeArgs& a, const RopePlan& p, cudaStream_t s) {
    const dim3 block(p.threads);
    void (*kernel)(RopeArgs) = nullptr;
    if (p.qk_norm) {
        kernel = pick<T, true>(p);
    } else {
        kernel = pick<T, false>(p);
    }
    if (!kernel) return cudaErrorInvalidValue;
    const dim3 grid(persistent_grid(kernel, p.threads, 0, p.num_sms, p.grid));
    return launch_kernel(kernel, grid, block, 0, s, p.pdl, 1, a);
}

}  // namespace rope

cudaError_t launch_rope_kv_store(const RopeArgs& a, const RopePlan& p, int dtype, cudaStream_t s) {
    if (p.variant != ROPE_TOKEN_CTA && p.variant != ROPE_TOKEN_CTA2) return cudaErrorInvalidValue;
    switch (dtype) {
        case DT_F32: return rope::launch_typed<float>(a, p, s);
        case DT_F16: return rope::launch_typed<__half>(a, p, s);
        case DT_BF16: return rope::launch_typed<__nv_bfloat16>(a, p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sra
