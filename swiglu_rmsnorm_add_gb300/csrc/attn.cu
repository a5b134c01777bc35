// Decode attention over the paged KV cache: the read side of rope_kv_store.
//
// For request b and query head h (kv head h / G, G = n_head / n_kv_head):
//   o = sum_t softmax_t(scale * q . K_t) V_t over the request's seq_lens[b]
// tokens, token t stored in cache block block_table[b, t / block_size] at
// offset t % block_size. mer.dev "AsyncT vllm 适配加速笔记（一）": section 1.1 (the
// FA cache layout [2, num_blocks, block_size, n_kv, head] with a block table
// and seq lens per request), section 2.2 (the K/V load is the bandwidth; the
// query heads that share a KV head should share its load), section 3.1 (a
// decode kernel reading that layout through the block table). m.lsln.cn
// 21-operator article, sections 2.1 and 5.3 (qk_score, scale + softmax and
// pv_agg fused over cache_kv_read) and section 3.2 (split the reduction and
// merge the parts through their (max, sum of exponentials)).
//
// Work: a CTA owns one (request, kv head, split). All G query heads of the kv
// head are computed together, so every K/V byte is read from HBM once. The
// request's cache blocks are dealt to the splits in contiguous ranges; a split
// streams its blocks through a STAGES-deep ring of shared-memory tiles filled
// by cp.async (16-byte copies, one tile = one cache block: block_size rows of K
// and of V). Per tile: every (head, token) pair gets one thread for its score
// (a head_dim-long dot product, with each token's start rotated across the row
// so the threads of one head hit different banks), an online-softmax update
// per head (running max m, running sum l, correction exp2(m_old - m_new)), and
// then the threads that own (head, 4-dim) output slices accumulate p * V.
// The splits of one (request, kv head) are the CTAs of one thread-block
// cluster: at the end each CTA leaves (m, l, acc) in its shared memory and the
// cluster merges them through distributed shared memory (no global scratch,
// no second kernel). Scores are kept in base 2: q is pre-scaled by
// scale * log2(e) and exponentials are exp2.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace sra {
namespace attn {

constexpr int kThreads = 128;

__host__ __device__ constexpr size_t r16(size_t b) { return (b + 15) / 16 * 16; }

// Shared-memory layout (byte offsets), the same on host and device.
struct Layout {
    size_t qs, kv, p, stat, pacc, total;
};
__host__ __device__ inline Layout layout(int G, int HD, int BS, int stages, int es) {
    Layout L{};
    size_t off = 0;
    L.qs = off;
    off += r16(static_cast<size_t>(G) * (HD + 4) * 4);  // q rows, fp32, padded by 4
    L.kv = off;
    off += r16(static_cast<size_t>(stages) * 2 * BS * HD * es);  // K and V tiles
    L.p = off;
    off += r16(static_cast<size_t>(G) * BS * 4);  // probabilities of the current tile
    L.stat = off;
    off += r16(static_cast<size_t>(3) * G * 4);  // running max, running sum, correction
    L.pacc = off;
    off += r16(static_cast<size_t>(G) * HD * 4);  // this CTA's partial output, for the merge
    L.total = off;
    return L;
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename T>
__device__ __forceinline__ T from_f32(float v) {
    if constexpr (sizeof(T) == 4) {
        return v;
    } else {
        const unsigned short b = Elem<T>::to_bits16(v);
        T r;
        memcpy(&r, &b, 2);
        return r;
    }
}

template <typename T, int HD, int STAGES>
__global__ void __launch_bounds__(kThreads) decode_kernel(AttnArgs a) {
    constexpr int IPT = HD / 64;                                  // (head, 4-dim) slices per thread, G <= 8
    constexpr int EPC = 16 / static_cast<int>(sizeof(T));         // elements per 16-byte copy
    constexpr int CPR = HD / EPC;                                 // copies per row
    extern __shared__ __align__(16) unsigned char smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int S = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int64_t grp = blockIdx.x / S;
    const int64_t b = grp / a.n_kv;
    const int kvh = static_cast<int>(grp - b * a.n_kv);
    const int G = a.group, BS = a.block_size;
    const Layout L = layout(G, HD, BS, STAGES, sizeof(T));
    float* qs = reinterpret_cast<float*>(smem + L.qs);
    T* kv = reinterpret_cast<T*>(smem + L.kv);
    float* ps = reinterpret_cast<float*>(smem + L.p);
    float* m_run = reinterpret_cast<float*>(smem + L.stat);
    float* l_run = m_run + G;
    float* corr = l_run + G;
    float* pacc = reinterpret_cast<float*>(smem + L.pacc);

    pdl_enter();
    int64_t len = a.seq_lens[b];
    const int64_t cap = a.max_blocks * BS;
    if ((len < 0 || len > cap) && kvh == 0 && rank == 0 && threadIdx.x == 0 && a.err) atomicAdd(a.err, 1);
    len = len < 0 ? 0 : (len > cap ? cap : len);
    const int64_t nblk = (len + BS - 1) / BS;
    const int64_t per = (nblk + S - 1) / S;
    const int64_t j0 = rank * per < nblk ? rank * per : nblk;
    const int64_t j1 = j0 + per < nblk ? j0 + per : nblk;

    for (int i = threadIdx.x; i < G * HD; i += kThreads) {
        const int g = i / HD, d = i - g * HD;
        const T* qp = static_cast<const T*>(a.q) + b * a.qs + static_cast<int64_t>(kvh * G + g) * HD + d;
        qs[g * (HD + 4) + d] = to_f32(*qp) * a.scale_log2;
    }
    if (threadIdx.x < G) {
        m_run[threadIdx.x] = -INFINITY;
        l_run[threadIdx.x] = 0.0f;
    }
    const int32_t* table = a.table + b * a.max_blocks;
    const int64_t tok_stride = static_cast<int64_t>(a.n_kv) * HD;          // elements between tokens
    const int64_t v_plane = a.num_blocks * BS * tok_stride;
    auto block_ok = [&](int32_t blk) { return blk >= 0 && blk < a.num_blocks; };
    auto issue = [&](int64_t j) {
        const int32_t blk = table[j];
        if (!block_ok(blk)) return;  // its tokens are skipped, the tile is never read
        T* dst = kv + static_cast<size_t>((j - j0) % STAGES) * 2 * BS * HD;
        const T* kb = static_cast<const T*>(a.cache) + (static_cast<int64_t>(blk) * BS * a.n_kv + kvh) * HD;
        for (int c = threadIdx.x; c < 2 * BS * CPR; c += kThreads) {
            const int plane = c / (BS * CPR);
            const int r = c - plane * BS * CPR;
            const int t = r / CPR, col = r - t * CPR;
            cp_async16(dst + plane * BS * HD + t * HD + col * EPC,
                       kb + (plane ? v_plane : 0) + t * tok_stride + col * EPC);
        }
    };
    for (int s = 0; s < STAGES - 1; ++s) {
        if (j0 + s < j1) issue(j0 + s);
        cp_async_commit();
    }

    float acc[IPT][4];
#pragma unroll
    for (int k = 0; k < IPT; ++k) acc[k][0] = acc[k][1] = acc[k][2] = acc[k][3] = 0.0f;
    const unsigned FULL = 0xffffffffu;

    for (int64_t j = j0; j < j1; ++j) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();  // tile j landed for every thread's copies; previous tile fully consumed
        if (j + STAGES - 1 < j1) issue(j + STAGES - 1);
        cp_async_commit();
        const int32_t blk = table[j];
        const bool ok = block_ok(blk);
        if (!ok && kvh == 0 && threadIdx.x == 0 && a.err) atomicAdd(a.err, 1);
        const int64_t left = len - j * BS;
        const int nvalid = ok ? static_cast<int>(left < BS ? left : BS) : 0;
        const T* Ks = kv + static_cast<size_t>((j - j0) % STAGES) * 2 * BS * HD;
        const T* Vs = Ks + BS * HD;

        // scores and the online-softmax update; item i = g * BS + t, BS-lane segments per head
        for (int i0 = 0; i0 < G * BS; i0 += kThreads) {
            const int i = i0 + threadIdx.x;
            const bool item = i < G * BS;
            const int g = item ? i / BS : 0, t = i - (i / BS) * BS;
            const bool valid = item && t < nvalid;
            const float m_old = item ? m_run[g] : -INFINITY;
            float sc = -INFINITY;
            if (valid) {
                const float* qg = qs + g * (HD + 4);
                const T* kt = Ks + t * HD;
                float d0 = 0.0f, d1 = 0.0f;
#pragma unroll 8
                for (int k = 0; k < HD; k += 4) {
                    const int d = (k + 4 * t) & (HD - 1);  // rotated start: bank spread over the tokens
                    float kf[4];
                    Vec<T, 4>::unpack(Vec<T, 4>::load(kt + d), kf);
                    const float4 qv = *reinterpret_cast<const float4*>(qg + d);
                    d0 = fmaf(qv.x, kf[0], d0);
                    d1 = fmaf(qv.y, kf[1], d1);
                    d0 = fmaf(qv.z, kf[2], d0);
                    d1 = fmaf(qv.w, kf[3], d1);
                }
                sc = d0 + d1;
            }
            float mx = sc;
            for (int o = BS >> 1; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
            const float m_new = fmaxf(m_old, mx);
            const float pr = valid ? exp2f(sc - m_new) : 0.0f;
            float sum = pr;
            for (int o = BS >> 1; o > 0; o >>= 1) sum += __shfl_xor_sync(FULL, sum, o);
            __syncwarp();
            if (item) {
                ps[i] = pr;
                if (t == 0) {
                    const float c = m_new == -INFINITY ? 1.0f : exp2f(m_old - m_new);
                    corr[g] = c;
                    l_run[g] = l_run[g] * c + sum;
                    m_run[g] = m_new;
                }
            }
        }
        __syncthreads();  // probabilities and corrections of this tile ready

#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            const int idx = threadIdx.x + k * kThreads;
            if (idx < G * (HD / 4)) {
                const int g = idx / (HD / 4), d = (idx - g * (HD / 4)) * 4;
                const float c = corr[g];
                float x0 = acc[k][0] * c, x1 = acc[k][1] * c, x2 = acc[k][2] * c, x3 = acc[k][3] * c;
                const float* pg = ps + g * BS;
                for (int t = 0; t < nvalid; ++t) {
                    const float pt = pg[t];
                    float vf[4];
                    Vec<T, 4>::unpack(Vec<T, 4>::load(Vs + t * HD + d), vf);
                    x0 = fmaf(pt, vf[0], x0);
                    x1 = fmaf(pt, vf[1], x1);
                    x2 = fmaf(pt, vf[2], x2);
                    x3 = fmaf(pt, vf[3], x3);
                }
                acc[k][0] = x0, acc[k][1] = x1, acc[k][2] = x2, acc[k][3] = x3;
            }
        }
    }
    cp_async_wait<0>();

    // this split's (m, l, acc) into shared memory, then merge across the cluster
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
        const int idx = threadIdx.x + k * kThreads;
        if (idx < G * (HD / 4)) {
            const int g = idx / (HD / 4), d = (idx - g * (HD / 4)) * 4;
            float* pa = pacc + g * HD + d;
            pa[0] = acc[k][0], pa[1] = acc[k][1], pa[2] = acc[k][2], pa[3] = acc[k][3];
        }
    }
    cluster.sync();
    T* out = static_cast<T*>(a.out) + b * a.os + static_cast<int64_t>(kvh * G) * HD;
    for (int idx = rank * kThreads + threadIdx.x; idx < G * HD; idx += S * kThreads) {
        const int g = idx / HD;
        float M = -INFINITY;
        for (int r = 0; r < S; ++r) M = fmaxf(M, cluster.map_shared_rank(m_run, r)[g]);
        float num = 0.0f, den = 0.0f;
        if (M != -INFINITY) {
            for (int r = 0; r < S; ++r) {
                const float mr = cluster.map_shared_rank(m_run, r)[g];
                if (mr == -INFINITY) continue;
                const float w = exp2f(mr - M);
                num = fmaf(w, cluster.map_shared_rank(pacc, r)[idx], num);
                den = fmaf(w, cluster.map_shared_rank(l_run, r)[g], den);
            }
        }
        out[idx] = from_f32<T>(den > 0.0f ? num / den : 0.0f);
    }
    cluster.sync();  // keep every CTA's shared memory alive until the merge has read it
}

template <typename T, int HD, int STAGES>
cudaError_t launch_hd(const AttnArgs& a, const AttnPlan& p, cudaStream_t s) {
    auto kernel = decode_kernel<T, HD, STAGES>;
    const size_t smem = layout(a.group, HD, a.block_size, STAGES, sizeof(T)).total;
    if (smem > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    const dim3 grid(static_cast<unsigned>(a.B * a.n_kv * p.splits)), block(kThreads);
    return launch_kernel(kernel, grid, block, smem, s, p.pdl, p.splits, a);
}

template <typename T, int STAGES>
cudaError_t launch_stages(const AttnArgs& a, const AttnPlan& p, cudaStream_t s) {
    switch (p.head_dim) {
        case 64: return launch_hd<T, 64, STAGES>(a, p, s);
        case 128: return launch_hd<T, 128, STAGES>(a, p, s);
        case 256: return launch_hd<T, 256, STAGES>(a, p, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t launch_typed(const AttnArgs& a, const AttnPlan& p, cudaStream_t s) {
    return p.stages >= 4 ? launch_stages<T, 4>(a, p, s) : launch_stages<T, 2>(a, p, s);
}

}  // namespace attn

size_t decode_attention_smem(int group, int head_dim, int block_size, int stages, int es) {
    return attn::layout(group, head_dim, block_size, stages, es).total;
}

cudaError_t launch_decode_attention(const AttnArgs& a, const AttnPlan& p, int dtype, cudaStream_t s) {
    switch (dtype) {
        case DT_F32: return attn::launch_typed<float>(a, p, s);
        case DT_F16: return attn::launch_typed<__half>(a, p, s);
        case DT_BF16: return attn::launch_typed<__nv_bfloat16>(a, p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sra
