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
// Two kernels. bf16 / fp16 with head_dim 64 or 128 run on the tensor cores
// (decode_mma_kernel below: warp-level mma.sync, each warp streaming its own
// 16-token tiles); fp32 and head_dim 256 run on the CUDA cores (decode_kernel,
// described next). Both share the split / cluster-merge structure.
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
#include "tma.cuh"

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

// ------------------------------------------------------------------------------------------
// Tensor-core path (bf16 / fp16, head_dim 64 or 128): warp-level mma.sync m16n8k16.
//
// The contraction per 16-token tile is S[16 x 16] = Q[16 x HD] K^T and
// O[16 x HD] += P[16 x 16] V with the G <= 8 query heads of the kv head as the
// rows 0..7 of the 16-row operands (rows 8..15 are zero). Each warp owns its
// own 16-token tiles and its own cp.async ring (K and V tiles of 16 rows,
// 16-byte chunks XOR-swizzled by row so ldmatrix reads are conflict-free;
// rows of tokens past the end or in a bad block are zero-filled and masked).
// Q stays in registers as A fragments for the whole kernel; K tiles feed the
// B operand directly (ldmatrix), V tiles through ldmatrix.trans. The
// probabilities are split into a T-rounded high part and a T-rounded residual,
// two MMAs per V fragment, so p keeps about 16 significant bits instead of the
// 8 (bf16) a single rounding would leave. Warps merge their (m, l, O) in
// shared memory, then the CTAs of the cluster as in the fp32 path.
// 2^x by the ex2.approx instruction (PTX ISA: about 2^-22 relative error); 2^-inf = 0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// mma.sync m16n8k16 with rows 8-15 of A zero (at most 8 query heads share a kv head): only
// the C / D fragment registers of rows 0-7 (c0, c1) are kept.
template <typename T>
struct Mma;
template <>
struct Mma<__nv_bfloat16> {
    __device__ __forceinline__ static void run(float (&d)[2], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
        // rows 8-15 of A are zero: their results go to registers local to the asm block
        asm volatile(
            "{\n\t.reg .f32 z0, z1;\n\t"
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,z0,z1}, {%2,%3,%4,%5}, {%6,%7}, "
            "{%0,%1,%8,%9};\n\t}"
            : "+f"(d[0]), "+f"(d[1])
            : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(0.0f), "f"(0.0f));
    }
};
template <>
struct Mma<__half> {
    __device__ __forceinline__ static void run(float (&d)[2], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
        // rows 8-15 of A are zero: their results go to registers local to the asm block
        asm volatile(
            "{\n\t.reg .f32 z0, z1;\n\t"
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,z0,z1}, {%2,%3,%4,%5}, {%6,%7}, "
            "{%0,%1,%8,%9};\n\t}"
            : "+f"(d[0]), "+f"(d[1])
            : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(0.0f), "f"(0.0f));
    }
};

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(s));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], const void* p) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(s));
}
// 16-byte copy; src_bytes = 0 fills the destination with zeros and reads nothing.
__device__ __forceinline__ void cp_async16_zfill(void* smem_dst, const void* gmem_src, int src_bytes) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem_src), "r"(src_bytes) : "memory");
}

// Two values rounded to T, packed (first value in the low half).
template <typename T>
__device__ __forceinline__ uint32_t pack2(float x, float y) {
    float f[2] = {x, y};
    return Elem<T>::pack_word(f);
}
template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
    float f[2];
    Elem<T>::unpack_word(w, f);
    return make_float2(f[0], f[1]);
}

// One 16-token tile of a warp: S = Q K^T (two 8-token halves), the online-softmax update of
// (m, l) on the rows this lane holds, and O = O * corr + P V with P split into a T-rounded high
// part and its residual. `addr(tok, chunk)` is the element offset of 16-byte chunk `chunk` of
// token `tok`'s row in the K (and V) tile, whatever layout the tile was staged in; `valid` has
// bit t set for the tile's tokens that count.
template <typename T, int HD, typename Addr>
__device__ __forceinline__ void tile_step(const T* Ks, const T* Vs, unsigned valid, const uint32_t (&qa)[HD / 16][2],
                                          float (&o)[HD / 8][2], float& m, float& l, float scale_log2, int lane,
                                          Addr addr) {
    constexpr int KS = HD / 16;
    constexpr int NB = HD / 8;
    const unsigned FULL = 0xffffffffu;
    const int ft = lane & 3;
    // S = Q K^T: two 8-token blocks
    float sc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    {
        const int mi = lane >> 3, rr = lane & 7;
        const int tok = 8 * (mi >> 1) + rr;
#pragma unroll
        for (int s = 0; s < KS; ++s) {
            uint32_t kb[4];
            const int chunk = 2 * s + (mi & 1);
            ldsm_x4(kb, Ks + addr(tok, chunk));
            Mma<T>::run(sc[0], qa[s][0], qa[s][1], kb[0], kb[1]);
            Mma<T>::run(sc[1], qa[s][0], qa[s][1], kb[2], kb[3]);
        }
    }
    // online softmax on row fg (this thread's tokens: 8 nb + 2 ft + e)
    float v[2][2];
    float mx = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            v[nb][e] = (valid >> (8 * nb + 2 * ft + e)) & 1u ? sc[nb][e] * scale_log2 : -INFINITY;
            mx = fmaxf(mx, v[nb][e]);
        }
    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 2));
    const float m_new = fmaxf(m, mx);
    const float corr = m_new == -INFINITY ? 1.0f : ex2(m - m_new);
    float p[2][2];
    float ps = 0.0f;
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            p[nb][e] = v[nb][e] == -INFINITY ? 0.0f : ex2(v[nb][e] - m_new);
            ps += p[nb][e];
        }
    l = l * corr + ps;
    m = m_new;
    // P as A fragments, high part and residual
    uint32_t ph0 = pack2<T>(p[0][0], p[0][1]), ph1 = pack2<T>(p[1][0], p[1][1]);
    const float2 h0 = unpack2<T>(ph0), h1 = unpack2<T>(ph1);
    uint32_t pl0 = pack2<T>(p[0][0] - h0.x, p[0][1] - h0.y), pl1 = pack2<T>(p[1][0] - h1.x, p[1][1] - h1.y);
    // O = O * corr + P V (the rescale only when some row's max moved)
    if (__any_sync(FULL, corr != 1.0f)) {
#pragma unroll
        for (int d = 0; d < NB; ++d) o[d][0] *= corr, o[d][1] *= corr;
    }
    {
        const int mi = lane >> 3, rr = lane & 7;
        const int tok = 8 * (mi & 1) + rr;
#pragma unroll
        for (int d2 = 0; d2 < NB / 2; ++d2) {
            uint32_t vb[4];
            const int chunk = 2 * d2 + (mi >> 1);
            ldsm_x4_trans(vb, Vs + addr(tok, chunk));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                Mma<T>::run(o[2 * d2 + h], ph0, ph1, vb[2 * h], vb[2 * h + 1]);
                Mma<T>::run(o[2 * d2 + h], pl0, pl1, vb[2 * h], vb[2 * h + 1]);
            }
        }
    }
}

constexpr int kMmaTile = 16;    // tokens per warp tile
constexpr int kMmaStages = 3;   // tiles per warp ring

// The cluster merge's inbox (outside the rings, so other CTAs of the cluster may write it while
// this CTA still streams): every split's maxima and sums [16][8] each, then its partial output
// columns for the slice of columns this CTA owns, [splits][slice] (slices of HD * 8 / splits
// columns rounded up to 4: at most 8 * HD + 64 floats in all).
__host__ __device__ constexpr size_t inbox_floats(int HD) { return 16 * 8 * 2 + 8 * static_cast<size_t>(HD) + 64; }

// Shared memory of an NW-warp CTA: the warps' rings, over which the merges later run (the
// warps' partials; with a workspace split, the last CTA's merge buffers), then the row masks.
__host__ __device__ inline size_t mma_ring_bytes(int HD, int NW) {
    const size_t ring = static_cast<size_t>(NW) * kMmaStages * 2 * kMmaTile * HD * 2;
    const size_t merge = (static_cast<size_t>(NW) * 8 * (HD + 11) + 8 * (HD + 2) + 17 * 8) * 4;
    const size_t gmerge = static_cast<size_t>(kMaxGsplits) * 24 * 4 + 64 + 16 * 8 * static_cast<size_t>(HD) * 4;
    size_t need = ring > merge ? ring : merge;
    return need > gmerge ? need : gmerge;
}
__host__ __device__ inline size_t mma_inbox_offset(int HD, int NW) {  // after the per-slot row masks
    return (mma_ring_bytes(HD, NW) + static_cast<size_t>(NW) * kMmaStages * 4 + 15) / 16 * 16;
}
__host__ __device__ inline size_t mma_smem(int HD, int NW) { return mma_inbox_offset(HD, NW) + inbox_floats(HD) * 4; }

// The end of a (request, kv head, split) CTA of the tensor-core kernels: the warps' (m, l, O)
// merged in shared memory (over the drained rings), then the splits merged through distributed
// shared memory (a cluster) or, with GMERGE, through the workspace by the CTA that finishes
// last. NW warps hold partials; warps past them (a copy-issuing warp) only join the barriers.
template <typename T, int HD, bool GMERGE, int NW>
__device__ __forceinline__ void finish_mma(const AttnArgs& a, unsigned char* smem, float* inbox, float m, float l,
                                           float (&o)[HD / 8][2], int lane, int warp, int64_t grp, int64_t b,
                                           int kvh, int S, int rank, int G, cg::cluster_group& cluster) {
    constexpr int NB = HD / 8;
    const unsigned FULL = 0xffffffffu;
    const int fg = lane >> 2, ft = lane & 3;
    l += __shfl_xor_sync(FULL, l, 1);
    l += __shfl_xor_sync(FULL, l, 2);

    // warp partials into shared memory (over the rings, which are done). A row of O is HD + 8
    // floats apart and each lane stores its pair as one 8-byte store, so the 16 lanes of a
    // half-warp hit 16 different bank pairs (rows HD apart would put the 8 rows of a fragment
    // in the same banks and serialise the stores 8-fold).
    constexpr int WS = HD + 8;
    __syncthreads();
    float* wm = reinterpret_cast<float*>(smem);  // [warps][8]
    float* wl = wm + NW * 8;                     // [warps][8]
    float* wo = wl + NW * 8;                     // [warps][8][WS]
    float* pm = wo + NW * 8 * WS;                // [8]  CTA partials for the cluster merge
    float* pl = pm + 8;                          // [8]
    float* pacc = pl + 8;                        // [8][HD]
    if (warp < NW) {
        if (ft == 0) {
            wm[warp * 8 + fg] = m;
            wl[warp * 8 + fg] = l;
        }
#pragma unroll
        for (int d = 0; d < NB; ++d)
            *reinterpret_cast<float2*>(wo + (warp * 8 + fg) * WS + 8 * d + 2 * ft) = make_float2(o[d][0], o[d][1]);
    }
    __syncthreads();
    // the warps' merge weights 2^(m_w - M) and the denominator, once per query head (they do
    // not depend on the output column); warps that saw no token weigh 0 and hold O = 0
    float* sw = pacc + 8 * HD;  // [warps][8]
    if (threadIdx.x < G) {
        const int gg = threadIdx.x;
        float M = -INFINITY;
        for (int w = 0; w < NW; ++w) M = fmaxf(M, wm[w * 8 + gg]);
        float den = 0.0f;
        for (int w = 0; w < NW; ++w) {
            const float mw = wm[w * 8 + gg];
            const float e = (M == -INFINITY || mw == -INFINITY) ? 0.0f : exp2f(mw - M);
            sw[w * 8 + gg] = e;
            den = fmaf(e, wl[w * 8 + gg], den);
        }
        pm[gg] = M;
        pl[gg] = den;
        if (!GMERGE && S > 1) {
            // this split's maxima and sums into every CTA's inbox
            for (int q = 0; q < S; ++q) {
                float* ib = cluster.map_shared_rank(inbox, q);
                ib[rank * 8 + gg] = M;
                ib[128 + rank * 8 + gg] = den;
            }
        }
    }
    __syncthreads();
    T* out = static_cast<T*>(a.out) + b * a.os + static_cast<int64_t>(kvh * G) * HD;
    const bool alone = !GMERGE && S == 1;  // one CTA holds the whole (request, kv head)
    // cluster merge: CTA q owns output columns [q * C, (q + 1) * C) and receives every split's
    // partials for them in its inbox (stores into other CTAs' shared memory, no round trip)
    const int C = (G * HD + 4 * S - 1) / (4 * S) * 4;
    for (int idx = threadIdx.x; idx < G * HD; idx += blockDim.x) {
        const int gg = idx / HD, d = idx - gg * HD;
        float num = 0.0f;
        for (int w = 0; w < NW; ++w) num = fmaf(sw[w * 8 + gg], wo[(w * 8 + gg) * WS + d], num);
        if (alone) {
            const float den = pl[gg];
            out[idx] = from_f32<T>(den > 0.0f ? num / den : 0.0f);
        } else if (GMERGE) {
            pacc[idx] = num;
        } else {
            const int q = idx / C;
            cluster.map_shared_rank(inbox, q)[256 + rank * C + (idx - q * C)] = num;
        }
    }
    if (alone) return;
    if constexpr (GMERGE) {
        // this split's partial into the workspace, [8 max][8 sum][8 x HD output]; the merge kernel
        // that follows in the stream (decode_merge_kernel) combines the splits
        float* slot = a.ws_part + (static_cast<int64_t>(grp) * S + rank) * (16 + 8 * HD);
        for (int i = threadIdx.x; i < G * HD; i += blockDim.x) slot[16 + i] = pacc[i];
        if (threadIdx.x < G) slot[threadIdx.x] = pm[threadIdx.x], slot[8 + threadIdx.x] = pl[threadIdx.x];
        return;
    }
    cluster.sync();  // every split's partials are in the owners' inboxes (release / acquire)
    // the splits' merge weights and the denominator, once per query head, from the inbox
    float* cw = sw + NW * 8;    // [S][8]
    float* cden = cw + 16 * 8;  // [8]
    if (threadIdx.x < G) {
        const int gg = threadIdx.x;
        float M = -INFINITY;
        for (int r = 0; r < S; ++r) M = fmaxf(M, inbox[r * 8 + gg]);
        float den = 0.0f;
        for (int r = 0; r < S; ++r) {
            const float mr = inbox[r * 8 + gg];
            const float e = (M == -INFINITY || mr == -INFINITY) ? 0.0f : exp2f(mr - M);
            cw[r * 8 + gg] = e;
            den = fmaf(e, inbox[128 + r * 8 + gg], den);
        }
        cden[gg] = den;
    }
    __syncthreads();
    const int c0 = rank * C, c1 = c0 + C < G * HD ? c0 + C : G * HD;
    for (int idx = c0 + threadIdx.x; idx < c1; idx += blockDim.x) {
        const int gg = idx / HD;
        float num = 0.0f;
        for (int r = 0; r < S; ++r) num = fmaf(cw[r * 8 + gg], inbox[256 + r * C + (idx - c0)], num);
        const float den = cden[gg];
        out[idx] = from_f32<T>(den > 0.0f ? num / den : 0.0f);
    }
}

// GMERGE: the splits of a (request, kv head) are independent CTAs (a.gsplits of them, more
// than a cluster holds): each writes its (max, sum, partial output) to the workspace, and
// decode_merge_kernel, launched after them, combines the records.
// NW warps per CTA: 8 (one CTA per SM) or 4 (two CTAs per SM, so a CTA of the next launch can
// start beside one of this launch).
template <typename T, int HD, bool GMERGE, int NW>
__global__ void __launch_bounds__(NW * 32, NW == 4 ? 2 : 1) decode_mma_kernel(AttnArgs a) {
    constexpr int CPR = HD * 2 / 16;      // 16-byte chunks per row
    constexpr int KS = HD / 16;           // k-steps of Q K^T
    constexpr int NB = HD / 8;            // 8-dim blocks of O
    constexpr int TE = kMmaTile * HD;     // elements of one K or V tile
    extern __shared__ __align__(16) unsigned char smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int S = GMERGE ? a.gsplits : static_cast<int>(cluster.num_blocks());
    const int rank = GMERGE ? static_cast<int>(blockIdx.x % a.gsplits) : static_cast<int>(cluster.block_rank());
    const int64_t grp = blockIdx.x / S;
    const int64_t b = grp / a.n_kv;
    const int kvh = static_cast<int>(grp - b * a.n_kv);
    const int G = a.group, BS = a.block_size;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int fg = lane >> 2, ft = lane & 3;  // fragment row group and thread-in-group
    T* ring = reinterpret_cast<T*>(smem) + static_cast<size_t>(warp) * kMmaStages * 2 * TE;

    {
        // Before the dependency wait: warm what the first tiles need. First the loads that
        // depend on nothing: this request's seq_len and this split's whole slice of the block
        // table (so the later tiles' table reads hit the L2 and each tile costs one DRAM round
        // trip, not two). Then the K and V rows of this warp's first two tiles: the split is a
        // static slice of the table's capacity, so the tiles' tokens are known; their block ids
        // are read relaxed (the previous kernel may still be writing them) and only steer
        // prefetches. Everything used below is read again after the wait.
        const int64_t cap0 = a.max_blocks * BS;
        const int64_t per0 = ((cap0 + S - 1) / S + kMmaTile - 1) / kMmaTile * kMmaTile;
        const int64_t s0 = rank * per0, s1 = cap0 < s0 + per0 ? cap0 : s0 + per0;
        if (warp == 0 && lane == 0) prefetch_lines(a.seq_lens + b, 4, 0, 1);
        if (warp == NW - 1 && s0 < s1)
            prefetch_lines(a.table + b * a.max_blocks + s0 / BS, ((s1 - 1) / BS - s0 / BS + 1) * 4, lane, 32);
        int blk[2] = {-1, -1};
        int64_t tok[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            tok[j] = s0 + (warp + j * NW) * kMmaTile + (lane & (kMmaTile - 1));
            if (tok[j] < s1)
                asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];"
                             : "=r"(blk[j])
                             : "l"(a.table + b * a.max_blocks + tok[j] / BS));
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            if (tok[j] < s1 && blk[j] >= 0 && blk[j] < a.num_blocks) {
                const T* row = static_cast<const T*>(a.cache) +
                               ((static_cast<int64_t>(blk[j]) * BS + tok[j] % BS) * a.n_kv + kvh) * HD +
                               (lane >= kMmaTile ? a.num_blocks * BS * static_cast<int64_t>(a.n_kv) * HD : 0);
                prefetch_lines(row, HD * 2, 0, 1);
            }
        }
    }
    pdl_enter();
    const int64_t cap = a.max_blocks * BS;
    // static split of the table's capacity (not of seq_len), so the block-table reads of the
    // first tiles need not wait for seq_len; tokens at or past seq_len are masked
    const int64_t per = ((cap + S - 1) / S + kMmaTile - 1) / kMmaTile * kMmaTile;
    const int64_t t_begin = rank * per < cap ? rank * per : cap;
    const int64_t t_lim = t_begin + per < cap ? t_begin + per : cap;
    const int32_t* table = a.table + b * a.max_blocks;
    const int bs_log2 = __ffs(BS) - 1;  // block_size is a power of two
    // Block-table entry of token `lane` of tile u (lanes < 16; 0 past the static range). It is
    // read one tile ahead of its use, so the copy issue never waits on the table's latency.
    auto load_blk = [&](int64_t u) -> int32_t {
        const int64_t tok = t_begin + u * kMmaTile + lane;
        return lane < kMmaTile && tok < t_lim ? table[tok >> bs_log2] : 0;
    };
    // the first tiles' block ids and seq_len are requested together: one round trip, not two
    int32_t blk0[kMmaStages];
#pragma unroll
    for (int k = 0; k < kMmaStages; ++k) blk0[k] = load_blk(warp + static_cast<int64_t>(k) * NW);
    int64_t len = a.seq_lens[b];
    if ((len < 0 || len > cap) && kvh == 0 && rank == 0 && threadIdx.x == 0 && a.err) atomicAdd(a.err, 1);
    len = len < 0 ? 0 : (len > cap ? cap : len);
    const int64_t t_end = len < t_begin ? t_begin : (len < t_lim ? len : t_lim);
    auto block_ok = [&](int32_t blk) { return blk >= 0 && blk < a.num_blocks; };
    const int64_t tok_stride = static_cast<int64_t>(a.n_kv) * HD;
    const int64_t v_plane = a.num_blocks * BS * tok_stride;
    const T* cache = static_cast<const T*>(a.cache);
    const int64_t n_tiles = (t_end - t_begin + kMmaTile - 1) / kMmaTile;
    const int64_t n_static = (t_lim - t_begin + kMmaTile - 1) / kMmaTile;
    unsigned* vmask = reinterpret_cast<unsigned*>(smem + mma_ring_bytes(HD, NW)) + warp * kMmaStages;
    const unsigned FULL = 0xffffffffu;
    // This warp's tile u into ring slot (u / warps) % stages: lane r < 16 finds token r's row
    // once; the 16-byte copies then go row by row, LPR lanes per row (contiguous), and each
    // lane's destination offsets in a slot are fixed, computed once. Chunks are XOR-swizzled
    // by row so the 8 rows one ldmatrix reads sit in 8 different bank groups. Rows past
    // seq_len or in a bad block are zero-filled (no read) and masked.
    constexpr int LPR = CPR < 32 ? CPR : 32;  // lanes per row
    constexpr int RPI = 32 / LPR;              // rows per instruction
    const int col = lane % LPR, rr0 = lane / LPR;
    const int64_t kvh_off = static_cast<int64_t>(kvh) * HD;
    int dst_off[kMmaTile / RPI][CPR / LPR];
#pragma unroll
    for (int i = 0; i < kMmaTile / RPI; ++i)
#pragma unroll
        for (int cc = 0; cc < CPR / LPR; ++cc) {
            const int r = rr0 + RPI * i, ch = col + cc * LPR;
            dst_off[i][cc] = r * HD + ((ch ^ (r & 7)) * 8);
        }
    auto issue = [&](int64_t u, int32_t blk) {
        const int slot = static_cast<int>((u / NW) % kMmaStages);
        T* dst = ring + static_cast<size_t>(slot) * 2 * TE;
        int64_t off = -1;  // element offset of token `lane`'s K row in the cache, -1: no row
        if (lane < kMmaTile) {
            const int64_t tok = t_begin + u * kMmaTile + lane;
            if (tok < t_end) {
                if (block_ok(blk)) {
                    off = ((static_cast<int64_t>(blk) << bs_log2) + (tok & (BS - 1))) * tok_stride + kvh_off;
                } else if (kvh == 0 && (tok & (BS - 1)) == 0 && a.err) {
                    atomicAdd(a.err, 1);  // a bad block entry, counted once (kv head 0, its first token)
                }
            }
        }
        const unsigned valid = __ballot_sync(FULL, off >= 0) & 0xffffu;
        if (lane == 0) vmask[slot] = valid;
#pragma unroll
        for (int i = 0; i < kMmaTile / RPI; ++i) {
            const int64_t ro = __shfl_sync(FULL, off, rr0 + RPI * i);
            const T* src = ro >= 0 ? cache + ro + col * 8 : cache;
            const int n = ro >= 0 ? 16 : 0;
#pragma unroll
            for (int cc = 0; cc < CPR / LPR; ++cc) {
                T* d = dst + dst_off[i][cc];
                cp_async16_zfill(d, src + cc * LPR * 8, n);
                cp_async16_zfill(d + TE, ro >= 0 ? src + cc * LPR * 8 + v_plane : cache, n);
            }
        }
    };
#pragma unroll
    for (int k = 0; k < kMmaStages - 1; ++k) {
        const int64_t u = warp + static_cast<int64_t>(k) * NW;
        if (u < n_static) issue(u, blk0[k]);
        cp_async_commit();
    }
    int32_t blk_next = blk0[kMmaStages - 1];
    // Q as A fragments (loaded while the first tiles are in flight): rows = query heads
    // (zero past G), columns = dims of k-step s
    uint32_t qa[KS][2];
    {
        const T* qrow = static_cast<const T*>(a.q) + b * a.qs + static_cast<int64_t>(kvh * G + fg) * HD;
#pragma unroll
        for (int s = 0; s < KS; ++s) {
            qa[s][0] = fg < G ? *reinterpret_cast<const uint32_t*>(qrow + 16 * s + 2 * ft) : 0u;
            qa[s][1] = fg < G ? *reinterpret_cast<const uint32_t*>(qrow + 16 * s + 8 + 2 * ft) : 0u;
        }
    }

    float o[NB][2];  // C fragments of O (rows fg: c0, c1)
#pragma unroll
    for (int d = 0; d < NB; ++d) o[d][0] = o[d][1] = 0.0f;
    float m = -INFINITY, l = 0.0f;
    for (int64_t u = warp, k = 0; u < n_tiles; u += NW, ++k) {
        cp_async_wait<kMmaStages - 2>();
        __syncwarp();
        if (u + (kMmaStages - 1) * NW < n_tiles) {
            issue(u + (kMmaStages - 1) * NW, blk_next);
            blk_next = load_blk(u + kMmaStages * NW);
        }
        cp_async_commit();
        const T* Ks = ring + static_cast<size_t>(k % kMmaStages) * 2 * TE;
        const T* Vs = Ks + TE;
        const unsigned valid = vmask[k % kMmaStages];

        tile_step<T, HD>(Ks, Vs, valid, qa, o, m, l, a.scale_log2, lane,
                         [](int tok, int chunk) { return tok * HD + ((chunk ^ (tok & 7)) * 8); });
    }
    cp_async_wait<0>();
    finish_mma<T, HD, GMERGE, NW>(a, smem, reinterpret_cast<float*>(smem + mma_inbox_offset(HD, NW)), m, l, o, lane,
                                  warp, grp, b, kvh, S, rank, G, cluster);
}

// The merge of a workspace split: CTA (pair, chunk) combines the S splits' partials of 32
// output columns (one query head: head_dim is a multiple of 32). Thread (p, j) reads column j of
// splits p, p + 8, ... with all its loads issued together and before the weights are known; the
// headers (each split's max and sum for the chunk's head) arrive in the same round trip. The
// eight partial sums of a column meet in shared memory in split order, so the result does not
// depend on timing. Launched right after the split kernel, with programmatic dependent launch:
// its CTAs start early and wait for the splits' records.
constexpr int kMergeCols = 32;
template <typename T, int HD>
__global__ void __launch_bounds__(256) decode_merge_kernel(AttnArgs a) {
    constexpr int PS = 16 + 8 * HD;        // floats per split's record
    constexpr int PER = kMaxGsplits / 8;  // splits one thread reads at most
    __shared__ float wgt[kMaxGsplits];
    __shared__ float red[8][kMergeCols];
    __shared__ float wmax[8], wsum[8], stat[2];
    const int S = a.gsplits, G = a.group;
    const int64_t grp = blockIdx.x;
    const int64_t b = grp / a.n_kv;
    const int kvh = static_cast<int>(grp - b * a.n_kv);
    const int c0 = blockIdx.y * kMergeCols, gg = c0 / HD;
    const int j = threadIdx.x % kMergeCols, p = threadIdx.x / kMergeCols;
    const unsigned FULL = 0xffffffffu;
    pdl_enter();
    const float* parts = a.ws_part + grp * S * PS;
    float v[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int r = p + 8 * i;
        v[i] = r < S ? __ldcg(parts + r * PS + 16 + c0 + j) : 0.0f;
    }
    float mr = -INFINITY, lr = 0.0f;
    if (threadIdx.x < S) {
        mr = __ldcg(parts + threadIdx.x * PS + gg);
        lr = __ldcg(parts + threadIdx.x * PS + 8 + gg);
    }
    // M over the splits (threads of split r hold its max), then the weights and the denominator
    float M = mr;
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, o));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = M;
    __syncthreads();
    if (threadIdx.x == 0) {
        float mm = -INFINITY;
        for (int w = 0; w < 8; ++w) mm = fmaxf(mm, wmax[w]);
        stat[0] = mm;
    }
    __syncthreads();
    M = stat[0];
    const float e = (threadIdx.x < S && M != -INFINITY && mr != -INFINITY) ? exp2f(mr - M) : 0.0f;
    if (threadIdx.x < S) wgt[threadIdx.x] = e;
    // the denominator: the same fixed reduction tree every call (a warp's butterfly, then the
    // warps' sums in order)
    float d = e * lr;
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(FULL, d, o);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = d;
    __syncthreads();  // the weights and the warps' sums are in shared memory
    if (threadIdx.x == 0) {
        float t = 0.0f;
        for (int w = 0; w < 8; ++w) t += wsum[w];
        stat[1] = t;
    }
    float num = 0.0f;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int r = p + 8 * i;
        if (r < S) num = fmaf(wgt[r], v[i], num);
    }
    red[p][j] = num;
    __syncthreads();
    if (p == 0) {
        float t = 0.0f;
#pragma unroll
        for (int q = 0; q < 8; ++q) t += red[q][j];
        const float den = stat[1];
        T* out = static_cast<T*>(a.out) + b * a.os + static_cast<int64_t>(kvh * G) * HD;
        out[c0 + j] = from_f32<T>(den > 0.0f ? t / den : 0.0f);
    }
}

template <typename T, int HD>
cudaError_t launch_merge(const AttnArgs& a, const AttnPlan& p, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.B * a.n_kv), static_cast<unsigned>(a.group * HD / kMergeCols));
    return launch_kernel(decode_merge_kernel<T, HD>, grid, dim3(256), 0, s, p.pdl, 1, a);
}

template <typename T, int HD, int NW>
cudaError_t launch_mma(const AttnArgs& a, const AttnPlan& p, cudaStream_t s) {
    const size_t smem = mma_smem(HD, NW);
    if (a.gsplits > 0) {
        auto kg = decode_mma_kernel<T, HD, true, NW>;
        const cudaError_t eg =
            cudaFuncSetAttribute(kg, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (eg != cudaSuccess) return eg;
        const dim3 grid(static_cast<unsigned>(a.B * a.n_kv * a.gsplits)), block(NW * 32);
        const cudaError_t el = launch_kernel(kg, grid, block, smem, s, p.pdl, 1, a);
        return el != cudaSuccess ? el : launch_merge<T, HD>(a, p, s);
    }
    auto kernel = decode_mma_kernel<T, HD, false, NW>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int splits = p.splits;
    if (splits > 8) {
        // a 16-CTA cluster is a non-portable size: use it only where the device can place one
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        int clusters = 0;
        if (e == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = static_cast<unsigned>(splits);
            attr.val.clusterDim.y = attr.val.clusterDim.z = 1;
            cfg.gridDim = dim3(static_cast<unsigned>(splits));
            cfg.blockDim = dim3(NW * 32);
            cfg.dynamicSmemBytes = smem;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
        }
        if (e != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            splits = 8;
        }
    }
    const dim3 grid(static_cast<unsigned>(a.B * a.n_kv * splits)), block(NW * 32);
    return launch_kernel(kernel, grid, block, smem, s, p.pdl, splits, a);
}


// ------------------------------------------------------------------------------------------
// Tensor-core path with the K / V tiles moved by TMA (bf16 / fp16, head_dim 64 or 128).
//
// The same work split, per-tile contraction and merge as decode_mma_kernel, with the data
// movement taken off the compute warps: a ninth warp streams the tiles. It reads the
// split's block-table entries 32 tiles at a time (one coalesced load, the entries passed by
// shuffles) and for each 16-token tile issues the TMA box copies of its cache rows (a 4-D
// tensor map over the cache: [HD][n_kv][num_blocks * block_size][K | V plane], boxes of 64
// dims x 1 head x 16 rows (8 for blocks of 8 tokens), 128-byte swizzle) into ring slot
// u % R, completing on the slot's full barrier, together with the tile's row mask. Compute
// warp u % 8 waits for the slot, zeroes the V rows of tokens that do not count (past
// seq_len, or in a bad block, whose rows are not copied), runs tile_step, and releases the
// slot on its empty barrier. R = 96 KB of slots, so two CTAs share an SM.
constexpr int kTmaWarps = 8;  // compute warps; warp 8 issues the copies
constexpr int kTmaTile = 16;  // tokens per tile
template <int HD>
__host__ __device__ constexpr int tma_slots() { return HD == 128 ? 12 : 24; }
template <int HD>
__host__ __device__ constexpr size_t tma_slot_bytes() { return 2u * kTmaTile * HD * 2; }  // K and V tiles
__host__ __device__ inline size_t tma_smem(int HD) {
    const size_t ring = HD == 128 ? tma_slots<128>() * tma_slot_bytes<128>() : tma_slots<64>() * tma_slot_bytes<64>();
    const size_t merge = (static_cast<size_t>(kTmaWarps) * 8 * (HD + 11) + 8 * (HD + 2) + 17 * 8) * 4;
    const size_t gmerge = static_cast<size_t>(kMaxGsplits) * 24 * 4 + 64 + 16 * 8 * static_cast<size_t>(HD) * 4;
    size_t need = ring > merge ? ring : merge;
    need = need > gmerge ? need : gmerge;
    return 1024 + need + inbox_floats(HD) * 4;
}

template <typename T, int HD, bool GMERGE>
__global__ void __maxnreg__(112) decode_tma_kernel(AttnArgs a,
                                                                         const __grid_constant__ CUtensorMap tmC) {
    constexpr int R = tma_slots<HD>();
    constexpr int HALVES = HD / 64;
    constexpr int KS = HD / 16, NB = HD / 8;
    constexpr size_t SLOT = tma_slot_bytes<HD>();
    constexpr size_t PLANE = SLOT / 2;          // bytes of the K (or V) tile
    constexpr size_t HALF = kTmaTile * 128;     // bytes of one 64-dim half of a tile
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ uint64_t full[R], empty[R];
    __shared__ unsigned vmask[R];
    cg::cluster_group cluster = cg::this_cluster();
    const int S = GMERGE ? a.gsplits : static_cast<int>(cluster.num_blocks());
    const int rank = GMERGE ? static_cast<int>(blockIdx.x % a.gsplits) : static_cast<int>(cluster.block_rank());
    const int64_t grp = blockIdx.x / S;
    const int64_t b = grp / a.n_kv;
    const int kvh = static_cast<int>(grp - b * a.n_kv);
    const int G = a.group, BS = a.block_size;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int fg = lane >> 2, ft = lane & 3;
    const unsigned FULL = 0xffffffffu;
    if (threadIdx.x == 0) {
        for (int i = 0; i < R; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init_fence();
    }
    {
        // Before the dependency wait, hints only: this request's seq_len and this split's slice of
        // the block table into L2 (the split is a static slice of the table's capacity).
        const int64_t cap0 = a.max_blocks * BS;
        const int64_t per0 = ((cap0 + S - 1) / S + kTmaTile - 1) / kTmaTile * kTmaTile;
        const int64_t s0 = rank * per0, s1 = cap0 < s0 + per0 ? cap0 : s0 + per0;
        if (warp == kTmaWarps && lane == 0) prefetch_lines(a.seq_lens + b, 4, 0, 1);
        if (warp == kTmaWarps && s0 < s1)
            prefetch_lines(a.table + b * a.max_blocks + s0 / BS, ((s1 - 1) / BS - s0 / BS + 1) * 4, lane, 32);
    }
    __syncthreads();  // the barriers are initialised
    pdl_enter();
    int64_t len = a.seq_lens[b];
    const int64_t cap = a.max_blocks * BS;
    if ((len < 0 || len > cap) && kvh == 0 && rank == 0 && threadIdx.x == 0 && a.err) atomicAdd(a.err, 1);
    len = len < 0 ? 0 : (len > cap ? cap : len);
    const int64_t per = ((cap + S - 1) / S + kTmaTile - 1) / kTmaTile * kTmaTile;
    const int64_t t_begin = rank * per < cap ? rank * per : cap;
    const int64_t t_lim = t_begin + per < cap ? t_begin + per : cap;
    const int64_t t_end = len < t_begin ? t_begin : (len < t_lim ? len : t_lim);
    const int64_t n_tiles = (t_end - t_begin + kTmaTile - 1) / kTmaTile;
    const int bs_log2 = __ffs(BS) - 1;           // block_size is a power of two (8, 16 or 32)
    const int RB = BS < kTmaTile ? BS : kTmaTile;  // cache rows per box
    const int NBX = kTmaTile / RB;                // boxes (cache blocks) per tile: 1 or 2

    float o[NB][2];
#pragma unroll
    for (int d = 0; d < NB; ++d) o[d][0] = o[d][1] = 0.0f;
    float m = -INFINITY, l = 0.0f;
    // A wait that gives up (counted in g_wait_timeouts) marks this thread: it waits no more, so a
    // stalled copy costs one wait limit, not one per tile.
    bool dead = false;
    if (warp == kTmaWarps) {
        const int32_t* table = a.table + b * a.max_blocks;
        for (int64_t base = 0; base < n_tiles; base += 32) {
            // lane i: the block ids of tile base + i (a second one for blocks of 8 tokens)
            int32_t e0 = -1, e1 = -1;
            if (base + lane < n_tiles) {
                const int64_t t0 = t_begin + (base + lane) * kTmaTile;
                e0 = table[t0 >> bs_log2];
                if (NBX == 2 && t0 + RB < t_end) e1 = table[(t0 + RB) >> bs_log2];
            }
            const int cnt = n_tiles - base < 32 ? static_cast<int>(n_tiles - base) : 32;
            for (int i = 0; i < cnt; ++i) {
                const int32_t blk0 = __shfl_sync(FULL, e0, i), blk1 = __shfl_sync(FULL, e1, i);
                if (lane == 0) {
                    const int64_t u = base + i;
                    const int slot = static_cast<int>(u % R);
                    // the slot's previous tile (u - R) has been released by its warp
                    if (u >= R && !dead) dead = !mbar_wait(&empty[slot], static_cast<uint32_t>(((u / R) - 1) & 1));
                    const int64_t t0 = t_begin + u * kTmaTile;
                    unsigned valid = 0;
                    uint32_t bytes = 0;
                    int32_t rows[2] = {-1, -1};
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        const int64_t tx = t0 + x * RB;  // first token of box x
                        if (x >= NBX || tx >= t_end) break;
                        const int32_t blk = x == 0 ? blk0 : blk1;
                        if (blk < 0 || blk >= a.num_blocks) {
                            // a bad block entry, counted once (kv head 0, the block's first token)
                            if (kvh == 0 && (tx & (BS - 1)) == 0 && a.err) atomicAdd(a.err, 1);
                            continue;
                        }
                        const int nv = t_end - tx < RB ? static_cast<int>(t_end - tx) : RB;
                        valid |= ((1u << nv) - 1u) << (x * RB);
                        bytes += static_cast<uint32_t>(2 * HALVES * RB * 128);
                        rows[x] = static_cast<int32_t>((static_cast<int64_t>(blk) << bs_log2) + (tx & (BS - 1)));
                    }
                    vmask[slot] = valid;
                    mbar_arrive_expect_tx(&full[slot], bytes);
                    unsigned char* st = smem + static_cast<size_t>(slot) * SLOT;
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        if (rows[x] < 0) continue;
#pragma unroll
                        for (int plane = 0; plane < 2; ++plane)
#pragma unroll
                            for (int h = 0; h < HALVES; ++h)
                                tma_load_4d(st + plane * PLANE + h * HALF + x * RB * 128, &tmC, h * 64, kvh, rows[x],
                                            plane, &full[slot]);
                    }
                }
                __syncwarp();
            }
        }
    } else {
        // Q as A fragments: rows = query heads (zero past G), columns = dims of k-step s
        uint32_t qa[KS][2];
        const T* qrow = static_cast<const T*>(a.q) + b * a.qs + static_cast<int64_t>(kvh * G + fg) * HD;
#pragma unroll
        for (int s2 = 0; s2 < KS; ++s2) {
            qa[s2][0] = fg < G ? *reinterpret_cast<const uint32_t*>(qrow + 16 * s2 + 2 * ft) : 0u;
            qa[s2][1] = fg < G ? *reinterpret_cast<const uint32_t*>(qrow + 16 * s2 + 8 + 2 * ft) : 0u;
        }
        // chunk c of token t's row: 64-dim half c / 8, its 16-byte chunk (c % 8) XOR t % 8 (the swizzle)
        auto addr = [](int tok, int chunk) {
            return (chunk >> 3) * (kTmaTile * 64) + tok * 64 + (((chunk & 7) ^ (tok & 7)) * 8);
        };
        for (int64_t u = warp; u < n_tiles; u += kTmaWarps) {
            const int slot = static_cast<int>(u % R);
            if (!dead) dead = !mbar_wait(&full[slot], static_cast<uint32_t>((u / R) & 1));
            __syncwarp();
            unsigned char* st = smem + static_cast<size_t>(slot) * SLOT;
            const unsigned valid = vmask[slot];
            if (valid != 0xffffu) {
                // V rows of tokens that do not count hold stale bytes (never copied, or past the end
                // of the request): zero them so that p = 0 meets 0, not whatever they hold
                for (int c = lane; c < kTmaTile * HALVES * 8; c += 32) {
                    const int r = c / (HALVES * 8), rest = c - r * (HALVES * 8);
                    if (!((valid >> r) & 1u))
                        *reinterpret_cast<uint4*>(st + PLANE + (rest >> 3) * HALF + r * 128 + (rest & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async();  // before the copy engine refills the slot
                __syncwarp();
            }
            tile_step<T, HD>(reinterpret_cast<const T*>(st), reinterpret_cast<const T*>(st + PLANE), valid, qa, o, m,
                             l, a.scale_log2, lane, addr);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
    }
    finish_mma<T, HD, GMERGE, kTmaWarps>(a, smem, reinterpret_cast<float*>(smem + tma_smem(HD) - 1024 - inbox_floats(HD) * 4),
                                         m, l, o, lane, warp, grp, b, kvh, S, rank, G, cluster);
}

template <typename T, int HD>
cudaError_t launch_tma(const AttnArgs& a, const AttnPlan& p, cudaStream_t s) {
    // the cache as [HD][n_kv][num_blocks * block_size][2 planes], boxes of 64 dims x 1 head x up to 16 rows
    const int BS = a.block_size;
    const uint64_t dims[4] = {static_cast<uint64_t>(HD), static_cast<uint64_t>(a.n_kv),
                              static_cast<uint64_t>(a.num_blocks) * BS, 2};
    const uint64_t strides[3] = {static_cast<uint64_t>(HD) * 2, static_cast<uint64_t>(a.n_kv) * HD * 2,
                                 static_cast<uint64_t>(a.num_blocks) * BS * a.n_kv * HD * 2};
    const uint32_t box[4] = {64, 1, static_cast<uint32_t>(BS < kTmaTile ? BS : kTmaTile), 1};
    CUtensorMap tm;
    if (!encode_tmap_16_nd(&tm, a.cache, 4, dims, strides, box, std::is_same<T, __nv_bfloat16>::value, true))
        return cudaErrorNotSupported;
    const size_t smem = tma_smem(HD);
    const dim3 block((kTmaWarps + 1) * 32);
    if (a.gsplits > 0) {
        auto kg = decode_tma_kernel<T, HD, true>;
        const cudaError_t eg =
            cudaFuncSetAttribute(kg, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (eg != cudaSuccess) return eg;
        const cudaError_t el =
            launch_kernel(kg, dim3(static_cast<unsigned>(a.B * a.n_kv * a.gsplits)), block, smem, s, p.pdl, 1, a, tm);
        return el != cudaSuccess ? el : launch_merge<T, HD>(a, p, s);
    }
    auto kernel = decode_tma_kernel<T, HD, false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int splits = p.splits;
    if (splits > 8) {
        // a 16-CTA cluster is a non-portable size: use it only where the device can place one
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        int clusters = 0;
        if (e == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = static_cast<unsigned>(splits);
            attr.val.clusterDim.y = attr.val.clusterDim.z = 1;
            cfg.gridDim = dim3(static_cast<unsigned>(splits));
            cfg.blockDim = block;
            cfg.dynamicSmemBytes = smem;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
        }
        if (e != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            splits = 8;
        }
    }
    return launch_kernel(kernel, dim3(static_cast<unsigned>(a.B * a.n_kv * splits)), block, smem, s, p.pdl, splits,
                         a, tm);
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
    if constexpr (sizeof(T) == 2) {
        if (p.tma) return p.head_dim == 64 ? launch_tma<T, 64>(a, p, s) : launch_tma<T, 128>(a, p, s);
        if (p.tensor_cores) {
            if (p.mma_warps == 4) return p.head_dim == 64 ? launch_mma<T, 64, 4>(a, p, s) : launch_mma<T, 128, 4>(a, p, s);
            return p.head_dim == 64 ? launch_mma<T, 64, 8>(a, p, s) : launch_mma<T, 128, 8>(a, p, s);
        }
    }
    return p.stages >= 4 ? launch_stages<T, 4>(a, p, s) : launch_stages<T, 2>(a, p, s);
}

}  // namespace attn

size_t decode_attention_mma_smem(int head_dim, int warps) { return attn::mma_smem(head_dim, warps); }
size_t decode_attention_tma_smem(int head_dim) { return attn::tma_smem(head_dim); }

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

// Bounded waits of this file's kernels (the TMA-fed attention variant) that ran out: the
// counter in tma.cuh is per translation unit, so each file that waits reports its own copy.
unsigned int attn_wait_timeouts() {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_wait_timeouts, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return v;
}

}  // namespace sra
