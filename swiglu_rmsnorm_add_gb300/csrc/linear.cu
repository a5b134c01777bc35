// The decoder's projections with their elementwise producer fused in as a
// prologue: y = prologue(x) @ W^T, W in nn.Linear's [N, K] layout.
//
// m.lsln.cn 21-operator article, section 2.2: the RMSNorm before the
// attention feeds qkv_proj directly, so the norm runs inside the projection
// and its output never goes to memory (3-5 % of the step); the same holds for
// the activation before the MLP's down projection (silu(gate) * up, or relu).
// The prologue's rows are rounded to the dtype, as the separate kernel would
// store them, before they meet W.
//
// At decode batch sizes the cost is the weight read (N * K * 2 bytes per call),
// so W is streamed once. Three kernels:
//  - linear16_kernel (up to 16 rows): a CTA owns 16 columns of y over the whole
//    of K; its warps split K, stream their W tiles through private cp.async
//    rings, and h for all of K is built once up front.
//  - linear_kernel (more rows): a CTA owns a 64-column slice of y for 16, 32 or
//    64 rows, K is split over the CTAs of a thread-block cluster and the partial
//    products are summed through distributed shared memory (no global scratch).
//    W tiles and the prologue's input tiles arrive by TMA tensor copies (128-byte
//    swizzle) into two mbarrier rings, W's deep (from DRAM) and the input's short
//    (from L2); h is built tile by tile from the input tiles into one of two h
//    buffers while the other is multiplied. For the RMSNorm each CTA first sums
//    the squares of its K range and the cluster exchanges the partial sums.
//  - linear_h_kernel (the workspace path, where the prologue ran in its own
//    kernel): a producer warp streams W and h tiles by TMA, the other warps
//    multiply and release each slot on an empty barrier; no CTA barrier per tile.
// The products run on the tensor cores as mma.sync m16n8k16 with fp32
// accumulators (h as the A operand, W tiles as the B operand, both through
// ldmatrix from swizzled shared memory).
#include <cooperative_groups.h>

#include <atomic>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace cg = cooperative_groups;

namespace sra {
namespace lin {

constexpr int kNT = 64;      // columns of y per CTA
constexpr int kKT = 64;      // K per W tile

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(s));
}

template <typename T>
struct Mma;
template <>
struct Mma<__nv_bfloat16> {
    __device__ __forceinline__ static void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};
template <>
struct Mma<__half> {
    __device__ __forceinline__ static void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};

template <typename T>
__device__ __forceinline__ T to_t(float v) {
    const unsigned short b = Elem<T>::to_bits16(v);
    T r;
    memcpy(&r, &b, 2);
    return r;
}

// Shared memory (from a 1024-byte aligned base, as the 128-byte swizzle of the tile copies
// needs): two rings. The W ring holds W tiles [64][64]; it runs far ahead (its tiles come
// from DRAM). The input ring holds, for the same 64 columns of K, the prologue's input tile:
// x [MT*16][64] and the norm weight's 64 entries (RMSNorm), or gate and up [2][MT*16][64]
// (GLU); its tiles are re-read by every column slice, so they come from L2 and a short ring
// covers them. Tiles are swizzled (16-byte chunk c of row r at c ^ (r % 8)). Then two h tiles
// [MT*16][64] (built while the other is multiplied). The epilogue's partial tile reuses the
// rings once they have drained. Sizes keep two CTAs per SM.
__host__ __device__ constexpr int warps_for(int MT) { return MT == 1 ? 4 : 8; }
__host__ __device__ constexpr bool glu_input(int PRO) { return PRO == 1 || PRO == 2; }  // gate and up tiles
__host__ __device__ constexpr int wstages_for(int MT, int PRO) { return MT == 4 && glu_input(PRO) ? 5 : 8; }
__host__ __device__ constexpr int xstages_for(int MT, int PRO) { return 3; }
__host__ __device__ constexpr size_t wtile_bytes() { return static_cast<size_t>(kNT) * kKT * 2; }
__host__ __device__ constexpr size_t xtile_bytes(int MT) { return static_cast<size_t>(MT) * 16 * kKT * 2; }
__host__ __device__ constexpr size_t xstage_bytes(int MT, int PRO) {
    return (static_cast<size_t>(glu_input(PRO) ? 2 : 1) * xtile_bytes(MT) + (PRO == 0 ? kKT * 2 : 0) + 1023) / 1024 * 1024;
}
__host__ __device__ constexpr size_t rings_bytes(int MT, int PRO) {
    return wstages_for(MT, PRO) * wtile_bytes() + xstages_for(MT, PRO) * xstage_bytes(MT, PRO);
}
__host__ __device__ constexpr size_t htile_bytes(int MT) { return static_cast<size_t>(MT) * 16 * kKT * 2; }
__host__ __device__ constexpr size_t ring_area(int MT, int PRO) {
    return rings_bytes(MT, PRO) > static_cast<size_t>(MT) * 16 * kNT * 4 ? rings_bytes(MT, PRO)
                                                                           : static_cast<size_t>(MT) * 16 * kNT * 4;
}
__host__ __device__ constexpr size_t smem_bytes(int MT, int PRO) {
    return 1024 + ring_area(MT, PRO) + 2 * htile_bytes(MT);  // + the alignment slack
}

// 16-byte chunk c of row r of a row-major tile whose rows hold `cpr` chunks.
__device__ __forceinline__ int swz(int r, int c) { return c ^ (r & 7); }

// PRO: 0 = RMSNorm prologue, 1 = SwiGLU, 2 = ReGLU, 3 = none (the input rows are h, already
// produced by the prologue's own kernel). The tensor maps: tmW over W [N][K] and tmX over the
// input rows [B][K] (GLU: [B][2K]), both with 64 x 64 (rows: MT*16) boxes and the 128-byte
// swizzle; tmN over the norm weight [K], 64-entry boxes (RMSNorm only).
template <typename T, int MT, int PRO>
__global__ void __launch_bounds__(warps_for(MT) * 32) linear_kernel(LinArgs a, const __grid_constant__ CUtensorMap tmW,
                                                              const __grid_constant__ CUtensorMap tmX,
                                                              const __grid_constant__ CUtensorMap tmN) {
    using V8 = Vec<T, 8>;
    using R8 = typename V8::Raw;
    constexpr int XR = MT * 16;                  // rows of an input / h tile
    constexpr int NW = warps_for(MT);            // warps
    constexpr int SW = wstages_for(MT, PRO);  // W ring stages
    constexpr int SX = xstages_for(MT, PRO);  // input ring stages
    constexpr size_t XB = xstage_bytes(MT, PRO);
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ uint64_t wfull[SW];  // W tile t lands in slot t % SW and completes on wfull[t % SW]
    __shared__ uint64_t xfull[SX];  // input tile t: slot t % SX, xfull[t % SX]
    __shared__ float stat[64];
    __shared__ float inv[64];
    __shared__ float pre[64];     // RMSNorm rows past fp32's sum range: a power-of-two pre-scale
    __shared__ double dstat[64];  // ... and their sums of squares again, in double
    cg::cluster_group cluster = cg::this_cluster();
    const int SK = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t n0 = (blockIdx.x / SK) * static_cast<int64_t>(kNT);
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * XR;
    const int rows = static_cast<int>(a.B - r0 < XR ? a.B - r0 : XR);
    const int KT = static_cast<int>(a.K / kKT);
    const int per = (KT + SK - 1) / SK;
    const int kt0 = rank * per < KT ? rank * per : KT;
    const int kt1 = kt0 + per < KT ? kt0 + per : KT;
    const int ntiles = kt1 - kt0;
    const int64_t kbase = static_cast<int64_t>(kt0) * kKT;
    float* part = reinterpret_cast<float*>(smem);  // the epilogue's partial tile, after the ring drains
    T* hbuf = reinterpret_cast<T*>(smem + ring_area(MT, PRO));  // [2][XR][64]
    const T* W = static_cast<const T*>(a.W);
    const T* X = static_cast<const T*>(a.x);
    auto wslot = [&](int t) { return reinterpret_cast<T*>(smem + static_cast<size_t>(t % SW) * wtile_bytes()); };
    auto xslot = [&](int t) {
        return reinterpret_cast<T*>(smem + SW * wtile_bytes() + static_cast<size_t>(t % SX) * XB);
    };

    // Thread 0 issues the tile copies. W tile t: W's 64 x 64 tile at columns (kt0 + t) * 64 of
    // rows n0 ..; input tile t: the input rows' same 64 columns of K (x; or gate and up) and,
    // for the RMSNorm, the norm weight's 64 entries. Rows past B arrive as zeros.
    constexpr uint32_t kXTx =
        static_cast<uint32_t>((glu_input(PRO) ? 2 : 1) * xtile_bytes(MT) + (PRO == 0 ? kKT * 2 : 0));
    auto issue_w = [&](int t) {
        uint64_t* bar = &wfull[t % SW];
        fence_proxy_async();  // the slot's earlier reads come before the copy
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(wtile_bytes()));
        tma_load_2d(wslot(t), &tmW, static_cast<int>(kbase) + t * kKT, static_cast<int>(n0), bar);
    };
    auto issue_x = [&](int t) {
        uint64_t* bar = &xfull[t % SX];
        const int k0 = static_cast<int>(kbase) + t * kKT;
        T* xd = xslot(t);
        fence_proxy_async();
        mbar_arrive_expect_tx(bar, kXTx);
        tma_load_2d(xd, &tmX, k0, static_cast<int>(r0), bar);
        if constexpr (glu_input(PRO)) {
            tma_load_2d(xd + XR * kKT, &tmX, static_cast<int>(a.K) + k0, static_cast<int>(r0), bar);
        } else if constexpr (PRO == 0) {
            tma_load_1d(xd + XR * kKT, &tmN, k0, bar);
        }
    };
    if (threadIdx.x == 0) {
        for (int i = 0; i < SW; ++i) mbar_init(&wfull[i], 1);
        for (int i = 0; i < SX; ++i) mbar_init(&xfull[i], 1);
        mbar_init_fence();
    }
    // Before the dependency wait: this CTA's slice of W (64 rows x its K range) and of the
    // prologue's input into L2 (hints only; both are read again after the wait).
    if (threadIdx.x < kNT && n0 + threadIdx.x < a.N)
        prefetch_l2(W + (n0 + threadIdx.x) * a.K + kbase, static_cast<int64_t>(ntiles) * kKT * 2);
    else if (threadIdx.x >= kNT && threadIdx.x - kNT < rows) {
        const T* xr = X + (r0 + threadIdx.x - kNT) * a.xs + kbase;
        prefetch_l2(xr, static_cast<int64_t>(ntiles) * kKT * 2);
        if (glu_input(PRO)) prefetch_l2(xr + a.K, static_cast<int64_t>(ntiles) * kKT * 2);
    }
    __syncthreads();  // the barriers are initialised
    pdl_enter();
    if (threadIdx.x == 0) {
        for (int t = 0; t < SX && t < ntiles; ++t) issue_x(t);
        for (int t = 0; t < SW - 1 && t < ntiles; ++t) issue_w(t);
    }

    // h tile t from input tile t: thread owns chunks c = tid + 32 NW i of the [XR][64] tile:
    // row c / 8, 8-element chunk c % 8; rows past B are zero.
    auto build = [&](int t) {
        T* hb = hbuf + static_cast<size_t>(t & 1) * XR * kKT;
        const T* xs = xslot(t);
#pragma unroll
        for (int i = 0; i < XR * 8 / (NW * 32); ++i) {
            const int c = threadIdx.x + NW * 32 * i, r = c >> 3, ch = c & 7;
            float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if constexpr (PRO == 1) {
                // a chunk holding a gate below -64 (never on the configured inputs): each
                // element through glu_mul, scalar, straight into the h tile
                if (r < rows && __builtin_expect(needs_careful<T, 8>(
                                                     *reinterpret_cast<const R8*>(xs + r * kKT + swz(r, ch) * 8)),
                                                 0)) {
                    const T* gp = xs + r * kKT + swz(r, ch) * 8;
                    const T* up = xs + (XR + r) * kKT + swz(r, ch) * 8;
                    T* hp = hb + r * kKT + swz(r, ch) * 8;
#pragma unroll 1
                    for (int e = 0; e < 8; ++e) hp[e] = to_t<T>(glu_mul<0>(to_f32(gp[e]), to_f32(up[e])));
                    continue;
                }
            }
            if (r < rows) {
                float g[8];
                V8::unpack(*reinterpret_cast<const R8*>(xs + r * kKT + swz(r, ch) * 8), f);
                if constexpr (PRO == 3) {
                    // h as given
                } else if constexpr (PRO == 0) {
                    V8::unpack(*reinterpret_cast<const R8*>(xs + XR * kKT + ch * 8), g);
                    const float iv = inv[r], pv = pre[r];
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = f[e] * pv * iv * g[e];
                } else {
                    V8::unpack(*reinterpret_cast<const R8*>(xs + (XR + r) * kKT + swz(r, ch) * 8), g);
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = glu_mul_fast<PRO - 1>(f[e], g[e]);
                }
            }
            *reinterpret_cast<R8*>(hb + r * kKT + swz(r, ch) * 8) = V8::pack(f);
        }
    };
    if constexpr (PRO == 0) {
        // each rank sums the squares of its K range; the cluster exchanges the partial sums.
        // A warp owns rows warp, warp + 4, ...: the loads of all its rows go out together,
        // one 16-byte chunk per lane and row per 256 columns
        constexpr int RPW = MT * 16 / NW;
        float ss[RPW];
#pragma unroll
        for (int i = 0; i < RPW; ++i) ss[i] = 0.0f;
        for (int k = lane * 8; k < ntiles * kKT; k += 256) {
            R8 v[RPW];
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const int r = warp + NW * i;
                if (r < rows) v[i] = V8::load(X + (r0 + r) * a.xs + kbase + k);
            }
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                if (warp + NW * i < rows) {
                    float f[8];
                    V8::unpack(v[i], f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss[i] = fmaf(f[e], f[e], ss[i]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            const float t = warp_sum(ss[i]);
            if (lane == 0) stat[warp + NW * i] = t;
        }
        cluster.sync();  // every rank's partial sums are in its shared memory
        int wide = 0;
        for (int r = threadIdx.x; r < MT * 16; r += NW * 32) {
            float tot = 0.0f;
            for (int q = 0; q < SK; ++q) tot += cluster.map_shared_rank(stat, q)[r];
            inv[r] = rsqrtf(tot / static_cast<float>(a.K) + a.eps);
            pre[r] = 1.0f;
            wide |= r < rows && !ss_in_range(tot, a.K, a.eps);
        }
        // inv complete before the first h tile. Every rank adds the same partials in the
        // same order, so `wide` is the same on all ranks of the cluster.
        if (__syncthreads_or(wide)) {
            // rows whose fp32 sum left fp32's range: each rank sums its K range again in
            // double, and the cluster exchanges those sums
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const int r = warp + NW * i;
                double sd = 0.0;
                if (r < rows) {
                    for (int k = lane * 8; k < ntiles * kKT; k += 256) {
                        float f[8];
                        V8::unpack(V8::load(X + (r0 + r) * a.xs + kbase + k), f);
#pragma unroll
                        for (int e = 0; e < 8; ++e) sd += static_cast<double>(f[e]) * static_cast<double>(f[e]);
                    }
                }
                sd = warp_sum_d(sd);
                if (lane == 0) dstat[r] = sd;
            }
            cluster.sync();
            for (int r = threadIdx.x; r < rows; r += NW * 32) {
                float tot = 0.0f;
                for (int q = 0; q < SK; ++q) tot += cluster.map_shared_rank(stat, q)[r];
                if (!ss_in_range(tot, a.K, a.eps)) {
                    double sd = 0.0;
                    for (int q = 0; q < SK; ++q) sd += cluster.map_shared_rank(dstat, q)[r];
                    const WideScale sc = wide_scale(sd, a.K, a.eps);
                    inv[r] = sc.rinv, pre[r] = sc.pre;
                }
            }
            __syncthreads();
        }
    }
    if (ntiles > 0) {
        mbar_wait(&xfull[0], 0);
        build(0);
    }

    constexpr int NGROUPS = NW / MT;   // warps sharing an m-tile split its 64 columns
    constexpr int NBW = 8 / NGROUPS;       // n8 blocks per warp
    const int mt = warp % MT, ng = warp / MT;
    float acc[NBW][4];
#pragma unroll
    for (int j = 0; j < NBW; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
    const int li = lane & 7, lm = lane >> 3;  // ldmatrix: row within a matrix, matrix index
    for (int t = 0; t < ntiles; ++t) {
        // W tile t landed (for this iteration's products), input tile t + 1 landed (for h
        // tile t + 1, built at the end of this iteration)
        mbar_wait(&wfull[t % SW], static_cast<uint32_t>((t / SW) & 1));
        if (t + 1 < ntiles) mbar_wait(&xfull[(t + 1) % SX], static_cast<uint32_t>(((t + 1) / SX) & 1));
        // h tile t is built and every warp is done with tile t - 1 and input tile t: W tile
        // t - 1's slot takes W tile t + SW - 1, input tile t's slot takes input tile t + SX,
        // h tile t - 1's buffer takes h tile t + 1
        __syncthreads();
        if (threadIdx.x == 0) {
            if (t + SW - 1 < ntiles) issue_w(t + SW - 1);
            if (t + SX < ntiles) issue_x(t + SX);
        }
        const T* wt = wslot(t);
        const T* ht = hbuf + static_cast<size_t>(t & 1) * XR * kKT;
#pragma unroll
        for (int ks = 0; ks < kKT / 16; ++ks) {
            uint32_t af[4];
            {
                const int r = mt * 16 + (lm & 1) * 8 + li;
                ldsm_x4(af, ht + r * kKT + swz(r, ks * 2 + (lm >> 1)) * 8);
            }
#pragma unroll
            for (int j = 0; j < NBW; j += 2) {
                uint32_t bf[4];
                const int n = (ng * NBW + j) * 8 + (lm >> 1) * 8 + li;
                ldsm_x4(bf, wt + n * kKT + swz(n, ks * 2 + (lm & 1)) * 8);
                Mma<T>::run(acc[j], af, bf[0], bf[1]);
                Mma<T>::run(acc[j + 1], af, bf[2], bf[3]);
            }
        }
        if (t + 1 < ntiles) build(t + 1);
    }
    __syncthreads();  // every warp is done with the ring: its space takes the partial tile

    // ---- epilogue: partial tile into shared memory, then summed over the cluster
    {
        const int g = lane >> 2, q = lane & 3;
#pragma unroll
        for (int j = 0; j < NBW; ++j) {
            const int col = (ng * NBW + j) * 8 + 2 * q;
            const int row = mt * 16 + g;
            part[row * kNT + col] = acc[j][0];
            part[row * kNT + col + 1] = acc[j][1];
            part[(row + 8) * kNT + col] = acc[j][2];
            part[(row + 8) * kNT + col + 1] = acc[j][3];
        }
    }
    cluster.sync();
    T* y = static_cast<T*>(a.y);
    for (int idx = rank * NW * 32 + threadIdx.x; idx < rows * kNT; idx += SK * NW * 32) {
        const int r = idx / kNT, c = idx - r * kNT;
        // every rank's value requested before the first add (the cluster holds at most 8 ranks)
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = q < SK ? cluster.map_shared_rank(part, q)[r * kNT + c] : 0.0f;
        float sum = 0.0f;
#pragma unroll
        for (int q = 0; q < 8; ++q) sum += v[q];
        y[(r0 + r) * a.ys + n0 + c] = to_t<T>(sum);
    }
    cluster.sync();
}

// ---- the projection of rows that are already h (the workspace path: the prologue ran in its
// own kernel). No prologue work is left, so nothing is shared between warps inside a tile and
// the CTA needs no barrier per tile: a producer warp streams stage t (W's 64 x 64 tile and
// h's [MT*16][64] tile, both by TMA with the 128-byte swizzle) into slot t % SH and the
// compute warps, each on its own 16 rows x (64 / NGROUPS) columns, wait for that stage's
// full barrier, multiply, and release the slot on its empty barrier (one arrival per
// warp). The K range, the cluster and the epilogue are those of linear_kernel.
constexpr int kStagesH = 6;
__host__ __device__ constexpr size_t hstage_bytes(int MT) { return wtile_bytes() + xtile_bytes(MT); }
__host__ __device__ constexpr size_t smemh_bytes(int MT) {
    return 1024 + (kStagesH * hstage_bytes(MT) > static_cast<size_t>(MT) * 16 * kNT * 4
                       ? kStagesH * hstage_bytes(MT)
                       : static_cast<size_t>(MT) * 16 * kNT * 4);
}

template <typename T, int MT>
__global__ void __launch_bounds__((warps_for(MT) + 1) * 32) linear_h_kernel(LinArgs a,
                                                                         const __grid_constant__ CUtensorMap tmW,
                                                                         const __grid_constant__ CUtensorMap tmX) {
    constexpr int XR = MT * 16;
    constexpr int NW = warps_for(MT);  // compute warps; warp NW issues the copies
    constexpr int S = kStagesH;
    constexpr size_t SB = hstage_bytes(MT);
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ uint64_t full[S], empty[S];
    cg::cluster_group cluster = cg::this_cluster();
    const int SK = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t n0 = (blockIdx.x / SK) * static_cast<int64_t>(kNT);
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * XR;
    const int rows = static_cast<int>(a.B - r0 < XR ? a.B - r0 : XR);
    const int KT = static_cast<int>(a.K / kKT);
    const int per = (KT + SK - 1) / SK;
    const int kt0 = rank * per < KT ? rank * per : KT;
    const int kt1 = kt0 + per < KT ? kt0 + per : KT;
    const int ntiles = kt1 - kt0;
    const int64_t kbase = static_cast<int64_t>(kt0) * kKT;
    float* part = reinterpret_cast<float*>(smem);  // the epilogue's partial tile, after the ring drains
    const T* W = static_cast<const T*>(a.W);
    const T* X = static_cast<const T*>(a.x);
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NW);
        }
        mbar_init_fence();
    }
    // Before the dependency wait: this CTA's slice of W and of h into L2 (hints only).
    if (threadIdx.x < kNT && n0 + threadIdx.x < a.N)
        prefetch_l2(W + (n0 + threadIdx.x) * a.K + kbase, static_cast<int64_t>(ntiles) * kKT * 2);
    else if (threadIdx.x >= kNT && threadIdx.x - kNT < rows)
        prefetch_l2(X + (r0 + threadIdx.x - kNT) * a.xs + kbase, static_cast<int64_t>(ntiles) * kKT * 2);
    __syncthreads();  // the barriers are initialised
    pdl_enter();

    constexpr int NGROUPS = NW / MT;   // warps sharing an m-tile split its 64 columns
    constexpr int NBW = 8 / NGROUPS;   // n8 blocks per warp
    float acc[NBW][4];
#pragma unroll
    for (int j = 0; j < NBW; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
    const int mt = warp % MT, ng = warp / MT;
    if (warp == NW) {
        if (lane == 0) {
            for (int t = 0; t < ntiles; ++t) {
                const int slot = t % S;
                // the slot's previous tile (t - S) is released by every compute warp
                if (t >= S) mbar_wait(&empty[slot], static_cast<uint32_t>(((t / S) - 1) & 1));
                unsigned char* st = smem + static_cast<size_t>(slot) * SB;
                const int k0 = static_cast<int>(kbase) + t * kKT;
                mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(SB));
                tma_load_2d(st, &tmW, k0, static_cast<int>(n0), &full[slot]);
                tma_load_2d(st + wtile_bytes(), &tmX, k0, static_cast<int>(r0), &full[slot]);
            }
        }
    } else {
        const int li = lane & 7, lm = lane >> 3;  // ldmatrix: row within a matrix, matrix index
        for (int t = 0; t < ntiles; ++t) {
            const int slot = t % S;
            mbar_wait(&full[slot], static_cast<uint32_t>((t / S) & 1));
            const T* wt = reinterpret_cast<const T*>(smem + static_cast<size_t>(slot) * SB);
            const T* ht = reinterpret_cast<const T*>(smem + static_cast<size_t>(slot) * SB + wtile_bytes());
            // every fragment of the tile first, then the products: the shared-memory loads
            // overlap instead of each waiting for the products before it
            uint32_t af[kKT / 16][4], bf[kKT / 16][NBW / 2][4];
#pragma unroll
            for (int ks = 0; ks < kKT / 16; ++ks) {
                const int r = mt * 16 + (lm & 1) * 8 + li;
                ldsm_x4(af[ks], ht + r * kKT + swz(r, ks * 2 + (lm >> 1)) * 8);
#pragma unroll
                for (int j = 0; j < NBW; j += 2) {
                    const int n = (ng * NBW + j) * 8 + (lm >> 1) * 8 + li;
                    ldsm_x4(bf[ks][j / 2], wt + n * kKT + swz(n, ks * 2 + (lm & 1)) * 8);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);  // the fragments are in registers: the slot is free
#pragma unroll
            for (int ks = 0; ks < kKT / 16; ++ks) {
#pragma unroll
                for (int j = 0; j < NBW; j += 2) {
                    Mma<T>::run(acc[j], af[ks], bf[ks][j / 2][0], bf[ks][j / 2][1]);
                    Mma<T>::run(acc[j + 1], af[ks], bf[ks][j / 2][2], bf[ks][j / 2][3]);
                }
            }
        }
    }
    __syncthreads();  // every stage has landed and been read: the ring's space takes the partial tile

    // ---- epilogue: partial tile into shared memory, then summed over the cluster
    if (warp < NW) {
        const int g = lane >> 2, q = lane & 3;
#pragma unroll
        for (int j = 0; j < NBW; ++j) {
            const int col = (ng * NBW + j) * 8 + 2 * q;
            const int row = mt * 16 + g;
            part[row * kNT + col] = acc[j][0];
            part[row * kNT + col + 1] = acc[j][1];
            part[(row + 8) * kNT + col] = acc[j][2];
            part[(row + 8) * kNT + col + 1] = acc[j][3];
        }
    }
    cluster.sync();
    T* y = static_cast<T*>(a.y);
    constexpr int NT = (NW + 1) * 32;
    for (int idx = rank * NT + threadIdx.x; idx < rows * kNT; idx += SK * NT) {
        const int r = idx / kNT, c = idx - r * kNT;
        // every rank's value requested before the first add (the cluster holds at most 8 ranks)
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = q < SK ? cluster.map_shared_rank(part, q)[r * kNT + c] : 0.0f;
        float sum = 0.0f;
#pragma unroll
        for (int q = 0; q < 8; ++q) sum += v[q];
        y[(r0 + r) * a.ys + n0 + c] = to_t<T>(sum);
    }
    cluster.sync();
}

// ---- the projection of rows that are already h on the fifth-generation tensor cores
// (tcgen05), for up to 64 rows. The MMA's operands are swapped so that no accumulator lane is
// padding: A is a 128-row tile of W (128 output columns of y), B the [64][64] tile of h (its
// rows past B arrive as zeros from the tensor map's bounds), and D = W_tile . h_tile^T is
// [128 output columns][64 rows], held in 64 columns of tensor memory with output column
// n0 + i in lane i. One thread issues the TMA copies of stage t (W's [128][64] tile and h's
// [64][64] tile, both with the 128-byte swizzle) into slot t % S; another waits for the
// stage, issues its four MMAs (K = 16 each, operands read from shared memory through matrix
// descriptors) and commits them to the slot's empty barrier, which the producer waits on
// before it refills the slot. After the last stage the MMA thread commits to the accumulator
// barrier; each warp then reads its quarter of the lanes (32 output columns x 64 rows) into a
// partial tile in shared memory, and the cluster (K split over its CTAs) sums its ranks'
// partial tiles as the other projection kernels do. No thread holds a fragment; the tensor
// core reads the staged tiles itself.
constexpr int kTcM = 128;    // output columns of y per CTA: the MMA's M
constexpr int kTcN = 64;     // rows of h (at most): the MMA's N
// Ring depth: 4 stages (97 KB of shared memory, two CTAs per SM) or 8 (193 KB, one CTA per SM
// with about twice the bytes in flight).
__host__ __device__ constexpr size_t tc_wtile_bytes() { return static_cast<size_t>(kTcM) * kKT * 2; }
__host__ __device__ constexpr size_t tc_htile_bytes() { return static_cast<size_t>(kTcN) * kKT * 2; }
// A stage: the W tile, then h's tile (prologue 3), or the gate and up tiles the activation warps
// turn into h's tile in place (prologue 1 / 2: the GLU fused into the projection), or the W tile
// alone (prologue 0: the RMSNorm fused, h's tiles held apart, `nx` of them, after the ring).
__host__ __device__ constexpr size_t tc_stage_bytes(int pro) {
    return tc_wtile_bytes() + (pro == 0 ? 0 : (pro == 3 ? 1 : 2)) * tc_htile_bytes();
}
__host__ __device__ constexpr size_t tc_smem_bytes(int stages, int pro = 3, int nx = 0) {
    return 1024 + (stages * tc_stage_bytes(pro) + nx * tc_htile_bytes() > static_cast<size_t>(kTcN) * kTcM * 4
                       ? stages * tc_stage_bytes(pro) + nx * tc_htile_bytes()
                       : static_cast<size_t>(kTcN) * kTcM * 4);
}
// Most K tiles a CTA of the fused RMSNorm holds (its whole K range stays in shared memory).
constexpr int kTcNormMaxTiles = 16;

// Threads of the tcgen05 projection: warp 0 issues the MMAs, warp 1 the copies, warps 0-3 read
// the accumulator back (a warp reaches only its quarter of the tensor-memory lanes); with the GLU
// fused, warps 2-9 compute it (two warps on each of the SM's four schedulers: a tile's products
// are short dependent chains, so the time per tile falls with the warps that share it); with the
// RMSNorm fused, all ten warps take the norm before the roles split.
__host__ __device__ constexpr int tc_threads(int pro) { return pro == 3 ? 128 : 320; }  // 0: the norm's threads
constexpr int kTcActWarps = 8;

// silu(g) * u on the fused projection's fast path (gates at or above kSiluFar; the rest take
// glu_mul): sigma(g) = 1 / (1 + 2^(-g log2 e)) from two approximate instructions of the PTX ISA,
// ex2.approx.ftz (relative error about 2^-22) and rcp.approx.ftz (about one ulp). Their operands
// stay in range there: -g log2 e <= 92.4, so 1 + e^-g lies in [1, 2^93); an e^-g that flushes to
// zero (g large) leaves 1, and a subnormal -g log2 e flushed to zero gives e^-g = 1, its value to
// fp32's precision. The products g * sigma * u are ordinary (non-flushing) multiplies.
__device__ __forceinline__ float silu_mul_mufu(float g, float u) {
    float e, r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(g * -1.4426950408889634f));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
    return g * r * u;
}

// PRO 3: h comes from the workspace (its own prologue kernel ran before). PRO 1 / 2: the GLU
// (SwiGLU / ReGLU) is fused: each stage brings the gate and up tiles of this CTA's K range, warps
// 2-9 turn them into h's tile in place (the same 128-byte swizzle, so the element-wise product
// needs no index arithmetic) and release it to the MMA thread on a barrier of its own. PRO 0:
// the RMSNorm is fused: the CTA's x tiles (its whole K range) arrive in a region of their own,
// every thread sums the squares of its share of a row, the cluster's ranks exchange their
// partial sums, and each CTA normalises its tiles in place into h's tiles before the first MMA;
// the ring then streams W alone.
template <typename T, int S, int PRO>
__global__ void __launch_bounds__(tc_threads(PRO)) linear_tc_kernel(LinArgs a, const __grid_constant__ CUtensorMap tmW,
                                                        const __grid_constant__ CUtensorMap tmX) {
    constexpr size_t SB = tc_stage_bytes(PRO);
    constexpr uint32_t kCols = 64;  // tensor-memory columns: one fp32 accumulator column per row of h
    constexpr uint32_t IDESC = tc::idesc_f16(std::is_same<T, __nv_bfloat16>::value, kTcM, kTcN);
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ uint64_t full[S], empty[S], hready[S], accb, xfull;
    __shared__ uint32_t tmem_slot;
    // the fused RMSNorm's row statistics: every rank's partial sums, pushed here by the ranks
    // (stat[q][r]: rank q's sum of row r), this rank's fp64 sums for rows past fp32's range, each
    // row's 1 / rms and pre-scale
    __shared__ float stat[PRO == 0 ? 16 : 1][PRO == 0 ? kTcN : 1], inv[PRO == 0 ? kTcN : 1], prev[PRO == 0 ? kTcN : 1];
    __shared__ double dstat[PRO == 0 ? kTcN : 1];
    __shared__ __align__(16) T wsl[PRO == 0 ? kTcNormMaxTiles * kKT : 8];  // the norm weight of the K range
    cg::cluster_group cluster = cg::this_cluster();
    const int SK = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t n0 = (blockIdx.x / SK) * static_cast<int64_t>(kTcM);
    const int rows = static_cast<int>(a.B < kTcN ? a.B : kTcN);
    const int KT = static_cast<int>(a.K / kKT);
    const int per = (KT + SK - 1) / SK;
    const int kt0 = rank * per < KT ? rank * per : KT;
    const int kt1 = kt0 + per < KT ? kt0 + per : KT;
    const int ntiles = kt1 - kt0;
    const int64_t kbase = static_cast<int64_t>(kt0) * kKT;
    float* part = reinterpret_cast<float*>(smem);  // the K split's reduction, after the ring drains
    unsigned char* xreg = smem + static_cast<size_t>(S) * SB;  // prologue 0: the CTA's x / h tiles
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
            mbar_init(&hready[i], kTcActWarps);  // the activation warps (prologue 1 / 2)
        }
        mbar_init(&accb, 1);
        mbar_init(&xfull, 1);
        mbar_init_fence();
    }
    if (warp == 0) {
        tc::alloc(&tmem_slot, kCols);
        tc::relinquish();
    }
    // (Before the dependency wait at most the first stages are prefetched into L2 below, never the
    // CTA's whole W slice: that measured slower, its traffic competing with the tiles the pipeline
    // needs.)
    __syncthreads();  // barriers initialised, the tensor-memory address in shared memory
    tc::fence_after();
    const uint32_t tmem = tmem_slot;
    // With h from the workspace, the first stages' W tiles are requested before the dependency
    // wait: that kernel runs only right after the prologue kernel of the same call, which writes
    // h, not W, and which itself waited for everything before it in the stream before this kernel
    // could start. (The fused GLU follows whatever the caller ran before: no copies before the wait.)
    // (prologue 0: the first stages are requested right after the wait, with the x tiles)
    const int pre = PRO == 1 || PRO == 2 ? 0 : (ntiles < S ? ntiles : S);
    if (warp == 1 && lane == 0) {
        for (int t = 0; PRO == 3 && t < pre; ++t) {
            mbar_arrive_expect_tx(&full[t], static_cast<uint32_t>(SB));
            tma_load_2d(smem + static_cast<size_t>(t) * SB, &tmW, static_cast<int>(kbase) + t * kKT,
                        static_cast<int>(n0), &full[t]);
        }
        // With the GLU fused, the first stages' W, gate and up boxes are only prefetched into the
        // L2 before the wait (hints, read again after it): their first copies then come from L2.
        if (PRO == 1 || PRO == 2) {
            for (int t = 0; t < S && t < ntiles; ++t) {
                const int k0 = static_cast<int>(kbase) + t * kKT;
                tma_prefetch_2d(&tmW, k0, static_cast<int>(n0));
                tma_prefetch_2d(&tmX, k0, 0);
                tma_prefetch_2d(&tmX, static_cast<int>(a.K) + k0, 0);
            }
        }
        // With the RMSNorm fused: the first stages' W boxes and all of the CTA's x boxes.
        if (PRO == 0) {
            for (int t = 0; t < ntiles; ++t) {
                const int k0 = static_cast<int>(kbase) + t * kKT;
                if (t < S) tma_prefetch_2d(&tmW, k0, static_cast<int>(n0));
                tma_prefetch_2d(&tmX, k0, 0);
            }
        }
    }
    pdl_enter();

    if constexpr (PRO == 0) {
        using V8 = Vec<T, 8>;
        using R8 = typename V8::Raw;
        if (warp == 1 && lane == 0) {
            // the x tiles of the CTA's K range, then the first stages of W
            mbar_arrive_expect_tx(&xfull, static_cast<uint32_t>(ntiles * tc_htile_bytes()));
            for (int t = 0; t < ntiles; ++t)
                tma_load_2d(xreg + static_cast<size_t>(t) * tc_htile_bytes(), &tmX, static_cast<int>(kbase) + t * kKT,
                            0, &xfull);
            for (int t = 0; t < ntiles && t < S; ++t) {
                mbar_arrive_expect_tx(&full[t], static_cast<uint32_t>(SB));
                tma_load_2d(smem + static_cast<size_t>(t) * SB, &tmW, static_cast<int>(kbase) + t * kKT,
                            static_cast<int>(n0), &full[t]);
            }
        }
        // the norm weight of the CTA's K range, staged while the x tiles arrive
        for (int c = static_cast<int>(threadIdx.x); c < ntiles * (kKT / 8); c += tc_threads(0))
            reinterpret_cast<R8*>(wsl)[c] = V8::load(static_cast<const T*>(a.w_ln) + kbase + c * 8);
        mbar_wait(&xfull, 0);
        // Partial sums of squares over the CTA's K range: thread i < 256 takes row i / 4 and its
        // 16-byte chunks i % 4 and i % 4 + 4 of every tile (the 128-byte swizzle moves a row's
        // chunks only within the row's 128 bytes), four lanes meeting by shuffles.
        const int sr = static_cast<int>(threadIdx.x >> 2), sq = static_cast<int>(threadIdx.x & 3);
        if (threadIdx.x < 4 * kTcN) {
            float ss = 0.0f;
            for (int t = 0; t < ntiles; ++t) {
                const unsigned char* rp = xreg + static_cast<size_t>(t) * tc_htile_bytes() + sr * (kKT * 2);
                float f[8], g[8];
                V8::unpack(*reinterpret_cast<const R8*>(rp + sq * 16), f);
                V8::unpack(*reinterpret_cast<const R8*>(rp + (sq + 4) * 16), g);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    ss = fmaf(f[e], f[e], ss);
                    ss = fmaf(g[e], g[e], ss);
                }
            }
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            ss += __shfl_xor_sync(0xffffffffu, ss, 2);
            // into every rank's stat[rank][row] (remote stores: nothing waits for a round trip)
            if (sq == 0)
                for (int q = 0; q < SK; ++q) dsmem_st_f32(dsmem_addr(&stat[rank][sr], static_cast<uint32_t>(q)), ss);
        }
        cluster.sync();  // (release / acquire) every rank's partial sums are in this CTA's stat
        int wide = 0;
        if (threadIdx.x < kTcN) {
            const int r = static_cast<int>(threadIdx.x);
            float tot = 0.0f;
            for (int q = 0; q < SK; ++q) tot += stat[q][r];
            inv[r] = r < rows ? rsqrtf(tot / static_cast<float>(a.K) + a.eps) : 0.0f;
            prev[r] = 1.0f;
            wide = r < rows && !ss_in_range(tot, a.K, a.eps);
        }
        // Every rank adds the same partials in the same order, so `wide` is the same on all the
        // cluster's ranks and the barrier below is reached by all of them or by none.
        if (__syncthreads_or(wide)) {
            // rows whose fp32 sum left fp32's range: the squares again in double, exchanged the same way
            if (threadIdx.x < 4 * kTcN) {
                double sd = 0.0;
                for (int t = 0; t < ntiles; ++t) {
                    const unsigned char* rp = xreg + static_cast<size_t>(t) * tc_htile_bytes() + sr * (kKT * 2);
                    float f[8], g[8];
                    V8::unpack(*reinterpret_cast<const R8*>(rp + sq * 16), f);
                    V8::unpack(*reinterpret_cast<const R8*>(rp + (sq + 4) * 16), g);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        sd += static_cast<double>(f[e]) * f[e] + static_cast<double>(g[e]) * g[e];
                }
                sd += __shfl_xor_sync(0xffffffffu, sd, 1);
                sd += __shfl_xor_sync(0xffffffffu, sd, 2);
                if (sq == 0) dstat[sr] = sd;
            }
            cluster.sync();
            if (threadIdx.x < rows) {
                const int r = static_cast<int>(threadIdx.x);
                float tot = 0.0f;
                for (int q = 0; q < SK; ++q) tot += stat[q][r];
                if (!ss_in_range(tot, a.K, a.eps)) {
                    double sd = 0.0;
                    for (int q = 0; q < SK; ++q) sd += cluster.map_shared_rank(dstat, q)[r];
                    const WideScale sc = wide_scale(sd, a.K, a.eps);
                    inv[r] = sc.rinv, prev[r] = sc.pre;
                }
            }
            __syncthreads();
        }
        // h = x * pre * (1 / rms) * w, rounded to T, in place: chunk p of row r in a tile holds
        // the row's columns 8 (p ^ (r % 8)) ... + 7 of the tile (the 128-byte swizzle). (The
        // barriers above made the staged weight visible.)
        // Thread i < 256 owns the (row, chunk) positions i and i + 256 of every tile (consecutive
        // threads: consecutive 16-byte chunks), so a position's row scale and weight column are
        // found once and the tiles are an inner loop of plain address steps.
        if (threadIdx.x < 4 * kTcN) {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int q = static_cast<int>(threadIdx.x) + h2 * 4 * kTcN, r = q >> 3, pch = q & 7;
                const float iv = inv[r], pv = prev[r];
                unsigned char* hp0 = xreg + r * (kKT * 2) + pch * 16;
                const R8* wp = reinterpret_cast<const R8*>(wsl) + (pch ^ (r & 7));
                for (int t = 0; t < ntiles; ++t) {
                    R8* hp = reinterpret_cast<R8*>(hp0 + static_cast<size_t>(t) * tc_htile_bytes());
                    float f[8], g[8];
                    V8::unpack(*hp, f);
                    V8::unpack(wp[t * (kKT / 8)], g);
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = f[e] * pv * iv * g[e];
                    *hp = V8::pack(f);
                }
            }
        }
        fence_proxy_async();  // h's tiles are read by the tensor core (the async proxy)
        __syncthreads();
    }

    // Lanes 1-31 of the producer and MMA warps wait at the warp barrier (not in a poll loop,
    // which would take the warp's issue slots from lane 0) until lane 0 has left its loop.
    if (warp == 1) {
        if (lane == 0) {
            for (int t = 0; t < ntiles; ++t) {
                const int slot = t % S;
                unsigned char* st = smem + static_cast<size_t>(slot) * SB;
                const int k0 = static_cast<int>(kbase) + t * kKT;
                if (t >= pre) {
                    // the slot's previous stage (t - S) has been read by its MMAs
                    if (t >= S) mbar_wait(&empty[slot], static_cast<uint32_t>(((t / S) - 1) & 1));
                    mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(SB));
                    tma_load_2d(st, &tmW, k0, static_cast<int>(n0), &full[slot]);
                }
                if (PRO != 0) tma_load_2d(st + tc_wtile_bytes(), &tmX, k0, 0, &full[slot]);
                if (PRO == 1 || PRO == 2)
                    tma_load_2d(st + tc_wtile_bytes() + tc_htile_bytes(), &tmX, static_cast<int>(a.K) + k0, 0,
                                &full[slot]);
            }
        }
        __syncwarp();
    } else if (warp == 0) {
        if (lane == 0) {
            for (int t = 0; t < ntiles; ++t) {
                const int slot = t % S;
                mbar_wait(PRO == 1 || PRO == 2 ? &hready[slot] : &full[slot], static_cast<uint32_t>((t / S) & 1));
                tc::fence_after();
                const unsigned char* st = smem + static_cast<size_t>(slot) * SB;
                const unsigned char* hb = PRO == 0 ? xreg + static_cast<size_t>(t) * tc_htile_bytes() : st + tc_wtile_bytes();
#pragma unroll
                for (int k = 0; k < kKT / 16; ++k)
                    tc::mma_f16(tmem, tc::sdesc_sw128(st, 32 * k), tc::sdesc_sw128(hb, 32 * k), IDESC,
                                (t | k) != 0 ? 1u : 0u);
                tc::commit(&empty[slot]);  // the slot is free once these MMAs have read it
            }
            tc::commit(&accb);  // the accumulator is complete once every MMA above has
        }
        __syncwarp();
    } else if (PRO == 1 || PRO == 2) {
        // activation warps 2-9: h = act(gate) * up over each stage's [64 rows][64] tiles, in
        // place of the gate tile; a chunk holding a gate below -64 (never on the configured
        // inputs) goes through glu_mul element by element
        // The thread's 8 gate vectors are read and checked first; unless a lane of the warp found
        // a far-negative gate, the products run in one branch-free unrolled pass (8 independent
        // vectors in flight), else vector by vector with the check.
        using V8 = Vec<T, 8>;
        using R8 = typename V8::Raw;
        constexpr int NA = 32 * kTcActWarps;                                // activation threads
        constexpr int NQ = static_cast<int>(tc_htile_bytes() / 16) / NA;  // vectors per thread
        const int at = threadIdx.x - 64;
        for (int t = 0; t < ntiles; ++t) {
            const int slot = t % S;
            mbar_wait(&full[slot], static_cast<uint32_t>((t / S) & 1));
            unsigned char* st = smem + static_cast<size_t>(slot) * SB + tc_wtile_bytes();
            R8* gt = reinterpret_cast<R8*>(st);
            const R8* ut = reinterpret_cast<const R8*>(st + tc_htile_bytes());
            R8 gv[NQ];
            bool careful = false;
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
                gv[i] = gt[at + NA * i];
                if (PRO == 1) careful |= needs_careful<T, 8>(gv[i]);
            }
            if (PRO == 1 && __any_sync(0xffffffffu, careful)) {
#pragma unroll 1
                for (int i = 0; i < NQ; ++i) {
                    float g[8], u[8];
                    V8::unpack(gv[i], g);
                    V8::unpack(ut[at + NA * i], u);
                    if (needs_careful<T, 8>(gv[i])) {
#pragma unroll 1
                        for (int e = 0; e < 8; ++e) g[e] = glu_mul<PRO - 1>(g[e], u[e]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) g[e] = glu_mul_fast<PRO - 1>(g[e], u[e]);
                    }
                    gt[at + NA * i] = V8::pack(g);
                }
            } else {
#pragma unroll
                for (int i = 0; i < NQ; ++i) {
                    float g[8], u[8];
                    V8::unpack(gv[i], g);
                    V8::unpack(ut[at + NA * i], u);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        g[e] = PRO == 1 ? silu_mul_mufu(g[e], u[e]) : glu_mul_fast<1>(g[e], u[e]);
                    gt[at + NA * i] = V8::pack(g);
                }
            }
            fence_proxy_async();  // the tile is read by the tensor core (the async proxy)
            __syncwarp();
            if (lane == 0) mbar_arrive(&hready[slot]);
        }
    }
    mbar_wait(&accb, 0);
    __syncwarp();  // the warp-wide accumulator loads below need all 32 lanes together
    tc::fence_after();
    // the K split's sum: rank q sums float4s [q share4, (q + 1) share4) of the [rows][128] tile
    const int tot4 = rows * kTcM / 4, share4 = (tot4 + SK - 1) / SK;
    const int end4 = (rank + 1) * share4 < tot4 ? (rank + 1) * share4 : tot4;

    if (a.ws_part) {
        // ---- epilogue through L2: this CTA's partial [64 rows][128 columns] goes straight from
        // tensor memory to the workspace (lane = column: each row a coalesced 128-byte store per
        // warp); after a cluster barrier (release / acquire: the cluster's global stores are
        // visible to its CTAs) each CTA sums 4 adjacent columns at a time over the cluster's
        // partials, every rank's 16-byte load issued before the first add
        float* mine = a.ws_part + (static_cast<int64_t>(blockIdx.x / SK) * SK + rank) * (kTcN * kTcM);
#pragma unroll
        for (int c0 = 0; c0 < kTcN && warp < 4; c0 += 16) {
            uint32_t v[16];
            tc::ld16(tmem + (static_cast<uint32_t>(32 * warp) << 16) + static_cast<uint32_t>(c0), v);
            tc::wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (c0 + j < rows) mine[(c0 + j) * kTcM + 32 * warp + lane] = ntiles > 0 ? __uint_as_float(v[j]) : 0.0f;
        }
        tc::fence_before();
        __syncthreads();
        if (warp == 0) tc::dealloc(tmem, kCols);
        cluster.sync();
        const float* base = a.ws_part + static_cast<int64_t>(blockIdx.x / SK) * SK * (kTcN * kTcM);
        T* y = static_cast<T*>(a.y);
        for (int s4 = rank * share4 + threadIdx.x; s4 < end4; s4 += tc_threads(PRO)) {
            const int r = (4 * s4) / kTcM, c = 4 * s4 - r * kTcM;
            float4 v[16];
#pragma unroll
            for (int q = 0; q < 16; ++q)
                v[q] = q < SK ? __ldcg(reinterpret_cast<const float4*>(base + q * (kTcN * kTcM)) + s4)
                              : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                sum.x += v[q].x;
                sum.y += v[q].y;
                sum.z += v[q].z;
                sum.w += v[q].w;
            }
            const float f[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (n0 + c + e < a.N) y[r * a.ys + n0 + c + e] = to_t<T>(f[e]);
        }
        return;
    }

    // ---- epilogue: warp w (< 4) reads output columns n0 + 32 w + lane, one 16-column (row) group at a time
#pragma unroll
    for (int c0 = 0; c0 < kTcN && warp < 4; c0 += 16) {
        uint32_t v[16];
        tc::ld16(tmem + (static_cast<uint32_t>(32 * warp) << 16) + static_cast<uint32_t>(c0), v);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) part[(c0 + j) * kTcM + 32 * warp + lane] = ntiles > 0 ? __uint_as_float(v[j]) : 0.0f;
    }
    tc::fence_before();
    __syncthreads();  // every accumulator read is done: the tensor memory can go
    if (warp == 0) tc::dealloc(tmem, kCols);
    cluster.sync();
    // the K split's sum: each thread 4 adjacent columns of y at a time, every rank's 16-byte
    // partial requested before the first add (the cluster holds at most 16 ranks)
    T* y = static_cast<T*>(a.y);
    for (int s4 = rank * share4 + threadIdx.x; s4 < end4; s4 += tc_threads(PRO)) {
        const int r = (4 * s4) / kTcM, c = 4 * s4 - r * kTcM;
        // (the fused prologues read the ranks' partials with explicit shared::cluster loads, which
        // measured faster there; the projection of h keeps the generic ones, with which the
        // compiler schedules its L2 path better: 8.2 against 7.7 us for ln1 + qkv_proj at batch 64)
        float4 v[16];
        if constexpr (PRO == 3) {
#pragma unroll
            for (int q = 0; q < 16; ++q)
                v[q] = q < SK ? reinterpret_cast<const float4*>(cluster.map_shared_rank(part, q))[s4]
                              : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        } else {
            const uint32_t pa = smem_u32(reinterpret_cast<const float4*>(part) + s4);
#pragma unroll
            for (int q = 0; q < 16; ++q)
                v[q] = q < SK ? dsmem_ld_f4(dsmem_addr(pa, static_cast<uint32_t>(q))) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            sum.x += v[q].x;
            sum.y += v[q].y;
            sum.z += v[q].z;
            sum.w += v[q].w;
        }
        const float f[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (n0 + c + e < a.N) y[r * a.ys + n0 + c + e] = to_t<T>(f[e]);
    }
    cluster.sync();
}

// ---- decode batches: a cluster of SK CTAs owns 16 columns of y, each CTA a 1 / SK slice of
// K (SK = 1: the whole of K, no cluster); a CTA's eight warps split its slice between them
// (each streaming its own W tiles through a private cp.async ring) and meet at the end in
// shared memory, and the cluster's CTAs then sum their slices' partials through distributed
// shared memory. h for the CTA's slice of K is built once, up front, while the first W tiles
// are in flight: the RMSNorm takes each row's norm over the full row itself (B x K values),
// the GLU activates the slice. Only the B real rows are stored; the A fragments of the
// padding rows read one zero row.
constexpr int kNW16 = 8;       // warps
constexpr int kStages16 = 6;   // W tiles in flight per warp
constexpr int kTile16 = 16 * kKT;  // elements of a W tile (16 columns x 64 of K)

__host__ __device__ inline size_t ring16_bytes() {
    const size_t ring = static_cast<size_t>(kNW16) * kStages16 * kTile16 * 2;
    const size_t part = static_cast<size_t>(kNW16) * 16 * 16 * 4;
    return ring > part ? ring : part;
}
// K elements of h one CTA of an SK-CTA cluster holds (its slice of K tiles, rounded up)
__host__ __device__ inline int64_t kslice16(int64_t K, int SK) { return (K / kKT + SK - 1) / SK * kKT; }
__host__ __device__ inline size_t smem16_bytes(int rows, int64_t K, int SK) {
    return ring16_bytes() + static_cast<size_t>(rows + 1) * kslice16(K, SK) * 2 + 2 * 64 * 4;
}

template <typename T, int PRO>
__global__ void __launch_bounds__(kNW16 * 32) linear16_kernel(LinArgs a) {
    using V8 = Vec<T, 8>;
    using R8 = typename V8::Raw;
    extern __shared__ __align__(16) unsigned char smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int SK = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x / SK) * 16;
    const int rows = static_cast<int>(a.B < 16 ? a.B : 16);
    // this CTA's slice of K: tiles [kt0, kt0 + KT), h columns [kb, kb + KL)
    const int KTall = static_cast<int>(a.K / kKT);
    const int per = (KTall + SK - 1) / SK;
    const int kt0 = rank * per < KTall ? rank * per : KTall;
    const int KT = (kt0 + per < KTall ? kt0 + per : KTall) - kt0;
    const int64_t kb = static_cast<int64_t>(kt0) * kKT, KL = static_cast<int64_t>(KT) * kKT;
    const int64_t HS = kslice16(a.K, SK);  // row stride of h in shared memory
    T* ring = reinterpret_cast<T*>(smem) + static_cast<size_t>(warp) * kStages16 * kTile16;
    float* part = reinterpret_cast<float*>(smem);  // [warps][16][16], after the rings drain
    float* csum = part + kNW16 * 256;              // [16][16] this CTA's sum, for the cluster
    T* hsm = reinterpret_cast<T*>(smem + ring16_bytes());  // [rows][HS], then one zero row
    T* zrow = hsm + static_cast<int64_t>(rows) * HS;
    float* inv = reinterpret_cast<float*>(smem + ring16_bytes() + static_cast<size_t>(rows + 1) * HS * 2);
    float* pre = inv + 64;  // RMSNorm rows past fp32's sum range: a power-of-two pre-scale
    const T* W = static_cast<const T*>(a.W);
    const T* X = static_cast<const T*>(a.x);
    // this warp's tiles: t = warp, warp + 8, ...; j-th of them into ring slot j % stages
    const int mine = KT > warp ? (KT - warp + kNW16 - 1) / kNW16 : 0;
    auto issue = [&](int j) {
        const int t = warp + j * kNW16;
        T* dst = ring + static_cast<size_t>(j % kStages16) * kTile16;
        const T* src = W + n0 * a.K + kb + static_cast<int64_t>(t) * kKT;
#pragma unroll
        for (int c = lane; c < 16 * 8; c += 32) {
            const int r = c >> 3, ch = c & 7;
            cp_async16(dst + r * kKT + swz(r, ch) * 8, src + static_cast<int64_t>(r) * a.K + ch * 8);
        }
    };
    // Before the dependency wait: this CTA's slice of its 16 rows of W and the prologue's input
    // (whole rows for the RMSNorm's norms, the slice of gate and up for the GLU) into L2 (hints
    // only; both are read again after the wait).
    if (threadIdx.x < 16) {
        prefetch_l2(W + (n0 + threadIdx.x) * a.K + kb, KL * 2);
    } else if (threadIdx.x >= 32 && threadIdx.x - 32 < rows) {
        const T* xr = X + (threadIdx.x - 32) * a.xs;
        if (PRO == 0) {
            prefetch_l2(xr, a.K * 2);
        } else {
            prefetch_l2(xr + kb, KL * 2);
            prefetch_l2(xr + a.K + kb, KL * 2);
        }
    }
    pdl_enter();
    for (int j = 0; j < kStages16 - 1; ++j) {
        if (j < mine) issue(j);
        cp_async_commit();
    }

    const int cpr = static_cast<int>(KL / 8);  // 16-byte chunks of a row's slice
    for (int c = threadIdx.x; c < cpr; c += kNW16 * 32) reinterpret_cast<uint4*>(zrow)[c] = make_uint4(0, 0, 0, 0);
    if constexpr (PRO == 0) {
        // full-row sums of squares: a warp per row, four 16-byte loads per lane in flight
        for (int r = warp; r < rows; r += kNW16) {
            const T* xr = X + r * a.xs;
            float ss = 0.0f;
            for (int64_t k0 = lane * 8; k0 < a.K; k0 += 4 * 256) {
                R8 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (k0 + u * 256 < a.K) v[u] = V8::load(xr + k0 + u * 256);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (k0 + u * 256 < a.K) {
                        float f[8];
                        V8::unpack(v[u], f);
#pragma unroll
                        for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
                    }
                }
            }
            ss = warp_sum(ss);
            float iv = rsqrtf(ss / static_cast<float>(a.K) + a.eps), pv = 1.0f;
            if (!ss_in_range(ss, a.K, a.eps)) {  // the row again, in double
                double sd = 0.0;
                for (int64_t k0 = lane * 8; k0 < a.K; k0 += 256) {
                    float f[8];
                    V8::unpack(V8::load(xr + k0), f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) sd += static_cast<double>(f[e]) * static_cast<double>(f[e]);
                }
                const WideScale sc = wide_scale(warp_sum_d(sd), a.K, a.eps);
                iv = sc.rinv, pv = sc.pre;
            }
            if (lane == 0) inv[r] = iv, pre[r] = pv;
        }
        __syncthreads();
    }
    // h for the slice: thread chunks c = tid + 256 u, the inputs of HB chunks loaded together
    constexpr int HB = 8;
    const int total = rows * cpr;
    for (int c0 = threadIdx.x; c0 < total; c0 += HB * kNW16 * 32) {
        R8 xv[HB], gv[HB];
#pragma unroll
        for (int u = 0; u < HB; ++u) {
            const int c = c0 + u * kNW16 * 32;
            if (c < total) {
                const int r = c / cpr, ch = c - r * cpr;
                const T* xr = X + r * a.xs + kb + ch * 8;
                xv[u] = V8::load(xr);
                gv[u] = PRO == 0 ? V8::load(static_cast<const T*>(a.w_ln) + kb + ch * 8) : V8::load(xr + a.K);
            }
        }
#pragma unroll
        for (int u = 0; u < HB; ++u) {
            const int c = c0 + u * kNW16 * 32;
            if (c < total) {
                const int r = c / cpr, ch = c - r * cpr;
                if constexpr (PRO == 1) {
                    // a chunk holding a gate below -64 (never on the configured inputs): each
                    // element through glu_mul, scalar, re-read from x
                    if (__builtin_expect(needs_careful<T, 8>(xv[u]), 0)) {
                        const T* xr = X + r * a.xs + kb + ch * 8;
                        T* hp = hsm + static_cast<int64_t>(r) * HS + swz(r, ch) * 8;
#pragma unroll 1
                        for (int e = 0; e < 8; ++e) hp[e] = to_t<T>(glu_mul<0>(to_f32(xr[e]), to_f32(xr[e + a.K])));
                        continue;
                    }
                }
                float f[8], g[8];
                V8::unpack(xv[u], f);
                V8::unpack(gv[u], g);
                if constexpr (PRO == 0) {
                    const float iv = inv[r], pv = pre[r];
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = f[e] * pv * iv * g[e];
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = glu_mul_fast<PRO - 1>(f[e], g[e]);
                }
                *reinterpret_cast<R8*>(hsm + static_cast<int64_t>(r) * HS + swz(r, ch) * 8) = V8::pack(f);
            }
        }
    }
    __syncthreads();

    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const int li = lane & 7, lm = lane >> 3;
    const int ar = (lm & 1) * 8 + li;  // this lane's A row in ldmatrix
    const T* arow = ar < rows ? hsm + static_cast<int64_t>(ar) * HS : zrow;
    for (int j = 0; j < mine; ++j) {
        const int t = warp + j * kNW16;
        cp_async_wait<kStages16 - 2>();
        __syncwarp();
        if (j + kStages16 - 1 < mine) issue(j + kStages16 - 1);
        cp_async_commit();
        const T* wt = ring + static_cast<size_t>(j % kStages16) * kTile16;
#pragma unroll
        for (int ks = 0; ks < kKT / 16; ++ks) {
            uint32_t af[4], bf[4];
            const int ach = (t * kKT + ks * 16) / 8 + (lm >> 1);
            ldsm_x4(af, arow + (ar < rows ? swz(ar, ach) : ach) * 8);
            const int n = (lm >> 1) * 8 + li;
            ldsm_x4(bf, wt + n * kKT + swz(n, ks * 2 + (lm & 1)) * 8);
            Mma<T>::run(acc[0], af, bf[0], bf[1]);
            Mma<T>::run(acc[1], af, bf[2], bf[3]);
        }
    }
    cp_async_wait<0>();
    __syncthreads();  // every warp is done with its ring: the space takes the partial tiles
    {
        const int g = lane >> 2, q = lane & 3;
        float* pw = part + warp * 256;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            pw[g * 16 + j * 8 + 2 * q] = acc[j][0];
            pw[g * 16 + j * 8 + 2 * q + 1] = acc[j][1];
            pw[(g + 8) * 16 + j * 8 + 2 * q] = acc[j][2];
            pw[(g + 8) * 16 + j * 8 + 2 * q + 1] = acc[j][3];
        }
    }
    __syncthreads();
    T* y = static_cast<T*>(a.y);
    for (int idx = threadIdx.x; idx < rows * 16; idx += kNW16 * 32) {
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < kNW16; ++w) sum += part[w * 256 + idx];
        if (SK == 1)
            y[(idx >> 4) * a.ys + n0 + (idx & 15)] = to_t<T>(sum);
        else
            csum[idx] = sum;
    }
    if (SK == 1) return;
    // the cluster's slices of K: each CTA sums every SK-th output over the ranks, in rank order
    cluster.sync();
    for (int idx = rank + SK * static_cast<int>(threadIdx.x); idx < rows * 16; idx += SK * kNW16 * 32) {
        float sum = 0.0f;
        for (int q = 0; q < SK; ++q) sum += cluster.map_shared_rank(csum, q)[idx];
        y[(idx >> 4) * a.ys + n0 + (idx & 15)] = to_t<T>(sum);
    }
    cluster.sync();  // every CTA's sums have been read
}

template <typename T, int PRO>
cudaError_t launch16(const LinArgs& a, const LinPlan& p, cudaStream_t s) {
    auto kernel = linear16_kernel<T, PRO>;
    const int SK = p.splits;  // CTAs of a cluster along K
    const size_t smem = smem16_bytes(static_cast<int>(a.B < 16 ? a.B : 16), a.K, SK);
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_kernel(kernel, dim3(static_cast<unsigned>(a.N / 16 * SK)), dim3(kNW16 * 32), smem, s, p.pdl, SK,
                         a);
}

template <typename T, int MT, int PRO>
cudaError_t launch_mt(const LinArgs& a, const LinPlan& p, cudaStream_t s, const CUtensorMap& tmW,
                      const CUtensorMap& tmX, const CUtensorMap& tmN) {
    auto kernel = linear_kernel<T, MT, PRO>;
    const size_t smem = smem_bytes(MT, PRO);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>(a.N / kNT * p.splits), static_cast<unsigned>((a.B + MT * 16 - 1) / (MT * 16)));
    return launch_kernel(kernel, grid, dim3(warps_for(MT) * 32), smem, s, p.pdl, p.splits, a, tmW, tmX, tmN);
}

template <typename T, int MT>
cudaError_t launch_h_mt(const LinArgs& a, const LinPlan& p, cudaStream_t s, const CUtensorMap& tmW,
                        const CUtensorMap& tmX) {
    auto kernel = linear_h_kernel<T, MT>;
    const size_t smem = smemh_bytes(MT);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>(a.N / kNT * p.splits), static_cast<unsigned>((a.B + MT * 16 - 1) / (MT * 16)));
    return launch_kernel(kernel, grid, dim3((warps_for(MT) + 1) * 32), smem, s, p.pdl, p.splits, a, tmW, tmX);
}

template <typename T, int STAGES, int PRO>
cudaError_t launch_tc(const LinArgs& a, const LinPlan& p, cudaStream_t s) {
    // W [N][K] in [128][64] boxes and h [B][K] (or gate_up [B][2K]) in [64][64] boxes, both with
    // the 128-byte swizzle
    const bool bf16 = std::is_same<T, __nv_bfloat16>::value;
    CUtensorMap tmW, tmX;
    if (!encode_tmap_16(&tmW, a.W, 2, a.K, a.N, a.K * 2, kKT, kTcM, bf16, true) ||
        !encode_tmap_16(&tmX, a.x, 2, PRO == 1 || PRO == 2 ? 2 * a.K : a.K, a.B, a.xs * 2, kKT, kTcN, bf16, true))
        return cudaErrorNotSupported;
    auto kernel = linear_tc_kernel<T, STAGES, PRO>;
    // prologue 0 holds the CTA's K range of x beside the ring: its size follows the split
    const int64_t KT = a.K / kKT;
    auto smem_for = [&](int sk) {
        return tc_smem_bytes(STAGES, PRO, PRO == 0 ? static_cast<int>((KT + sk - 1) / sk) : 0);
    };
    if (PRO == 0 && (KT + p.splits - 1) / p.splits > kTcNormMaxTiles) return cudaErrorInvalidValue;
    size_t smem = smem_for(p.splits);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int splits = p.splits;
    if (splits > 8) {
        // a cluster of more than 8 CTAs is a non-portable size: use it only where the device can place one
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        int clusters = 0;
        if (e == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = static_cast<unsigned>(splits);
            attr.val.clusterDim.y = attr.val.clusterDim.z = 1;
            cfg.gridDim = dim3(static_cast<unsigned>(splits));
            cfg.blockDim = dim3(tc_threads(PRO));
            cfg.dynamicSmemBytes = smem;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
        }
        if (e != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            splits = 8;
            if (PRO == 0) {
                if ((KT + splits - 1) / splits > kTcNormMaxTiles) return cudaErrorInvalidValue;
                smem = smem_for(splits);
                e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
                if (e != cudaSuccess) return e;
            }
        }
    }
    const dim3 grid(static_cast<unsigned>((a.N + kTcM - 1) / kTcM * splits));
    return launch_kernel(kernel, grid, dim3(tc_threads(PRO)), smem, s, p.pdl, splits, a, tmW, tmX);
}

template <typename T, int PRO>
cudaError_t launch_pro(const LinArgs& a, const LinPlan& p, cudaStream_t s) {
    // tensor maps: W [N][K] and the input rows [B][K or 2K] in 64 x (64 or MT*16) boxes with the
    // 128-byte swizzle, the norm weight [K] in 64-entry boxes
    const bool bf16 = sizeof(T) == 2 && std::is_same<T, __nv_bfloat16>::value;
    const uint32_t xr = static_cast<uint32_t>(p.mt) * 16;
    CUtensorMap tmW, tmX, tmN;
    memset(&tmN, 0, sizeof(tmN));
    if (!encode_tmap_16(&tmW, a.W, 2, a.K, a.N, a.K * 2, kKT, kNT, bf16, true) ||
        !encode_tmap_16(&tmX, a.x, 2, glu_input(PRO) ? 2 * a.K : a.K, a.B, a.xs * 2, kKT, xr, bf16, true) ||
        (PRO == 0 && !encode_tmap_16(&tmN, a.w_ln, 1, a.K, 1, 0, kKT, 1, bf16, false)))
        return cudaErrorNotSupported;
    if constexpr (PRO == 3) {
        switch (p.mt) {
            case 1: return launch_h_mt<T, 1>(a, p, s, tmW, tmX);
            case 2: return launch_h_mt<T, 2>(a, p, s, tmW, tmX);
            case 4: return launch_h_mt<T, 4>(a, p, s, tmW, tmX);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (p.mt) {
        case 1: return launch_mt<T, 1, PRO>(a, p, s, tmW, tmX, tmN);
        case 2: return launch_mt<T, 2, PRO>(a, p, s, tmW, tmX, tmN);
        case 4: return launch_mt<T, 4, PRO>(a, p, s, tmW, tmX, tmN);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t launch_typed(const LinArgs& a, const LinPlan& p, cudaStream_t s) {
    if (p.tcgen05) {
        switch (p.prologue) {
            case 0: return launch_tc<T, 4, 0>(a, p, s);  // the RMSNorm fused: a 4-stage W ring
            case 1: return launch_tc<T, 3, 1>(a, p, s);  // the GLU fused: 3 stages of 32 KB, two CTAs per SM
            case 2: return launch_tc<T, 3, 2>(a, p, s);
            case 3: return p.tc_stages == 8 ? launch_tc<T, 8, 3>(a, p, s) : launch_tc<T, 4, 3>(a, p, s);
            default: return cudaErrorInvalidValue;
        }
    }
    if (p.narrow) {
        switch (p.prologue) {
            case 0: return launch16<T, 0>(a, p, s);
            case 1: return launch16<T, 1>(a, p, s);
            case 2: return launch16<T, 2>(a, p, s);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (p.prologue) {
        case 0: return launch_pro<T, 0>(a, p, s);
        case 1: return launch_pro<T, 1>(a, p, s);
        case 2: return launch_pro<T, 2>(a, p, s);
        case 3: return launch_pro<T, 3>(a, p, s);
        default: return cudaErrorInvalidValue;
    }
}

// ---- the general path (fp32, unaligned layouts, K or N not a multiple of 64): CUDA cores.
// CTA (column chunk, row): the row's h (rounded to T) in shared memory as fp32, then one
// warp per output column, lanes striding over K.
template <typename T, int PRO>
__global__ void __launch_bounds__(128) linear_simple_kernel(LinArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    float* h = reinterpret_cast<float*>(smem);
    __shared__ float red[33];
    __shared__ double dred[33];
    const int64_t b = blockIdx.y;
    const T* xr = static_cast<const T*>(a.x) + b * a.xs;
    pdl_enter();
    if constexpr (PRO == 0) {
        float ss = 0.0f;
        for (int64_t k = threadIdx.x; k < a.K; k += blockDim.x) {
            const float v = to_f32(xr[k]);
            ss = fmaf(v, v, ss);
        }
        ss = block_sum(ss, red);
        float iv = rsqrtf(ss / static_cast<float>(a.K) + a.eps), pv = 1.0f;
        if (!ss_in_range(ss, a.K, a.eps)) {  // the row again, in double
            double sd = 0.0;
            for (int64_t k = threadIdx.x; k < a.K; k += blockDim.x) {
                const double v = to_f32(xr[k]);
                sd += v * v;
            }
            const WideScale sc = wide_scale(block_sum_d(sd, dred), a.K, a.eps);
            iv = sc.rinv, pv = sc.pre;
        }
        const T* wl = static_cast<const T*>(a.w_ln);
        for (int64_t k = threadIdx.x; k < a.K; k += blockDim.x)
            h[k] = round_trip<T>(to_f32(xr[k]) * pv * iv * to_f32(wl[k]));
    } else {
        for (int64_t k = threadIdx.x; k < a.K; k += blockDim.x)
            h[k] = round_trip<T>(glu_mul<PRO - 1>(to_f32(xr[k]), to_f32(xr[k + a.K])));
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const T* W = static_cast<const T*>(a.W);
    for (int64_t n = blockIdx.x * 128 + warp; n < a.N && n < (blockIdx.x + 1) * 128; n += 4) {
        float acc = 0.0f;
        for (int64_t k = lane; k < a.K; k += 32) acc = fmaf(h[k], to_f32(W[n * a.K + k]), acc);
        acc = warp_sum(acc);
        if (lane == 0) static_cast<T*>(a.y)[b * a.ys + n] = from_f32<T>(acc);
    }
}

template <typename T, int PRO>
cudaError_t launch_simple(const LinArgs& a, const LinPlan& p, cudaStream_t s) {
    auto kernel = linear_simple_kernel<T, PRO>;
    const size_t smem = static_cast<size_t>(a.K) * 4;
    if (smem > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    const dim3 grid(static_cast<unsigned>((a.N + 127) / 128), static_cast<unsigned>(a.B));
    return launch_kernel(kernel, grid, dim3(128), smem, s, p.pdl, 1, a);
}

template <typename T>
cudaError_t launch_simple_typed(const LinArgs& a, const LinPlan& p, cudaStream_t s) {
    switch (p.prologue) {
        case 0: return launch_simple<T, 0>(a, p, s);
        case 1: return launch_simple<T, 1>(a, p, s);
        case 2: return launch_simple<T, 2>(a, p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lin

namespace {
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeFn encoder() {
    static const EncodeFn encode = [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return static_cast<EncodeFn>(nullptr);
        }
        return reinterpret_cast<EncodeFn>(fn);
    }();
    return encode;
}
}  // namespace

bool encode_tmap_16_nd(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                       const uint32_t* box, bool bf16, bool swizzle128) {
    const EncodeFn encode = encoder();
    if (!encode || rank < 1 || rank > 4) return false;
    cuuint64_t d[4], st[3];
    cuuint32_t bx[4], estr[4];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        estr[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    return encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, st, bx, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_16(CUtensorMap* map, const void* base, int rank, uint64_t dim0, uint64_t dim1, uint64_t stride1,
                    uint32_t box0, uint32_t box1, bool bf16, bool swizzle128) {
    if (rank < 1 || rank > 2) return false;
    const uint64_t dims[2] = {dim0, dim1}, strides[1] = {stride1};
    const uint32_t box[2] = {box0, box1};
    return encode_tmap_16_nd(map, base, rank, dims, strides, box, bf16, swizzle128);
}

namespace lin {
// One thread waits on a barrier that nothing arrives at: the bounded wait has to give up,
// count the timeout and return, leaving the GPU usable.
__global__ void wait_selftest_kernel(int32_t* out) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0) out[0] = mbar_wait(&bar, 0) ? 1 : 0;
}
}  // namespace lin

cudaError_t launch_wait_selftest(int32_t* out, cudaStream_t s) {
    lin::wait_selftest_kernel<<<1, 32, 0, s>>>(out);
    return cudaGetLastError();
}

unsigned int linear_wait_timeouts() {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_wait_timeouts, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return v;
}

size_t linear_smem(int mt, int prologue) {
    return prologue == 3 ? lin::smemh_bytes(mt) : lin::smem_bytes(mt, prologue);
}
size_t linear16_smem(int rows, int64_t K, int splits) { return lin::smem16_bytes(rows, K, splits); }
size_t linear_tc_smem(int stages, int prologue, int nx) { return lin::tc_smem_bytes(stages, prologue, nx); }

// CTAs of the tcgen05 projection with the RMSNorm fused (nx x tiles held) one SM holds at once
// (its static shared memory included), kept per (device, dtype, nx).
int linear_tc_norm_ctas_per_sm(int nx, bool bf16) {
    static std::atomic<int> memo[16][2][lin::kTcNormMaxTiles + 1];
    static std::once_flag once;
    std::call_once(once, [] {
        for (auto& a : memo)
            for (auto& b : a)
                for (auto& c : b) c.store(-1);
    });
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (nx < 0 || nx > lin::kTcNormMaxTiles) return 0;
    std::atomic<int>* slot = dev >= 0 && dev < 16 ? &memo[dev][bf16 ? 1 : 0][nx] : nullptr;
    if (slot && slot->load() >= 0) return slot->load();
    const size_t smem = lin::tc_smem_bytes(4, 0, nx);
    int n = 0;
    auto query = [&](auto kernel) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
                cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, lin::tc_threads(0), smem) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
    };
    bf16 ? query(lin::linear_tc_kernel<__nv_bfloat16, 4, 0>) : query(lin::linear_tc_kernel<__half, 4, 0>);
    if (slot) slot->store(n);
    return n;
}

// Clusters of `splits` CTAs of the tcgen05 projection (ring of `stages`) the device can hold at once.
int linear_tc_max_clusters(int splits, int stages, bool bf16, int prologue, int nx) {
    // answers kept per (device, dtype, kernel kind, x tiles held, cluster size): the query sets
    // kernel attributes. Kinds: 0 / 1 the 4 / 8-stage projection of h, 2 the GLU fused, 3 the
    // RMSNorm fused (with nx of its x tiles beside the ring)
    static std::atomic<int> memo[16][2][4][lin::kTcNormMaxTiles + 1][17];
    static std::once_flag once;
    std::call_once(once, [] {
        for (auto& a : memo)
            for (auto& b : a)
                for (auto& c : b)
                    for (auto& d : c)
                        for (auto& e : d) e.store(-1);
    });
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (splits < 1 || splits > 16) return 0;
    if (prologue != 0) nx = 0;
    if (nx < 0 || nx > lin::kTcNormMaxTiles) return 0;
    const int kind = prologue == 0 ? 3 : (prologue != 3 ? 2 : (stages == 8 ? 1 : 0));
    std::atomic<int>* slot = dev >= 0 && dev < 16 ? &memo[dev][bf16 ? 1 : 0][kind][nx][splits] : nullptr;
    if (slot && slot->load() >= 0) return slot->load();
    const size_t smem = kind == 3 ? lin::tc_smem_bytes(4, 0, nx)
                                  : lin::tc_smem_bytes(kind == 2 ? 3 : stages, prologue != 3 ? 1 : 3);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = static_cast<unsigned>(splits);
    attr.val.clusterDim.y = attr.val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(splits));
    cfg.blockDim = dim3(lin::tc_threads(prologue == 3 ? 3 : prologue));
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    auto query = [&](auto kernel) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
                cudaSuccess ||
            (splits > 8 && cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                               cudaSuccess) ||
            cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
    };
    if (kind == 3)
        bf16 ? query(lin::linear_tc_kernel<__nv_bfloat16, 4, 0>) : query(lin::linear_tc_kernel<__half, 4, 0>);
    else if (kind == 2)
        bf16 ? query(lin::linear_tc_kernel<__nv_bfloat16, 3, 1>) : query(lin::linear_tc_kernel<__half, 3, 1>);
    else if (kind == 1)
        bf16 ? query(lin::linear_tc_kernel<__nv_bfloat16, 8, 3>) : query(lin::linear_tc_kernel<__half, 8, 3>);
    else
        bf16 ? query(lin::linear_tc_kernel<__nv_bfloat16, 4, 3>) : query(lin::linear_tc_kernel<__half, 4, 3>);
    if (slot) slot->store(n);
    return n;
}

cudaError_t launch_linear(const LinArgs& a, const LinPlan& p, int dtype, cudaStream_t s) {
    if (!p.tensor_cores) {
        switch (dtype) {
            case DT_F32: return lin::launch_simple_typed<float>(a, p, s);
            case DT_F16: return lin::launch_simple_typed<__half>(a, p, s);
            case DT_BF16: return lin::launch_simple_typed<__nv_bfloat16>(a, p, s);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (dtype) {
        case DT_F16: return lin::launch_typed<__half>(a, p, s);
        case DT_BF16: return lin::launch_typed<__nv_bfloat16>(a, p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sra
