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
// Variants (chosen per shape by the host planner; 16-byte layouts):
//   warp_rows  a warp per row, the row in registers          (short rows, many)
//   cta_row    a CTA per row, the row in registers           (long rows; decode)
//   cta_pair   a 2-CTA cluster per row, half the row in each CTA's registers;
//              the partial sums of squares meet through distributed shared
//              memory (wide rows that one CTA per row cannot spread evenly)
//   warp_smem, cta_smem, pair_smem
//              the same three row groupings with the row landed in shared memory
//              by cp.async (16-byte asynchronous copies that hold no registers in
//              flight; cp.async.wait_all is a hardware wait, not a software spin),
//              the weight slice copied in the same round trip; the resident row
//              count is then bounded by shared memory instead of registers
//   two_pass   a CTA per row, the scale pass re-reads the row (any width)
//   warps_row  G = 2, 4 or 8 warps per row, the row in registers and w read in
//              the scale loop; the warps' partial sums meet in shared memory
//              behind a named barrier of just those G warps (rows of 513 to
//              2048 accesses at a few hundred rows: no CTA-wide barrier, and
//              the rows dealt evenly over all SMs)
// Layouts that are not 16-byte aligned use scalar register kernels.
// A predicated scalar tail covers D % VEC; nothing is padded to a power of two.
// Every thread reads back and writes only its own elements, so in-place use
// (out == x) is safe. A row whose fp32 sum of squares overflows, or is too small
// for fp32 to hold its digits (ss_in_range, common.cuh), is summed again in
// double from the values the thread already holds, and scaled by wide_scale's
// power of two `pre` and fp32 `rinv` (out = ((x * pre) * rinv) * w; pre is 1 on
// every other row): the same result the exact formula gives, for every finite
// input. Each translation unit instantiates one ADD value only (norm_rms.cu:
// false, norm_add.cu: true), so no kernel is registered from two modules.
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

// How a row's sum of squares is reduced, and which threads share a row.
enum Reduce { RED_WARP = 0, RED_CTA = 1, RED_PAIR = 2, RED_GROUP = 3 };

// Barrier of the G warps of this warp's group (id 1 + group; id 0 is the CTA's).
template <int G>
__device__ __forceinline__ void group_barrier() {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + static_cast<int>(threadIdx.x >> 5) / G), "r"(32 * G) : "memory");
}

__host__ __device__ constexpr size_t round16(size_t b) { return (b + 15) / 16 * 16; }

// Sum of squares of one row reduced over the group; every thread gets it.
// RED_GROUP (G warps per row): each warp's sum goes to its slot of the row's
// parity, scratch[32 * parity + warp]; one barrier of the group publishes them.
// The next row writes the other parity's slots, and the row after that can only
// reach its own writes once every warp of the group has passed the next row's
// barrier, i.e. has read this row's slots: one barrier per row suffices.
template <int RED, int G = 1>
__device__ __forceinline__ float group_sum(float ss, float* scratch, float* pair_slot, int parity) {
    if constexpr (RED == RED_WARP) {
        return warp_sum(ss);
    } else if constexpr (RED == RED_GROUP) {
        const int warp = static_cast<int>(threadIdx.x >> 5), first = warp / G * G;
        ss = warp_sum(ss);
        if ((threadIdx.x & 31) == 0) scratch[32 * parity + warp] = ss;
        group_barrier<G>();
        float tot = 0.0f;
#pragma unroll
        for (int i = 0; i < G; ++i) tot += scratch[32 * parity + first + i];  // the same order in every warp
        return tot;
    } else if constexpr (RED == RED_CTA) {
        return block_sum(ss, scratch);
    } else {
        // Each CTA's partial goes to its own slot (double-buffered by row parity so
        // the next row cannot overwrite a value the peer has yet to read); the
        // cluster barrier publishes both; each CTA adds the peer's.
        const float part = block_sum(ss, scratch);
        cg::cluster_group cl = cg::this_cluster();
        if (threadIdx.x == 0) pair_slot[parity] = part;
        cl.sync();
        const float peer = *cl.map_shared_rank(pair_slot + parity, static_cast<int>(cl.block_rank()) ^ 1);
        return part + peer;  // the same value on both CTAs (addition commutes exactly)
    }
}

// The same in double (rare rows only). `scratch` is the float scratch of
// group_sum, 8-byte aligned and >= 66 floats; `pair_slot` >= 6 floats (the
// doubles live in its floats 2..5, double-buffered by row parity).
// RED_GROUP: `pair_slot` holds 32 doubles, one per warp; the next use of a slot
// comes after at least one more group_sum barrier, which every warp passes only
// after reading this one.
template <int RED, int G = 1>
__device__ __forceinline__ double group_sum_d(double v, float* scratch, float* pair_slot, int parity) {
    if constexpr (RED == RED_WARP) {
        return warp_sum_d(v);
    } else if constexpr (RED == RED_GROUP) {
        double* slot = reinterpret_cast<double*>(pair_slot);
        const int warp = static_cast<int>(threadIdx.x >> 5), first = warp / G * G;
        v = warp_sum_d(v);
        if ((threadIdx.x & 31) == 0) slot[warp] = v;
        group_barrier<G>();
        double tot = 0.0;
#pragma unroll
        for (int i = 0; i < G; ++i) tot += slot[first + i];
        return tot;
    } else if constexpr (RED == RED_CTA) {
        return block_sum_d(v, reinterpret_cast<double*>(scratch));
    } else {
        const double part = block_sum_d(v, reinterpret_cast<double*>(scratch));
        double* slot = reinterpret_cast<double*>(pair_slot + 2);
        cg::cluster_group cl = cg::this_cluster();
        if (threadIdx.x == 0) slot[parity] = part;
        cl.sync();
        const double peer = *cl.map_shared_rank(slot + parity, static_cast<int>(cl.block_rank()) ^ 1);
        return part + peer;
    }
}

__device__ __forceinline__ double sq_d(float v) { return static_cast<double>(v) * static_cast<double>(v); }

// ------------------------------------------------------------------ staged
// T with 16-byte accesses (VEC = 16 / sizeof(T)). Shared memory:
//   [ws: the w slice if a.stage_w] [per group: x slice][per group: res slice (ADD)]
// each slice round16(slice_accesses * 16) bytes.
template <typename T, bool ADD, int RED>
__global__ void __launch_bounds__(1024) staged_rows_kernel(NormArgs a) {
    constexpr int VEC = vec16<T>();
    using V = Vec<T, VEC>;
    extern __shared__ __align__(16) unsigned char dyn_smem[];
    __shared__ __align__(8) float scratch[66];
    __shared__ __align__(8) float pair_slot[6];
    pdl_enter();

    const int64_t nvec = a.D / VEC;
    int rank = 0;
    if constexpr (RED == RED_PAIR) rank = static_cast<int>(cg::this_cluster().block_rank());
    const int64_t half = norm_pair_half(nvec);
    const int64_t a0 = (RED == RED_PAIR && rank == 1) ? half : 0;
    const int64_t a1 = (RED == RED_PAIR && rank == 0) ? half : nvec;
    const int64_t slice_max = RED == RED_PAIR ? half : nvec;
    const size_t slice_bytes = round16(static_cast<size_t>(slice_max) * 16);
    const int tail = (RED != RED_PAIR || rank == 1) ? static_cast<int>(a.D - nvec * VEC) : 0;

    int tid, threads, group, groups;
    if constexpr (RED == RED_WARP) {
        tid = threadIdx.x & 31, threads = 32, group = threadIdx.x >> 5, groups = blockDim.x >> 5;
    } else {
        tid = threadIdx.x, threads = blockDim.x, group = 0, groups = 1;
    }
    int64_t r0, step;
    if constexpr (RED == RED_WARP) {
        // rows dealt to CTAs round-robin: CTAs (and SMs) differ by one row at most
        r0 = static_cast<int64_t>(group) * gridDim.x + blockIdx.x, step = static_cast<int64_t>(gridDim.x) * groups;
    } else if constexpr (RED == RED_CTA) {
        r0 = blockIdx.x, step = gridDim.x;
    } else {
        r0 = blockIdx.x / 2, step = gridDim.x / 2;
    }

    const bool stage_w = a.stage_w != 0;
    T* ws = reinterpret_cast<T*>(dyn_smem);
    unsigned char* gbase = dyn_smem + (stage_w ? slice_bytes : 0) + group * slice_bytes * (ADD ? 2 : 1);
    T* xs = reinterpret_cast<T*>(gbase);
    T* rs = reinterpret_cast<T*>(gbase + slice_bytes);
    const T* w = static_cast<const T*>(a.w);

    auto issue_row = [&](int64_t r) {
        const T* xr = static_cast<const T*>(a.x) + r * a.xs;
        const T* rr = static_cast<const T*>(a.res) + r * a.rs;
        for (int64_t idx = a0 + tid; idx < a1; idx += threads) {
            cp_async16(xs + (idx - a0) * VEC, xr + idx * VEC);
            if constexpr (ADD) cp_async16(rs + (idx - a0) * VEC, rr + idx * VEC);
        }
    };

    // The D % VEC trailing elements travel by plain loads, issued with the copies.
    float xt = 0.0f, rt = 0.0f, wt = 0.0f;
    auto load_tail = [&](int64_t r) {
        if (tid < tail) {
            const int64_t j = nvec * VEC + tid;
            xt = to_f32(static_cast<const T*>(a.x)[r * a.xs + j]);
            if constexpr (ADD) rt = to_f32(static_cast<const T*>(a.res)[r * a.rs + j]);
            wt = to_f32(w[j]);
        }
    };

    // Prologue: the w slice and this group's first row are in flight together.
    if (stage_w) {
        for (int64_t i = threadIdx.x; i < a1 - a0; i += blockDim.x) cp_async16(ws + i * VEC, w + (a0 + i) * VEC);
    }
    if (r0 < a.rows) {
        issue_row(r0);
        load_tail(r0);
    }
    cp_async_wait_all();
    __syncthreads();  // every thread's w chunks are visible to the whole CTA

    int parity = 0;
    for (int64_t r = r0; r < a.rows; r += step) {
        if (r != r0) {
            issue_row(r);
            load_tail(r);
            cp_async_wait_all();  // this thread's own chunks only: no barrier needed
        }
        T* xr = static_cast<T*>(a.x) + r * a.xs;
        T* orow = static_cast<T*>(a.out) + r * a.os;

        float ss = 0.0f;
        for (int64_t idx = a0 + tid; idx < a1; idx += threads) {
            float xf[VEC];
            V::unpack(V::load(xs + (idx - a0) * VEC), xf);
            if constexpr (ADD) {
                float rf[VEC];
                V::unpack(V::load(rs + (idx - a0) * VEC), rf);
#pragma unroll
                for (int i = 0; i < VEC; ++i) xf[i] += rf[i];
                const typename V::Raw p = V::pack(xf);  // the rounded sum
                V::store(xr + idx * VEC, p);
                V::store(xs + (idx - a0) * VEC, p);
                V::unpack(p, xf);
            }
#pragma unroll
            for (int i = 0; i < VEC; ++i) ss = fmaf(xf[i], xf[i], ss);
        }
        if (tid < tail) {
            if constexpr (ADD) {
                const T s = from_f32<T>(xt + rt);
                xr[nvec * VEC + tid] = s;
                xt = to_f32(s);
            }
            ss = fmaf(xt, xt, ss);
        }
        ss = group_sum<RED>(ss, scratch, pair_slot, parity);
        float rinv = rsqrtf(ss / static_cast<float>(a.D) + a.eps), pre = 1.0f;
        if (__builtin_expect(!ss_in_range(ss, a.D, a.eps), 0)) {
            double sd = tid < tail ? sq_d(xt) : 0.0;
            for (int64_t idx = a0 + tid; idx < a1; idx += threads) {
                float xf[VEC];
                V::unpack(V::load(xs + (idx - a0) * VEC), xf);
#pragma unroll
                for (int i = 0; i < VEC; ++i) sd += sq_d(xf[i]);
            }
            const WideScale sc = wide_scale(group_sum_d<RED>(sd, scratch, pair_slot, parity), a.D, a.eps);
            pre = sc.pre, rinv = sc.rinv;
        }
        parity ^= 1;

        for (int64_t idx = a0 + tid; idx < a1; idx += threads) {
            float xf[VEC], wf[VEC];
            V::unpack(V::load(xs + (idx - a0) * VEC), xf);
            V::unpack(stage_w ? V::load(ws + (idx - a0) * VEC) : V::load(w + idx * VEC), wf);
#pragma unroll
            for (int i = 0; i < VEC; ++i) xf[i] = xf[i] * pre * rinv * wf[i];
            V::store(orow + idx * VEC, V::pack(xf));
        }
        if (tid < tail) orow[nvec * VEC + tid] = from_f32<T>(xt * pre * rinv * wt);
    }
    if constexpr (RED == RED_PAIR) {
        cg::this_cluster().sync();  // no CTA exits while its peer may still read its pair_slot
    }
}

// ------------------------------------------------------------------ registers
// 16-byte accesses, the row (or the CTA's half of it) in registers: thread tid
// of the group owns accesses idx = a0 + v * threads + tid, v < NV. The weights
// are loaded once the residual sum is formed, so their latency hides behind
// the reduction and their registers reuse the residual's.
// LEAN: w is read in the scale loop, one access at a time, instead of being
// held in registers across the reduction; fewer registers, so more CTAs are
// resident.
template <typename T, int NV, bool ADD, int RED, bool LEAN = false, int G = 1>
__device__ __forceinline__ void reg_row(const NormArgs& a, int64_t r, int tid, int threads, int64_t a0, int64_t a1,
                                        bool tail_owner, float* scratch, float* pair_slot, int parity) {
    constexpr int VEC = vec16<T>();
    using V = Vec<T, VEC>;
    using R = typename V::Raw;
    const int64_t nvec = a.D / VEC;
    const int tail = tail_owner ? static_cast<int>(a.D - nvec * VEC) : 0;
    const T* w = static_cast<const T*>(a.w);
    T* xr = static_cast<T*>(a.x) + r * a.xs;
    T* orow = static_cast<T*>(a.out) + r * a.os;

    R xv[NV];
    float xt = 0.0f, wt = 0.0f;
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

    R wv[LEAN ? 1 : NV];
    if constexpr (!LEAN) {
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int64_t idx = a0 + static_cast<int64_t>(v) * threads + tid;
            if (idx < a1) wv[v] = V::load(w + idx * VEC);
        }
    }
    if (tid < tail) wt = to_f32(w[nvec * VEC + tid]);

    ss = group_sum<RED, G>(ss, scratch, pair_slot, parity);
    float rinv = rsqrtf(ss / static_cast<float>(a.D) + a.eps), pre = 1.0f;
    if (__builtin_expect(!ss_in_range(ss, a.D, a.eps), 0)) {
        double sd = tid < tail ? sq_d(xt) : 0.0;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            if (a0 + static_cast<int64_t>(v) * threads + tid < a1) {
                float xf[VEC];
                V::unpack(xv[v], xf);
#pragma unroll
                for (int i = 0; i < VEC; ++i) sd += sq_d(xf[i]);
            }
        }
        const WideScale sc = wide_scale(group_sum_d<RED, G>(sd, scratch, pair_slot, parity), a.D, a.eps);
        pre = sc.pre, rinv = sc.rinv;
    }

#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int64_t idx = a0 + static_cast<int64_t>(v) * threads + tid;
        if (idx < a1) {
            float xf[VEC], wf[VEC];
            V::unpack(xv[v], xf);
            V::unpack(LEAN ? V::load(w + idx * VEC) : wv[LEAN ? 0 : v], wf);
#pragma unroll
            for (int i = 0; i < VEC; ++i) xf[i] = xf[i] * pre * rinv * wf[i];
            V::store(orow + idx * VEC, V::pack(xf));
        }
    }
    if (tid < tail) orow[nvec * VEC + tid] = from_f32<T>(xt * pre * rinv * wt);
}

// Prefetch row r of x (and res) and, if `with_w`, w, into L2 (one thread).
// Few rows per SM (decode batches, a few hundred rows): one thread issues bulk
// prefetches. Many rows per SM: bulk requests would queue behind each other, so
// the group's threads prefetch the row's cache lines themselves.
template <typename T, bool ADD>
__device__ __forceinline__ void prefetch_row(const NormArgs& a, int64_t r, int64_t e0, int64_t e1, bool with_w,
                                             int i, int n) {
    if (r >= a.rows) return;
    const int64_t bytes = (e1 - e0) * static_cast<int64_t>(sizeof(T));
    const T* x = static_cast<const T*>(a.x) + r * a.xs + e0;
    const T* res = static_cast<const T*>(a.res) + r * a.rs + e0;
    if (a.prefetch) {
        if (i != 0) return;
        prefetch_l2(x, bytes);
        if constexpr (ADD) prefetch_l2(res, bytes);
        if (with_w) prefetch_l2(static_cast<const T*>(a.w) + e0, bytes);
    } else {
        prefetch_lines(x, bytes, i, n);
        if constexpr (ADD) prefetch_lines(res, bytes, i, n);
    }
}

// A group that will process another row after this one prefetches that row's
// lines into L2 now, so the DRAM queue stays full across the boundary between
// one round of resident rows and the next. Off when rows are so many that they
// stream back to back anyway.
template <typename T, bool ADD>
__device__ __forceinline__ void next_row_prefetch(const NormArgs& a, int64_t r, int64_t e0, int64_t e1, int i,
                                                  int n) {
    if (!a.next_prefetch || r >= a.rows) return;
    const int64_t bytes = (e1 - e0) * static_cast<int64_t>(sizeof(T));
    prefetch_lines(static_cast<const T*>(a.x) + r * a.xs + e0, bytes, i, n);
    if constexpr (ADD) prefetch_lines(static_cast<const T*>(a.res) + r * a.rs + e0, bytes, i, n);
}

template <typename T, int NV, bool ADD>
__global__ void __launch_bounds__(256) reg_warp_kernel(NormArgs a) {
    prefetch_row<T, ADD>(a, static_cast<int64_t>(threadIdx.x >> 5) * gridDim.x + blockIdx.x, 0, a.D,
                         threadIdx.x == 0, threadIdx.x & 31, 32);
    pdl_enter();
    const int wpc = blockDim.x >> 5;
    const int64_t nvec = a.D / vec16<T>();
    // Rows are dealt to CTAs round-robin, so CTAs (and SMs) differ by one row at most.
    const int64_t step = static_cast<int64_t>(gridDim.x) * wpc;
    for (int64_t r = static_cast<int64_t>(threadIdx.x >> 5) * gridDim.x + blockIdx.x; r < a.rows; r += step) {
        next_row_prefetch<T, ADD>(a, r + step, 0, a.D, threadIdx.x & 31, 32);
        reg_row<T, NV, ADD, RED_WARP>(a, r, threadIdx.x & 31, 32, 0, nvec, true, nullptr, nullptr, 0);
    }
}

// Largest CTA the register-resident CTA variants are compiled for, per NV.
template <int NV> constexpr int cta_row_max_threads() { return NV >= 8 ? 256 : (NV >= 4 ? 512 : 1024); }

template <typename T, int NV, bool ADD>
__global__ void __launch_bounds__(cta_row_max_threads<NV>()) reg_cta_kernel(NormArgs a) {
    __shared__ __align__(8) float scratch[66];
    prefetch_row<T, ADD>(a, blockIdx.x, 0, a.D, true, threadIdx.x, blockDim.x);
    pdl_enter();
    const int64_t nvec = a.D / vec16<T>();
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        next_row_prefetch<T, ADD>(a, r + gridDim.x, 0, a.D, threadIdx.x, blockDim.x);
        reg_row<T, NV, ADD, RED_CTA>(a, r, threadIdx.x, blockDim.x, 0, nvec, true, scratch, nullptr, 0);
    }
}

// A CTA per row like reg_cta_kernel, with w read in the scale loop and at most
// 256 threads held to 64 registers, so four CTAs (rows) or more share an SM:
// 4 x 152 = 608 rows resident at once, and a second launch's CTAs can become
// resident beside a first one's while it drains.
template <typename T, int NV, bool ADD>
__global__ void __launch_bounds__(256, 4) reg_lean_kernel(NormArgs a) {
    __shared__ __align__(8) float scratch[66];
    prefetch_row<T, ADD>(a, blockIdx.x, 0, a.D, true, threadIdx.x, blockDim.x);
    pdl_enter();
    const int64_t nvec = a.D / vec16<T>();
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        next_row_prefetch<T, ADD>(a, r + gridDim.x, 0, a.D, threadIdx.x, blockDim.x);
        reg_row<T, NV, ADD, RED_CTA, true>(a, r, threadIdx.x, blockDim.x, 0, nvec, true, scratch, nullptr, 0);
    }
}

// G warps per row (warps_row): the CTA's warps form groups of G, each group takes
// rows dealt round-robin over all groups of the grid (CTAs, and so SMs, differ by
// one row at most), thread tid = 32 * (warp % G) + lane of its group owns accesses
// idx = tid + v * 32 G. w is read in the scale loop, as in the lean CTA kernel.
template <typename T, int NV, bool ADD, int G>
__global__ void __launch_bounds__(256) reg_group_kernel(NormArgs a) {
    __shared__ __align__(8) float scratch[66];    // [parity][warp] partial sums
    __shared__ __align__(8) float dslots[66];     // [warp] double partial sums (rare rows)
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int gpc = static_cast<int>(blockDim.x >> 5) / G;  // groups per CTA
    const int tid = static_cast<int>(threadIdx.x) - warp / G * G * 32;
    const int64_t step = static_cast<int64_t>(gridDim.x) * gpc;
    const int64_t r0 = static_cast<int64_t>(warp / G) * gridDim.x + blockIdx.x;
    prefetch_row<T, ADD>(a, r0, 0, a.D, tid == 0, tid, 32 * G);
    pdl_enter();
    const int64_t nvec = a.D / vec16<T>();
    int parity = 0;
    for (int64_t r = r0; r < a.rows; r += step) {
        next_row_prefetch<T, ADD>(a, r + step, 0, a.D, tid, 32 * G);
        reg_row<T, NV, ADD, RED_GROUP, true, G>(a, r, tid, 32 * G, 0, nvec, true, scratch, dslots, parity);
        parity ^= 1;
    }
}

template <typename T, int NV, bool ADD>
__global__ void __launch_bounds__(cta_row_max_threads<NV>()) reg_pair_kernel(NormArgs a) {
    __shared__ __align__(8) float scratch[66];
    __shared__ __align__(8) float pair_slot[6];
    const int rank = static_cast<int>(cg::this_cluster().block_rank());
    const int64_t nvec = a.D / vec16<T>();
    const int64_t half = norm_pair_half(nvec);
    const int64_t a0 = rank == 0 ? 0 : half;
    const int64_t a1 = rank == 0 ? half : nvec;
    prefetch_row<T, ADD>(a, blockIdx.x / 2, a0 * vec16<T>(), rank == 0 ? a1 * vec16<T>() : a.D, true, threadIdx.x,
                         blockDim.x);
    pdl_enter();
    int parity = 0;
    for (int64_t r = blockIdx.x / 2; r < a.rows; r += gridDim.x / 2) {
        next_row_prefetch<T, ADD>(a, r + gridDim.x / 2, a0 * vec16<T>(), rank == 0 ? a1 * vec16<T>() : a.D,
                                  threadIdx.x, blockDim.x);
        reg_row<T, NV, ADD, RED_PAIR>(a, r, threadIdx.x, blockDim.x, a0, a1, rank == 1, scratch, pair_slot, parity);
        parity ^= 1;
    }
    cg::this_cluster().sync();  // no CTA exits while its peer may still read its pair_slot
}

// ------------------------------------------------------------------ registers
// Scalar accesses (layouts that are not 16-byte aligned): the row in registers,
// NV elements per thread, w loaded beside it.
template <typename T, int NV, bool ADD, int RED>
__device__ __forceinline__ void scalar_row(const NormArgs& a, int64_t r, int tid, int threads, float* scratch) {
    T* xr = static_cast<T*>(a.x) + r * a.xs;
    const T* rr = static_cast<const T*>(a.res) + r * a.rs;
    const T* w = static_cast<const T*>(a.w);
    T* orow = static_cast<T*>(a.out) + r * a.os;
    float xv[NV], wv[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int64_t j = static_cast<int64_t>(v) * threads + tid;
        xv[v] = 0.0f;
        if (j < a.D) {
            xv[v] = to_f32(xr[j]);
            if constexpr (ADD) xv[v] += to_f32(rr[j]);
            wv[v] = to_f32(w[j]);
        }
    }
    float ss = 0.0f;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int64_t j = static_cast<int64_t>(v) * threads + tid;
        if (j < a.D) {
            if constexpr (ADD) {
                const T s = from_f32<T>(xv[v]);  // the rounded sum
                xr[j] = s;
                xv[v] = to_f32(s);
            }
            ss = fmaf(xv[v], xv[v], ss);
        }
    }
    ss = group_sum<RED>(ss, scratch, nullptr, 0);
    float rinv = rsqrtf(ss / static_cast<float>(a.D) + a.eps), pre = 1.0f;
    if (__builtin_expect(!ss_in_range(ss, a.D, a.eps), 0)) {
        double sd = 0.0;
#pragma unroll
        for (int v = 0; v < NV; ++v) sd += sq_d(xv[v]);  // xv is 0 past the row's end
        const WideScale sc = wide_scale(group_sum_d<RED>(sd, scratch, nullptr, 0), a.D, a.eps);
        pre = sc.pre, rinv = sc.rinv;
    }
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int64_t j = static_cast<int64_t>(v) * threads + tid;
        if (j < a.D) orow[j] = from_f32<T>(xv[v] * pre * rinv * wv[v]);
    }
}

template <typename T, int NV, bool ADD>
__global__ void __launch_bounds__(256) scalar_warp_kernel(NormArgs a) {
    prefetch_row<T, ADD>(a, static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5), 0, a.D,
                         threadIdx.x == 0, threadIdx.x & 31, 32);
    pdl_enter();
    const int wpc = blockDim.x >> 5;
    const int64_t step = static_cast<int64_t>(gridDim.x) * wpc;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * wpc + (threadIdx.x >> 5); r < a.rows; r += step)
        scalar_row<T, NV, ADD, RED_WARP>(a, r, threadIdx.x & 31, 32, nullptr);
}

template <typename T, int NV, bool ADD>
__global__ void __launch_bounds__(1024) scalar_cta_kernel(NormArgs a) {
    __shared__ __align__(8) float scratch[66];
    prefetch_row<T, ADD>(a, blockIdx.x, 0, a.D, true, threadIdx.x, blockDim.x);
    pdl_enter();
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x)
        scalar_row<T, NV, ADD, RED_CTA>(a, r, threadIdx.x, blockDim.x, scratch);
}

// ------------------------------------------------------------------ two-pass
// Any width: the statistics pass keeps nothing; the scale pass re-reads the
// row (from L2). Each thread revisits only its own elements.
template <typename T, int VEC, bool ADD>
__global__ void __launch_bounds__(1024) two_pass_kernel(NormArgs a) {
    using V = Vec<T, VEC>;
    using R = typename V::Raw;
    __shared__ __align__(8) float scratch[66];
    prefetch_row<T, ADD>(a, blockIdx.x, 0, a.D, true, threadIdx.x, blockDim.x);
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
        float rinv = rsqrtf(ss / static_cast<float>(a.D) + a.eps), pre = 1.0f;
        if (__builtin_expect(!ss_in_range(ss, a.D, a.eps), 0)) {
            // the statistics pass again in double (each thread its own, already updated, elements)
            double sd = tid < tail ? sq_d(xt) : 0.0;
            for (int64_t idx = tid; idx < nvec; idx += threads) {
                float xf[VEC];
                V::unpack(V::load(xr + idx * VEC), xf);
#pragma unroll
                for (int i = 0; i < VEC; ++i) sd += sq_d(xf[i]);
            }
            const WideScale sc = wide_scale(block_sum_d(sd, reinterpret_cast<double*>(scratch)), a.D, a.eps);
            pre = sc.pre, rinv = sc.rinv;
        }
        for (int64_t idx = tid; idx < nvec; idx += threads) {
            float xf[VEC], wf[VEC];
            V::unpack(V::load(xr + idx * VEC), xf);
            V::unpack(V::load(w + idx * VEC), wf);
#pragma unroll
            for (int i = 0; i < VEC; ++i) xf[i] = xf[i] * pre * rinv * wf[i];
            V::store(orow + idx * VEC, V::pack(xf));
        }
        if (tid < tail) {
            const int64_t j = nvec * VEC + tid;
            orow[j] = from_f32<T>(xt * pre * rinv * to_f32(w[j]));
        }
    }
}

// ------------------------------------------------------------------ launch
template <typename KArgs>
cudaError_t smem_opt_in(void (*kernel)(KArgs), size_t smem) {
    // The static shared memory counts against the 48 KB default too.
    if (smem <= 32 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
}

template <typename KArgs>
cudaError_t launch_persistent(void (*kernel)(KArgs), const NormArgs& a, const NormPlan& p, bool pairs,
                              cudaStream_t s) {
    const cudaError_t e = smem_opt_in(kernel, p.smem);
    if (e != cudaSuccess) return e;
    unsigned g = persistent_grid(kernel, p.threads, p.smem, p.num_sms, p.grid);
    if (pairs) {
        g &= ~1u;  // whole clusters only
        if (g < 2) g = 2;
    }
    return launch_kernel(kernel, dim3(g), dim3(p.threads), p.smem, s, p.pdl, pairs ? 2 : 1, a);
}

template <typename T, bool ADD>
cudaError_t launch_vector(const NormArgs& a, const NormPlan& p, cudaStream_t s) {
    switch (p.variant) {
        case NORM_WARP_ROWS:
            switch (p.nv) {
                case 1: return launch_persistent(reg_warp_kernel<T, 1, ADD>, a, p, false, s);
                case 2: return launch_persistent(reg_warp_kernel<T, 2, ADD>, a, p, false, s);
                case 3: return launch_persistent(reg_warp_kernel<T, 3, ADD>, a, p, false, s);
                case 4: return launch_persistent(reg_warp_kernel<T, 4, ADD>, a, p, false, s);
                case 6: return launch_persistent(reg_warp_kernel<T, 6, ADD>, a, p, false, s);
                case 8: return launch_persistent(reg_warp_kernel<T, 8, ADD>, a, p, false, s);
                case 12: return launch_persistent(reg_warp_kernel<T, 12, ADD>, a, p, false, s);
                case 16: return launch_persistent(reg_warp_kernel<T, 16, ADD>, a, p, false, s);
                default: return cudaErrorInvalidValue;
            }
        case NORM_CTA_ROW:
            switch (p.nv) {
                case 1: return launch_persistent(reg_cta_kernel<T, 1, ADD>, a, p, false, s);
                case 2: return launch_persistent(reg_cta_kernel<T, 2, ADD>, a, p, false, s);
                case 4: return launch_persistent(reg_cta_kernel<T, 4, ADD>, a, p, false, s);
                case 8: return launch_persistent(reg_cta_kernel<T, 8, ADD>, a, p, false, s);
                default: return cudaErrorInvalidValue;
            }
        case NORM_CTA_LEAN:
            switch (p.nv) {
                case 2: return launch_persistent(reg_lean_kernel<T, 2, ADD>, a, p, false, s);
                case 4: return launch_persistent(reg_lean_kernel<T, 4, ADD>, a, p, false, s);
                case 8: return launch_persistent(reg_lean_kernel<T, 8, ADD>, a, p, false, s);
                default: return cudaErrorInvalidValue;
            }
        case NORM_WARPS_ROW:
            switch (p.nv * 16 + p.group_warps) {
                case 8 * 16 + 2: return launch_persistent(reg_group_kernel<T, 8, ADD, 2>, a, p, false, s);
                case 8 * 16 + 4: return launch_persistent(reg_group_kernel<T, 8, ADD, 4>, a, p, false, s);
                case 8 * 16 + 8: return launch_persistent(reg_group_kernel<T, 8, ADD, 8>, a, p, false, s);
                case 16 * 16 + 2: return launch_persistent(reg_group_kernel<T, 16, ADD, 2>, a, p, false, s);
                case 16 * 16 + 4: return launch_persistent(reg_group_kernel<T, 16, ADD, 4>, a, p, false, s);
                case 16 * 16 + 8: return launch_persistent(reg_group_kernel<T, 16, ADD, 8>, a, p, false, s);
                default: return cudaErrorInvalidValue;
            }
        case NORM_CTA_PAIR:
            switch (p.nv) {
                case 2: return launch_persistent(reg_pair_kernel<T, 2, ADD>, a, p, true, s);
                case 4: return launch_persistent(reg_pair_kernel<T, 4, ADD>, a, p, true, s);
                case 8: return launch_persistent(reg_pair_kernel<T, 8, ADD>, a, p, true, s);
                default: return cudaErrorInvalidValue;
            }
        case NORM_WARP_SMEM: return launch_persistent(staged_rows_kernel<T, ADD, RED_WARP>, a, p, false, s);
        case NORM_CTA_SMEM: return launch_persistent(staged_rows_kernel<T, ADD, RED_CTA>, a, p, false, s);
        case NORM_PAIR_SMEM: return launch_persistent(staged_rows_kernel<T, ADD, RED_PAIR>, a, p, true, s);
        case NORM_TWO_PASS: return launch_persistent(two_pass_kernel<T, vec16<T>(), ADD>, a, p, false, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, bool ADD>
cudaError_t launch_scalar(const NormArgs& a, const NormPlan& p, cudaStream_t s) {
    switch (p.variant) {
        case NORM_WARP_ROWS:
            switch (p.nv) {
                case 1: return launch_persistent(scalar_warp_kernel<T, 1, ADD>, a, p, false, s);
                case 2: return launch_persistent(scalar_warp_kernel<T, 2, ADD>, a, p, false, s);
                case 4: return launch_persistent(scalar_warp_kernel<T, 4, ADD>, a, p, false, s);
                case 8: return launch_persistent(scalar_warp_kernel<T, 8, ADD>, a, p, false, s);
                default: return cudaErrorInvalidValue;
            }
        case NORM_CTA_ROW:
            switch (p.nv) {
                case 1: return launch_persistent(scalar_cta_kernel<T, 1, ADD>, a, p, false, s);
                case 2: return launch_persistent(scalar_cta_kernel<T, 2, ADD>, a, p, false, s);
                case 4: return launch_persistent(scalar_cta_kernel<T, 4, ADD>, a, p, false, s);
                case 8: return launch_persistent(scalar_cta_kernel<T, 8, ADD>, a, p, false, s);
                default: return cudaErrorInvalidValue;
            }
        case NORM_TWO_PASS: return launch_persistent(two_pass_kernel<T, 1, ADD>, a, p, false, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, bool ADD>
cudaError_t launch_typed(const NormArgs& a, const NormPlan& p, cudaStream_t s) {
    if (p.vec == vec16<T>()) return launch_vector<T, ADD>(a, p, s);
    if (p.vec == 1) return launch_scalar<T, ADD>(a, p, s);
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
