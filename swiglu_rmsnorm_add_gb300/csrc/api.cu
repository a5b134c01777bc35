// C-ABI entry points (include/sra.h): argument validation, per-shape kernel
// planning and launch on the caller's stream. Host code only.
//
// Validation happens entirely before the first CUDA runtime call, so a bad call
// enqueues nothing and touches no device state. Planning is a pure function of
// the sizes, the alignment of every pointer and stride, and the SM count.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>

#include "internal.h"
#include "sra.h"

namespace sra {
namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_smem_optin[kMaxDevices];
std::atomic<int> g_force_norm{-1}, g_force_rope{-1}, g_force_glu{-1}, g_force_attn{-1}, g_force_lin{-1},
    g_force_narrow{-1};
thread_local bool g_pdl = false;  // programmatic dependent launch for this thread's calls
thread_local int g_force_nv = 0;  // accesses per thread forced for A/B measurement (0 = planner's)
thread_local int g_force_g = 0;   // warps per row forced for warps_row A/B measurement (0 = planner's)

// SM count of the current device (cached per device).
int current_sm_count(int* dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (dev_out) *dev_out = dev;
    if (dev >= 0 && dev < kMaxDevices) {
        int c = g_sm_count[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return -1;
    }
    if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

int smem_per_sm(int dev) {
    static std::atomic<int> cache[kMaxDevices];
    if (dev >= 0 && dev < kMaxDevices) {
        int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 100 * 1024;
    }
    if (dev >= 0 && dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

int smem_optin(int dev) {
    if (dev >= 0 && dev < kMaxDevices) {
        int c = g_smem_optin[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 48 * 1024;
    }
    if (dev >= 0 && dev < kMaxDevices) g_smem_optin[dev].store(n, std::memory_order_relaxed);
    return n;
}

bool valid_dtype(int dt) { return dt == DT_F32 || dt == DT_F16 || dt == DT_BF16; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool stride_aligned16(int64_t stride_elems, int es) { return ((stride_elems * es) & 15) == 0; }

// Byte span [lo, hi) of a strided [rows, width] region.
struct Span {
    uintptr_t lo, hi;
};
Span span_of(const void* p, int64_t rows, int64_t stride, int64_t width, int es) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    const int64_t n = rows <= 0 ? 0 : ((rows - 1) * stride + width);
    return {lo, lo + static_cast<uintptr_t>(n) * static_cast<uintptr_t>(es)};
}
bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

// Whether two strided row sets [p + r*stride, p + r*stride + width) (r < rows,
// element units of size es) share a byte. Exact for equal strides (interleaved
// views of one fused buffer, e.g. q / k / v of a fused QKV); otherwise the
// conservative span test.
bool rows_overlap(const void* p1, int64_t rows1, int64_t s1, int64_t w1, const void* p2, int64_t rows2, int64_t s2,
                  int64_t w2, int es) {
    const Span a = span_of(p1, rows1, s1, w1, es), b = span_of(p2, rows2, s2, w2, es);
    if (!overlap(a, b)) return false;
    if (s1 != s2 || rows1 <= 1 || rows2 <= 1 || s1 < w1 || s1 < w2) return true;
    const int64_t S = s1 * es, W1 = w1 * es, W2 = w2 * es;
    const int64_t d = static_cast<int64_t>(reinterpret_cast<intptr_t>(p2) - reinterpret_cast<intptr_t>(p1));
    const int64_t dm = ((d % S) + S) % S;  // row 2's start within row 1's period
    return dm < W1 || dm + W2 > S;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int round_up32(int64_t v) { return static_cast<int>(((v + 31) / 32) * 32); }

// ------------------------------------------------------------------ RMSNorm plan
size_t round_up16(int64_t bytes) { return static_cast<size_t>((bytes + 15) / 16 * 16); }

// Shared memory the planner may use per CTA, and per SM (CTAs resident by memory).
struct SmemBudget {
    int per_cta;  // opt-in limit minus the kernels' static shared memory and a margin
    int per_sm;   // shared memory of one SM
};
constexpr int kCtaReserve = 1024;  // per-CTA shared memory the system keeps

int64_t resident_by_smem(const SmemBudget& b, size_t smem, int threads) {
    const int64_t by_smem = b.per_sm / static_cast<int64_t>(smem + kCtaReserve + 256);
    const int64_t by_threads = 2048 / threads;
    return std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(by_smem, by_threads), 32));
}

// Scalar (unaligned) register kernels: warp NV in {1,2,4,8}; CTA NV in {1,2,4,8}.
bool plan_norm_scalar(int variant, int64_t rows, int64_t D, int num_sms, NormPlan* p) {
    switch (variant) {
        case NORM_WARP_ROWS: {
            if (D > 256) return false;
            int nv = 1;
            while (nv * 32 < D) nv <<= 1;
            p->nv = nv;
            p->threads = rows >= 4LL * num_sms ? 128 : 32;
            p->grid = std::max<int64_t>(1, ceil_div(rows, p->threads / 32));
            return true;
        }
        case NORM_CTA_ROW: {
            if (D > 8192) return false;
            int nv = 1;
            while (nv < 8 && ceil_div(D, nv) > 1024) nv <<= 1;
            if (rows >= 2LL * num_sms) {
                while (nv < 8 && ceil_div(D, nv) > 256) nv <<= 1;
            }
            p->nv = nv;
            p->threads = std::max(32, round_up32(ceil_div(D, nv)));
            p->grid = std::max<int64_t>(1, rows);
            return true;
        }
        case NORM_TWO_PASS:
            p->nv = 0;
            p->threads = static_cast<int>(std::min<int64_t>(1024, std::max(32, round_up32(D))));
            p->grid = std::max<int64_t>(1, rows);
            return true;
        default:
            return false;  // cta_smem and cta_pair need 16-byte layouts
    }
}

// Threads for `acc` 16-byte accesses of one row slice in the staged kernels: few
// rows (decode) get one access per thread; many rows eight, so CTAs stay small
// and many of them are resident.
int staged_threads(int64_t acc, bool few_rows) {
    const int64_t per = few_rows ? 1 : 8;
    return static_cast<int>(std::min<int64_t>(1024, std::max(32, round_up32(ceil_div(acc, per)))));
}

// Register kernels: NV accesses per thread and threads for `nacc` accesses over
// one CTA. Few rows favour many threads with short chains; many rows four
// accesses per thread.
constexpr int kCtaMaxAccesses = 2048;  // 256 threads x 8, 512 x 4, 1024 x 2
int cta_max_threads_for_nv(int nv) { return nv >= 8 ? 256 : (nv >= 4 ? 512 : 1024); }
// Measured on GB300 (bench.py --sweep-variants): one access per thread is best
// for a few rows (decode latency); for hundreds of rows the smallest NV >= 2
// that keeps the CTA at <= 512 threads.
bool cta_shape(int64_t nacc, bool few_rows, int min_nv, int* nv_out, int* threads_out) {
    if (g_force_nv) {
        const int nv = g_force_nv;
        if ((nv & (nv - 1)) || nv < min_nv || nv > 8 || ceil_div(nacc, nv) > cta_max_threads_for_nv(nv)) return false;
        *nv_out = nv;
        *threads_out = std::max(32, round_up32(ceil_div(nacc, nv)));
        return true;
    }
    int nv = std::max(min_nv, few_rows ? 1 : 2);
    while (nv < 8 && ceil_div(nacc, nv) > (few_rows ? cta_max_threads_for_nv(nv) : 512)) nv <<= 1;
    while (nv > min_nv && ceil_div(nacc, nv) < 64) nv >>= 1;
    if (ceil_div(nacc, nv) > cta_max_threads_for_nv(nv)) return false;
    *nv_out = nv;
    *threads_out = std::max(32, round_up32(ceil_div(nacc, nv)));
    return true;
}

// Warps per CTA for warp-per-row kernels: the smallest per-SM row load when CTAs
// are dealt evenly (ties to larger CTAs).
int balanced_wpc(int64_t rows, int num_sms) {
    int best = 8;
    int64_t best_load = -1;
    for (int wpc : {8, 4, 2, 1}) {
        const int64_t load = ceil_div(ceil_div(rows, wpc), num_sms) * wpc;
        if (best_load < 0 || load < best_load) best_load = load, best = wpc;
    }
    return best;
}

bool plan_norm_vector(int variant, int64_t rows, int64_t D, int vec, bool add, int num_sms, const SmemBudget& b,
                      NormPlan* p) {
    const int64_t nvec = D / vec;
    const int64_t nacc = ceil_div(D, vec);  // accesses per row, tail included
    const int copies = add ? 2 : 1;         // x (and res) slices per group, staged kernels
    const bool few_rows = rows < 2LL * num_sms;
    switch (variant) {
        case NORM_WARP_ROWS: {
            const int64_t per_lane = ceil_div(nacc, 32);
            if (per_lane > 16) return false;
            int nv = 16;
            for (int c : {1, 2, 3, 4, 6, 8, 12, 16}) {
                if (c >= per_lane && (g_force_nv == 0 || c == g_force_nv)) {
                    nv = c;
                    break;
                }
            }
            if (nv < per_lane || (g_force_nv && nv != g_force_nv)) return false;
            const int wpc = balanced_wpc(rows, num_sms);
            p->nv = nv;
            p->threads = 32 * wpc;
            p->grid = std::max<int64_t>(1, ceil_div(rows, wpc));
            return true;
        }
        case NORM_CTA_ROW:
            if (nacc > kCtaMaxAccesses) return false;
            if (!cta_shape(nacc, few_rows, 1, &p->nv, &p->threads)) return false;
            p->grid = std::max<int64_t>(1, rows);
            return true;
        case NORM_CTA_LEAN: {
            // at most 256 threads: the fewest accesses per thread (2, 4 or 8) that fit
            int nv = 0;
            for (int c : {2, 4, 8}) {
                if ((g_force_nv == 0 || c == g_force_nv) && ceil_div(nacc, c) <= 256) {
                    nv = c;
                    break;
                }
            }
            if (!nv) return false;
            p->nv = nv;
            p->threads = std::max(32, round_up32(ceil_div(nacc, nv)));
            p->grid = std::max<int64_t>(1, rows);
            return true;
        }
        case NORM_WARPS_ROW: {
            // G warps per row with NV (8 or 16) accesses per lane: the fewest warps that hold
            // the row, then the fewest accesses per lane
            int G = 0, nv = 0;
            for (int g : {2, 4, 8}) {
                if (g_force_g && g != g_force_g) continue;
                for (int c : {8, 16}) {
                    if (g_force_nv && c != g_force_nv) continue;
                    if (32LL * g * c >= nacc) {
                        G = g, nv = c;
                        break;
                    }
                }
                if (G) break;
            }
            if (!G || nacc <= 32 * 16 / 2) return false;  // rows a single warp holds take warp_rows
            // groups per CTA (<= 256 threads): the smallest per-SM row load, ties to larger CTAs
            int best = 1;
            int64_t best_load = -1;
            for (int gpc = 8 / G; gpc >= 1; gpc >>= 1) {
                const int64_t load = ceil_div(ceil_div(rows, gpc), num_sms) * gpc;
                if (best_load < 0 || load < best_load) best_load = load, best = gpc;
            }
            p->nv = nv;
            p->group_warps = G;
            p->threads = 32 * G * best;
            p->grid = std::max<int64_t>(1, ceil_div(rows, best));
            return true;
        }
        case NORM_CTA_PAIR: {
            if (nvec < 2) return false;
            const int64_t half = norm_pair_half(nvec);
            const int64_t per_cta = std::max<int64_t>(half, nacc - half);
            if (per_cta > kCtaMaxAccesses) return false;
            if (!cta_shape(per_cta, few_rows, 2, &p->nv, &p->threads)) return false;
            p->grid = 2 * std::max<int64_t>(1, rows);
            return true;
        }
        case NORM_WARP_SMEM: {
            if (nacc > 256) return false;
            const size_t slice = round_up16(nvec * 16);
            // Warps per CTA: the smallest per-SM row load that is resident in one
            // round (shared memory, threads); ties go to larger CTAs.
            int best = 0;
            int64_t best_load = 0, best_cap = 0;
            for (int wpc : {8, 4, 2, 1}) {
                const size_t smem = slice + wpc * slice * copies;
                if (static_cast<int64_t>(smem) > b.per_cta) continue;
                const int64_t cap = resident_by_smem(b, smem, 32 * wpc) * wpc;
                const int64_t load = ceil_div(ceil_div(rows, wpc), num_sms) * wpc;
                const bool fits = load <= cap;
                const bool best_fits = best && best_load <= best_cap;
                if (!best || (fits && (!best_fits || load < best_load)) || (!fits && !best_fits && cap > best_cap))
                    best = wpc, best_load = load, best_cap = cap;
            }
            if (!best) return false;
            p->threads = 32 * best;
            p->grid = std::max<int64_t>(1, ceil_div(rows, best));
            p->smem = slice + best * slice * copies;
            p->stage_w = 1;
            return true;
        }
        case NORM_CTA_SMEM: {
            const size_t slice = round_up16(nvec * 16);
            // stage w beside the row when both fit, else read it from L2
            const bool stage = static_cast<int64_t>(slice + slice * copies) <= b.per_cta;
            const size_t smem = (stage ? slice : 0) + slice * copies;
            if (static_cast<int64_t>(smem) > b.per_cta) return false;
            p->threads = staged_threads(nvec, few_rows);
            p->grid = std::max<int64_t>(1, rows);
            p->smem = smem;
            p->stage_w = stage ? 1 : 0;
            return true;
        }
        case NORM_PAIR_SMEM: {
            if (nvec < 2) return false;
            const int64_t half = norm_pair_half(nvec);
            const size_t slice = round_up16(half * 16);
            const size_t smem = slice + slice * copies;
            if (static_cast<int64_t>(smem) > b.per_cta) return false;
            p->threads = staged_threads(half, few_rows);
            p->grid = 2 * std::max<int64_t>(1, rows);
            p->smem = smem;
            p->stage_w = 1;
            return true;
        }
        case NORM_TWO_PASS:
            p->threads = static_cast<int>(std::min<int64_t>(1024, std::max(32, round_up32(nacc))));
            p->grid = std::max<int64_t>(1, rows);
            return true;
        default:
            return false;
    }
}

bool plan_norm_variant(int variant, int64_t rows, int64_t D, int vec, bool add, int num_sms, const SmemBudget& b,
                       NormPlan* p) {
    p->variant = variant;
    p->vec = vec;
    p->nv = 0;
    p->smem = 0;
    p->pdl = g_pdl;
    p->num_sms = num_sms;
    p->stage_w = 0;
    p->group_warps = 0;
    p->prefetch = rows <= 4LL * num_sms ? 1 : 0;
    // groups with a next row exist only past one row per resident group; with very
    // many rows they stream back to back anyway (measured: bench.py --sweep-variants)
    p->next_prefetch = rows >= 2LL * num_sms && rows <= 64LL * num_sms ? 1 : 0;
    if (vec == 1) return plan_norm_scalar(variant, rows, D, num_sms, p);
    return plan_norm_vector(variant, rows, D, vec, add, num_sms, b, p);
}

// Automatic choice: the preferred variants for the shape, in order.
int plan_norm(int64_t rows, int64_t D, int vec, bool add, int num_sms, const SmemBudget& b, NormPlan* p) {
    const int forced = g_force_norm.load(std::memory_order_relaxed);
    if (forced >= 0) {
        g_force_nv = (forced >> 8) & 0xFF;
        g_force_g = (forced >> 16) & 0xFF;
        const bool ok = plan_norm_variant(forced & 0xFF, rows, D, vec, add, num_sms, b, p);
        g_force_nv = 0;
        g_force_g = 0;
        // bits 24..27: at most that many CTAs per SM (the grid shrinks; every kernel strides
        // over its rows, so any grid is correct)
        const int cps = (forced >> 24) & 0xF;
        if (ok && cps) {
            const bool pairs = p->variant == NORM_CTA_PAIR || p->variant == NORM_PAIR_SMEM;
            p->grid = std::min<int64_t>(p->grid, static_cast<int64_t>(cps) * num_sms * (pairs ? 2 : 1));
        }
        return ok ? SRA_OK : SRA_ERR_VARIANT;
    }
    const int64_t nacc = ceil_div(D, vec);
    const bool few_rows = rows < 2LL * num_sms;
    // Order from the variant sweep on GB300 (bench.py --sweep-variants): the
    // register variants beat the shared-memory ones on every configured shape
    // but one (within 2%), and a CTA per row beats the CTA pair.
    int order[7];
    int n = 0;
    // a warp per row from 256 rows (add_rmsnorm [256, 1536]: 15 % faster than a CTA per row), or
    // for short rows once every SM has two. Rows of 257 to 512 accesses (12 or 16 per lane) take
    // a warp each at a few hundred rows: 512 rows of fp32 1536 / 2048, 16-bit 2176 / 4096 measured
    // 35 / 28 / 21 / 9 % faster than the CTA variants
    if (nacc <= 256 && (rows >= 256 || (!few_rows && nacc <= 64))) order[n++] = NORM_WARP_ROWS;
    else if (nacc <= 512 && rows >= 256 && rows <= 8LL * num_sms) order[n++] = NORM_WARP_ROWS;
    // 16-bit rows of 512 to 1024 accesses (4096 to 8192 elements), hundreds of rows: the lean
    // CTA (w read in the scale loop) measured 3-4 % faster than cta_row
    if (!few_rows && vec == 8 && nacc >= 512 && nacc <= 1024) order[n++] = NORM_CTA_LEAN;
    order[n++] = NORM_CTA_ROW;
    order[n++] = NORM_CTA_SMEM;
    order[n++] = NORM_TWO_PASS;
    for (int i = 0; i < n; ++i) {
        if (plan_norm_variant(order[i], rows, D, vec, add, num_sms, b, p)) return SRA_OK;
    }
    return SRA_ERR_VARIANT;
}

int norm_vec(int dt, const void* const* ptrs, int nptr, const int64_t* strides, int nstr) {
    const int es = elem_bytes(dt);
    bool ok = true;
    for (int i = 0; i < nptr; ++i) ok = ok && aligned16(ptrs[i]);
    for (int i = 0; i < nstr; ++i) ok = ok && stride_aligned16(strides[i], es);
    return ok ? 16 / es : 1;
}

// ------------------------------------------------------------------ RoPE plan
int plan_rope(int64_t T, int n_head, int n_kv, int head_dim, int pairs, int style, bool qk_norm, int num_sms,
              RopePlan* p) {
    const int forced = g_force_rope.load(std::memory_order_relaxed);
    const int h = head_dim / 2;
    const int n_units = n_head + 2 * n_kv;
    // two tasks per thread need the token's tasks to split into two equal sets of whole heads
    const bool two_ok = n_units % 2 == 0;
    // Two tasks per thread once the tokens outnumber what one round of the one-task kernel holds
    // (about 9 tokens per SM at Qwen2.5-1.5B bf16 shapes). Measured on GB300, bf16, 12 / 2 heads:
    // T = 2048 and 32768 faster (neox and interleaved), T = 1 and 64 slower; with the Q/K UClip
    // fused the two-task kernel runs out of registers and is slower at every T.
    int variant = two_ok && !qk_norm && T > 8LL * num_sms ? ROPE_TOKEN_CTA2 : ROPE_TOKEN_CTA;
    if (forced >= 0) {
        if (forced >= ROPE_NUM_VARIANTS) return SRA_ERR_VARIANT;  // no accesses-per-thread setting here
        variant = forced;
    }
    if (variant == ROPE_TOKEN_CTA2 && !two_ok) return SRA_ERR_VARIANT;
    const int64_t U = static_cast<int64_t>(n_units) * (h / pairs) / (variant == ROPE_TOKEN_CTA2 ? 2 : 1);
    p->variant = variant;
    p->style = style;
    p->qk_norm = qk_norm;
    p->pairs = pairs;
    p->pdl = g_pdl;
    p->num_sms = num_sms;
    // the two-task kernel is compiled for at most 512 threads (its tasks loop past them)
    const int64_t max_threads = variant == ROPE_TOKEN_CTA2 ? 512 : 1024;
    p->threads = static_cast<int>(std::min<int64_t>(max_threads, std::max(32, round_up32(U))));
    p->grid = std::max<int64_t>(1, T);
    return SRA_OK;
}

// ------------------------------------------------------------------- GLU plan
int plan_glu(int64_t T, int64_t I, int vec, int act, int num_sms, GluPlan* p) {
    const int forced = g_force_glu.load(std::memory_order_relaxed);
    const int64_t nv = I / vec;
    // Measured on GB300 (bench.py --sweep-variants, streaming): SiLU runs faster with the
    // registers the compiler picks (58 on 16-byte vectors, four CTAs per SM: T = 4096 53.2 against
    // 55.2 us, T = 512 8.2 against 8.8 us); ReLU at 48 (51.2 against 52.2 us at T = 4096)
    p->variant = forced >= 0 ? forced : (act == 0 ? GLU_COLS_ROWS_REGS : GLU_COLS_ROWS);
    p->vec = vec;
    p->pdl = g_pdl;
    p->num_sms = num_sms;
    // Few rows: narrow CTAs spread the columns over many SMs. Many rows: 256 threads.
    int threads = T >= 64 ? 256 : 128;
    threads = static_cast<int>(std::min<int64_t>(threads, std::max(32, round_up32(nv))));
    p->threads = threads;
    p->grid_x = ceil_div(nv, threads);
    const int64_t resident = static_cast<int64_t>(num_sms) * (2048 / threads);
    const int64_t gy = std::max<int64_t>(1, resident / std::max<int64_t>(1, p->grid_x));
    p->grid_y = std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(T, gy), 65535));
    return SRA_OK;
}

// Largest power-of-two vector width (elements, <= 16 bytes) that divides I and
// every stride and keeps every pointer aligned.
int glu_vec(int dt, const void* gu, const void* out, int64_t I, int64_t is, int64_t os) {
    const int es = elem_bytes(dt);
    for (int bytes = 16; bytes >= es * 2; bytes >>= 1) {
        const int vec = bytes / es;
        if ((reinterpret_cast<uintptr_t>(gu) % bytes) == 0 && (reinterpret_cast<uintptr_t>(out) % bytes) == 0 &&
            I % vec == 0 && is % vec == 0 && os % vec == 0)
            return vec;
    }
    return 1;
}

thread_local int g_last_cuda_error = 0;

int status_from(cudaError_t e) {
    if (e == cudaSuccess) return SRA_OK;
    g_last_cuda_error = static_cast<int>(e);
    cudaGetLastError();
    return SRA_ERR_LAUNCH;
}

int norm_common(void* x, const void* res, const void* w, void* out, int64_t rows, int64_t D, int64_t xs,
                int64_t rs, int64_t os, float eps, int dtype, void* stream, bool add) {
    if (!valid_dtype(dtype)) return SRA_ERR_DTYPE;
    if (rows < 0 || D <= 0) return SRA_ERR_SHAPE;
    if (xs < D || os < D || (add && rs < D)) return SRA_ERR_STRIDE;
    if (!(eps >= 0.0f) || !std::isfinite(eps)) return SRA_ERR_ARG;
    if (rows == 0) return SRA_OK;
    if (!x || !w || !out || (add && !res)) return SRA_ERR_NULL;
    const int es = elem_bytes(dtype);
    const Span sw = span_of(w, 1, D, D, es);
    const Span sx = span_of(x, rows, xs, D, es), so = span_of(out, rows, os, D, es);
    if (add) {
        const Span sr = span_of(res, rows, rs, D, es);
        if (rows_overlap(out, rows, os, D, x, rows, xs, D, es) || rows_overlap(out, rows, os, D, res, rows, rs, D, es) ||
            overlap(so, sw) || overlap(sx, sw))
            return SRA_ERR_ALIAS;
        if (!(res == x && rs == xs) && rows_overlap(x, rows, xs, D, res, rows, rs, D, es)) return SRA_ERR_ALIAS;
        (void)sr;
    } else {
        const bool in_place = out == x && os == xs;
        if ((!in_place && rows_overlap(out, rows, os, D, x, rows, xs, D, es)) || overlap(so, sw)) return SRA_ERR_ALIAS;
    }
    int dev = 0;
    const int sms = current_sm_count(&dev);
    if (sms <= 0) return SRA_ERR_DEVICE;
    const void* ptrs[4] = {x, w, out, add ? res : x};
    const int64_t strides[3] = {xs, os, add ? rs : xs};
    const int vec = norm_vec(dtype, ptrs, 4, strides, 3);
    NormPlan plan;
    SmemBudget budget;
    budget.per_cta = smem_optin(dev) - 1024;
    budget.per_sm = smem_per_sm(dev);
    int st = plan_norm(rows, D, vec, add, sms, budget, &plan);
    if (st != SRA_OK) return st;
    NormArgs a;
    a.x = x;
    a.res = res;
    a.w = w;
    a.out = out;
    a.rows = rows;
    a.D = D;
    a.xs = xs;
    a.rs = add ? rs : 0;
    a.os = os;
    a.eps = eps;
    a.stage_w = plan.stage_w;
    a.prefetch = plan.prefetch;
    a.next_prefetch = plan.next_prefetch;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return status_from(add ? launch_add_rmsnorm(a, plan, dtype, s) : launch_rmsnorm(a, plan, dtype, s));
}

std::atomic<int>* force_slot(const char* op) {
    if (!op) return nullptr;
    if (std::strcmp(op, "rmsnorm") == 0) return &g_force_norm;
    if (std::strcmp(op, "rope_kv_store") == 0) return &g_force_rope;
    if (std::strcmp(op, "glu") == 0) return &g_force_glu;
    if (std::strcmp(op, "decode_attention") == 0) return &g_force_attn;
    if (std::strcmp(op, "linear") == 0) return &g_force_lin;
    if (std::strcmp(op, "linear_narrow") == 0) return &g_force_narrow;
    return nullptr;
}

int variant_count(const char* op) {
    if (!op) return SRA_ERR_ARG;
    if (std::strcmp(op, "rmsnorm") == 0) return NORM_NUM_VARIANTS;
    if (std::strcmp(op, "rope_kv_store") == 0) return ROPE_NUM_VARIANTS;
    if (std::strcmp(op, "glu") == 0) return GLU_NUM_VARIANTS;
    if (std::strcmp(op, "decode_attention") == 0) return 3;  // CUDA cores, mma.sync, mma.sync fed by TMA
    if (std::strcmp(op, "linear") == 0) return 2;            // mma.sync, tcgen05 (projection over h)
    if (std::strcmp(op, "linear_narrow") == 0) return 1;     // the decode-batch kernel (K split forced)
    return SRA_ERR_ARG;
}

// ------------------------------------------------------------------- UClip plan

// Whether the rows of an [N, H, D] view (element strides n_s, h_s, 1) are
// pairwise disjoint: heads nested inside tokens, or tokens inside heads.
// A dimension of size 1 places no constraint through its stride.
bool rows_disjoint(int64_t N, int64_t H, int64_t D, int64_t n_s, int64_t h_s) {
    const bool heads_ok = H <= 1 || h_s >= D;
    const int64_t tok_w = H <= 1 ? D : (H - 1) * h_s + D;
    if (heads_ok && (N <= 1 || n_s >= tok_w)) return true;
    const bool toks_ok = N <= 1 || n_s >= D;
    const int64_t head_w = N <= 1 ? D : (N - 1) * n_s + D;
    return toks_ok && (H <= 1 || h_s >= head_w);
}

int uclip_vec(int dt, const UclipArgs& a) {
    const int es = elem_bytes(dt);
    for (int bytes = 16; bytes >= es * 2; bytes >>= 1) {
        const int vec = bytes / es;
        const int pbytes = 4 * (vec >= 4 ? 4 : vec);
        bool ok = reinterpret_cast<uintptr_t>(a.x) % bytes == 0 && reinterpret_cast<uintptr_t>(a.out) % bytes == 0 &&
                  a.D % vec == 0 && (a.N <= 1 || (a.xn % vec == 0 && a.on % vec == 0)) &&
                  (a.H <= 1 || (a.xh % vec == 0 && a.oh % vec == 0));
        ok = ok && (!a.alpha_pc || reinterpret_cast<uintptr_t>(a.alpha) % pbytes == 0);
        ok = ok && (!a.gamma_pc || reinterpret_cast<uintptr_t>(a.gamma) % pbytes == 0);
        if (ok) return vec;
    }
    return 1;
}

void plan_uclip(int64_t rows, int64_t D, int vec, int num_sms, UclipPlan* p) {
    const int64_t nv = D / vec;
    p->vec = vec;
    p->bx = static_cast<int>(std::min<int64_t>(nv, 256));
    p->by = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(256 / p->bx, rows)));
    p->grid_x = ceil_div(nv, p->bx);
    p->grid_y = std::max<int64_t>(1, ceil_div(rows, p->by));
    p->pdl = g_pdl;
    p->num_sms = num_sms;
}

// RoPE + KV store, optionally with the UClip of Q and K (norm != nullptr: qa, qg,
// ka, kg per-channel fp32 parameters of head_dim entries, then the clip bounds).
struct QkNorm {
    const float *qa, *qg, *ka, *kg;
    float lo, hi;
};

int rope_impl(void* q, const void* k, const void* v, const float* cos, const float* sin, const int64_t* pos,
              const int64_t* slot_mapping, void* kv_cache, int64_t T, int n_head, int n_kv_head, int head_dim,
              int64_t q_tok_stride, int64_t k_tok_stride, int64_t v_tok_stride, int64_t max_pos, int64_t num_blocks,
              int block_size, int32_t* err_count, int style, const QkNorm* norm, int dtype, void* stream) {
    if (!valid_dtype(dtype)) return SRA_ERR_DTYPE;
    if (style != SRA_ROPE_NEOX && style != SRA_ROPE_INTERLEAVED) return SRA_ERR_ARG;
    if (T < 0 || n_head <= 0 || n_kv_head <= 0 || n_head % n_kv_head != 0 || head_dim <= 0 || head_dim % 2 != 0 ||
        block_size <= 0 || num_blocks < 0 || max_pos < 0)
        return SRA_ERR_SHAPE;
    const int64_t qw = static_cast<int64_t>(n_head) * head_dim, kw = static_cast<int64_t>(n_kv_head) * head_dim;
    if (q_tok_stride < qw || k_tok_stride < kw || v_tok_stride < kw) return SRA_ERR_STRIDE;
    if (T == 0) return SRA_OK;
    if (!q || !k || !v || !cos || !sin || !pos || !slot_mapping || !kv_cache) return SRA_ERR_NULL;
    if (norm && (!norm->qa || !norm->qg || !norm->ka || !norm->kg)) return SRA_ERR_NULL;
    const int es = elem_bytes(dtype);
    const Span sq = span_of(q, T, q_tok_stride, qw, es), sk = span_of(k, T, k_tok_stride, kw, es),
               sv = span_of(v, T, v_tok_stride, kw, es);
    const Span sc = span_of(kv_cache, 1, 0, 2 * num_blocks * block_size * kw, es);
    if (rows_overlap(q, T, q_tok_stride, qw, k, T, k_tok_stride, kw, es) ||
        rows_overlap(q, T, q_tok_stride, qw, v, T, v_tok_stride, kw, es) || overlap(sc, sq) || overlap(sc, sk) ||
        overlap(sc, sv))
        return SRA_ERR_ALIAS;
    if (norm) {
        // the parameters are read while q and the cache are written
        const float* ps[4] = {norm->qa, norm->qg, norm->ka, norm->kg};
        for (const float* pp : ps) {
            const Span sp = span_of(pp, 1, 0, head_dim, 4);
            if (overlap(sp, sq) || overlap(sp, sc)) return SRA_ERR_ALIAS;
        }
    }
    int dev = 0;
    const int sms = current_sm_count(&dev);
    if (sms <= 0) return SRA_ERR_DEVICE;
    const int h = head_dim / 2;
    // 16 / es pairs per task: two 16-byte accesses (one per half for neox, two
    // consecutive ones for interleaved)
    int pairs = 16 / es;
    const bool vec_ok = h % pairs == 0 && h % 4 == 0 && aligned16(q) && aligned16(k) && aligned16(v) &&
                        aligned16(kv_cache) && aligned16(cos) && aligned16(sin) &&
                        stride_aligned16(q_tok_stride, es) && stride_aligned16(k_tok_stride, es) &&
                        stride_aligned16(v_tok_stride, es) &&
                        (!norm || (aligned16(norm->qa) && aligned16(norm->qg) && aligned16(norm->ka) &&
                                   aligned16(norm->kg)));
    if (!vec_ok) pairs = 1;
    RopePlan plan;
    int st = plan_rope(T, n_head, n_kv_head, head_dim, pairs, style, norm != nullptr, sms, &plan);
    if (st != SRA_OK) return st;
    RopeArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.cos = cos;
    a.sin = sin;
    a.pos = pos;
    a.slot = slot_mapping;
    a.cache = kv_cache;
    a.err = err_count;
    a.T = T;
    a.n_head = n_head;
    a.n_kv = n_kv_head;
    a.head_dim = head_dim;
    a.qs = q_tok_stride;
    a.ks = k_tok_stride;
    a.vs = v_tok_stride;
    a.max_pos = max_pos;
    a.num_blocks = num_blocks;
    a.block_size = block_size;
    if (norm) {
        a.qa = norm->qa, a.qg = norm->qg, a.ka = norm->ka, a.kg = norm->kg;
        a.clip_lo = norm->lo, a.clip_hi = norm->hi;
    }
    return status_from(launch_rope_kv_store(a, plan, dtype, static_cast<cudaStream_t>(stream)));
}

}  // namespace

// Global splits of a decode-attention call: used when the cluster splits cannot give every SM
// work (fewer than SMs / 16 (request, kv head) pairs) and the context is long enough for more
// than 16 splits of at least 512 tokens; one CTA per SM at most.
int decode_attention_gsplits(int64_t B, int n_kv, int64_t max_blocks, int block_size, int num_sms) {
    const int64_t groups = B * n_kv;
    if (groups <= 0 || groups * 16 >= num_sms) return 0;
    const int64_t gs = std::min<int64_t>({num_sms / groups, max_blocks * block_size / 512, kMaxGsplits});
    return gs > 16 ? static_cast<int>(gs) : 0;
}

int64_t decode_attention_ws_bytes(int64_t B, int n_kv, int head_dim, int gsplits) {
    if (gsplits <= 0) return 0;
    const int64_t groups = B * n_kv;
    return (groups * 4 + 255) / 256 * 256 + groups * gsplits * (16 + 8 * static_cast<int64_t>(head_dim)) * 4;
}

}  // namespace sra

using namespace sra;

extern "C" {

int sra_version(void) { return SRA_VERSION; }

int sra_last_cuda_error(void) { return g_last_cuda_error; }

unsigned int sra_wait_timeouts(void) { return linear_wait_timeouts() + attn_wait_timeouts(); }

int sra_wait_selftest(int32_t* result, void* stream) {
    if (!result) return SRA_ERR_NULL;
    return status_from(launch_wait_selftest(result, static_cast<cudaStream_t>(stream)));
}

int sra_set_pdl(int enable) {
    const int prev = g_pdl ? 1 : 0;
    g_pdl = enable != 0;
    return prev;
}

const char* sra_status_string(int status) {
    switch (status) {
        case SRA_OK: return "ok";
        case SRA_ERR_NULL: return "a required pointer is NULL";
        case SRA_ERR_SHAPE: return "a size is out of range";
        case SRA_ERR_STRIDE: return "a stride is smaller than the row it must hold";
        case SRA_ERR_DTYPE: return "unsupported dtype";
        case SRA_ERR_ALIAS: return "an output overlaps an input in a way the operator forbids";
        case SRA_ERR_ARG: return "invalid argument";
        case SRA_ERR_VARIANT: return "the forced kernel variant cannot handle this call";
        case SRA_ERR_LAUNCH: return "CUDA kernel launch failed";
        case SRA_ERR_DEVICE: return "could not query the CUDA device";
        default: return "unknown status";
    }
}

int sra_rmsnorm(const void* x, const void* w, void* out, int64_t rows, int64_t D, int64_t x_row_stride,
                int64_t out_row_stride, float eps, int dtype, void* stream) {
    return norm_common(const_cast<void*>(x), nullptr, w, out, rows, D, x_row_stride, 0, out_row_stride, eps,
                       dtype, stream, false);
}

int sra_add_rmsnorm(void* x, const void* res, const void* w, void* out, int64_t rows, int64_t D,
                    int64_t x_row_stride, int64_t res_row_stride, int64_t out_row_stride, float eps, int dtype,
                    void* stream) {
    return norm_common(x, res, w, out, rows, D, x_row_stride, res_row_stride, out_row_stride, eps, dtype, stream,
                       true);
}

int sra_rope_kv_store_ex(void* q, const void* k, const void* v, const float* cos, const float* sin,
                         const int64_t* pos, const int64_t* slot_mapping, void* kv_cache, int64_t T, int n_head,
                         int n_kv_head, int head_dim, int64_t q_tok_stride, int64_t k_tok_stride,
                         int64_t v_tok_stride, int64_t max_pos, int64_t num_blocks, int block_size,
                         int32_t* err_count, int style, int dtype, void* stream) {
    return rope_impl(q, k, v, cos, sin, pos, slot_mapping, kv_cache, T, n_head, n_kv_head, head_dim, q_tok_stride,
                     k_tok_stride, v_tok_stride, max_pos, num_blocks, block_size, err_count, style, nullptr, dtype,
                     stream);
}

int sra_rope_kv_store_qk_uclip(void* q, const void* k, const void* v, const float* cos, const float* sin,
                               const int64_t* pos, const int64_t* slot_mapping, void* kv_cache, int64_t T,
                               int n_head, int n_kv_head, int head_dim, int64_t q_tok_stride, int64_t k_tok_stride,
                               int64_t v_tok_stride, int64_t max_pos, int64_t num_blocks, int block_size,
                               int32_t* err_count, int style, const float* q_alpha, const float* q_gamma,
                               const float* k_alpha, const float* k_gamma, float clip_min, float clip_max,
                               int dtype, void* stream) {
    if (std::isnan(clip_min) || std::isnan(clip_max) || clip_min > clip_max) return SRA_ERR_ARG;
    const QkNorm norm{q_alpha, q_gamma, k_alpha, k_gamma, clip_min, clip_max};
    return rope_impl(q, k, v, cos, sin, pos, slot_mapping, kv_cache, T, n_head, n_kv_head, head_dim, q_tok_stride,
                     k_tok_stride, v_tok_stride, max_pos, num_blocks, block_size, err_count, style, &norm, dtype,
                     stream);
}

int sra_rope_kv_store(void* q, const void* k, const void* v, const float* cos, const float* sin,
                      const int64_t* pos, const int64_t* slot_mapping, void* kv_cache, int64_t T, int n_head,
                      int n_kv_head, int head_dim, int64_t q_tok_stride, int64_t k_tok_stride,
                      int64_t v_tok_stride, int64_t max_pos, int64_t num_blocks, int block_size,
                      int32_t* err_count, int dtype, void* stream) {
    return sra_rope_kv_store_ex(q, k, v, cos, sin, pos, slot_mapping, kv_cache, T, n_head, n_kv_head, head_dim,
                                q_tok_stride, k_tok_stride, v_tok_stride, max_pos, num_blocks, block_size,
                                err_count, SRA_ROPE_NEOX, dtype, stream);
}

int sra_glu(const void* gate_up, void* out, int64_t T, int64_t I, int64_t in_row_stride, int64_t out_row_stride,
            int act, int dtype, void* stream) {
    if (!valid_dtype(dtype)) return SRA_ERR_DTYPE;
    if (act != SRA_ACT_SILU && act != SRA_ACT_RELU) return SRA_ERR_ARG;
    if (T < 0 || I <= 0) return SRA_ERR_SHAPE;
    if (in_row_stride < 2 * I || out_row_stride < I) return SRA_ERR_STRIDE;
    if (T == 0) return SRA_OK;
    if (!gate_up || !out) return SRA_ERR_NULL;
    const int es = elem_bytes(dtype);
    if (rows_overlap(gate_up, T, in_row_stride, 2 * I, out, T, out_row_stride, I, es)) return SRA_ERR_ALIAS;
    int dev = 0;
    const int sms = current_sm_count(&dev);
    if (sms <= 0) return SRA_ERR_DEVICE;
    GluPlan plan;
    int st = plan_glu(T, I, glu_vec(dtype, gate_up, out, I, in_row_stride, out_row_stride), act, sms, &plan);
    if (st != SRA_OK) return st;
    GluArgs a;
    a.gate_up = gate_up;
    a.out = out;
    a.T = T;
    a.I = I;
    a.is = in_row_stride;
    a.os = out_row_stride;
    return status_from(launch_glu(a, plan, act, dtype, static_cast<cudaStream_t>(stream)));
}

int sra_swiglu(const void* gate_up, void* out, int64_t T, int64_t I, int64_t in_row_stride,
               int64_t out_row_stride, int dtype, void* stream) {
    return sra_glu(gate_up, out, T, I, in_row_stride, out_row_stride, SRA_ACT_SILU, dtype, stream);
}

// ------------------------------------------------------------------- decode attention
static int attention_impl(const void* q, const void* kv_cache, const int32_t* block_table, const int32_t* seq_lens,
                          void* out, int64_t B, int n_head, int n_kv_head, int head_dim, int64_t q_tok_stride,
                          int64_t out_tok_stride, int64_t num_blocks, int block_size, int64_t max_blocks_per_seq,
                          float scale, void* workspace, int64_t workspace_bytes, int32_t* err_count, int dtype,
                          void* stream) {
    if (!valid_dtype(dtype)) return SRA_ERR_DTYPE;
    if (B < 0 || n_head <= 0 || n_kv_head <= 0 || n_head % n_kv_head != 0 || n_head / n_kv_head > 8 ||
        (head_dim != 64 && head_dim != 128 && head_dim != 256) ||
        (block_size != 8 && block_size != 16 && block_size != 32) || num_blocks < 0 || max_blocks_per_seq < 0)
        return SRA_ERR_SHAPE;
    const int64_t w = static_cast<int64_t>(n_head) * head_dim;
    if (q_tok_stride < w || out_tok_stride < w) return SRA_ERR_STRIDE;
    if (!std::isfinite(scale)) return SRA_ERR_ARG;
    if (B == 0) return SRA_OK;
    if (!q || !kv_cache || !block_table || !seq_lens || !out) return SRA_ERR_NULL;
    if (!aligned16(kv_cache)) return SRA_ERR_ARG;
    const int es = elem_bytes(dtype);
    const Span so = span_of(out, B, out_tok_stride, w, es);
    const Span sc = span_of(kv_cache, 1, 0, 2 * num_blocks * block_size * static_cast<int64_t>(n_kv_head) * head_dim, es);
    const Span st = span_of(block_table, 1, 0, B * max_blocks_per_seq, 4), sl = span_of(seq_lens, 1, 0, B, 4);
    if (rows_overlap(out, B, out_tok_stride, w, q, B, q_tok_stride, w, es) || overlap(so, sc) || overlap(so, st) ||
        overlap(so, sl))
        return SRA_ERR_ALIAS;
    int dev = 0;
    const int sms = current_sm_count(&dev);
    if (sms <= 0) return SRA_ERR_DEVICE;
    const int group = n_head / n_kv_head;
    AttnPlan plan;
    plan.head_dim = head_dim;
    plan.threads = 128;
    plan.pdl = g_pdl;
    plan.num_sms = sms;
    // splits of one (request, kv head): a cluster of up to 8 CTAs, enough CTAs for two per SM,
    // and at least 4 cache blocks per split
    const int64_t groups = B * n_kv_head;
    const int64_t limit = smem_optin(dev) - 1024;
    // tensor cores for 16-bit data when q rows allow 4-byte fragment loads
    plan.tensor_cores = dtype != DT_F32 && (head_dim == 64 || head_dim == 128) &&
                        (reinterpret_cast<uintptr_t>(q) & 3u) == 0 && q_tok_stride % 2 == 0 &&
                        num_blocks * block_size < (int64_t(1) << 31) &&
                        static_cast<int64_t>(decode_attention_mma_smem(head_dim, 8)) <= limit;
    const int forced_all = g_force_attn.load(std::memory_order_relaxed);
    const int forced = forced_all < 0 ? -1 : (forced_all & 0xFF);  // variant; bits 8-15: splits (A/B only)
    if ((forced == 1 || forced == 2) && !plan.tensor_cores) return SRA_ERR_VARIANT;
    if (forced == 0) plan.tensor_cores = false;
    // the TMA-fed kernel: a 4-D tensor map over the cache (16-byte strides hold for head_dim
    // 64 and 128), its ring in one CTA's shared memory
    plan.tma = forced == 2;
    if (plan.tma && static_cast<int64_t>(decode_attention_tma_smem(head_dim)) > limit) return SRA_ERR_VARIANT;
    // mma.sync kernel: 8 warps per CTA (one CTA per SM) unless forced to 4 (two per SM)
    const int forced_warps = forced_all < 0 ? 0 : (forced_all >> 16) & 0xFF;
    if (forced_warps) {
        if ((forced_warps != 4 && forced_warps != 8) || forced != 1) return SRA_ERR_VARIANT;
        plan.mma_warps = forced_warps;
    }
    int splits = 1;
    if (plan.tensor_cores) {
        // as many CTAs as the SMs hold at once (the K/V rings fill an SM's shared memory with one
        // 8-warp CTA or two 4-warp ones), and at least two 16-token tiles per warp per split
        const int64_t per_sm = plan.mma_warps == 4 ? 2 : 1;
        const int64_t min_tok = 32 * static_cast<int64_t>(plan.mma_warps);
        while (splits < 16 && groups * splits * 2 <= per_sm * sms &&
               max_blocks_per_seq * block_size >= min_tok * splits * 2)
            splits *= 2;
    } else {
        while (splits < 8 && groups * splits < 2 * static_cast<int64_t>(sms) && max_blocks_per_seq >= 4 * splits)
            splits *= 2;
    }
    if (forced_all > 0 && ((forced_all >> 8) & 0xFF)) {
        const int fs = (forced_all >> 8) & 0xFF;
        if ((fs & (fs - 1)) || fs > (plan.tensor_cores ? 16 : 8)) return SRA_ERR_VARIANT;
        splits = fs;
    }
    plan.splits = splits;
    plan.stages = 4;
    if (static_cast<int64_t>(decode_attention_smem(group, head_dim, block_size, 4, es)) > limit) plan.stages = 2;
    plan.smem = plan.tma            ? decode_attention_tma_smem(head_dim)
                : plan.tensor_cores ? decode_attention_mma_smem(head_dim, plan.mma_warps)
                                    : decode_attention_smem(group, head_dim, block_size, plan.stages, es);
    if (static_cast<int64_t>(plan.smem) > limit) return SRA_ERR_SHAPE;
    AttnArgs a;
    a.q = q;
    a.cache = kv_cache;
    a.table = block_table;
    a.seq_lens = seq_lens;
    a.out = out;
    a.err = err_count;
    a.B = B;
    a.qs = q_tok_stride;
    a.os = out_tok_stride;
    a.num_blocks = num_blocks;
    a.max_blocks = max_blocks_per_seq;
    a.n_head = n_head;
    a.n_kv = n_kv_head;
    a.group = group;
    a.block_size = block_size;
    a.scale_log2 = scale * 1.4426950408889634f;
    if (workspace && plan.tensor_cores && forced != 0) {
        const int gs = decode_attention_gsplits(B, n_kv_head, max_blocks_per_seq, block_size, sms);
        const int64_t need = decode_attention_ws_bytes(B, n_kv_head, head_dim, gs);
        if (gs > 0) {
            if (workspace_bytes < need || !aligned16(workspace)) return SRA_ERR_ARG;
            const Span sws = span_of(workspace, 1, 0, need, 1);
            if (overlap(sws, so) || overlap(sws, sc) || overlap(sws, st) || overlap(sws, sl) ||
                overlap(sws, span_of(q, B, q_tok_stride, w, es)))
                return SRA_ERR_ALIAS;
            a.gsplits = gs;
            a.ws_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((B * n_kv_head * 4 + 255) / 256) * 256);
        }
    }
    return status_from(launch_decode_attention(a, plan, dtype, static_cast<cudaStream_t>(stream)));
}


int sra_paged_decode_attention(const void* q, const void* kv_cache, const int32_t* block_table,
                               const int32_t* seq_lens, void* out, int64_t B, int n_head, int n_kv_head,
                               int head_dim, int64_t q_tok_stride, int64_t out_tok_stride, int64_t num_blocks,
                               int block_size, int64_t max_blocks_per_seq, float scale, int32_t* err_count,
                               int dtype, void* stream) {
    return attention_impl(q, kv_cache, block_table, seq_lens, out, B, n_head, n_kv_head, head_dim, q_tok_stride,
                          out_tok_stride, num_blocks, block_size, max_blocks_per_seq, scale, nullptr, 0, err_count,
                          dtype, stream);
}

int64_t sra_paged_decode_attention_workspace_size(int64_t B, int n_head, int n_kv_head, int head_dim,
                                                  int64_t max_blocks_per_seq, int block_size, int dtype) {
    if (!valid_dtype(dtype)) return SRA_ERR_DTYPE;
    if (B < 0 || n_head <= 0 || n_kv_head <= 0 || n_head % n_kv_head != 0 || n_head / n_kv_head > 8 ||
        (head_dim != 64 && head_dim != 128 && head_dim != 256) ||
        (block_size != 8 && block_size != 16 && block_size != 32) || max_blocks_per_seq < 0)
        return SRA_ERR_SHAPE;
    if (dtype == DT_F32 || head_dim > 128 || B == 0) return 0;
    int dev = 0;
    const int sms = current_sm_count(&dev);
    if (sms <= 0) return SRA_ERR_DEVICE;
    return decode_attention_ws_bytes(B, n_kv_head, head_dim,
                                     decode_attention_gsplits(B, n_kv_head, max_blocks_per_seq, block_size, sms));
}

int sra_paged_decode_attention_ws(const void* q, const void* kv_cache, const int32_t* block_table,
                                  const int32_t* seq_lens, void* out, int64_t B, int n_head, int n_kv_head,
                                  int head_dim, int64_t q_tok_stride, int64_t out_tok_stride, int64_t num_blocks,
                                  int block_size, int64_t max_blocks_per_seq, float scale, void* workspace,
                                  int64_t workspace_bytes, int32_t* err_count, int dtype, void* stream) {
    if (workspace_bytes < 0) return SRA_ERR_ARG;
    return attention_impl(q, kv_cache, block_table, seq_lens, out, B, n_head, n_kv_head, head_dim, q_tok_stride,
                          out_tok_stride, num_blocks, block_size, max_blocks_per_seq, scale, workspace,
                          workspace_bytes, err_count, dtype, stream);
}

// ------------------------------------------------------------------- fused linear
// prologue: 0 RMSNorm, 1 SwiGLU, 2 ReGLU, 3 none (x holds h; internal, from linear_ws)
static int linear_common(const void* x, const void* w_ln, const void* W, void* y, int64_t B, int64_t K, int64_t N,
                      int64_t xs, int64_t ys, float eps, int prologue, int dtype, void* stream,
                      float* ws_part = nullptr) {
    if (!valid_dtype(dtype)) return SRA_ERR_DTYPE;
    if (B < 0 || K <= 0 || N <= 0) return SRA_ERR_SHAPE;
    const int64_t xw = prologue == 1 || prologue == 2 ? 2 * K : K;
    if (xs < xw || ys < N) return SRA_ERR_STRIDE;
    if (prologue == 0 && (!(eps >= 0.0f) || !std::isfinite(eps))) return SRA_ERR_ARG;
    if (B == 0) return SRA_OK;
    if (!x || !W || !y || (prologue == 0 && !w_ln)) return SRA_ERR_NULL;
    const int es = elem_bytes(dtype);
    const Span sy = span_of(y, B, ys, N, es);
    if (rows_overlap(y, B, ys, N, x, B, xs, xw, es) || overlap(sy, span_of(W, 1, 0, N * K, es)) ||
        (prologue == 0 && overlap(sy, span_of(w_ln, 1, 0, K, es))))
        return SRA_ERR_ALIAS;
    int dev = 0;
    const int sms = current_sm_count(&dev);
    if (sms <= 0) return SRA_ERR_DEVICE;
    const int64_t limit = smem_optin(dev) - 1024;
    LinPlan plan;
    plan.prologue = prologue;
    plan.pdl = g_pdl;
    plan.mt = B <= 16 ? 1 : (B <= 32 ? 2 : 4);
    plan.tensor_cores = dtype != DT_F32 && K % 64 == 0 && N % 64 == 0 && aligned16(x) && aligned16(W) &&
                        xs % 8 == 0 && (prologue != 0 || aligned16(w_ln));
    plan.narrow = false;
    plan.splits = 1;
    plan.tcgen05 = false;
    // decode batches: 16-column CTAs over all of K, when the B rows of h for all of K fit in
    // shared memory beside the W rings. (The kernel can also split K over a cluster of up to 8
    // CTAs, forced only: measured slower at every split count, e.g. SwiGLU + down_proj
    // [8960 -> 1536] at batch 1 8.3 us unsplit against 9.5-16.2 us split 2-8 ways.)
    plan.narrow = plan.tensor_cores && B <= 16 &&
                  static_cast<int64_t>(linear16_smem(static_cast<int>(B), K, 1)) <= std::min<int64_t>(limit, 200 * 1024);
    if (plan.narrow) {
        const int64_t KT = K / 64;
        const int nf = g_force_narrow.load(std::memory_order_relaxed);
        if (nf >= 0) {
            const int fs = (nf >> 8) & 0xFF;  // variant 0; bits 8-15: the cluster's K split (1..8)
            if (fs) {
                if (fs > 8 || fs > KT) return SRA_ERR_VARIANT;
                plan.splits = fs;
            }
        }
    }
    // the projection of h (the workspace path) on tcgen05: up to 64 rows, 128-column slices.
    // Chosen from K = 4096 up (measured on GB300 at batch 64: SwiGLU + down_proj [8960 -> 1536]
    // 14.3 against 18.1 us with mma.sync; ln1 + qkv_proj [1536 -> 2048] 10.9 against 8.5 us,
    // too few W tiles per CTA to amortise the tensor-memory set-up and the cluster epilogue);
    // sra_force_variant("linear", 0 or 1) overrides it
    const int lin_all = g_force_lin.load(std::memory_order_relaxed);
    const int lin_forced = lin_all < 0 ? -1 : (lin_all & 0xFF);  // bits 8-15: K splits (A/B only)
    // (measured at batch 64: from K = 4096 up always; from K = 1024 up when the partials go through
    // L2, e.g. ln1 + qkv_proj [1536 -> 2048] 8.5 -> 7.6 us)
    const bool tc_wanted = lin_forced == 1 || (lin_forced < 0 && (K >= 4096 || (ws_part && K >= 1024)));
    if (plan.tensor_cores && prologue == 3 && B <= 64 && N % 128 == 0 && tc_wanted &&
        static_cast<int64_t>(linear_tc_smem(4)) <= limit) {
        plan.tcgen05 = true;
        // 128-column slices x K splits (a cluster of up to 16 CTAs): a 4-stage ring, two CTAs per
        // SM, and as many splits as fill those two slots once, with at least 4 W tiles per CTA.
        // (An 8-stage ring at one CTA per SM measured slower at every split count: batch 64 x
        // 8960 -> 1536 best 15.9 us against 14.3 us.)
        const int64_t slices = N / 128, KT = K / 64;
        plan.tc_stages = 4;
        const int fst = lin_all < 0 ? 0 : (lin_all >> 16) & 0xFF;  // forced ring depth
        if (fst) {
            if (fst != 4 && fst != 8) return SRA_ERR_VARIANT;
            if (static_cast<int64_t>(linear_tc_smem(fst)) > limit) return SRA_ERR_VARIANT;
            plan.tc_stages = fst;
        }
        const int64_t per_sm = plan.tc_stages == 8 ? 1 : 2;
        plan.splits = static_cast<int>(std::max<int64_t>(
            1, std::min<int64_t>({16, per_sm * sms / slices, KT / 4})));
        const int fs = lin_all < 0 ? 0 : (lin_all >> 8) & 0xFF;
        if (fs) {
            if (fs > 16 || fs > KT) return SRA_ERR_VARIANT;
            plan.splits = fs;
        }
        // a cluster the device cannot place at all takes the largest size it can
        while (plan.splits > 1 && linear_tc_max_clusters(plan.splits, plan.tc_stages, dtype == DT_BF16) < 1) {
            if (fs) return SRA_ERR_VARIANT;
            --plan.splits;
        }
    } else if (lin_forced == 1 && prologue == 3) {
        return SRA_ERR_VARIANT;
    }
    // the GLU fused into the tcgen05 projection (no workspace, one launch): from 4 to 64 rows (or
    // forced onto it, from 1 row; not while the decode-batch kernel's split is forced), N a
    // multiple of 128; 3 stages of 32 KB, two CTAs per SM. Measured on GB300 (CUDA-graph replay, us
    // per call, decode-batch or mma.sync kernel against tcgen05): SwiGLU + down_proj [8960 -> 1536]
    // batch 1 8.65 / 12.31, 3 11.88 / 12.42, 4 13.82 / 12.21, 16 17.17 / 12.42, 64 28.59 / 14.15;
    // [14336 -> 4096] batch 2 35.97 / 45.18, 4 51.83 / 45.18, 64 88.18 / 48.26
    const bool narrow_forced = g_force_narrow.load(std::memory_order_relaxed) >= 0;
    if (plan.tensor_cores && (prologue == 1 || prologue == 2) && B <= 64 && N % 128 == 0 &&
        (lin_forced == 1 || (lin_forced < 0 && !narrow_forced && B >= 4)) &&
        static_cast<int64_t>(linear_tc_smem(3, 1)) <= limit) {
        plan.tcgen05 = true;
        plan.narrow = false;
        const int64_t slices = N / 128, KT = K / 64;
        plan.splits = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>({16, 2 * sms / slices, KT / 4})));
        const int fs = lin_all < 0 ? 0 : (lin_all >> 8) & 0xFF;
        if (fs) {
            if (fs > 16 || fs > KT) return SRA_ERR_VARIANT;
            plan.splits = fs;
        }
        while (plan.splits > 1 && linear_tc_max_clusters(plan.splits, 3, dtype == DT_BF16, 1) < 1) {
            if (fs) return SRA_ERR_VARIANT;
            --plan.splits;
        }
    }
    // the RMSNorm fused into the tcgen05 projection (one launch), N a multiple of 128: a CTA holds
    // its whole K range of x (at most 16 tiles) beside a 4-stage W ring, so the split is at least
    // K / (16 x 64). Chosen from 33 rows, or from 17 with K >= 4096, at the largest split whose grid
    // is one wave (two CTAs per SM up to 5 x tiles each, one beyond). Measured on GB300 (CUDA-graph
    // replay, us per call, mma.sync against tcgen05): batch 64 [1536 -> 2048] 9.7 / 8.1, [4096 ->
    // 4096] 26.4 / 17.4; batch 32 [4096 -> 4096] 19.5 / 16.9 but [1536 -> 2048] 7.5 / 8.4, batch 17
    // 7.3 / 8.9. Forced onto it, from 1 row and at any split that fits.
    if (plan.tensor_cores && prologue == 0 && B <= 64 && N % 128 == 0 &&
        (lin_forced == 1 || (lin_forced < 0 && (B > 32 || (B > 16 && K >= 4096))))) {
        const int64_t slices = N / 128, KT = K / 64;
        const int64_t min_split = (KT + 15) / 16;
        const bool bf = dtype == DT_BF16;
        auto nx_of = [&](int k) { return static_cast<int>((KT + k - 1) / k); };
        auto fits = [&](int k) { return static_cast<int64_t>(linear_tc_smem(4, 0, nx_of(k))) <= limit; };
        auto placed = [&](int k) { return linear_tc_max_clusters(k, 4, bf, 0, nx_of(k)) >= 1; };
        const int fs = lin_all < 0 ? 0 : (lin_all >> 8) & 0xFF;
        int sk = 0;
        if (fs) {
            if (fs > 16 || fs > KT || fs < min_split || !fits(fs) || !placed(fs)) return SRA_ERR_VARIANT;
            sk = fs;
        } else {
            // the largest split with at least 4 K tiles a CTA whose grid is one wave; forced onto
            // the kernel without one, the smallest split that fits
            for (int k = static_cast<int>(std::min<int64_t>(16, std::max<int64_t>(1, KT / 4))); k >= min_split && !sk;
                 --k) {
                if (!fits(k)) continue;
                const int per_sm = linear_tc_norm_ctas_per_sm(nx_of(k), bf);
                if (per_sm >= 1 && slices * k <= static_cast<int64_t>(per_sm) * sms && placed(k)) sk = k;
            }
            if (!sk && lin_forced == 1)
                for (int k = static_cast<int>(std::max<int64_t>(1, min_split)); k <= 16 && k <= KT && !sk; ++k)
                    if (fits(k) && placed(k)) sk = k;
        }
        if (sk) {
            plan.tcgen05 = true;
            plan.narrow = false;
            plan.splits = sk;
        } else if (lin_forced == 1) {
            return SRA_ERR_VARIANT;
        }
    }
    if (plan.tensor_cores && !plan.narrow && !plan.tcgen05) {
        // 64-column slices x row blocks x K splits (a cluster); two CTAs per SM fit (45 to 113 KB
        // each): aim for one wave of 1-2 CTAs per SM with at least four W tiles per CTA
        const int64_t slices = (N / 64) * ((B + plan.mt * 16 - 1) / (plan.mt * 16));
        const int64_t KT = K / 64;
        while (plan.splits < 8 && slices * plan.splits * 2 <= 2 * static_cast<int64_t>(sms) &&
               KT >= 4 * plan.splits)
            plan.splits *= 2;
        if (static_cast<int64_t>(linear_smem(plan.mt, prologue)) > limit) plan.tensor_cores = false;
    }
    if (!plan.tensor_cores) {
        plan.splits = 1;
        if (K * 4 > limit) return SRA_ERR_SHAPE;
    }
    LinArgs a;
    a.x = x;
    a.w_ln = w_ln;
    a.W = W;
    a.y = y;
    a.B = B;
    a.K = K;
    a.N = N;
    a.xs = xs;
    a.ys = ys;
    a.eps = eps;
    a.ws_part = plan.tcgen05 ? ws_part : nullptr;
    return status_from(launch_linear(a, plan, dtype, static_cast<cudaStream_t>(stream)));
}

int sra_rmsnorm_linear(const void* x, const void* w_ln, const void* W, void* y, int64_t B, int64_t K, int64_t N,
                       int64_t x_row_stride, int64_t y_row_stride, float eps, int dtype, void* stream) {
    return linear_common(x, w_ln, W, y, B, K, N, x_row_stride, y_row_stride, eps, 0, dtype, stream);
}

// Rows from which the workspace entry points split the prologue off: the fused kernel rebuilds
// the prologue's rows once per 64-column slice of y (24 times for N = 1536). Measured on GB300
// at 64 rows: ln1 + qkv_proj 9.4 -> 8.3 us, SwiGLU + down_proj 30.0 -> 19.0 us.
constexpr int64_t kLinearSplitRows = 32;

// The workspace path: the prologue's own kernel writes h [B, K] into the workspace, then the
// projection streams W against h (prologue 3). Falls back to the fused kernel (workspace
// untouched) below kLinearSplitRows rows or where the tensor-core path does not apply.
static int linear_ws(const void* x, const void* w_ln, const void* W, void* y, int64_t B, int64_t K, int64_t N,
                     int64_t xs, int64_t ys, float eps, int prologue, void* ws, int64_t ws_bytes, int dtype,
                     void* stream) {
    // validate exactly as the fused call does (nothing is enqueued on error)
    if (!valid_dtype(dtype)) return SRA_ERR_DTYPE;
    if (B < 0 || K <= 0 || N <= 0) return SRA_ERR_SHAPE;
    const int64_t xw = prologue == 0 ? K : 2 * K;
    if (xs < xw || ys < N) return SRA_ERR_STRIDE;
    if (prologue == 0 && (!(eps >= 0.0f) || !std::isfinite(eps))) return SRA_ERR_ARG;
    if (ws_bytes < 0) return SRA_ERR_ARG;
    if (B == 0) return SRA_OK;
    if (!x || !W || !y || (prologue == 0 && !w_ln)) return SRA_ERR_NULL;
    const int es = elem_bytes(dtype);
    const bool split = ws != nullptr && B >= kLinearSplitRows && dtype != DT_F32 && K % 64 == 0 && N % 64 == 0 &&
                       aligned16(W) && aligned16(ws);
    if (!split)
        return linear_common(x, w_ln, W, y, B, K, N, xs, ys, eps, prologue, dtype, stream);
    if (ws_bytes < B * K * es) return SRA_ERR_ARG;
    // a workspace with room past h for the tcgen05 projection's partials lets it sum its K split
    // through L2 instead of the cluster's shared memory
    const int64_t hb = linear_ws_h_bytes(B, K, es);
    const bool part = B <= 64 && N % 128 == 0 && ws_bytes >= hb + linear_ws_part_bytes(N);
    const Span sw = span_of(ws, 1, 0, part ? hb + linear_ws_part_bytes(N) : B * K * es, 1);
    if (overlap(sw, span_of(x, B, xs, xw, es)) || overlap(sw, span_of(W, 1, 0, N * K, es)) ||
        overlap(sw, span_of(y, B, ys, N, es)) || (prologue == 0 && overlap(sw, span_of(w_ln, 1, 0, K, es))))
        return SRA_ERR_ALIAS;
    // the fused call's own checks (alias of y with x, W, w_ln; strides), before anything runs
    {
        const Span sy = span_of(y, B, ys, N, es);
        if (rows_overlap(y, B, ys, N, x, B, xs, xw, es) || overlap(sy, span_of(W, 1, 0, N * K, es)) ||
            (prologue == 0 && overlap(sy, span_of(w_ln, 1, 0, K, es))))
            return SRA_ERR_ALIAS;
    }
    // a forced tcgen05 projection that cannot serve this call: nothing is enqueued
    if (g_force_lin.load(std::memory_order_relaxed) == 1 && (B > 64 || N % 128 != 0)) return SRA_ERR_VARIANT;
    const int st = prologue == 0 ? sra_rmsnorm(x, w_ln, ws, B, K, xs, K, eps, dtype, stream)
                                 : sra_glu(x, ws, B, K, xs, K, prologue - 1, dtype, stream);
    if (st != SRA_OK) return st;
    return linear_common(ws, nullptr, W, y, B, K, N, K, ys, 0.0f, 3, dtype, stream,
                         part ? reinterpret_cast<float*>(static_cast<char*>(ws) + hb) : nullptr);
}

int64_t sra_linear_workspace_size(int64_t B, int64_t K, int64_t N, int dtype) {
    if (!valid_dtype(dtype)) return SRA_ERR_DTYPE;
    if (B < 0 || K <= 0 || N <= 0) return SRA_ERR_SHAPE;
    const int es = elem_bytes(dtype);
    const int64_t h = linear_ws_h_bytes(B, K, es);
    return B <= 64 && N % 128 == 0 && dtype != DT_F32 ? h + linear_ws_part_bytes(N) : h;
}

int sra_rmsnorm_linear_ws(const void* x, const void* w_ln, const void* W, void* y, int64_t B, int64_t K, int64_t N,
                          int64_t x_row_stride, int64_t y_row_stride, float eps, void* workspace,
                          int64_t workspace_bytes, int dtype, void* stream) {
    return linear_ws(x, w_ln, W, y, B, K, N, x_row_stride, y_row_stride, eps, 0, workspace, workspace_bytes, dtype,
                     stream);
}

int sra_glu_linear_ws(const void* gate_up, const void* W, void* y, int64_t B, int64_t I, int64_t N,
                      int64_t in_row_stride, int64_t y_row_stride, int act, void* workspace, int64_t workspace_bytes,
                      int dtype, void* stream) {
    if (act != SRA_ACT_SILU && act != SRA_ACT_RELU) return valid_dtype(dtype) ? SRA_ERR_ARG : SRA_ERR_DTYPE;
    return linear_ws(gate_up, nullptr, W, y, B, I, N, in_row_stride, y_row_stride, 0.0f, 1 + act, workspace,
                     workspace_bytes, dtype, stream);
}

int sra_glu_linear(const void* gate_up, const void* W, void* y, int64_t B, int64_t I, int64_t N,
                   int64_t in_row_stride, int64_t y_row_stride, int act, int dtype, void* stream) {
    if (act != SRA_ACT_SILU && act != SRA_ACT_RELU) return valid_dtype(dtype) ? SRA_ERR_ARG : SRA_ERR_DTYPE;
    return linear_common(gate_up, nullptr, W, y, B, I, N, in_row_stride, y_row_stride, 0.0f, 1 + act, dtype,
                             stream);
}

// ------------------------------------------------------------------- UClip
int sra_uclip(const void* x, const float* alpha, const float* gamma, void* out, int64_t N, int64_t H, int64_t D,
              int64_t x_n_stride, int64_t x_h_stride, int64_t out_n_stride, int64_t out_h_stride,
              int alpha_per_channel, int gamma_per_channel, float clip_min, float clip_max, int dtype, void* stream) {
    if (!valid_dtype(dtype)) return SRA_ERR_DTYPE;
    if (N < 0 || H < 0 || H > INT32_MAX || D <= 0) return SRA_ERR_SHAPE;
    if ((alpha_per_channel != 0 && alpha_per_channel != 1) || (gamma_per_channel != 0 && gamma_per_channel != 1) ||
        std::isnan(clip_min) || std::isnan(clip_max) || clip_min > clip_max)
        return SRA_ERR_ARG;
    if (x_n_stride < 0 || x_h_stride < 0 || out_n_stride < 0 || out_h_stride < 0 ||
        !rows_disjoint(N, H, D, out_n_stride, out_h_stride))
        return SRA_ERR_STRIDE;
    if (N == 0 || H == 0) return SRA_OK;
    if (!x || !alpha || !gamma || !out) return SRA_ERR_NULL;
    const int es = elem_bytes(dtype);
    // tokens as rows of width (H - 1) * h_stride + D: exact for the equal token
    // strides of views into one fused buffer, conservative otherwise
    const int64_t xw = H <= 1 ? D : (H - 1) * x_h_stride + D, ow = H <= 1 ? D : (H - 1) * out_h_stride + D;
    const bool in_place = out == x && (N <= 1 || out_n_stride == x_n_stride) && (H <= 1 || out_h_stride == x_h_stride);
    const Span so = span_of(out, N, out_n_stride, ow, es);
    const Span sa = span_of(alpha, 1, 0, alpha_per_channel ? D : 1, 4), sg = span_of(gamma, 1, 0, gamma_per_channel ? D : 1, 4);
    if ((!in_place && rows_overlap(out, N, out_n_stride, ow, x, N, x_n_stride, xw, es)) || overlap(so, sa) ||
        overlap(so, sg))
        return SRA_ERR_ALIAS;
    int dev = 0;
    const int sms = current_sm_count(&dev);
    if (sms <= 0) return SRA_ERR_DEVICE;
    UclipArgs a;
    a.x = x;
    a.alpha = alpha;
    a.gamma = gamma;
    a.out = out;
    a.N = N;
    a.H = H;
    a.D = D;
    a.xn = N <= 1 ? 0 : x_n_stride;
    a.xh = H <= 1 ? 0 : x_h_stride;
    a.on = N <= 1 ? 0 : out_n_stride;
    a.oh = H <= 1 ? 0 : out_h_stride;
    a.alpha_pc = alpha_per_channel != 0;
    a.gamma_pc = gamma_per_channel != 0;
    a.lo = clip_min;
    a.hi = clip_max;
    UclipPlan plan;
    plan_uclip(N * H, D, uclip_vec(dtype, a), sms, &plan);
    return status_from(launch_uclip(a, plan, dtype, static_cast<cudaStream_t>(stream)));
}

int sra_force_variant(const char* op, int variant) {
    std::atomic<int>* slot = force_slot(op);
    if (!slot) return SRA_ERR_ARG;
    if (variant < -1 || (variant >= 0 && ((variant & 0xFF) >= variant_count(op) || (variant >> 28) != 0)))
        return SRA_ERR_ARG;
    slot->store(variant, std::memory_order_relaxed);
    return SRA_OK;
}

int sra_variant_count(const char* op) { return variant_count(op); }

const char* sra_variant_name(const char* op, int variant) {
    static const char* const norm_names[] = {"warp_rows", "cta_row",   "cta_smem",  "two_pass", "cta_pair",
                                             "warp_smem", "pair_smem", "cta_lean",  "warps_row"};
    static const char* const rope_names[] = {"token_cta", "token_cta2"};
    static const char* const glu_names[] = {"cols_rows", "cols_rows_regs"};
    static const char* const attn_names[] = {"cuda_cores", "mma_sync", "mma_sync_tma"};
    static const char* const lin_names[] = {"mma_sync", "tcgen05"};
    static const char* const narrow_names[] = {"cluster_k_split"};
    const int n = variant_count(op);
    if (n < 0 || variant < 0 || variant >= n) return nullptr;
    if (std::strcmp(op, "rmsnorm") == 0) return norm_names[variant];
    if (std::strcmp(op, "rope_kv_store") == 0) return rope_names[variant];
    if (std::strcmp(op, "decode_attention") == 0) return attn_names[variant];
    if (std::strcmp(op, "linear") == 0) return lin_names[variant];
    if (std::strcmp(op, "linear_narrow") == 0) return narrow_names[variant];
    return glu_names[variant];
}

int sra_pick_variant(const char* op, int64_t a, int64_t b, int64_t c, int64_t d, int dtype, int num_sms) {
    if (!valid_dtype(dtype) || variant_count(op) < 0) return SRA_ERR_ARG;
    int dev = 0;
    if (num_sms <= 0) {
        num_sms = current_sm_count(&dev);
        if (num_sms <= 0) return SRA_ERR_DEVICE;
    }
    const int es = elem_bytes(dtype);
    if (std::strcmp(op, "rmsnorm") == 0) {
        if (a < 0 || b <= 0) return SRA_ERR_SHAPE;
        NormPlan p;
        SmemBudget budget;
        budget.per_cta = 227 * 1024 - 1024;
        budget.per_sm = 228 * 1024;
        const int st = plan_norm(a, b, 16 / es, false, num_sms, budget, &p);
        return st == SRA_OK ? p.variant : st;
    }
    if (std::strcmp(op, "rope_kv_store") == 0) {
        if (a < 0 || b <= 0 || c <= 0 || d <= 0 || d % 2) return SRA_ERR_SHAPE;
        RopePlan p;
        const int st =
            plan_rope(a, static_cast<int>(b), static_cast<int>(c), static_cast<int>(d), 1, 0, false, num_sms, &p);
        return st == SRA_OK ? p.variant : st;
    }
    if (std::strcmp(op, "decode_attention") == 0) {
        if (a < 0 || b <= 0 || c <= 0 || b % c || b / c > 8 || (d != 64 && d != 128 && d != 256))
            return SRA_ERR_SHAPE;
        return dtype != DT_F32 && d <= 128 ? 1 : 0;
    }
    if (std::strcmp(op, "glu") != 0) return SRA_ERR_ARG;  // the projections' plans depend on more than four sizes
    if (a < 0 || b <= 0) return SRA_ERR_SHAPE;
    GluPlan p;
    const int st = plan_glu(a, b, 16 / es, c == 1 ? 1 : 0, num_sms, &p);
    return st == SRA_OK ? p.variant : st;
}

}  // extern "C"
