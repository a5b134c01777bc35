// Internal interface between the C-ABI host layer (api.cu) and the kernel
// launchers. Plain host types only.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sra {

enum Dtype { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2 };

inline int elem_bytes(int dt) { return dt == DT_F32 ? 4 : 2; }

// ----------------------------------------------------------------- RMSNorm
struct NormArgs {
    void* x;          // [rows, D], in/out for add_rmsnorm
    const void* res;  // [rows, D] residual (add_rmsnorm only)
    const void* w;    // [D]
    void* out;        // [rows, D]
    int64_t rows, D;
    int64_t xs, rs, os;  // row strides, elements
    float eps;
    int stage_w;         // staged kernels: 1 = w slice staged in shared memory
    int prefetch;        // 1 = prefetch each CTA's first rows into L2 before the launch wait
    int next_prefetch;   // 1 = prefetch a group's next row while it processes the current one
};

enum NormVariant {
    NORM_WARP_ROWS = 0,  // one warp per row, row held in registers
    NORM_CTA_ROW = 1,    // one CTA per row, row held in registers
    NORM_CTA_SMEM = 2,   // one CTA per row, row landed in shared memory (cp.async)
    NORM_TWO_PASS = 3,   // one CTA per row, second pass re-reads the row (any D)
    NORM_CTA_PAIR = 4,   // a 2-CTA cluster per row, half the row in each CTA's registers
    NORM_WARP_SMEM = 5,  // one warp per row, row landed in shared memory (cp.async)
    NORM_PAIR_SMEM = 6,  // a 2-CTA cluster per row, half the row in each CTA's shared memory
    NORM_CTA_LEAN = 7,   // one CTA (<= 256 threads) per row, row in registers, w read in the scale loop
    NORM_WARPS_ROW = 8,  // 2, 4 or 8 warps per row, row in registers, w read in the scale loop;
                         // the warps' partial sums meet behind a named barrier of just those warps
    NORM_NUM_VARIANTS = 9
};

#ifdef __CUDACC__
#define SRA_HD __host__ __device__
#else
#define SRA_HD
#endif
// Accesses of a row taken by rank 0 of a cta_pair cluster (rank 1 takes the rest
// and the scalar tail).
inline SRA_HD int64_t norm_pair_half(int64_t nvec) { return (nvec + 1) / 2; }

struct NormPlan {
    int variant;
    int vec;        // elements per access: 16 bytes' worth, or 1
    int nv;         // accesses per thread held in registers (warp / cta variants)
    int threads;    // threads per CTA
    int64_t grid;   // CTAs wanted; the launcher caps it at the resident count
    size_t smem;    // dynamic shared memory, bytes
    bool pdl;       // launch with programmatic stream serialization
    int num_sms;
    int stage_w;    // staged kernels: stage the w slice in shared memory
    int prefetch;   // L2 prefetch of the first rows before the launch wait
    int next_prefetch;  // L2 prefetch of each group's next row
    int group_warps;    // warps_row: warps per row (2, 4 or 8)
};

cudaError_t launch_rmsnorm(const NormArgs& a, const NormPlan& p, int dtype, cudaStream_t s);
cudaError_t launch_add_rmsnorm(const NormArgs& a, const NormPlan& p, int dtype, cudaStream_t s);

// ------------------------------------------------------------ RoPE + KV store
struct RopeArgs {
    void* q;
    const void* k;
    const void* v;
    const float* cos;
    const float* sin;
    const int64_t* pos;
    const int64_t* slot;
    void* cache;
    int32_t* err;
    int64_t T;
    int n_head, n_kv, head_dim;
    int64_t qs, ks, vs;  // token strides, elements
    int64_t max_pos, num_blocks;
    int block_size;
    // optional UClip of Q and K before the rotation (per-channel fp32, head_dim entries)
    const float* qa = nullptr;
    const float* qg = nullptr;
    const float* ka = nullptr;
    const float* kg = nullptr;
    float clip_lo = 0.0f, clip_hi = 0.0f;
};

// TOKEN_CTA: one task of P pairs per thread; TOKEN_CTA2: two tasks per thread sharing one
// cos / sin load (needs an even number of head units, n_head + 2 n_kv_head)
enum RopeVariant { ROPE_TOKEN_CTA = 0, ROPE_TOKEN_CTA2 = 1, ROPE_NUM_VARIANTS = 2 };

struct RopePlan {
    int variant;
    int style;      // 0 = neox (i, i + h), 1 = interleaved (2i, 2i + 1)
    bool qk_norm;   // UClip Q and K heads before rotating (RopeArgs::qa..kg)
    int pairs;      // rotation pairs per task: 16 bytes of elements per access, or 1
    int threads;    // threads per CTA
    int64_t grid;   // CTAs wanted (tokens are strided over the grid); capped at the resident count
    bool pdl;
    int num_sms;
};

cudaError_t launch_rope_kv_store(const RopeArgs& a, const RopePlan& p, int dtype, cudaStream_t s);

// ------------------------------------------------------------------- GLU
struct GluArgs {
    const void* gate_up;  // [T, 2I]
    void* out;            // [T, I]
    int64_t T, I;
    int64_t is, os;       // row strides, elements
};

enum GluVariant {
    GLU_COLS_ROWS = 0,       // columns over threads, rows over CTAs; 48 registers (five 256-thread CTAs per SM)
    GLU_COLS_ROWS_REGS = 1,  // the same kernel with the registers the compiler wants (A/B)
    GLU_NUM_VARIANTS = 2
};

struct GluPlan {
    int variant;
    int vec;        // elements per access (power of two, <= 16 bytes)
    int threads;    // threads per CTA (x)
    int64_t grid_x; // CTAs across the column vectors
    int64_t grid_y; // CTAs across rows (rows strided over grid_y); the launcher sizes it from occupancy
    bool pdl;
    int num_sms;
};

cudaError_t launch_glu(const GluArgs& a, const GluPlan& p, int act, int dtype, cudaStream_t s);

// ------------------------------------------------------------------- decode attention
struct AttnArgs {
    const void* q;             // [B, n_head, head_dim], token stride qs
    const void* cache;         // [2, num_blocks, block_size, n_kv, head_dim]
    const int32_t* table;      // [B, max_blocks]
    const int32_t* seq_lens;   // [B]
    void* out;                 // [B, n_head, head_dim], token stride os
    int32_t* err;              // nullable
    int64_t B, qs, os, num_blocks, max_blocks;
    int n_head, n_kv, group, block_size;
    float scale_log2;          // softmax scale * log2(e)
    // global split (tensor-core kernel): gsplits > 0 CTAs per (request, kv head), their partials
    // in the workspace, combined by the merge kernel launched after them
    int gsplits = 0;
    float* ws_part = nullptr;  // [B * n_kv][gsplits][16 + 8 * head_dim]
};

struct AttnPlan {
    int head_dim;  // 64, 128 or 256 (template)
    int splits;    // CTAs per (request, kv head): the cluster size
    int threads;
    int stages;    // K/V tiles in flight per CTA (CUDA-core path)
    bool tensor_cores;  // bf16 / fp16, head_dim 64 or 128: the mma.sync path
    bool tma = false;   // ... with the K / V tiles moved by TMA (decode_tma_kernel)
    int mma_warps = 8;  // warps per CTA of the mma.sync kernel: 8 (one CTA per SM) or 4 (two)
    size_t smem;
    bool pdl;
    int num_sms;
};

cudaError_t launch_decode_attention(const AttnArgs& a, const AttnPlan& p, int dtype, cudaStream_t s);
size_t decode_attention_smem(int group, int head_dim, int block_size, int stages, int es);
size_t decode_attention_mma_smem(int head_dim, int warps);
size_t decode_attention_tma_smem(int head_dim);
// Global-split plan of a decode-attention call: splits per (request, kv head) (0: none) and the
// workspace bytes it needs.
// at most this many global splits: the last CTA's merge buffers fit over its drained rings
constexpr int kMaxGsplits = 256;
int decode_attention_gsplits(int64_t B, int n_kv, int64_t max_blocks, int block_size, int num_sms);
int64_t decode_attention_ws_bytes(int64_t B, int n_kv, int head_dim, int gsplits);

// ------------------------------------------------------------------- fused linear
struct LinArgs {
    const void* x;     // [B, K] (RMSNorm prologue, or h itself) or gate_up [B, 2K] (GLU prologue), row stride xs
    const void* w_ln;  // [K] RMSNorm weight (RMSNorm prologue only)
    const void* W;     // [N, K] row-major (nn.Linear)
    void* y;           // [B, N], row stride ys
    int64_t B, K, N, xs, ys;
    float eps;
    // tcgen05 projection: where its K split's fp32 partials go through L2 ([N / 128][16][64][128]
    // in the caller's workspace), or null to sum them through the cluster's shared memory
    float* ws_part = nullptr;
};
// Workspace of the _ws projections: h [B, K] (rounded up to 256 bytes), then the tcgen05
// projection's partials where it serves the call.
inline int64_t linear_ws_h_bytes(int64_t B, int64_t K, int es) { return (B * K * es + 255) / 256 * 256; }
inline int64_t linear_ws_part_bytes(int64_t N) { return N / 128 * 16 * 64 * 128 * 4; }

struct LinPlan {
    int prologue;       // 0 RMSNorm, 1 SwiGLU, 2 ReGLU, 3 none (the input rows are h)
    bool tensor_cores;  // bf16 / fp16, K and N multiples of 64, 16-byte aligned layouts
    bool narrow;        // B <= 16: CTAs of 16 columns over all of K, no cluster
    int mt;             // 16-row m-tiles per CTA (1, 2 or 4)
    int splits;         // CTAs per cluster along K
    bool pdl;
    bool tcgen05;       // <= 64 rows, N a multiple of 128: the tcgen05 kernel (prologue 3, or the GLU or RMSNorm fused)
    int tc_stages = 4;  // its ring depth: 4 (two CTAs per SM) or 8 (one)
};

cudaError_t launch_linear(const LinArgs& a, const LinPlan& p, int dtype, cudaStream_t s);
size_t linear_smem(int mt, int prologue);
size_t linear_tc_smem(int stages, int prologue = 3, int nx = 0);
// nx: with the RMSNorm fused (prologue 0), the K tiles of x a CTA holds (at most 16)
int linear_tc_max_clusters(int splits, int stages, bool bf16, int prologue = 3, int nx = 0);
int linear_tc_norm_ctas_per_sm(int nx, bool bf16);  // the fused-RMSNorm kernel's CTAs per SM
unsigned int linear_wait_timeouts();  // bounded waits of the fused-projection kernels that ran out
unsigned int attn_wait_timeouts();    // bounded waits of the TMA-fed attention kernel that ran out
cudaError_t launch_wait_selftest(int32_t* out, cudaStream_t s);  // a wait on a barrier nothing completes
size_t linear16_smem(int rows, int64_t K, int splits);

// ------------------------------------------------------------------- UClip
struct UclipArgs {
    const void* x;       // [N, H, D], strides (xn, xh, 1)
    const float* alpha;  // D entries if alpha_pc, else 1
    const float* gamma;  // D entries if gamma_pc, else 1
    void* out;           // [N, H, D], strides (on, oh, 1)
    int64_t N, H, D;
    int64_t xn, xh, on, oh;  // elements
    bool alpha_pc, gamma_pc;
    float lo, hi;
};

struct UclipPlan {
    int vec;         // elements per access (power of two, <= 16 bytes)
    int bx, by;      // CTA shape: column groups x rows
    int64_t grid_x;  // CTAs across the column groups
    int64_t grid_y;  // CTAs across rows (upper bound; the launcher caps it at one resident wave)
    bool pdl;
    int num_sms;
};

cudaError_t launch_uclip(const UclipArgs& a, const UclipPlan& p, int dtype, cudaStream_t s);

}  // namespace sra
