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
};

enum NormVariant {
    NORM_WARP_ROWS = 0,  // one warp per row, row held in registers
    NORM_CTA_ROW = 1,    // one CTA per row, row held in registers
    NORM_CTA_SMEM = 2,   // one CTA per row, row staged in shared memory
    NORM_TWO_PASS = 3,   // one CTA per row, second pass re-reads the row (any D)
    NORM_NUM_VARIANTS = 4
};

struct NormPlan {
    int variant;
    int vec;        // elements per access: 16 bytes' worth, or 1
    int nv;         // accesses per thread held in registers (warp / cta variants)
    int threads;    // threads per CTA
    int64_t grid;   // CTAs
    size_t smem;    // dynamic shared memory, bytes
};

cudaError_t launch_rmsnorm(const NormArgs& a, const NormPlan& p, int dtype, cudaStream_t s);
cudaError_t launch_add_rmsnorm(const NormArgs& a, const NormPlan& p, int dtype, cudaStream_t s);
// Largest dynamic shared memory the CTA_SMEM variant may request on this device.
cudaError_t norm_smem_prepare(int dtype, bool add, int vec, size_t bytes);

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
};

enum RopeVariant { ROPE_TOKEN_CTA = 0, ROPE_NUM_VARIANTS = 1 };

struct RopePlan {
    int variant;
    int pairs;      // rotation pairs per task: 16 bytes of elements per half, or 1
    int threads;    // threads per CTA
    int64_t grid;   // CTAs (tokens are strided over the grid)
};

cudaError_t launch_rope_kv_store(const RopeArgs& a, const RopePlan& p, int dtype, cudaStream_t s);

// ------------------------------------------------------------------- GLU
struct GluArgs {
    const void* gate_up;  // [T, 2I]
    void* out;            // [T, I]
    int64_t T, I;
    int64_t is, os;       // row strides, elements
};

enum GluVariant { GLU_COLS_ROWS = 0, GLU_NUM_VARIANTS = 1 };

struct GluPlan {
    int variant;
    int vec;        // elements per access (power of two, <= 16 bytes)
    int threads;    // threads per CTA (x)
    int64_t grid_x; // CTAs across the column vectors
    int64_t grid_y; // CTAs across rows (rows strided over grid_y)
};

cudaError_t launch_glu(const GluArgs& a, const GluPlan& p, int act, int dtype, cudaStream_t s);

}  // namespace sra
