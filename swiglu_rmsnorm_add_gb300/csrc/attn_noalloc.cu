// Paged decode attention for callers that cannot allocate device memory.
//
// sra_paged_decode_attention_ws splits a long context over many CTAs and merges
// their partial results through a workspace the caller allocates. Some callers
// cannot make that allocation: code running inside a memory pool it does not own
// (an inference server whose allocator hands out only KV-cache blocks), a plugin
// loaded into another framework's process that must not call cudaMalloc behind
// that framework's back, or a latency-bound decode loop that cannot afford the
// device-wide synchronisation a cudaMalloc or cudaFree may bring. This file gives
// them the same kernel with its scratch in one fixed device array that the library
// itself holds.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "sra.h"

// Room for the partials of every split this library plans on a GPU of up to 252 SMs
// at head_dim 128 (a leading area of at most 256 bytes plus one (16 + 8 * head_dim)
// float record per CTA, and it plans at most one CTA per SM).
static constexpr int64_t kScratchBytes = SRA_NOALLOC_SCRATCH_BYTES;

// Every GPU that loads this library holds this array until the process exits.
// Each call writes the records it then reads; nothing carries over between calls.
static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

// The context a cached address belongs to: the driver's process-unique context id
// (cuCtxGetId; a handle value can be reused by a context created after a reset, an
// id never is). 0 when the driver cannot tell, and then nothing is cached.
unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static const GetCurrent get_current = [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return static_cast<GetCurrent>(nullptr);
        }
        return reinterpret_cast<GetCurrent>(fn);
    }();
    static const GetId get_id = [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return static_cast<GetId>(nullptr);
        }
        return reinterpret_cast<GetId>(fn);
    }();
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

std::mutex g_mu;
unsigned long long g_ctx_id[kMaxDevices];
void* g_addr[kMaxDevices];

// Device address of the array in the current device's context. Host code sees only a
// host-side stand-in for g_attn_scratch, so the address comes from the runtime, with the
// device current: once per device, and again whenever that device's context has
// changed since (after cudaDeviceReset the array lives in a new context). A call made
// before the runtime has made the device's context current is answered but not cached.
// Returns nullptr when the runtime cannot give the address.
void* scratch_on_current_device(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(g_mu);
    if (id != 0 && g_ctx_id[dev] == id && g_addr[dev]) return g_addr[dev];
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return nullptr;
    }
    g_ctx_id[dev] = id;
    g_addr[dev] = id != 0 ? p : nullptr;
    return p;
}

}  // namespace

extern "C" {

int sra_paged_decode_attention_noalloc(const void* q, const void* kv_cache, const int32_t* block_table,
                                       const int32_t* seq_lens, void* out, int64_t B, int n_head, int n_kv_head,
                                       int head_dim, int64_t q_tok_stride, int64_t out_tok_stride,
                                       int64_t num_blocks, int block_size, int64_t max_blocks_per_seq, float scale,
                                       int32_t* err_count, int dtype, void* stream) {
    const int64_t need = sra_paged_decode_attention_workspace_size(B, n_head, n_kv_head, head_dim,
                                                                    max_blocks_per_seq, block_size, dtype);
    if (need < 0) return static_cast<int>(need);
    if (need > kScratchBytes) return SRA_ERR_SHAPE;
    if (need == 0)  // this shape takes the cluster kernel, which needs no scratch
        return sra_paged_decode_attention(q, kv_cache, block_table, seq_lens, out, B, n_head, n_kv_head, head_dim,
                                          q_tok_stride, out_tok_stride, num_blocks, block_size, max_blocks_per_seq,
                                          scale, err_count, dtype, stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SRA_ERR_DEVICE;
    }
    void* scratch = scratch_on_current_device(dev);
    if (!scratch) return SRA_ERR_DEVICE;
    return sra_paged_decode_attention_ws(q, kv_cache, block_table, seq_lens, out, B, n_head, n_kv_head, head_dim,
                                         q_tok_stride, out_tok_stride, num_blocks, block_size, max_blocks_per_seq,
                                         scale, scratch, kScratchBytes, err_count, dtype, stream);
}

}  // extern "C"
