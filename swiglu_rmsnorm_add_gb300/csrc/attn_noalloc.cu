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

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "sra.h"

// Room for the partials of every split this library plans on a GPU of up to 252 SMs
// at head_dim 128 (the merge needs at most 256 bytes of counters plus one
// (16 + 8 * head_dim) float record per CTA, and it plans at most one CTA per SM).
static constexpr int64_t kScratchBytes = SRA_NOALLOC_SCRATCH_BYTES;

// Every GPU that loads this library holds this array until the process exits.
// Zero at load; each call clears its counters before the kernel runs.
static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of the array on the current device. Host code sees only a host-side
// stand-in for g_attn_scratch, so the address comes from the runtime, once per device,
// with that device current. Returns nullptr when the runtime cannot give it.
void* scratch_on_current_device(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p) return p;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return nullptr;
    }
    g_scratch_addr[dev].store(p, std::memory_order_release);
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
    // the per-(request, kv head) arrival counters lead the scratch; the kernel's last CTA
    // leaves them at zero, but they are cleared here too, so a call never depends on how
    // an earlier one ended
    const size_t counters = static_cast<size_t>((B * n_kv_head * 4 + 255) / 256 * 256);
    if (cudaMemsetAsync(scratch, 0, counters, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return SRA_ERR_LAUNCH;
    }
    return sra_paged_decode_attention_ws(q, kv_cache, block_table, seq_lens, out, B, n_head, n_kv_head, head_dim,
                                         q_tok_stride, out_tok_stride, num_blocks, block_size, max_blocks_per_seq,
                                         scale, scratch, kScratchBytes, err_count, dtype, stream);
}

}  // extern "C"
