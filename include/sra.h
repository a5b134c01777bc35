/*
 * sra.h — C ABI of the GB300 (sm_103a) per-token decoder-path library.
 *
 * Bandwidth-bound operators of a transformer decoder layer, each a
 * hand-written CUDA kernel chosen per shape:
 *
 *   sra_rmsnorm        row-wise RMSNorm, fp32 accumulation
 *   sra_add_rmsnorm    residual add (in place) + RMSNorm
 *   sra_rope_kv_store  neox RoPE of Q and K + paged KV-cache store through slot_mapping (GQA)
 *                      (sra_rope_kv_store_ex: also the interleaved GPT-J pairing;
 *                      sra_rope_kv_store_qk_uclip: with the Q/K UClip norms fused in)
 *   sra_glu            SwiGLU silu(gate) * up, or ReGLU relu(gate) * up, over a fused gate_up
 *   sra_uclip          UClip / DyHT clamp(alpha * x, lo, hi) * gamma over [N, H, D] views
 *   sra_paged_decode_attention  softmax decode attention read through the paged cache's block table
 *   sra_rmsnorm_linear / sra_glu_linear  RMSNorm / GLU fused into the projection they feed
 *   sra_rmsnorm_linear_ws / sra_glu_linear_ws  the same, given a workspace for larger batches
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers to tensors are DEVICE pointers (any memory the current device can
 *    load from and store to). The caller owns every buffer; the library never
 *    allocates, frees, zero-fills or keeps a pointer after the call returns.
 *    Two exceptions, both library-owned device arrays in the library's own
 *    module: the scratch array of sra_paged_decode_attention_noalloc (which that
 *    call writes its partial results into, and whose address it keeps per
 *    device), and the counter of bounded device waits that ran out
 *    (sra_wait_timeouts).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). Every call only enqueues work on that stream and returns at once;
 *    results are visible after the stream is synchronised. The kernel runs on
 *    the device that is current for the calling thread.
 *  - Strides are in ELEMENTS, not bytes; the innermost (column) stride is 1.
 *  - Any pointer alignment is accepted. 16-byte aligned rows and strides get the
 *    128-bit vector kernels; other layouts get narrower accesses.
 *  - Return value: SRA_OK (0) or a negative sra_status. Argument errors are
 *    found on the host BEFORE anything is enqueued: on error nothing runs and
 *    no output byte changes. SRA_ERR_LAUNCH reports a failed kernel launch
 *    (cudaGetLastError after the launch). A zero-sized call (rows == 0 or
 *    T == 0) validates its arguments, enqueues nothing and returns SRA_OK.
 *  - No call waits for the device to finish, and no kernel traps or asserts. The
 *    device-side waits are the fused projections' and the TMA-fed attention
 *    variant's waits for their own tile copies, each bounded and counted when it
 *    runs out (sra_wait_timeouts), and the cluster kernels' barriers among the
 *    CTAs of one cluster, which the hardware schedules together.
 *  - Thread safety: calls may be made concurrently from several host threads.
 *    sra_force_variant changes process-wide state and is meant for A/B
 *    measurement only.
 *
 * Sources. The operators are those of these web pages (cited by title and section):
 *  [koas] koas-w.github.io "preformanceimprovement": sec. 1 fused RoPE + paged KV
 *         cache store; sec. 2 fused SwiGLU; sec. 3 Triton RMSNorm; sec. 4 fused add + norm.
 *  [lsln] m.lsln.cn/news/61269 "21 个算子": sec. 2.2 fusion choices (ln1 + qkv_proj);
 *         sec. 2.3 RMSNorm and RoPE details; sec. 3 split reductions; sec. 5.3 cache read.
 *  [mer]  mer.dev "AsyncT vllm 适配加速笔记（一）": sec. 0 DyHT replacing RMSNorm;
 *         sec. 1.1 KV-cache layout; sec. 3.3 kernel fusion (ReGLU as relu_and_mul;
 *         the UClip kernel; stride-aware Q/K views).
 *  [csdn] agent.csdn.net "使用Triton实现RMSNorm算子": RMSNorm kernels and pitfalls.
 */
#ifndef SRA_H_
#define SRA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SRA_VERSION 1

#if defined(__GNUC__)
#define SRA_API __attribute__((visibility("default")))
#else
#define SRA_API
#endif

typedef enum sra_dtype {
    SRA_F32 = 0,  /* IEEE binary32 */
    SRA_F16 = 1,  /* IEEE binary16 */
    SRA_BF16 = 2  /* bfloat16 */
} sra_dtype_t;

typedef enum sra_status {
    SRA_OK = 0,
    SRA_ERR_NULL = -1,     /* a required pointer is NULL */
    SRA_ERR_SHAPE = -2,    /* a size is out of range (negative count, D <= 0, odd head_dim, ...) */
    SRA_ERR_STRIDE = -3,   /* a row / token stride is smaller than the row it must hold */
    SRA_ERR_DTYPE = -4,    /* dtype is not one of sra_dtype_t */
    SRA_ERR_ALIAS = -5,    /* outputs overlap inputs in a way the operator forbids */
    SRA_ERR_ARG = -6,      /* any other invalid argument (unknown activation, op name, ...) */
    SRA_ERR_VARIANT = -7,  /* a forced kernel variant cannot handle this call */
    SRA_ERR_LAUNCH = -8,   /* the CUDA launch failed (no device, bad context, ...) */
    SRA_ERR_DEVICE = -9    /* the device could not be queried */
} sra_status_t;

typedef enum sra_rope_style {
    SRA_ROPE_NEOX = 0,        /* pairs (i, i + head_dim/2): rotate halves       [koas] sec. 1 */
    SRA_ROPE_INTERLEAVED = 1  /* pairs (2i, 2i + 1): GPT-J even/odd partners    [lsln] sec. 2.3 */
} sra_rope_style_t;

typedef enum sra_act {
    SRA_ACT_SILU = 0,  /* SwiGLU: silu(g) * u, silu(g) = g / (1 + e^-g)   [koas] sec. 2 */
    SRA_ACT_RELU = 1   /* ReGLU:  max(g, 0) * u                            [mer] sec. 3.3 */
} sra_act_t;

/*
 * sra_rmsnorm — [koas] sec. 3, [lsln] sec. 2.3, [csdn].
 *
 *   out[r, j] = x[r, j] * rsqrt( (1/D) * sum_k x[r, k]^2 + eps ) * w[j]
 *
 * x:    [rows, D] of dtype, row r at x + r * x_row_stride (x_row_stride >= D).
 * w:    [D] of dtype, contiguous.
 * out:  [rows, D] of dtype, row r at out + r * out_row_stride (>= D).
 *       out may equal x exactly (in-place); any other overlap with x or w is
 *       SRA_ERR_ALIAS.
 * eps:  added to the mean of squares inside the root (eps >= 0).
 * Arithmetic: inputs widened to fp32, fp32 sum of squares, one round-to-nearest-
 * even to dtype on the store.
 * Errors: NULL x/w/out (unless rows == 0) -> SRA_ERR_NULL; rows < 0 or D <= 0 ->
 * SRA_ERR_SHAPE; stride < D -> SRA_ERR_STRIDE; eps < 0 or not finite -> SRA_ERR_ARG.
 */
SRA_API int sra_rmsnorm(const void* x, const void* w, void* out, int64_t rows, int64_t D,
                int64_t x_row_stride, int64_t out_row_stride, float eps, int dtype,
                void* stream);

/*
 * sra_add_rmsnorm — [koas] sec. 4 (x updated in place with the residual, the
 * normalised result returned; read once, write twice).
 *
 *   x[r, j]   <- round_dtype( x[r, j] + res[r, j] )        (stored in place)
 *   out[r, j]  = rmsnorm of the ROUNDED, stored x[r, :] as in sra_rmsnorm
 *
 * x:    [rows, D] in/out, row stride x_row_stride (>= D).
 * res:  [rows, D] input, row stride res_row_stride (>= D). res may equal x exactly.
 * w:    [D] contiguous.
 * out:  [rows, D] output, row stride out_row_stride (>= D). out must not overlap
 *       x, res or w (SRA_ERR_ALIAS).
 * The stored sum is the correctly rounded x + res (fp32 add of two dtype values,
 * then one RNE to dtype).
 * Errors: as sra_rmsnorm, plus NULL res.
 */
SRA_API int sra_add_rmsnorm(void* x, const void* res, const void* w, void* out, int64_t rows, int64_t D,
                    int64_t x_row_stride, int64_t res_row_stride, int64_t out_row_stride,
                    float eps, int dtype, void* stream);

/*
 * sra_rope_kv_store — [koas] sec. 1 (RoPE fused with the paged KV-cache store,
 * GQA through kv_head = head / (n_head / n_kv_head)); cache layout from [mer]
 * sec. 1.1.
 *
 * For token t with p = pos[t], h = head_dim / 2, c = cos[p*h + i], s = sin[p*h + i]
 * (neox half rotation, i < h):
 *   y[i]     = x[i] * c - x[i + h] * s
 *   y[i + h] = x[i + h] * c + x[i] * s
 * - every Q head of token t is rotated IN PLACE in q;
 * - every K head is rotated and written to kv_cache[0, b, o, kvh, :] and every
 *   V head copied bit-for-bit to kv_cache[1, b, o, kvh, :], where
 *   b = slot_mapping[t] / block_size and o = slot_mapping[t] % block_size.
 * No other byte of the cache or of q changes; k and v are read-only.
 *
 * q:        [T, n_head, head_dim] of dtype; token t at q + t * q_tok_stride
 *           (>= n_head * head_dim); heads contiguous within a token.
 * k, v:     [T, n_kv_head, head_dim]; token strides k_tok_stride, v_tok_stride
 *           (>= n_kv_head * head_dim). q, k and v may be views of one fused QKV
 *           buffer; q must not overlap k or v.
 * cos, sin: fp32 tables [max_pos, head_dim / 2], contiguous.
 * pos, slot_mapping: int64 [T].
 * kv_cache: [2, num_blocks, block_size, n_kv_head, head_dim] of dtype, contiguous.
 * err_count: NULL, or a device int32 the kernel atomically increments by one for
 *           every token whose position is outside [0, max_pos) and one more for
 *           every token whose slot is >= num_blocks * block_size. The caller
 *           zeroes it; the library only adds.
 * Token rules: a position outside [0, max_pos) leaves q[t] unchanged and writes
 * nothing to the cache; slot < 0 marks a padding token (Q still rotated, nothing
 * written to the cache, not an error); a slot past the cache is skipped (and
 * counted). Two tokens with the same valid slot race (undefined which wins).
 * Errors (host): NULL pointers (err_count may be NULL) -> SRA_ERR_NULL;
 * T < 0, n_head <= 0, n_kv_head <= 0, n_head % n_kv_head != 0, head_dim <= 0 or
 * odd, block_size <= 0, num_blocks < 0, max_pos < 0 -> SRA_ERR_SHAPE;
 * short strides -> SRA_ERR_STRIDE.
 */
SRA_API int sra_rope_kv_store(void* q, const void* k, const void* v, const float* cos, const float* sin,
                      const int64_t* pos, const int64_t* slot_mapping, void* kv_cache, int64_t T,
                      int n_head, int n_kv_head, int head_dim, int64_t q_tok_stride,
                      int64_t k_tok_stride, int64_t v_tok_stride, int64_t max_pos,
                      int64_t num_blocks, int block_size, int32_t* err_count, int dtype,
                      void* stream);

/*
 * sra_rope_kv_store_ex — sra_rope_kv_store with the rotation pairing chosen by
 * `style` (sra_rope_style_t). SRA_ROPE_INTERLEAVED rotates the pairs (2i, 2i + 1)
 * with c = cos[p*h + i], s = sin[p*h + i] ([lsln] sec. 2.3: each even dimension and
 * the next odd one form a pair); the tables, cache layout, token rules and errors
 * are those of sra_rope_kv_store. An unknown style -> SRA_ERR_ARG.
 */
SRA_API int sra_rope_kv_store_ex(void* q, const void* k, const void* v, const float* cos, const float* sin,
                                 const int64_t* pos, const int64_t* slot_mapping, void* kv_cache, int64_t T,
                                 int n_head, int n_kv_head, int head_dim, int64_t q_tok_stride,
                                 int64_t k_tok_stride, int64_t v_tok_stride, int64_t max_pos,
                                 int64_t num_blocks, int block_size, int32_t* err_count, int style, int dtype,
                                 void* stream);

/*
 * sra_rope_kv_store_qk_uclip — sra_rope_kv_store_ex with the Q and K norms of
 * [mer] sec. 3.3 fused into the load: every Q head and every K head is first
 * replaced by UClip clamp(alpha_d * x_d, clip_min, clip_max) * gamma_d (fp32,
 * rounded once to the dtype, exactly as sra_uclip would store it) and then rotated;
 * the normed, rotated K goes to the cache, q holds the normed, rotated Q. V is
 * copied unchanged. A token whose position is out of range is left as it is (q
 * not normed either) and counted, as in sra_rope_kv_store.
 * q_alpha, q_gamma, k_alpha, k_gamma: fp32 device arrays of head_dim entries,
 * shared by all heads of their kind (pass head_dim copies for a scalar).
 * Errors: those of sra_rope_kv_store_ex; a NULL parameter -> SRA_ERR_NULL; a NaN
 * bound or clip_min > clip_max -> SRA_ERR_ARG; a parameter array overlapping q or
 * the cache -> SRA_ERR_ALIAS.
 */
SRA_API int sra_rope_kv_store_qk_uclip(void* q, const void* k, const void* v, const float* cos, const float* sin,
                                       const int64_t* pos, const int64_t* slot_mapping, void* kv_cache, int64_t T,
                                       int n_head, int n_kv_head, int head_dim, int64_t q_tok_stride,
                                       int64_t k_tok_stride, int64_t v_tok_stride, int64_t max_pos,
                                       int64_t num_blocks, int block_size, int32_t* err_count, int style,
                                       const float* q_alpha, const float* q_gamma, const float* k_alpha,
                                       const float* k_gamma, float clip_min, float clip_max, int dtype,
                                       void* stream);

/*
 * sra_glu — [koas] sec. 2 (SwiGLU: gate and up loaded together, activation and
 * product in registers, one write), [mer] sec. 3.3 (ReGLU, relu_and_mul).
 *
 *   out[t, j] = act( gate_up[t, j] ) * gate_up[t, I + j],   0 <= j < I
 *
 * gate_up: [T, 2I] of dtype (gate = first I columns, up = last I), row stride
 *          in_row_stride (>= 2I).
 * out:     [T, I] of dtype, row stride out_row_stride (>= I); must not overlap gate_up.
 * act:     SRA_ACT_SILU or SRA_ACT_RELU. fp32 arithmetic, one RNE on the store.
 * Errors: NULL -> SRA_ERR_NULL; T < 0 or I <= 0 -> SRA_ERR_SHAPE; short strides
 * -> SRA_ERR_STRIDE; unknown act -> SRA_ERR_ARG; overlap -> SRA_ERR_ALIAS.
 */
SRA_API int sra_glu(const void* gate_up, void* out, int64_t T, int64_t I, int64_t in_row_stride,
            int64_t out_row_stride, int act, int dtype, void* stream);

/* sra_swiglu — sra_glu with act = SRA_ACT_SILU (the call swiglu(gate_up, out, T, I) on contiguous rows). */
SRA_API int sra_swiglu(const void* gate_up, void* out, int64_t T, int64_t I, int64_t in_row_stride,
               int64_t out_row_stride, int dtype, void* stream);

/*
 * sra_paged_decode_attention — the read side of the paged cache: [mer] sec. 1.1
 * (cache [2, num_blocks, block_size, n_kv, head] with a block table and seq lens
 * per request), sec. 2.2 (the K/V load is the cost; query heads sharing a KV head
 * share its load) and sec. 3.1 (a decode kernel reading that layout through the
 * block table); [lsln] sec. 2.1 and 5.3 (qk_score, scale + softmax and pv_agg over
 * cache_kv_read) and sec. 3.2 (a split reduction merged through each part's max
 * and sum of exponentials).
 *
 *   out[b, h, :] = sum_{t < seq_lens[b]} softmax_t(scale * q[b, h, :] . K_t) V_t
 *
 * with K_t / V_t the rows of kv head h / (n_head / n_kv_head) at block
 * block_table[b, t / block_size], offset t % block_size. fp32 arithmetic (scores
 * in base 2, an online softmax per split, the splits merged in fp32), one RNE to
 * the dtype.
 *
 * q:           [B, n_head, head_dim] of `dtype`, heads contiguous, token stride
 *              q_tok_stride. Read only.
 * kv_cache:    [2, num_blocks, block_size, n_kv_head, head_dim] of `dtype`,
 *              contiguous and 16-byte aligned; plane 0 = K, plane 1 = V (what
 *              sra_rope_kv_store writes). Read only.
 * block_table: int32 [B, max_blocks_per_seq], row-major. Read only.
 * seq_lens:    int32 [B]. Read only.
 * out:         [B, n_head, head_dim] of `dtype`, token stride out_tok_stride; it
 *              must not overlap q, the cache, the table or seq_lens.
 * scale:       any finite float (1 / sqrt(head_dim) for the usual attention).
 * err_count:   nullable device int32, incremented (atomically) once per request
 *              whose seq_len lies outside [0, max_blocks_per_seq * block_size]
 *              (it is clamped into that range) and once per used block entry
 *              outside [0, num_blocks) (that block's tokens are skipped). A request
 *              left with no token gets zeros.
 * Supported shapes: head_dim 64, 128 or 256; block_size 8, 16 or 32; n_head /
 * n_kv_head <= 8. Others -> SRA_ERR_SHAPE.
 * Errors: unknown dtype -> SRA_ERR_DTYPE; bad sizes -> SRA_ERR_SHAPE; a token
 * stride below n_head * head_dim -> SRA_ERR_STRIDE; a non-finite scale or a cache
 * not 16-byte aligned -> SRA_ERR_ARG; NULL -> SRA_ERR_NULL; overlap ->
 * SRA_ERR_ALIAS. B == 0 is a no-op.
 */
SRA_API int sra_paged_decode_attention(const void* q, const void* kv_cache, const int32_t* block_table,
                                       const int32_t* seq_lens, void* out, int64_t B, int n_head, int n_kv_head,
                                       int head_dim, int64_t q_tok_stride, int64_t out_tok_stride,
                                       int64_t num_blocks, int block_size, int64_t max_blocks_per_seq, float scale,
                                       int32_t* err_count, int dtype, void* stream);

/*
 * sra_paged_decode_attention_ws — sra_paged_decode_attention with a caller-owned
 * workspace. When few (request, kv head) pairs meet a long context (the case a
 * cluster of up to 16 splits cannot spread over the GPU, e.g. one request with
 * 32 k cached tokens), the tensor-core kernel splits every pair over many
 * independent CTAs ([lsln] sec. 3: split the reduction, then merge the parts by
 * their max and sum of exponentials); each writes its partial result into the
 * workspace and a second kernel, launched right after them on the same stream,
 * merges them. Otherwise the workspace is unused and the call is
 * sra_paged_decode_attention.
 * workspace: device memory of at least
 *   sra_paged_decode_attention_workspace_size(B, n_head, n_kv_head, head_dim,
 *                                             max_blocks_per_seq, block_size, dtype)
 *   bytes, 16-byte aligned; its contents on entry do not matter (a leading area,
 *   kept for the layout, is never written). It must not overlap any other
 *   argument, and calls that share a workspace must not run concurrently (same
 *   stream, or ordered by events).
 * Errors: those of sra_paged_decode_attention; workspace_bytes below the size the
 * shape needs, a negative size or a misaligned workspace -> SRA_ERR_ARG.
 */
SRA_API int sra_paged_decode_attention_ws(const void* q, const void* kv_cache, const int32_t* block_table,
                                          const int32_t* seq_lens, void* out, int64_t B, int n_head,
                                          int n_kv_head, int head_dim, int64_t q_tok_stride,
                                          int64_t out_tok_stride, int64_t num_blocks, int block_size,
                                          int64_t max_blocks_per_seq, float scale, void* workspace,
                                          int64_t workspace_bytes, int32_t* err_count, int dtype, void* stream);

/*
 * Workspace bytes sra_paged_decode_attention_ws needs for this shape on the
 * current device (0: the shape takes the cluster kernel and needs none); a
 * negative sra_status for sizes sra_paged_decode_attention would reject.
 */
SRA_API int64_t sra_paged_decode_attention_workspace_size(int64_t B, int n_head, int n_kv_head, int head_dim,
                                                          int64_t max_blocks_per_seq, int block_size, int dtype);

/*
 * sra_paged_decode_attention_noalloc — sra_paged_decode_attention_ws for callers
 * that cannot allocate device memory: a library running inside a serving stack
 * whose allocator owns all of the GPU's memory, a plugin that must not call
 * cudaMalloc behind its host framework's back, or a decode loop that cannot take
 * the device-wide synchronisation cudaMalloc / cudaFree may cause. The pages this
 * library follows have no counterpart to it: it exists only for such callers.
 * Its scratch is one library-owned device array of SRA_NOALLOC_SCRATCH_BYTES,
 * present (and held until the process exits) on every GPU that loads the
 * library; the call allocates nothing and calls no allocating routine.
 * Arguments, layout and results are those of sra_paged_decode_attention; on this
 * library's planning the result equals sra_paged_decode_attention_ws's.
 * Set-up: the first call on a device looks up the array's device address on that
 * device (with it current); make that first call before any stream capture. The
 * address is kept per device and looked up again when the device's context has
 * changed (a call after cudaDeviceReset finds the array in the new context).
 * Every call writes the partial results it then merges; nothing carries over.
 * Races: all calls on a device share the one array, so two calls that may run at
 * the same time on the GPU (different streams without an event between them, or
 * different host threads) corrupt each other's partial results; order them on one
 * stream. Shapes that need no scratch run the cluster kernel and share nothing.
 * Errors: those of sra_paged_decode_attention_ws; a shape whose scratch would
 * exceed SRA_NOALLOC_SCRATCH_BYTES -> SRA_ERR_SHAPE (none does on a GPU of up to
 * 252 SMs); the array's address not available -> SRA_ERR_DEVICE.
 */
#define SRA_NOALLOC_SCRATCH_BYTES (1 << 20)
SRA_API int sra_paged_decode_attention_noalloc(const void* q, const void* kv_cache, const int32_t* block_table,
                                               const int32_t* seq_lens, void* out, int64_t B, int n_head,
                                               int n_kv_head, int head_dim, int64_t q_tok_stride,
                                               int64_t out_tok_stride, int64_t num_blocks, int block_size,
                                               int64_t max_blocks_per_seq, float scale, int32_t* err_count,
                                               int dtype, void* stream);

/*
 * sra_rmsnorm_linear — RMSNorm as the prologue of the projection it feeds
 * ([lsln] sec. 2.2: ln1 + qkv_proj fused, the normed rows never stored):
 *
 *   h[b, :] = RNE(x[b, :] * rsqrt(mean_k x[b, k]^2 + eps) * w_ln[:])   (as sra_rmsnorm)
 *   y[b, n] = RNE(sum_k h[b, k] * W[n, k])
 *
 * x:    [B, K] of `dtype`, row stride x_row_stride (>= K). Read only.
 * w_ln: [K] RMSNorm weight of `dtype`. Read only.
 * W:    [N, K] of `dtype`, row-major (nn.Linear's [out, in] layout). Read only.
 * y:    [B, N] of `dtype`, row stride y_row_stride (>= N); must not overlap x, w_ln or W.
 * bf16 / fp16 with K and N multiples of 64 and 16-byte aligned x, w_ln, W (x_row_stride a
 * multiple of 8) run on the tensor cores (fp32 accumulation; with N a multiple of 128, from
 * 33 to 64 rows, or from 17 with K >= 4096, on the fifth-generation tensor cores in one
 * kernel that also takes the norm); other layouts and fp32 run a CUDA-core kernel with the
 * same result up to the order of the fp32 sums.
 * Errors: unknown dtype -> SRA_ERR_DTYPE; B < 0, K <= 0 or N <= 0 (or K too long for
 * one CTA's shared memory on the CUDA-core path) -> SRA_ERR_SHAPE; short strides ->
 * SRA_ERR_STRIDE; eps negative or not finite -> SRA_ERR_ARG; NULL -> SRA_ERR_NULL;
 * overlap -> SRA_ERR_ALIAS. B == 0 is a no-op.
 */
SRA_API int sra_rmsnorm_linear(const void* x, const void* w_ln, const void* W, void* y, int64_t B, int64_t K,
                               int64_t N, int64_t x_row_stride, int64_t y_row_stride, float eps, int dtype,
                               void* stream);

/*
 * sra_glu_linear — the gated activation as the prologue of the down projection
 * ([lsln] sec. 2.2 applied to the MLP; [koas] sec. 2 / [mer] sec. 3.3 for the
 * activation):
 *
 *   h[b, i] = RNE(act(gate_up[b, i]) * gate_up[b, I + i])   (as sra_glu)
 *   y[b, n] = RNE(sum_i h[b, i] * W[n, i])
 *
 * gate_up: [B, 2I] of `dtype`, row stride in_row_stride (>= 2I). W: [N, I] row-major.
 * y: [B, N], row stride y_row_stride. act: sra_act_t. Layout rules, paths and errors
 * as sra_rmsnorm_linear (an unknown act -> SRA_ERR_ARG), except that the one kernel on the
 * fifth-generation tensor cores, computing the activation itself, serves from 4 rows.
 */
SRA_API int sra_glu_linear(const void* gate_up, const void* W, void* y, int64_t B, int64_t I, int64_t N,
                           int64_t in_row_stride, int64_t y_row_stride, int act, int dtype, void* stream);

/*
 * sra_rmsnorm_linear_ws / sra_glu_linear_ws — the same projections given a caller
 * workspace (the library allocates nothing). The fused kernels rebuild the prologue's
 * rows once per 64-column slice of y; at larger batches that repeated work dominates, so
 * from 32 rows (bf16 / fp16, K and N multiples of 64, 16-byte aligned W and workspace)
 * the prologue runs once in its own kernel (as sra_rmsnorm / sra_glu), writing
 * h [B, K] (row stride K) into the workspace, and the projection then streams W against
 * h. Below that, or for other layouts, the fused kernel runs and the workspace is not
 * touched. The result is the same computation (h rounded to the dtype, then one rounding
 * of the product; y may differ from the fused call's in the last bit where an h element
 * lands on the other side of a rounding midpoint).
 * workspace: device memory of at least B * K (sra_glu_linear_ws: B * I) elements of
 * `dtype`, 16-byte aligned, overlapping no other argument; its contents on return are
 * unspecified (from 32 rows it holds h). A NULL workspace runs the fused kernel; where the
 * split applies, a workspace smaller than B * K elements -> SRA_ERR_ARG and one that
 * overlaps another argument -> SRA_ERR_ALIAS. Other arguments and errors as
 * sra_rmsnorm_linear / sra_glu_linear. The projection over h runs a warp-specialised
 * kernel: a producer warp streams W and h tiles by TMA, the other warps multiply.
 * A workspace of sra_linear_workspace_size(B, K, N, dtype) bytes (more than B * K
 * elements where the tcgen05 projection serves the call: up to 64 rows, N a multiple
 * of 128) also holds that projection's K-split partials, which it then sums through
 * L2 rather than through the cluster's shared memory; the result is the same.
 * Calls that share a workspace must not overlap on the GPU.
 */
SRA_API int sra_rmsnorm_linear_ws(const void* x, const void* w_ln, const void* W, void* y, int64_t B, int64_t K,
                                  int64_t N, int64_t x_row_stride, int64_t y_row_stride, float eps, void* workspace,
                                  int64_t workspace_bytes, int dtype, void* stream);
SRA_API int sra_glu_linear_ws(const void* gate_up, const void* W, void* y, int64_t B, int64_t I, int64_t N,
                              int64_t in_row_stride, int64_t y_row_stride, int act, void* workspace,
                              int64_t workspace_bytes, int dtype, void* stream);
/* Bytes of the workspace the _ws projections use best for these sizes (K = I for the GLU
 * one): B * K elements of `dtype` rounded up to 256 bytes, plus the tcgen05 projection's
 * partials where it can serve the call. Negative sra_status for bad sizes or dtype. */
SRA_API int64_t sra_linear_workspace_size(int64_t B, int64_t K, int64_t N, int dtype);

/*
 * sra_uclip — [mer] sec. 0 (DyHT(x) = y * clamp(a x, -1, 1) in place of every
 * RMSNorm) and sec. 3.3 (one kernel: clamp(alpha * x, clip_min, clip_max) * gamma
 * with a scalar or per-channel alpha and gamma; Q/K norms on narrow 3-D views of
 * a fused QKV projection, whose head stride is free).
 *
 *   out[n, h, d] = clamp(alpha_d * x[n, h, d], clip_min, clip_max) * gamma_d
 *
 * computed in fp32 and rounded once (RNE) to the dtype. DyHT is clip_min = -1,
 * clip_max = 1. A NaN alpha * x becomes clip_min (the page's kernel clamps with
 * fmaxf then fminf, which keep the non-NaN operand); +-inf clips to a bound.
 *
 * x:      [N, H, D] of `dtype`, element strides (x_n_stride, x_h_stride, 1); a
 *         2-D [rows, D] tensor is N = rows, H = 1. Read only.
 * alpha:  fp32, D entries if alpha_per_channel (1) else 1 entry (0). Read only.
 * gamma:  fp32, D entries if gamma_per_channel (1) else 1 entry (0). Read only.
 * out:    [N, H, D] of `dtype`, strides (out_n_stride, out_h_stride, 1); its rows
 *         must be pairwise disjoint. out == x with equal strides (in place) is
 *         allowed; any other overlap of out with x, alpha or gamma is not.
 * The stride of a dimension of size 1 is ignored.
 * Errors: unknown dtype -> SRA_ERR_DTYPE; N < 0, H < 0, H >= 2^31 or D <= 0 -> SRA_ERR_SHAPE;
 * a per-channel flag other than 0 / 1, a NaN bound or clip_min > clip_max ->
 * SRA_ERR_ARG; a negative stride or out rows that overlap one another ->
 * SRA_ERR_STRIDE; NULL -> SRA_ERR_NULL; overlap -> SRA_ERR_ALIAS. N * H == 0 is
 * a no-op.
 */
SRA_API int sra_uclip(const void* x, const float* alpha, const float* gamma, void* out, int64_t N, int64_t H,
                      int64_t D, int64_t x_n_stride, int64_t x_h_stride, int64_t out_n_stride,
                      int64_t out_h_stride, int alpha_per_channel, int gamma_per_channel, float clip_min,
                      float clip_max, int dtype, void* stream);

/* Static text for a status code (never NULL). */
SRA_API const char* sra_status_string(int status);

/* SRA_VERSION of the loaded library. */
SRA_API int sra_version(void);

/*
 * The cudaError_t value behind the most recent SRA_ERR_LAUNCH returned to the
 * calling thread (0 if there has been none). Diagnostic only.
 */
SRA_API int sra_last_cuda_error(void);

/*
 * Bounded device waits that gave up, on the current device, since the library was
 * loaded. Kernels that stream tiles with tensor-memory-access copies
 * (sra_rmsnorm_linear, sra_glu_linear and their _ws forms; decode attention's
 * TMA-fed variant) wait on shared-memory barriers for those copies; each wait is bounded (about a second), and a wait that runs out is
 * counted here and the kernel goes on, so a copy that never completes cannot hang
 * the GPU (that call's output is then not valid). Reads the counter synchronously
 * (cudaMemcpyFromSymbol); 0 on a device that ran none of those kernels. No paper
 * section defines this; it is the library's own failure report.
 */
SRA_API unsigned int sra_wait_timeouts(void);

/*
 * Self-test of that bound: one GPU thread waits on a shared-memory barrier that nothing
 * completes. The wait gives up after about a second, the kernel writes 0 to *result
 * (device int32; 1 would mean the barrier completed) and sra_wait_timeouts() grows by
 * one. Enqueued on `stream`; NULL result -> SRA_ERR_NULL. No paper section defines it.
 */
SRA_API int sra_wait_selftest(int32_t* result, void* stream);

/*
 * Programmatic dependent launch for the CALLING THREAD's subsequent calls
 * (enable != 0: on; 0: off, the default). When on, each kernel is launched with
 * programmatic stream serialization: the GPU may schedule it while the kernel
 * before it in the stream is still finishing, which hides launch latency in
 * chains of short kernels (e.g. a decode step). Every kernel of this library
 * first waits for the preceding grid to complete and its writes to become
 * visible, so results are identical either way. The setting is captured into
 * CUDA graphs with the launches. Returns the previous setting.
 */
SRA_API int sra_set_pdl(int enable);

/*
 * Kernel-variant control, for A/B measurement of the per-shape dispatch.
 * op: "rmsnorm" (also used by add_rmsnorm), "rope_kv_store" (0 = one task of a
 * token per thread, 1 = two tasks per thread that read the same cos / sin chunk,
 * for an even n_head + 2 * n_kv_head), "glu" (0 = columns over threads and rows over
 * CTAs at 48 registers a thread, 1 = the same kernel with the registers the compiler
 * picks), "decode_attention" (0 = CUDA-core kernel,
 * 1 = mma.sync kernel for bf16 / fp16 with head_dim 64 or 128, 2 = the same
 * contraction with the K / V tiles moved by TMA; for 1 and 2, OR-ed with (s << 8),
 * s in 1, 2, 4, 8, 16, it also forces the CTAs per (request, kv head), and for 1,
 * OR-ed with (4 << 16), it runs 4-warp CTAs, two per SM), "linear" (the
 * projection kernels of the fused entry points and of the _ws entry points once
 * their prologue has run: 0 = mma.sync kernels, 1 = the tcgen05 kernel, for up to
 * 64 rows and N a multiple of 128, which for the fused entry points computes the
 * RMSNorm or the GLU itself; OR-ed with (s << 8), s in 1..16, it also forces the
 * tcgen05 kernel's K splits (with the RMSNorm fused, s >= K / 1024: a CTA holds at
 * most 1024 columns of x), and with (r << 16), r = 4 or 8, the ring depth in stages
 * of the projection over h), "linear_narrow" (the
 * decode-batch projection kernel of the fused entry points, up to 16 rows: variant 0,
 * OR-ed with (s << 8), s in 1..8, forces the CTAs of its cluster along K).
 * variant: -1 = automatic per-shape choice (the default); otherwise an index
 * < sra_variant_count(op), optionally OR-ed with (nv << 8) to also force the
 * number of 16-byte accesses each thread holds in the register variants of
 * "rmsnorm" (nv in 1, 2, 3, 4, 6, 8; also 12 and 16 for the warp-per-row
 * variant; 8 or 16 for warps_row), with (g << 16) to force the warps per row
 * of warps_row (g in 2, 4, 8), and with (c << 24) to launch at most c CTAs per
 * SM (c in 1..15; "rmsnorm" only). A forced setting that cannot serve a later
 * call makes that call return SRA_ERR_VARIANT without enqueueing anything.
 * Returns SRA_OK, or SRA_ERR_ARG for an unknown op or out-of-range variant.
 */
SRA_API int sra_force_variant(const char* op, int variant);
SRA_API int sra_variant_count(const char* op);
/* Name of a variant ("warp_rows", "cta_row", ...); NULL for bad arguments. */
SRA_API const char* sra_variant_name(const char* op, int variant);
/*
 * The variant the automatic dispatch would pick for a call with these sizes and
 * all pointers and strides 16-byte aligned, on a GPU with num_sms SMs
 * (num_sms <= 0: query the current device). rmsnorm: a = rows, b = D;
 * rope_kv_store: a = T, b = n_head, c = n_kv_head, d = head_dim; glu: a = T, b = I,
 * c = act (0 = SiLU, 1 = ReLU);
 * decode_attention: a = B, b = n_head, c = n_kv_head, d = head_dim ("linear" and
 * "linear_narrow" have no pick: SRA_ERR_ARG).
 * Negative sra_status on bad arguments. Enqueues nothing.
 */
SRA_API int sra_pick_variant(const char* op, int64_t a, int64_t b, int64_t c, int64_t d, int dtype,
                     int num_sms);

#ifdef __cplusplus
}
#endif

#endif /* SRA_H_ */
