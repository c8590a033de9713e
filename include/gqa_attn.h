/*
 * gqa_attn.h — C ABI of the GB300 (sm_103a) grouped-query attention block forward.
 *
 * The block is the Llama-3 / Llama-3.1 8B attention sub-block described on the page
 * "Llama 3.1 8B · Grouped-query attention" (step list "All 13 steps"; in/out contract
 * x [B,T,4096], R [T,64 pairs], M [T queries, T keys] -> Delta_attn [B,T,4096];
 * parameter table: W_Q 4096x4096, W_K and W_V 4096x(8x128), W_O 4096x4096).  It computes
 *
 *     Q = x W_Q,  K = x W_K,  V = x W_V                      (steps 1-3)
 *     Q_r, K_r = pair rotation of Q, K by R                  (steps 4-5)
 *     K_G[h] = K_r[h/4],  V_G[h] = V[h/4]                    (steps 6-7)
 *     S = Q_r K_G^T,  S_s = S / sqrt(128),  S_m = S_s + M    (steps 8-10)
 *     A = softmax over keys of S_m,  H = A V_G               (steps 11-12)
 *     H merged to [B,T,4096],  Delta_attn = H W_O            (steps 13-14)
 *
 * Dimensions are fixed by the model catalogue quoted on that page: dim 4096, 32 query
 * heads, 8 key/value heads, head width 128 (64 rotation pairs).  B, T, the cache length
 * S_max and start_pos are runtime values.
 *
 * Conventions shared by every call below
 *  - Every pointer argument named x, R, R_row, cache_k, cache_v, delta, wq, wk, wv, wo is
 *    a DEVICE pointer (cudaMalloc / torch CUDA storage on the current device).  The
 *    caller owns these buffers; the library borrows them for the duration of the
 *    asynchronous work it enqueues and never frees them.
 *  - bf16 tensors are IEEE bfloat16 bit patterns (uint16), row-major, densely packed.
 *  - Every device pointer must be 16-byte aligned (GQA_ERR_ALIGN otherwise).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  All work is enqueued on
 *    it and the call returns without synchronising, except where noted.
 *  - Arguments are validated on the host before anything is enqueued; on any error the
 *    call enqueues nothing and returns a non-zero gqa_status.
 *  - A context may be used from one stream at a time; calls on one context must not
 *    overlap on different streams (they share the context's workspace).
 *  - Kernels bound every wait on the device.  A wait that runs out records
 *    GQA_ERR_TIMEOUT in the context's device status word and the kernel returns; read
 *    it with attn_sync_status.
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */
typedef struct CUstream_st *gqa_stream_t;

typedef struct gqa_ctx gqa_ctx; /* opaque */

typedef enum {
    GQA_OK = 0,
    GQA_ERR_INVALID_ARG = 1, /* null pointer / null context / bad flag */
    GQA_ERR_SHAPE = 2,       /* B, T, S_max, start_pos out of range */
    GQA_ERR_ALIGN = 3,       /* a device pointer is not 16-byte aligned */
    GQA_ERR_CUDA = 4,        /* a CUDA runtime call failed (see attn_last_cuda_error) */
    GQA_ERR_TIMEOUT = 5,     /* a bounded device-side wait ran out (device status word) */
    GQA_ERR_OOM = 6,         /* workspace allocation failed */
    GQA_ERR_DEVICE = 7       /* current device is not an sm_103 GPU */
} gqa_status;

#define GQA_DIM 4096
#define GQA_N_HEADS 32
#define GQA_N_KV_HEADS 8
#define GQA_HEAD_DIM 128
#define GQA_QKV_DIM 6144 /* 4096 query + 1024 key + 1024 value features */

/*
 * attn_create — build a context for one block on the current CUDA device.
 *
 * wq [4096,4096], wk [1024,4096], wv [1024,4096], wo [4096,4096]: bf16 device tensors in
 * the [out, in] storage of the quoted fairscale ColumnParallelLinear / RowParallelLinear
 * layers ("F.linear performs XA^T ... we allocate the transpose").  They are COPIED into
 * memory the context owns (W_Q, W_K, W_V packed into one [6144,4096] matrix; W_O kept
 * [4096,4096]); the caller may free its copies once the stream has passed this call.
 * The copies are enqueued on `stream`.
 * On success *out receives the context (to be released with attn_destroy).
 * Errors: GQA_ERR_INVALID_ARG (null), GQA_ERR_ALIGN, GQA_ERR_DEVICE (not sm_103),
 * GQA_ERR_OOM, GQA_ERR_CUDA.
 */
gqa_status attn_create(const void *wq, const void *wk, const void *wv, const void *wo,
                       gqa_stream_t stream, gqa_ctx **out);

/*
 * attn_create_shard — a context for one tensor-parallel shard of the block: the query heads
 * of n_kv_local consecutive kv groups (4 n_kv_local query heads, n_kv_local key/value
 * heads), as the quoted Attention.__init__ splits the block over model-parallel ranks
 * (page "Llama 3.1 8B · Grouped-query attention", Query projection: n_local_heads =
 * n_heads / model_parallel_size, n_local_kv_heads likewise; wq, wk, wv are
 * ColumnParallelLinear(gather_output=False), whose weight is [output_size_per_partition,
 * in_features]) and the output projection is a RowParallelLinear(input_is_parallel=True)
 * whose weight is [out_features, input_size_per_partition] (page "Llama 3.1 8B · Merge and
 * project").  Rank r of a world of w ranks holds kv groups 8r/w .. 8(r+1)/w - 1.
 *
 * wq_shard [512 n,4096]: rows 512 g0 .. 512 (g0+n) - 1 of W_Q (query heads 4 g0 .. 4 (g0+n) - 1)
 * wk_shard, wv_shard [128 n,4096]: rows 128 g0 .. 128 (g0+n) - 1 of W_K, W_V
 * wo_shard [4096,512 n]: columns 512 g0 .. 512 (g0+n) - 1 of W_O, row-major (densely packed)
 * with n = n_kv_local in 1..8; all bf16 device tensors, copied into the context as by
 * attn_create.
 *
 * attn_prefill / attn_decode on a shard context compute that shard's heads only:
 *  - cache_k, cache_v are the shard's own caches [B,S_max,n,128] (its kv heads);
 *  - attn_debug_buffers' q_r and h are [B*T,512 n];
 *  - delta receives the shard's PARTIAL Delta_attn [B,T,4096] fp32 = H_shard W_O_shard^T:
 *    the block's Delta_attn is the sum of the partials of all shards, which the row-parallel
 *    output projection's all-reduce (a sum over ranks, done by the caller, e.g. with
 *    torch.distributed.all_reduce) produces.
 * The residual forms (attn_set_norm, attn_*_residual) need the whole sum and return
 * GQA_ERR_INVALID_ARG on a shard context: apply attention_norm before the shards and add x
 * after the all-reduce.  n_kv_local = 8 gives the same context as attn_create.
 * Errors: those of attn_create, and GQA_ERR_SHAPE for n_kv_local outside 1..8.
 */
gqa_status attn_create_shard(const void *wq_shard, const void *wk_shard, const void *wv_shard,
                             const void *wo_shard, int n_kv_local, gqa_stream_t stream, gqa_ctx **out);

/*
 * attn_prefill — Delta_attn for T new positions of B sequences (steps 1-14).
 *
 * x       [B,T,4096] bf16: the block input, already normalised by the caller
 *         (the page's x_attn = attention_norm(x)).
 * R       [T,64,2] fp32: (cos, sin) of the rotation for positions start_pos+t,
 *         t = 0..T-1, pair j (the page's R [T positions, 64 pairs]).
 * causal  non-zero: M[t,s] = -inf for keys s > start_pos+t, else 0 (the quoted
 *         triu(diagonal=1) mask hstacked after start_pos zero columns); zero: M = 0.
 * cache_k, cache_v  [B,S_max,8,128] bf16 key / value cache.  Positions
 *         0..start_pos-1 must already hold rotated keys (cache_k) and values (cache_v)
 *         of the earlier positions; this call writes K_r and V of its T positions at
 *         start_pos..start_pos+T-1, then attends over keys 0..start_pos+T-1.  Other
 *         positions are neither read nor written.
 * delta   [B,T,4096] fp32 output, fully overwritten.
 * Requires B >= 1, T >= 1, start_pos >= 0, start_pos + T <= S_max, and
 * B*T <= 262144, S_max <= 1048576.
 * Intermediates (Q_r and H, bf16) live in the context's workspace, which grows on
 * demand: a call that needs a larger workspace synchronises `stream` and reallocates
 * (so the first call at a new maximum size is not capturable in a CUDA graph).
 */
gqa_status attn_prefill(gqa_ctx *ctx, const void *x, int B, int T, const float *R, int causal,
                        void *cache_k, void *cache_v, int S_max, int start_pos, float *delta,
                        gqa_stream_t stream);

/*
 * attn_decode — one new position per sequence (T = 1, no mask: every cached key is
 * visible, as in the quoted forward when seqlen == 1).
 *
 * x       [B,1,4096] bf16 block input of the new token of each sequence.
 * R_row   [1,64,2] fp32: rotation for position start_pos (shared by all sequences).
 * cache_k, cache_v  [B,S_max,8,128] bf16; positions 0..start_pos-1 hold the earlier
 *         rotated keys / values.  The new K_r, V are written at position start_pos,
 *         then the token attends over keys 0..start_pos.
 * delta   [B,1,4096] fp32 output.
 * Requires 1 <= B <= 1024, 0 <= start_pos < S_max <= 1048576.
 */
gqa_status attn_decode(gqa_ctx *ctx, const void *x, int B, int start_pos, const float *R_row,
                       void *cache_k, void *cache_v, int S_max, float *delta,
                       gqa_stream_t stream);

/*
 * The block's residual form.  The transformer block around this attention block computes
 * h = x + Delta_attn(attention_norm(x)) (page "Llama 3.1 8B · Merge and project", code
 * excerpt model.py 236-248 and "Contextual evidence from Output projection"), with
 * attention_norm an RMSNorm of weight w and eps = norm_eps = 1e-05 (sku_list.py arch_args on
 * the same page).  The pages do not print the RMSNorm body; it is read as
 *     attention_norm(x)[t, j] = x[t, j] / sqrt(mean_k x[t, k]^2 + eps) * w[j].
 * The library folds w into a second copy of W_Q, W_K, W_V (made by attn_set_norm) and scales
 * each token row of the projections by 1 / rms in their epilogue; the residual add happens in
 * the epilogue of the W_O projection.
 */

/*
 * attn_set_norm — give the context the attention_norm weight.
 *
 * norm_w  [4096] bf16 device tensor, read during this call only (the folded copy it makes,
 *         W_QKV * diag(norm_w) in bf16, 48 MiB, is owned by the context; a later call
 *         replaces it).
 * eps     the RMSNorm epsilon (> 0; 1e-5 for the Llama 3 / 3.1 8B configurations).
 * Enqueued on `stream`.  Errors: GQA_ERR_INVALID_ARG (null, eps <= 0 or not finite),
 * GQA_ERR_ALIGN, GQA_ERR_DEVICE, GQA_ERR_OOM, GQA_ERR_CUDA.
 */
gqa_status attn_set_norm(gqa_ctx *ctx, const void *norm_w, float eps, gqa_stream_t stream);

/*
 * attn_prefill_residual — h_out = x + Delta_attn(attention_norm(x)) for T new positions of
 * B sequences: attn_prefill with the normalisation in front and the residual add behind.
 *
 * x       [B,T,4096] bf16: the residual stream entering the block (not normalised).
 * h_out   [B,T,4096] fp32 output (x widened to fp32 plus Delta_attn), fully overwritten;
 *         it must not overlap x.
 * Every other argument, requirement and the cache semantics are those of attn_prefill.
 * Errors: those of attn_prefill, and GQA_ERR_INVALID_ARG when attn_set_norm has not been
 * called on the context.
 */
gqa_status attn_prefill_residual(gqa_ctx *ctx, const void *x, int B, int T, const float *R, int causal,
                                 void *cache_k, void *cache_v, int S_max, int start_pos, float *h_out,
                                 gqa_stream_t stream);

/*
 * attn_decode_residual — attn_decode in the residual form: x [B,1,4096] bf16 residual
 * stream of the new token of each sequence, h_out [B,1,4096] fp32 = x + Delta_attn
 * (must not overlap x).  Other arguments and errors as attn_decode, plus
 * GQA_ERR_INVALID_ARG when attn_set_norm has not been called on the context.
 */
gqa_status attn_decode_residual(gqa_ctx *ctx, const void *x, int B, int start_pos, const float *R_row,
                                void *cache_k, void *cache_v, int S_max, float *h_out,
                                gqa_stream_t stream);

/*
 * attn_sync_status — synchronise `stream`, then read and clear the context's device
 * status word.  Returns GQA_OK, GQA_ERR_TIMEOUT (a bounded device wait ran out in some
 * earlier call) or GQA_ERR_CUDA (the synchronisation itself failed).
 */
gqa_status attn_sync_status(gqa_ctx *ctx, gqa_stream_t stream);

/*
 * attn_debug_buffers — device pointers to the context's intermediates after the last
 * call on it: q_r [B*T,4096] bf16 (rotated queries) and h [B*T,4096] bf16 (merged head
 * outputs, the page's H after step 13).  Valid until the next call on the context.
 * Either out-pointer may be NULL.  Returns GQA_ERR_INVALID_ARG for a null context.
 */
gqa_status attn_debug_buffers(gqa_ctx *ctx, const void **q_r, const void **h);

/*
 * Per-kernel device timing (tracing).  Kernel kinds:
 */
enum {
    GQA_KERNEL_QKV_GEMM = 0,       /* fused Q/K/V projection + RoPE + cache write (many tokens) */
    GQA_KERNEL_QKV_SPLITK = 1,     /* the same for few tokens: cluster split-K with its reduction */
    GQA_KERNEL_FLASH_PREFILL = 2,  /* causal GQA attention, prefill */
    GQA_KERNEL_DECODE_ATTN = 3,    /* split-KV attention with the fused merge, decode */
    GQA_KERNEL_OUT_GEMM = 4,       /* Delta = H W_O^T (many tokens) */
    GQA_KERNEL_OUT_SPLITK = 5,     /* the same for few tokens */
    GQA_KERNEL_RMS_NORM = 6,       /* 1 / rms of each token row (residual form only) */
    GQA_KERNEL_KINDS = 7
};

/*
 * attn_profile_begin — from now on, every kernel this context launches is bracketed by
 * two CUDA events recorded on the launch stream (up to 65536 launches).  Recording adds
 * two event records per launch and nothing else.
 * attn_profile_end — stop recording, synchronise `stream`, and write, per kernel kind,
 * the summed device time in milliseconds (ms_per_kind[GQA_KERNEL_KINDS]) and the number
 * of launches (launches_per_kind[GQA_KERNEL_KINDS]) since attn_profile_begin.  Either
 * output may be NULL.  Errors: GQA_ERR_INVALID_ARG (null context), GQA_ERR_CUDA.
 */
gqa_status attn_profile_begin(gqa_ctx *ctx);
gqa_status attn_profile_end(gqa_ctx *ctx, double *ms_per_kind, int *launches_per_kind,
                            gqa_stream_t stream);

/*
 * attn_decode_attention_noalloc — the decode attention of attn_decode (key/value head
 * sharing, scores, scaling, softmax over keys 0..kv_len-1, value product, head merge) for
 * callers that cannot let this library allocate device memory.  The pages have no
 * counterpart for this entry point: it exists for a serving engine that keeps all of HBM
 * in its own pool (for example for a paged KV cache) and gives a library only its inputs
 * and outputs, and for decode loops that cannot afford the device-wide synchronisation a
 * cudaMalloc implies.  It allocates nothing and needs no context.
 *
 * q_r     [B,4096] bf16: rotated queries of the new token of each sequence (what
 *         attn_debug_buffers returns as q_r after attn_decode).
 * cache_k, cache_v  [B,S_max,8,128] bf16: rotated keys / values; positions 0..kv_len-1
 *         are read (the new token's entry must already be written), nothing is written.
 * h       [B,4096] bf16 output: merged head outputs (the page's H after the merge).
 * Limits: 1 <= B <= 256, 1 <= kv_len <= S_max <= 1048576; larger B returns GQA_ERR_SHAPE.
 *
 * Scratch: the per-split partial results live in one file-scope device array of about
 * 4.3 MB (2048 units of (sequence, kv head, key split)), which every GPU that loads this
 * library holds until the process exits.  The first call on a device looks up that
 * array's device address (cudaGetSymbolAddress), the device's SM count and architecture,
 * and configures the kernels; make that first call before any stream capture.  Every call
 * shares the array and it keeps the last call's contents; calls whose work overlaps on the
 * GPU (other streams or host threads) race and must be serialised by the caller.
 * Time-outs: if a bounded device-side wait of this call runs out, every element of h is
 * written as NaN (never a mix of stale partial results) and the time-out is recorded in a
 * status word inside the array, which attn_decode_attention_noalloc_status reports.
 * Errors: GQA_ERR_INVALID_ARG, GQA_ERR_SHAPE, GQA_ERR_ALIGN, GQA_ERR_DEVICE (not sm_103),
 * GQA_ERR_CUDA (the cause via attn_last_cuda_error).
 */
gqa_status attn_decode_attention_noalloc(const void *q_r, const void *cache_k,
                                         const void *cache_v, int B, int kv_len, int S_max,
                                         void *h, gqa_stream_t stream);

/*
 * attn_decode_attention_noalloc_status — synchronise `stream`, then read and clear the
 * status word of attn_decode_attention_noalloc on the current device (allocates nothing).
 * Returns GQA_ERR_TIMEOUT if a device-side wait of any call since the last read ran out
 * (those calls wrote NaN into their h), GQA_OK otherwise, or GQA_ERR_DEVICE / GQA_ERR_CUDA.
 * The word is shared by every caller of the entry point on that device.
 */
gqa_status attn_decode_attention_noalloc_status(gqa_stream_t stream);

/*
 * attn_decode_attention_noalloc_debug_inject_timeout — test hook for that failure path (no
 * counterpart on the pages): the next call of attn_decode_attention_noalloc (in any thread)
 * makes its first work unit issue no loads, so that unit's bounded waits run out after about
 * 2 s; nothing faults or hangs.  Always returns GQA_OK.
 */
gqa_status attn_decode_attention_noalloc_debug_inject_timeout(void);

/*
 * attn_debug_inject_timeout — test hook for the failure path (no counterpart on the pages).
 * Arms a one-shot flag: on the next launch of kernel kind `kind` (GQA_KERNEL_QKV_GEMM,
 * _QKV_SPLITK, _FLASH_PREFILL, _DECODE_ATTN, _OUT_GEMM or _OUT_SPLITK) made through this
 * context, the first work unit's TMA producer issues no loads.  Its consumers' bounded
 * waits then run out (about 2 s), the unit records GQA_ERR_TIMEOUT in the status word,
 * releases its tensor memory and returns; kernels queued after it on the stream may time
 * out too.  Nothing faults or hangs.  The outputs of that call are undefined; the next
 * attn_sync_status returns GQA_ERR_TIMEOUT and resets the device-side state, after which
 * the context is usable again.  Errors: GQA_ERR_INVALID_ARG (null context, other kind).
 */
gqa_status attn_debug_inject_timeout(gqa_ctx *ctx, int kind);

/*
 * attn_debug_pair_schedule — the work schedule of the many-token projection GEMM, computed
 * on the host exactly as the library sizes a launch and as each CTA pair walks it (no
 * counterpart on the pages; for tests, no GPU needed).  Output tiles of 256 x 256:
 * m_tiles x n_tiles of them (n_tiles 24 for the Q/K/V projection, 16 for W_O), over n_pairs
 * co-resident CTA pairs.  Writes *full_rounds (rounds of whole tiles), *tail_w (width of the
 * pieces the last, partial round is cut into; 0: none) and *grid_ctas (CTAs launched), and
 * the items in launch order of pairs, each pair's items in the order it runs them, as
 * quadruples (pair, m tile, first column, width) into items[4 * max_items]; *n_items gets
 * their count.  Errors: GQA_ERR_INVALID_ARG (null pointer, m_tiles, n_tiles or n_pairs < 1,
 * max_items < 0), GQA_ERR_SHAPE (more than max_items items; *n_items holds the count).
 */
gqa_status attn_debug_pair_schedule(int m_tiles, int n_tiles, int n_pairs, int *full_rounds,
                                    int *tail_w, int *grid_ctas, int *items, int max_items,
                                    int *n_items);

/*
 * attn_debug_exp2 — the two exponentials the prefill softmax uses, on n fp32 device inputs a
 * (no counterpart on the pages; for tests): out_fma[i] = 2^a[i] by the FMA-pipe cubic
 * (range reduction, a minimax cubic fitted for relative error, exponent insertion; inputs
 * below -125 give 2^-125) and out_mufu[i] = ex2.approx.ftz(a[i]), both fp32 device arrays of
 * n elements.  Enqueued on `stream`.  Errors: GQA_ERR_INVALID_ARG (null, n < 1), GQA_ERR_CUDA.
 */
gqa_status attn_debug_exp2(const float *a, float *out_fma, float *out_mufu, int n, gqa_stream_t stream);

/* attn_destroy — free everything the context owns (after synchronising the device).
 * NULL is ignored. */
void attn_destroy(gqa_ctx *ctx);

/* attn_strerror — static description of a status code (never NULL). */
const char *attn_strerror(gqa_status status);

/* attn_last_cuda_error — the cudaError_t value of the last failing CUDA call made by
 * this library on the calling thread (0 if none). */
int attn_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H */
