/*
 * pagedkv.h - C ABI of the GB300 paged KV cache decode path (libpagedkv.so).
 *
 * Three calls make one decode step of one attention layer:
 *   kv_compute_slot_mapping   token positions + block tables -> cache slot per token
 *   kv_reshape_and_cache      scatter this step's new K/V rows into the paged cache
 *   kv_paged_attention_decode attention over each sequence's K/V, found through its block table
 *
 * The operations follow four web pages on vLLM's paged KV cache:
 *   "Deep Dive into vLLM Worker-Side GPU KV Cache Initialization" (kongchang.com/en),
 *   "vLLM의 KV cache 연결 흐름" (llm-engineer.pages.dev),
 *   "Understanding PageAttention Memory Optimization" (freaks.city),
 *   "vLLM Worker侧GPU KV Cache初始化流程深度解析" (kongchang.com).
 * Each declaration below names the section that defines its operation.
 *
 * Conventions shared by every call
 *   - All pointers are DEVICE pointers unless marked host.  The caller owns every buffer; the
 *     library allocates nothing, never synchronises and keeps no state between calls beyond
 *     cached device properties: work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Calls can be captured into CUDA graphs; make one uncaptured call on the
 *     stream's device first (a warm-up), since the stream's device cannot be queried while it
 *     is capturing.
 *   - Cache layout (vLLM Worker侧..., section "Worker与ModelRunner的协作"): two tensors, K and V,
 *     each [num_blocks, block_size, num_kv_heads, head_dim], row-major, densely packed.  They may
 *     be views of one byte allocation.  Slot s is (block s / block_size, offset s % block_size);
 *     the element offset of (slot, head h, dim d) is (s * num_kv_heads + h) * head_dim + d.
 *   - Errors found on the host are returned before anything is launched.  Errors that depend
 *     on device data (a bad block id, a slot out of range, a length past the table) set bits in
 *     *d_err (a device int32 the caller zeroes and reads after its own synchronisation; may be
 *     NULL) and the offending item is skipped; nothing traps, nothing waits without bound.
 *   - Supported: head_dim 64 or 128 (fp8 caches: 128), block_size 4, 8, 16 or 32, q_len 1..8,
 *     num_q_heads a multiple of num_kv_heads with (num_q_heads/num_kv_heads)*q_len <= 64.
 *     Anything else returns KV_ERR_UNSUPPORTED; there is no fallback path.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KV_API __attribute__((visibility("default")))
#else
#define KV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status returned synchronously by every call. */
typedef enum {
    KV_OK = 0,
    KV_ERR_INVALID_ARG = 1, /* null pointer, negative size, inconsistent shapes, misalignment */
    KV_ERR_UNSUPPORTED = 2, /* a valid request outside the supported set listed above */
    KV_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a launch failed */
    KV_ERR_WORKSPACE = 4,   /* workspace missing or smaller than the size query returned */
    KV_ERR_OUT_OF_BLOCKS = 5 /* the block manager's free pool holds too few blocks (nothing changed) */
} kv_status;

/* Element types.  Caches may be fp16, bf16, OCP FP8 E4M3 ("fn": bias 7, max 448, no inf), or
 * INT4 with group scales (two's-complement nibbles, two per byte; only through the calls of
 * pagedkv_int4.h, which take the scales: every other call rejects KV_INT4 as unsupported). */
typedef enum { KV_F16 = 0, KV_BF16 = 1, KV_FP8_E4M3 = 2, KV_INT4 = 3 } kv_dtype;

/* Bits set in *d_err by device code (atomicOr). */
#define KV_DERR_BAD_BLOCK   1  /* a block-table entry that is read is < 0 or >= num_blocks */
#define KV_DERR_BAD_SLOT    2  /* a slot >= num_blocks * block_size in kv_reshape_and_cache */
#define KV_DERR_PAST_TABLE  4  /* a position needs a logical block >= max_blocks_per_seq */
#define KV_DERR_TIMEOUT     8  /* a bounded wait inside a kernel expired (never expected) */
#define KV_DERR_BAD_LEN    16  /* seq_lens[b] < q_len, > max_seq_len, or past the table */
#define KV_DERR_BAD_UPDATE 32  /* a block-table update or zero-fill id out of range (skipped) */

/*
 * kv_compute_slot_mapping - cache slot of every token of this step.
 *
 * Defined by "Deep Dive into vLLM Worker-Side GPU KV Cache Initialization", section
 * "Pinpointing the Token Slot" (logical block = pos // block_size, offset = pos % block_size,
 * address = physical block * block_size + offset) and "vLLM의 KV cache 연결 흐름", section
 * "Slot mapping은 왜 필요한가" (position -> logical block + offset -> physical block -> slot).
 *
 * For token t of request r (query_start_loc[r] <= t < query_start_loc[r+1]):
 *   slot_mapping[t] = block_table[r * bt_stride + positions[t] / block_size] * block_size
 *                     + positions[t] % block_size
 * and slot_mapping[t] = -1 when positions[t] < 0 (padding), when t lies in no request's range,
 * or when the entry is invalid (then KV_DERR_BAD_BLOCK or KV_DERR_PAST_TABLE is set).
 *
 *   block_table      int32 [num_seqs, bt_stride] (row r's first max_blocks_per_seq entries used)
 *   query_start_loc  int32 [num_seqs + 1], non-decreasing, query_start_loc[num_seqs] <= num_tokens
 *   positions        int32 [num_tokens], 0-based
 *   slot_mapping     int64 [num_tokens], written for every token
 * Bit-exact integer arithmetic; one launch.
 */
KV_API kv_status kv_compute_slot_mapping(const int32_t *block_table, int64_t bt_stride,
                                  int32_t num_seqs, int32_t max_blocks_per_seq,
                                  const int32_t *query_start_loc, const int32_t *positions,
                                  int32_t num_tokens, int32_t block_size, int32_t num_blocks,
                                  int64_t *slot_mapping, int32_t *d_err, void *stream);

/*
 * kv_reshape_and_cache - write this step's new K/V rows into their slots.
 *
 * Defined by "vLLM의 KV cache 연결 흐름", section "Slot mapping은 왜 필요한가" (decode stores the
 * new token's K/V in its slot) with the layout of "vLLM Worker侧GPU KV Cache初始化流程深度解析",
 * section "Worker与ModelRunner的协作"; the FP8 variant is the FP8 KV cache of its section
 * "KV Cache技术背景".
 *
 * For every token t with slot_mapping[t] >= 0 and every head h, dim d:
 *   k_cache[slot][h][d] = cvt(key[t * key_row_stride + h * head_dim + d]), same for V,
 * where cvt is a bit copy when cache_dtype == src_dtype, and for an E4M3 cache
 *   cvt(x) = E4M3_RNE_satfinite(float(x) / scale)   (IEEE float32 division, k_scale for K,
 *                                                     v_scale for V; values past 448 saturate)
 *   key, value        fp16/bf16 [num_tokens, row stride], rows 16-byte aligned
 *                     (row strides in elements, multiples of 8, >= num_kv_heads * head_dim)
 *   slot_mapping      int64 [num_tokens]; -1 skips the token; >= num_blocks*block_size sets
 *                     KV_DERR_BAD_SLOT and skips it.  Duplicate slots in one call: undefined.
 *   k_cache, v_cache  [num_blocks, block_size, num_kv_heads, head_dim] of cache_dtype,
 *                     16-byte aligned
 * Bit-exact; one launch.
 */
KV_API kv_status kv_reshape_and_cache(const void *key, const void *value, kv_dtype src_dtype,
                               int64_t key_row_stride, int64_t value_row_stride,
                               int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                               const int64_t *slot_mapping, void *k_cache, void *v_cache,
                               kv_dtype cache_dtype, int32_t num_blocks, int32_t block_size,
                               float k_scale, float v_scale, int32_t *d_err, void *stream);

/*
 * kv_paged_attention_workspace_size - bytes of device workspace kv_paged_attention_decode
 * needs for these sizes (SIZE_MAX when the arguments are invalid or unsupported, or no device
 * can be queried).  Host-only; reads the current device's SM count and shared-memory limit.
 * Pass the same values to the decode call (cache_dtype KV_INT4 for
 * kv_paged_attention_decode_int4).  The size grows with num_seqs and the number of
 * workers, not with sequence length: about (num_seqs + workers) x rows x (head_dim + 1) x 4 B.
 */
KV_API size_t kv_paged_attention_workspace_size(int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
                                         int32_t num_kv_heads, int32_t head_dim,
                                         int32_t block_size, kv_dtype cache_dtype,
                                         int32_t max_seq_len, int32_t window,
                                         int32_t num_workers);

/*
 * kv_paged_attention_plan_info - the launch geometry kv_paged_attention_decode (and
 * kv_decode_step) would use for these sizes, for tuning and diagnostics.  Host-only; the
 * arguments are those of kv_paged_attention_workspace_size.  On KV_OK, info[0..7] holds:
 *   0 pipeline stages of the shared-memory ring   1 bytes of one stage (K and V boxes)
 *   2 kv heads per CTA                           3 CTAs (stream-K workers)
 *   4 threads per CTA (without the fused step's writer warp)
 *   5 query rows per consumer warp               6 (head group, sequence) items
 *   7 workspace bytes
 * Invalid or unsupported sizes return the status kv_paged_attention_workspace_size reports as
 * SIZE_MAX (the reason in kv_last_error()).  The pages have no counterpart of this query.
 */
KV_API kv_status kv_paged_attention_plan_info(int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
                                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                              kv_dtype cache_dtype, int32_t max_seq_len, int32_t window,
                                              int32_t num_workers, int64_t *info);

/*
 * kv_paged_attention_decode - attention of this step's queries over the paged cache.
 *
 * Defined by "vLLM의 KV cache 연결 흐름", sections "Slot mapping은 왜 필요한가" and
 * "Forward 직전의 metadata" (attention reads past K/V through the block table, not a contiguous
 * tensor); "Understanding PageAttention Memory Optimization", section "Handling Softmax Across
 * Blocks" (the softmax denominator needs every block: resolved with an online softmax, the
 * tiling + online softmax of "vLLM Worker侧...", section "Worker与ModelRunner的协作"); GQA of
 * "Deep Dive into vLLM Worker-Side...", section "Hybrid Attention Mechanisms"; sliding windows
 * of "vLLM Worker侧...", section "混合注意力机制"; speculative tokens of "vLLM의 KV cache 연결
 * 흐름", section "EngineCore가 하는 일".
 *
 * Sequence b has L = seq_lens[b] tokens including its q_len new ones, which sit at positions
 * p_i = L - q_len + i.  Query row (b, i, q head hq) attends kv head hq / (num_q_heads /
 * num_kv_heads) over keys j with lo_i <= j <= p_i, lo_i = max(0, p_i - window + 1) if
 * window > 0 else 0:
 *   out = sum_j softmax_j(scale * q.K_j) V_j,   lse = log(sum_j exp(scale * q.K_j))  (natural log)
 * E4M3 caches are dequantised as decode(code) * k_scale (V: * v_scale).  Accumulation is
 * float32; q.K and p.V run on tensor cores in the cache's 16-bit type (fp16 for E4M3 caches, with
 * q rounded to fp16).  The keys of the whole batch are split into num_workers equal shares
 * (0 = one persistent CTA per SM); a sequence that straddles shares is finished by a
 * log-sum-exp merge of its pieces.  Results depend on num_workers only through rounding.
 *
 *   q          [num_seqs * q_len, num_q_heads, head_dim] of q_dtype (fp16 or bf16; for a 16-bit
 *              cache it must equal cache_dtype), rows of one sequence consecutive, 16-B aligned
 *   block_table int32 [num_seqs, bt_stride]; entries past ceil(L/block_size), and entries of
 *              blocks wholly outside a window, are never read (they may hold -1)
 *   seq_lens   int32 [num_seqs]
 *   max_seq_len host bound on seq_lens (a longer sequence sets KV_DERR_BAD_LEN; its rows are 0)
 *   workspace  device buffer of at least kv_paged_attention_workspace_size(...) bytes, 256-B
 *              aligned; contents on entry do not matter
 *   out        [num_seqs * q_len, num_q_heads, head_dim] of q_dtype
 *   lse_out    float32 [num_seqs * q_len, num_q_heads] or NULL
 * Rows of a sequence whose length is rejected (KV_DERR_BAD_LEN) are written as 0 (lse -inf).
 * Two launches: the attention kernel and the log-sum-exp merge.
 */
KV_API kv_status kv_paged_attention_decode(const void *q, kv_dtype q_dtype, int32_t num_seqs,
                                    int32_t q_len, int32_t num_q_heads, const void *k_cache,
                                    const void *v_cache, kv_dtype cache_dtype,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                    int32_t num_blocks, const int32_t *block_table,
                                    int64_t bt_stride, int32_t max_blocks_per_seq,
                                    const int32_t *seq_lens, int32_t max_seq_len, float scale,
                                    int32_t window, float k_scale, float v_scale,
                                    int32_t num_workers, void *workspace,
                                    size_t workspace_bytes, void *out, float *lse_out,
                                    int32_t *d_err, void *stream);

/*
 * kv_decode_step - one whole decode step of one layer in a single launch: exactly
 *   kv_compute_slot_mapping(block_table, query_start_loc, positions, num_seqs*q_len tokens)
 *   kv_reshape_and_cache(key, value, those slots)            (key/value of the q dtype)
 *   kv_paged_attention_decode(q, caches, block_table, seq_lens, ...)
 * with the same arguments, results and error bits ("vLLM의 KV cache 연결 흐름", section
 * "Slot mapping은 왜 필요한가": decode stores the new tokens' K/V in their slots, then attention
 * reads past K/V through the block table; section "Forward 직전의 metadata" lists the inputs).
 * Two launches instead of four: the attention kernel's CTAs first write the new-token rows that
 * their own share of the keys will read (rows no attention reads are shared out by token), then
 * attend; the log-sum-exp merge follows.  No grid-wide barrier.  The new
 * tokens are the rows of query_start_loc (one sequence's q_len tokens consecutive,
 * num_seqs*q_len in all).  slot_mapping (int64 [num_seqs*q_len]) is an optional output.  The
 * workspace is kv_paged_attention_workspace_size for the same sizes.
 */
KV_API kv_status kv_decode_step(const int32_t *block_table, int64_t bt_stride,
                                int32_t max_blocks_per_seq, const int32_t *query_start_loc,
                                const int32_t *positions, int64_t *slot_mapping, const void *key,
                                const void *value, int64_t key_row_stride,
                                int64_t value_row_stride, const void *q, kv_dtype q_dtype,
                                int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
                                void *k_cache, void *v_cache, kv_dtype cache_dtype,
                                int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                int32_t num_blocks, const int32_t *seq_lens, int32_t max_seq_len,
                                float scale, int32_t window, float k_scale, float v_scale,
                                int32_t num_workers, void *workspace, size_t workspace_bytes,
                                void *out, float *lse_out, int32_t *d_err, void *stream);

/*
 * kv_paged_attention_decode_noalloc - kv_paged_attention_decode for callers that cannot allocate
 * device memory.  The pages have no counterpart of this call: it serves callers for which
 * cudaMalloc is not an option (a plugin inside a framework that owns every device allocation, a
 * real-time decode loop where an allocation could synchronise the device or fail, a C caller
 * with no allocator).  Arguments, results and errors are those of kv_paged_attention_decode
 * without the workspace: its scratch is a file-scope device array of KV_NOALLOC_SCRATCH_BYTES
 * inside the library, which every GPU that loads the library holds until the process exits.
 *   - The first call on a device (with that device current) looks up the array's device address
 *     (cudaGetSymbolAddress); the address is kept per device once a lookup succeeds, and a failed
 *     lookup is retried by the next call.  Make that first call before any stream capture.
 *   - Sizes whose workspace (kv_paged_attention_workspace_size) exceeds the array return
 *     KV_ERR_WORKSPACE with the sizes in kv_last_error(); nothing is launched.
 *   - All calls on a device share the array and it keeps the last call's contents; each call
 *     writes everything it reads, so nothing needs clearing.  Calls that overlap on the GPU (two
 *     streams without ordering) race on it: order them on one stream.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
#define KV_NOALLOC_SCRATCH_BYTES (32u << 20)

KV_API kv_status kv_paged_attention_decode_noalloc(
    const void *q, kv_dtype q_dtype, int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
    const void *k_cache, const void *v_cache, kv_dtype cache_dtype, int32_t num_kv_heads,
    int32_t head_dim, int32_t block_size, int32_t num_blocks, const int32_t *block_table,
    int64_t bt_stride, int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t max_seq_len,
    float scale, int32_t window, float k_scale, float v_scale, int32_t num_workers, void *out,
    float *lse_out, int32_t *d_err, void *stream);

/*
 * kv_paged_attention_prefill - attention of a chunk of new tokens per sequence (chunked prefill)
 * over the paged cache, on the tensor cores (tcgen05).
 *
 * Defined by "vLLM의 KV cache 연결 흐름", section "EngineCore가 하는 일" (a step computes the
 * request's num_new_tokens not yet in the cache) and section "Slot mapping은 왜 필요한가" (the
 * new tokens' K/V are written to their slots, then attention reads K/V through the block table),
 * with the GQA, window and softmax of kv_paged_attention_decode.  Sequence b has
 * n_b = query_start_loc[b+1] - query_start_loc[b] query rows (0 allowed) at positions
 * L_b - n_b .. L_b - 1, L_b = seq_lens[b] including them; their K/V must already be in the cache
 * (kv_reshape_and_cache first).  Row (token at position p, q head hq) attends kv head
 * hq / (num_q_heads / num_kv_heads) over keys lo <= j <= p (lo = max(0, p - window + 1) with a
 * window, else 0):  out = softmax(scale * q.K) V,  lse = log sum exp(scale * q.K).
 *   q            [num_tokens, num_q_heads, 128] of q_dtype (fp16 or bf16, equal to cache_dtype),
 *                16-byte aligned; num_tokens >= query_start_loc[num_seqs]
 *   query_start_loc int32 [num_seqs + 1], non-decreasing; max_query_len >= every n_b (host bound)
 *   block_table, seq_lens, max_seq_len, caches: as for kv_paged_attention_decode (entries of
 *                blocks wholly before a window are never read)
 *   out          [num_tokens, num_q_heads, 128] of q_dtype; lse_out float32 [num_tokens,
 *                num_q_heads] or NULL.  Rows of no sequence are not written.
 * Supported: head_dim 128, block_size 8, 16 or 32, num_q_heads / num_kv_heads a power of two
 * <= 128.  A sequence whose length is rejected sets KV_DERR_BAD_LEN and its rows are 0 (lse
 * -inf).  Accumulation in fp32 (TMEM); the softmax weights are rounded to the 16-bit type for
 * the second product, and the normaliser sums the rounded weights.  One launch; no workspace.
 */
KV_API kv_status kv_paged_attention_prefill(const void *q, kv_dtype q_dtype,
                                            const int32_t *query_start_loc, int32_t num_seqs,
                                            int32_t num_tokens, int32_t max_query_len,
                                            int32_t num_q_heads, const void *k_cache,
                                            const void *v_cache, kv_dtype cache_dtype,
                                            int32_t num_kv_heads, int32_t head_dim,
                                            int32_t block_size, int32_t num_blocks,
                                            const int32_t *block_table, int64_t bt_stride,
                                            int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                            int32_t max_seq_len, float scale, int32_t window,
                                            void *out, float *lse_out, int32_t *d_err,
                                            void *stream);

/* Human-readable name of a status (static string). */
KV_API const char *kv_status_string(kv_status s);

/* Last error detail recorded by this thread (static per-thread buffer, "" if none). */
KV_API const char *kv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
