/*
 * pagedkv_int4.h - INT4 paged KV cache with group scales (part of libpagedkv.so).
 *
 * "vLLM Worker侧GPU KV Cache初始化流程深度解析", section "KV Cache技术背景", lists an INT4 KV
 * cache at half a byte per element next to the FP8 one, with scales that a deployment calibrates.
 * The pages fix no encoding; this library's reading of it:
 *   - element (slot, head h, dim d) is a signed 4-bit two's-complement integer q in [-8, 7],
 *     value q * scale[h][d / group_size];
 *   - a cache is [num_blocks, block_size, num_kv_heads, head_dim / 2] bytes, row-major, the even
 *     dim of each pair in the low nibble (so slot s, head h, dims 2i, 2i+1 share byte
 *     (s * num_kv_heads + h) * head_dim / 2 + i);
 *   - scales are float32 [num_kv_heads, head_dim / group_size] on the device, one array for K and
 *     one for V, given by the caller (no calibration happens here); they must be finite and > 0;
 *   - encoding: q = clamp(rint(float(x) / scale), -8, 7), the division in IEEE float32, rint
 *     rounding half to even; +-inf saturate, NaN stores 0.
 * Conventions (device pointers, caller-owned buffers, stream semantics, d_err bits, host errors
 * returned before any launch) are those of pagedkv.h.
 * Supported: head_dim 128, group_size 8, 16, 32, 64 or 128, block_size 4, 8, 16 or 32, and the
 * q_len / GQA limits of kv_paged_attention_decode.
 */
#ifndef PAGEDKV_INT4_H
#define PAGEDKV_INT4_H

#include "pagedkv.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * kv_reshape_and_cache_int4 - write this step's new K/V rows into their slots of INT4 caches.
 *
 * The cache write of kv_reshape_and_cache ("vLLM의 KV cache 연결 흐름", section "Slot mapping은
 * 왜 필요한가") with the INT4 encoding above: for every token t with slot_mapping[t] >= 0, head h,
 * dim d, the nibble of (slot, h, d) in k_cache becomes
 *   clamp(rint(float(key[t * key_row_stride + h * head_dim + d]) / k_scales[h][d / group_size]), -8, 7)
 * (V alike with v_scales).
 *   key, value        fp16/bf16 (src_dtype) [num_tokens, row stride], 16-byte aligned rows
 *                     (strides in elements, multiples of 8, >= num_kv_heads * head_dim)
 *   slot_mapping      int64 [num_tokens]; -1 skips the token; >= num_blocks * block_size sets
 *                     KV_DERR_BAD_SLOT and skips it.  Duplicate slots in one call: undefined.
 *   k_cache, v_cache  uint8 [num_blocks, block_size, num_kv_heads, head_dim / 2], 16-byte aligned
 *   k_scales, v_scales float32 [num_kv_heads, head_dim / group_size], 4-byte aligned
 * Bit-exact; one launch.
 */
KV_API kv_status kv_reshape_and_cache_int4(const void *key, const void *value, kv_dtype src_dtype,
                                           int64_t key_row_stride, int64_t value_row_stride,
                                           int32_t num_tokens, int32_t num_kv_heads,
                                           int32_t head_dim, const int64_t *slot_mapping,
                                           void *k_cache, void *v_cache, int32_t num_blocks,
                                           int32_t block_size, const float *k_scales,
                                           const float *v_scales, int32_t group_size,
                                           int32_t *d_err, void *stream);

/*
 * kv_paged_attention_decode_int4 - kv_paged_attention_decode over INT4 caches.
 *
 * Same operation, arguments and results as kv_paged_attention_decode (its sections of the pages
 * define it), with K and V dequantised as code * scale of the element's (head, dim group):
 *   out = sum_j softmax_j(scale * sum_d q_d K_jd) V_j,  K_jd = kcode_jd * k_scales[h][d / group_size]
 * q.K and p.V run on tensor cores in fp16: q is multiplied by the K scales of its dims and
 * rounded to fp16; the V scales multiply the float32 result.  The workspace is
 * kv_paged_attention_workspace_size(..., KV_INT4, ...) for the same sizes.
 *   q, out            [num_seqs * q_len, num_q_heads, 128] of q_dtype (fp16 or bf16)
 *   k_cache, v_cache  uint8 [num_blocks, block_size, num_kv_heads, 64], 16-byte aligned
 *   k_scales, v_scales float32 [num_kv_heads, 128 / group_size], 4-byte aligned
 * Two launches: the attention kernel and the log-sum-exp merge.
 */
KV_API kv_status kv_paged_attention_decode_int4(
    const void *q, kv_dtype q_dtype, int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
    const void *k_cache, const void *v_cache, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int32_t num_blocks, const int32_t *block_table, int64_t bt_stride,
    int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t max_seq_len, float scale,
    int32_t window, const float *k_scales, const float *v_scales, int32_t group_size,
    int32_t num_workers, void *workspace, size_t workspace_bytes, void *out, float *lse_out,
    int32_t *d_err, void *stream);

/*
 * kv_decode_step_int4 - kv_decode_step over INT4 caches: exactly
 *   kv_compute_slot_mapping(block_table, query_start_loc, positions, num_seqs*q_len tokens)
 *   kv_reshape_and_cache_int4(key, value, those slots, k_scales, v_scales, group_size)
 *   kv_paged_attention_decode_int4(q, caches, block_table, seq_lens, ...)
 * with the same arguments, results (bit for bit) and error bits, in two launches (the attention
 * kernel's workers first write the new-token rows their own stages read, then attend; the merge
 * follows).  The new tokens are the rows of query_start_loc (one sequence's q_len tokens
 * consecutive); key/value are of q_dtype; slot_mapping (int64 [num_seqs*q_len]) is an optional
 * output; the workspace is kv_paged_attention_workspace_size(..., KV_INT4, ...).
 */
KV_API kv_status kv_decode_step_int4(
    const int32_t *block_table, int64_t bt_stride, int32_t max_blocks_per_seq,
    const int32_t *query_start_loc, const int32_t *positions, int64_t *slot_mapping, const void *key,
    const void *value, int64_t key_row_stride, int64_t value_row_stride, const void *q, kv_dtype q_dtype,
    int32_t num_seqs, int32_t q_len, int32_t num_q_heads, void *k_cache, void *v_cache,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
    const int32_t *seq_lens, int32_t max_seq_len, float scale, int32_t window, const float *k_scales,
    const float *v_scales, int32_t group_size, int32_t num_workers, void *workspace,
    size_t workspace_bytes, void *out, float *lse_out, int32_t *d_err, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_INT4_H */
