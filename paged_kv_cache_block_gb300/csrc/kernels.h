// Internal launch interface between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

cudaError_t launch_slot_mapping(const int32_t *block_table, int64_t bt_stride, int32_t num_seqs,
                                int32_t max_blocks_per_seq, const int32_t *query_start_loc,
                                const int32_t *positions, int32_t num_tokens, int32_t block_size,
                                int32_t num_blocks, int64_t *slot_mapping, int32_t *d_err,
                                cudaStream_t stream);

// src_dtype / cache_dtype use the kv_dtype numbering of pagedkv.h.
cudaError_t launch_reshape_and_cache(const void *key, const void *value, int src_dtype,
                                     int64_t key_row_stride, int64_t value_row_stride,
                                     int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                     const int64_t *slot_mapping, void *k_cache, void *v_cache,
                                     int cache_dtype, int64_t total_slots, float k_scale,
                                     float v_scale, int32_t *d_err, int sm_count,
                                     cudaStream_t stream);

// Launch geometry of the decode kernel, chosen on the host (see plan_decode in api.cu).
struct DecodePlan {
    int heads_per_cta;     // kv heads handled by one CTA (HG)
    int m_tiles;           // 16-row query tiles per kv head: ceil(group * q_len / 16)
    int blocks_per_stage;  // cache blocks per pipeline stage
    int stage_tokens;      // blocks_per_stage * block_size (16 or 32)
    int part_tokens;       // keys per partition (multiple of stage_tokens)
    int max_parts;         // partitions of the longest sequence (grid x)
    int num_stages;        // pipeline depth
    int box_bytes;         // bytes one TMA box writes: heads_per_cta * block_size * 128
    int box_stride;        // box_bytes rounded up to 1024 (swizzle atom)
    int threads;           // (consumer warps + 1 producer warp) * 32
    size_t smem_bytes;     // dynamic shared memory
    size_t workspace_bytes;
};

struct DecodeArgs {
    const void *q;
    void *out;
    float *lse_out;
    float *ws_o;            // [T, Hq, max_parts, D] partial outputs (normalised), or null
    float *ws_lse;          // [T, Hq, max_parts] partial log-sum-exp (natural log)
    const int32_t *block_table;
    int64_t bt_stride;
    int32_t max_blocks_per_seq;
    const int32_t *seq_lens;
    int32_t max_seq_len;
    int32_t *d_err;
    int32_t num_seqs, q_len, num_q_heads, num_kv_heads, head_dim;
    int32_t block_size, num_blocks, window;
    float scale_log2;       // softmax scale * k_scale * log2(e)
    float v_scale;
};

cudaError_t launch_paged_decode(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                                const DecodeArgs &a, const DecodePlan &plan, int q_dtype,
                                int cache_dtype, cudaStream_t stream);

}  // namespace pkv
