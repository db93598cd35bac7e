// Internal launch interface between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pagedkv.h"
#include "../../include/pagedkv_blocks.h"
#include "../../include/pagedkv_int4.h"
#include "../../include/pagedkv_selftest.h"

namespace pkv {

// Record a message for kv_last_error() and return the status (shared by the entry points).
kv_status record_error(kv_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));

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

// INT4 caches with float32 group scales [num_kv_heads, head_dim / group_size].
cudaError_t launch_reshape_and_cache_int4(const void *key, const void *value, int src_dtype,
                                          int64_t key_row_stride, int64_t value_row_stride,
                                          int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                          const int64_t *slot_mapping, void *k_cache, void *v_cache,
                                          int64_t total_slots, const float *k_scales,
                                          const float *v_scales, int32_t group_size, int32_t *d_err,
                                          int sm_count, cudaStream_t stream);

// Threads of the decode kernel for RN query rows per consumer warp (must match its launch
// bounds): up to 14 consumer warps with 8 rows each, or 8 with 16 rows, plus one producer warp
// and, in the fused step, one writer warp (at most 16 or 10 warps: 128 or 168 registers a
// thread).
template <int RN> struct DecodeLaunch {
    static constexpr int kMaxConsumers = RN == 8 ? 14 : 8;
    static constexpr int kThreads = (kMaxConsumers + 2) * 32;
    // each of the SM's four schedulers holds a quarter of the register file and up to
    // ceil(warps / 4) of the block's warps: 16 warps -> 128, 10 (3 a scheduler) -> 168
    static constexpr int kMaxRegs = (65536 / ((kThreads / 32 + 3) / 4 * 4 * 32)) & ~7;
};

// Launch geometry of the decode kernel, chosen on the host (plan_decode in api.cu).
struct DecodePlan {
    int rows_per_warp;     // RN: 8 or 16 query rows per consumer warp
    int warps_per_head;    // ceil(group * q_len / RN)
    int heads_per_cta;     // kv heads per CTA (HG); num_kv_heads / HG head groups
    int blocks_per_stage;  // cache blocks per pipeline stage
    int stage_tokens;      // blocks_per_stage * block_size (16 or 32)
    int num_stages;        // pipeline depth
    int box_bytes;         // bytes one TMA box writes: heads_per_cta * block_size * 128
    int box_stride;        // box_bytes rounded up to 1024 (swizzle atom)
    int threads;           // (consumer warps + 1 producer warp [+ 1 writer warp, fused step]) * 32
    int num_items;         // head groups * num_seqs
    int rows_per_item;     // heads_per_cta * group * q_len
    int num_ctas;          // persistent CTAs (equal shares of the flat stage list)
    int sets_per_cta;      // INT4 kernel: independent warp sets per CTA (1 otherwise)
    int num_workers;       // INT4 kernel: stream-K workers (sets) in all (num_ctas otherwise)
    int tile_ws;           // partial results as consumer-warp fragment tiles (no padding rows)
    int item_cost;         // a piece's fixed cost in quarter stages (shares by cost); 0: equal stages
    int lens_smem;         // the per-sequence length table is kept in shared memory
    size_t ws_pieces_off;  // the [num_items][2] share owners (16-bit / E4M3 kernel)
    size_t smem_bytes;     // dynamic shared memory
    size_t ws_prefix_off, ws_lse_off, ws_o_off, workspace_bytes;
};

// Inputs of the fused decode step's first part (slot mapping and cache write), which run in the
// attention kernel's own launch: each CTA writes the new-token rows its own stages read.
struct StepArgs {
    const int32_t *query_start_loc;
    const int32_t *positions;
    int32_t num_tokens;
    const void *key, *value;            // [num_tokens, row stride] of the q dtype
    int64_t key_row_stride, value_row_stride;
    void *k_cache, *v_cache;            // the caches the attention reads
    int64_t total_slots;                // num_blocks * block_size
    float k_scale, v_scale;             // E4M3 caches
    int64_t *slot_mapping;              // optional output
};

struct DecodeArgs {
    const void *q;
    void *out;
    float *lse_out;
    int32_t *ws_prefix;     // [num_items + 1] stage prefix, written by CTA 0
    int32_t *ws_pieces;     // [num_items][2] shares holding each item's first and last stage (16-bit /
                            // E4M3 kernel; nullptr: equal stage counts, computed by the merge)
    float *ws_lse;          // [num_items + num_ctas, rows_per_item] partial log-sum-exp
    float *ws_o;            // [num_items + num_ctas, rows_per_item, D] partial outputs (o / l)
    const int32_t *block_table;
    int64_t bt_stride;
    int32_t max_blocks_per_seq;
    const int32_t *seq_lens;
    int32_t max_seq_len;
    int32_t *d_err;
    int32_t num_seqs, q_len, num_q_heads, num_kv_heads, head_dim;
    int32_t block_size, num_blocks, window;
    float scale_log2;       // softmax scale * k_scale * log2(e) (INT4: * 2^24, the unit of its codes)
    float v_scale;
    // INT4 caches only: group scales and the log-sum-exp correction of the offset-binary codes
    const float *k_gscales, *v_gscales;  // [num_kv_heads, head_dim >> group_shift]
    int32_t group_shift;                 // log2(group_size)
    float lse_offset_scale;              // 8 * softmax scale
};

cudaError_t launch_paged_decode(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                                const DecodeArgs &a, const DecodePlan &plan, int q_dtype,
                                int cache_dtype, cudaStream_t stream);

// Decode attention over INT4 caches (paged_decode_int4.cu): warps with private TMA rings,
// int4_decode_warps(rows_per_warp) per CTA, then the merge kernel.
int int4_decode_warps(int rows_per_warp);
cudaError_t launch_paged_decode_int4(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                                     const DecodeArgs &a, const DecodePlan &plan, int q_dtype,
                                     cudaStream_t stream);
// The INT4 one-launch step: each worker writes (as INT4 codes) the new-token rows it reads.
cudaError_t launch_decode_step_int4(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                                    const DecodeArgs &a, const StepArgs &f, const DecodePlan &plan,
                                    int q_dtype, cudaStream_t stream);

// The whole decode step in two launches: each CTA writes the new-token rows it will read, then
// attends; the merge kernel combines split sequences.
cudaError_t launch_decode_step(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                               const DecodeArgs &a, const StepArgs &f, const DecodePlan &plan,
                               int q_dtype, int cache_dtype, cudaStream_t stream);

// Chunked-prefill attention on tcgen05 (kv_paged_attention_prefill).
struct PrefillArgs {
    const int32_t *query_start_loc;
    const int32_t *seq_lens;
    const int32_t *block_table;
    int64_t bt_stride;
    int32_t max_blocks_per_seq;
    int32_t num_seqs, num_tokens, max_query_len, num_q_heads, num_kv_heads;
    int32_t block_size, num_blocks, max_seq_len, window;
    float scale;
    void *out;
    float *lse_out;
    int32_t *d_err;
};

size_t prefill_smem_bytes();
cudaError_t launch_prefill(const CUtensorMap &tmap_q, const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                           const PrefillArgs &a, int q_dtype, cudaStream_t stream);

// kv_selftest_bounded_wait: one thread waits limit_us on an mbarrier nothing completes.
cudaError_t launch_selftest_bounded_wait(int32_t limit_us, int32_t *d_err, int32_t *d_waited_us,
                                         cudaStream_t stream);

// Block-table writes and zero fill of new blocks (kv_apply_block_updates); caches is a host
// array of num_caches device pointers, copied into the launch's parameters.
cudaError_t launch_block_updates(const int32_t *updates, int32_t num_updates, int32_t *block_table,
                                 int64_t bt_stride, int32_t num_rows, int32_t max_blocks,
                                 const int32_t *zero_ids, int32_t num_zero, void *const *caches,
                                 int32_t num_caches, int64_t block_bytes, int32_t num_blocks,
                                 int32_t *d_err, int sm_count, cudaStream_t stream);

}  // namespace pkv
