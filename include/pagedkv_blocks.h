/*
 * pagedkv_blocks.h - the block manager of the paged KV cache (host side) and the worker-side
 * block-table writes and zero fill (device side), in libpagedkv.so next to the decode path of
 * pagedkv.h.
 *
 * The manager is the allocator "vLLM의 KV cache 연결 흐름" describes in its section
 * "KVCacheManager가 하는 일": it tracks the blocks each request holds, works out whether new
 * tokens need a new block, hands blocks out of a free pool, takes them back when the request
 * ends, and produces the block ids the worker receives.  Shared prompt prefixes with a
 * reference count per block follow "vLLM Worker侧GPU KV Cache初始化流程深度解析", section
 * "PagedAttention与Block管理"; the release of blocks that left a sliding window follows its
 * section "混合注意力机制".  The worker side (section "GPU worker가 하는 일" of the first page:
 * append the new block ids to the request's block-table row, zero-fill new blocks) is one
 * kernel, kv_apply_block_updates.
 *
 * One decode step of a serving loop:
 *   host    kv_bm_allocate (or _batch) for each scheduled request; kv_bm_free for finished
 *           ones; kv_bm_share_prefix for a new request that starts with another's prompt
 *   host    kv_bm_flush -> staged (row, column, block id) writes and the ids of new blocks
 *   copy    both arrays to the device (cudaMemcpyAsync from pinned memory)
 *   device  kv_apply_block_updates (block table and zero fill), then kv_decode_step (pagedkv.h)
 *
 * Semantics (the pages leave these open; each is one plain choice):
 *   - Rows.  A request is a row r of the block table, 0 <= r < num_rows.  The row holding T
 *     tokens owns ceil(T / block_size) logical blocks (a block opens only when the previous one
 *     is full).  Entry j of the row names the physical block of positions j*bs .. j*bs+bs-1, or
 *     -1 once a window has released it; entries past the row's blocks are not maintained (the
 *     decode path never reads them).
 *   - Free pool: first in, first out.  It starts as 0, 1, ..., num_blocks-1; allocation takes
 *     from the front; a block whose reference count reaches zero joins the back (blocks
 *     released together in logical order).
 *   - kv_bm_allocate(row, n): room for n more tokens at positions T .. T+n-1, then the row holds
 *     T+n tokens.  All or nothing: with too few free blocks it returns KV_ERR_OUT_OF_BLOCKS and
 *     changes nothing (except the window release below).  With a window W > 0 the call first
 *     releases every live block whose last position is <= T - W (no query at >= T can see it:
 *     keys p-W < j <= p), staging -1 for its entry, so after a step of n tokens a row holds at
 *     most ceil((W + n - 1) / bs) + 1 live blocks.
 *   - kv_bm_share_prefix(dst, src, k): the empty row dst takes src's first k blocks, which must
 *     be full and live; each block's count rises by one; dst holds k * block_size tokens.
 *   - kv_bm_free(row): the row's live blocks lose one reference each; the row becomes empty.
 *     No table writes are staged.
 *   - Staged writes: one per (row, column) changed since the last flush, the last value
 *     winning; kv_bm_flush hands them out sorted by (row, column).  The zero-fill list holds
 *     the blocks taken from the pool since the last flush that are still held (sorted, each
 *     once; empty when zero fill is off).  Shared blocks are never in it.
 *   - A manager is single-threaded state: calls on one manager must not overlap; distinct
 *     managers are independent.  Layers of different attention kinds (full, windowed) use one
 *     manager each, as the pages' layer groups do; the block ids of one manager index every
 *     cache of its layers.
 *   - Host pointers only; the manager never touches the GPU.  Errors return a status and
 *     record a message for kv_last_error().
 */
#ifndef PAGEDKV_BLOCKS_H
#define PAGEDKV_BLOCKS_H

#include "pagedkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kv_block_manager kv_block_manager;

/*
 * kv_bm_create - a manager over num_blocks blocks of block_size tokens, for num_rows requests
 * of at most max_blocks_per_row blocks each.  window > 0 releases blocks that left a window of
 * that many tokens; zero_fill != 0 lists new blocks for zeroing.  *out receives the manager
 * (host memory: about 14 bytes per block plus 5 bytes per table entry).
 */
KV_API kv_status kv_bm_create(int32_t num_blocks, int32_t block_size, int32_t num_rows,
                              int32_t max_blocks_per_row, int32_t window, int32_t zero_fill,
                              kv_block_manager **out);

/* Frees the manager (NULL is ignored). */
KV_API void kv_bm_destroy(kv_block_manager *bm);

/* Room for num_new_tokens more tokens in row `row` (see the semantics above).
 * KV_ERR_OUT_OF_BLOCKS: too few free blocks, nothing allocated.  KV_ERR_INVALID_ARG: bad row,
 * negative count, or the row would need more than max_blocks_per_row blocks. */
KV_API kv_status kv_bm_allocate(kv_block_manager *bm, int32_t row, int32_t num_new_tokens);

/* kv_bm_allocate for n (row, count) pairs in order (host arrays).  Each pair succeeds or fails
 * on its own; status_out (host int32 [n], may be NULL) receives each status.  Returns KV_OK when
 * all succeeded, else the status of the first failure. */
KV_API kv_status kv_bm_allocate_batch(kv_block_manager *bm, const int32_t *rows,
                                      const int32_t *num_new_tokens, int32_t n,
                                      int32_t *status_out);

/* Returns the row's blocks (one reference each) and empties it. */
KV_API kv_status kv_bm_free(kv_block_manager *bm, int32_t row);

/* The empty row dst_row takes the first num_blocks blocks of src_row (full and live). */
KV_API kv_status kv_bm_share_prefix(kv_block_manager *bm, int32_t dst_row, int32_t src_row,
                                    int32_t num_blocks);

/* Blocks in the free pool (-1 for a NULL manager). */
KV_API int32_t kv_bm_num_free_blocks(const kv_block_manager *bm);

/* Reference count of a block (-1 when out of range). */
KV_API int32_t kv_bm_ref_count(const kv_block_manager *bm, int32_t block);

/* Tokens and logical blocks of a row; its entries (-1 = released) into blocks (host int32
 * [capacity], may be NULL; KV_ERR_WORKSPACE when capacity is smaller than the block count). */
KV_API kv_status kv_bm_row(const kv_block_manager *bm, int32_t row, int32_t *num_tokens,
                           int32_t *num_blocks, int32_t *blocks, int32_t capacity);

/* Sizes the next kv_bm_flush would hand out. */
KV_API kv_status kv_bm_pending(const kv_block_manager *bm, int32_t *num_updates,
                               int32_t *num_zero);

/*
 * kv_bm_flush - hand out and clear the staged writes: updates (host int32 [max_updates][3]) gets
 * (row, column, block id) triples, zero_ids (host int32 [max_zero]) the blocks to zero-fill.
 * KV_ERR_WORKSPACE (nothing handed out, nothing cleared) when either array is too small.
 */
KV_API kv_status kv_bm_flush(kv_block_manager *bm, int32_t *updates, int32_t max_updates,
                             int32_t *num_updates, int32_t *zero_ids, int32_t max_zero,
                             int32_t *num_zero);

/*
 * kv_apply_block_updates - the worker's side of a flush, one launch on `stream`:
 *   block_table[row * bt_stride + column] = id      for each (row, column, id) of updates
 *   every byte of block b of each cache = 0          for each b of zero_ids
 * ("vLLM의 KV cache 연결 흐름", section "GPU worker가 하는 일").
 *   updates     device int32 [num_updates][3]; rows >= num_rows, columns >= max_blocks_per_row
 *               and ids outside [-1, num_blocks) set KV_DERR_BAD_UPDATE and are skipped
 *   block_table device int32 [num_rows, bt_stride]
 *   zero_ids    device int32 [num_zero]; ids outside [0, num_blocks) set KV_DERR_BAD_UPDATE
 *   caches      HOST array of num_caches (<= KV_MAX_ZERO_CACHES) device pointers, each a cache
 *               of num_blocks blocks of block_bytes bytes (K and V of every layer of the
 *               manager's group); 16-byte aligned, block_bytes a multiple of 16
 * Duplicate (row, column) pairs in one call: undefined (kv_bm_flush never makes them).  The
 * zeroing is written by the tensor-memory-access engine (bulk stores from a zeroed shared-memory
 * tile); completion is ordered with later work on `stream` as for any kernel.
 */
#define KV_MAX_ZERO_CACHES 128

KV_API kv_status kv_apply_block_updates(const int32_t *updates, int32_t num_updates,
                                        int32_t *block_table, int64_t bt_stride,
                                        int32_t num_rows, int32_t max_blocks_per_row,
                                        const int32_t *zero_ids, int32_t num_zero,
                                        void *const *caches, int32_t num_caches,
                                        int64_t block_bytes, int32_t num_blocks, int32_t *d_err,
                                        void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_BLOCKS_H */
