// Host block manager of the paged KV cache (pagedkv_blocks.h): free pool, reference counts,
// per-request block-table rows, prefix sharing, sliding-window release and the staged
// block-table writes the worker applies.
//
// The allocator of "vLLM의 KV cache 연결 흐름", section "KVCacheManager가 하는 일" (track each
// request's blocks, decide whether new tokens need a block, hand blocks out of the free pool,
// take them back, produce the block ids for the worker), with the shared prefixes and reference
// counts of "vLLM Worker侧GPU KV Cache初始化流程深度解析", section "PagedAttention与Block管理",
// and the window release of its section "混合注意力机制".
//
// Layout, chosen for a scheduler that touches a few hundred rows per step:
//   - the free pool is a ring of num_blocks ids (first in, first out);
//   - the table is mirrored in one flat int32 array [num_rows * max_blocks_per_row] that holds
//     the last value staged for each entry, so a row's blocks are a contiguous slice;
//   - released blocks are always a prefix of a row (a window only moves forward), so a row is
//     (tokens, logical block count, first live index);
//   - staged writes are a dirty flag per table entry plus the list of dirty entries, sorted by
//     flat index (= (row, column) order) at flush; new blocks are a flag per block plus a list.
// Every operation is O(blocks it touches); nothing scans the pool or the table.
#include <algorithm>
#include <new>
#include <vector>

#include "kernels.h"
#include "../../include/pagedkv_blocks.h"

struct kv_block_manager {
    int32_t num_blocks, block_size, num_rows, max_blocks, window;
    bool zero_fill;
    std::vector<int32_t> ring;  // free pool, ring buffer: ring[(head + i) % num_blocks]
    int64_t head = 0;
    int32_t num_free = 0;
    std::vector<int32_t> ref;         // per block
    std::vector<uint8_t> fresh;       // per block: taken from the pool since the last flush
    std::vector<int32_t> fresh_list;  // blocks with fresh set
    std::vector<int32_t> table;       // [num_rows * max_blocks], last staged value per entry
    std::vector<uint8_t> dirty;       // per entry: staged since the last flush
    std::vector<int64_t> dirty_list;
    std::vector<int64_t> tokens;     // per row
    std::vector<int32_t> nblk;       // per row: logical blocks
    std::vector<int32_t> first_live;  // per row: entries below it were released by the window

    int32_t take() {
        const int32_t b = ring[head];
        head = head + 1 == num_blocks ? 0 : head + 1;
        --num_free;
        ref[b] = 1;
        if (!fresh[b]) {
            fresh[b] = 1;
            fresh_list.push_back(b);
        }
        return b;
    }
    void drop(int32_t b) {
        if (--ref[b] == 0) {
            int64_t tail = head + num_free;
            if (tail >= num_blocks) tail -= num_blocks;
            ring[tail] = b;
            ++num_free;
        }
    }
    void stage(int32_t row, int32_t col, int32_t value) {
        const int64_t i = static_cast<int64_t>(row) * max_blocks + col;
        table[i] = value;
        if (!dirty[i]) {
            dirty[i] = 1;
            dirty_list.push_back(i);
        }
    }
    int32_t *row_entries(int32_t row) { return table.data() + static_cast<int64_t>(row) * max_blocks; }
    const int32_t *row_entries(int32_t row) const {
        return table.data() + static_cast<int64_t>(row) * max_blocks;
    }

    // blocks whose last position is <= T - W are invisible to every query at position >= T
    void release_outside_window(int32_t row) {
        if (window <= 0) return;
        const int64_t first_query = tokens[row];
        int32_t *e = row_entries(row);
        int32_t j = first_live[row];
        while (j < nblk[row] && static_cast<int64_t>(j + 1) * block_size - 1 <= first_query - window) {
            drop(e[j]);
            stage(row, j, -1);
            ++j;
        }
        first_live[row] = j;
    }

    int32_t pending_zero() const {
        if (!zero_fill) return 0;
        int32_t n = 0;
        for (int32_t b : fresh_list) n += ref[b] > 0;
        return n;
    }
};

namespace {

kv_status check_bm(const kv_block_manager *bm, const char *fn) {
    if (!bm) return pkv::record_error(KV_ERR_INVALID_ARG, "%s: null manager", fn);
    return KV_OK;
}

kv_status check_row(const kv_block_manager *bm, int32_t row, const char *fn) {
    if (row < 0 || row >= bm->num_rows)
        return pkv::record_error(KV_ERR_INVALID_ARG, "%s: row %d outside [0, %d)", fn, row, bm->num_rows);
    return KV_OK;
}

}  // namespace

extern "C" {

kv_status kv_bm_create(int32_t num_blocks, int32_t block_size, int32_t num_rows,
                       int32_t max_blocks_per_row, int32_t window, int32_t zero_fill,
                       kv_block_manager **out) {
    if (!out) return pkv::record_error(KV_ERR_INVALID_ARG, "kv_bm_create: null out");
    *out = nullptr;
    if (num_blocks <= 0 || block_size <= 0 || num_rows <= 0 || max_blocks_per_row <= 0 || window < 0)
        return pkv::record_error(KV_ERR_INVALID_ARG,
                                 "kv_bm_create: sizes must be positive (window >= 0): blocks %d, "
                                 "block_size %d, rows %d, max_blocks_per_row %d, window %d",
                                 num_blocks, block_size, num_rows, max_blocks_per_row, window);
    kv_block_manager *bm = new (std::nothrow) kv_block_manager();
    if (!bm) return pkv::record_error(KV_ERR_INVALID_ARG, "kv_bm_create: out of host memory");
    try {
        bm->num_blocks = num_blocks;
        bm->block_size = block_size;
        bm->num_rows = num_rows;
        bm->max_blocks = max_blocks_per_row;
        bm->window = window;
        bm->zero_fill = zero_fill != 0;
        bm->ring.resize(num_blocks);
        for (int32_t b = 0; b < num_blocks; ++b) bm->ring[b] = b;
        bm->num_free = num_blocks;
        bm->ref.assign(num_blocks, 0);
        bm->fresh.assign(num_blocks, 0);
        const int64_t entries = static_cast<int64_t>(num_rows) * max_blocks_per_row;
        bm->table.assign(entries, -1);
        bm->dirty.assign(entries, 0);
        bm->tokens.assign(num_rows, 0);
        bm->nblk.assign(num_rows, 0);
        bm->first_live.assign(num_rows, 0);
    } catch (const std::bad_alloc &) {
        delete bm;
        return pkv::record_error(KV_ERR_INVALID_ARG, "kv_bm_create: out of host memory");
    }
    *out = bm;
    return KV_OK;
}

void kv_bm_destroy(kv_block_manager *bm) { delete bm; }

kv_status kv_bm_allocate(kv_block_manager *bm, int32_t row, int32_t num_new_tokens) {
    kv_status st = check_bm(bm, "kv_bm_allocate");
    if (st == KV_OK) st = check_row(bm, row, "kv_bm_allocate");
    if (st != KV_OK) return st;
    if (num_new_tokens < 0)
        return pkv::record_error(KV_ERR_INVALID_ARG, "kv_bm_allocate: negative token count %d", num_new_tokens);
    const int64_t total = bm->tokens[row] + num_new_tokens;
    const int64_t need = (total + bm->block_size - 1) / bm->block_size;
    if (need > bm->max_blocks)
        return pkv::record_error(KV_ERR_INVALID_ARG,
                                 "kv_bm_allocate: row %d would need %lld blocks, the table row holds %d",
                                 row, static_cast<long long>(need), bm->max_blocks);
    bm->release_outside_window(row);
    const int64_t missing = need - bm->nblk[row];
    if (missing > bm->num_free)
        return pkv::record_error(KV_ERR_OUT_OF_BLOCKS,
                                 "kv_bm_allocate: row %d needs %lld new blocks, %d free", row,
                                 static_cast<long long>(missing), bm->num_free);
    for (int64_t i = 0; i < missing; ++i) {
        const int32_t b = bm->take();
        bm->stage(row, bm->nblk[row], b);
        ++bm->nblk[row];
    }
    bm->tokens[row] = total;
    return KV_OK;
}

kv_status kv_bm_allocate_batch(kv_block_manager *bm, const int32_t *rows, const int32_t *num_new_tokens,
                               int32_t n, int32_t *status_out) {
    kv_status st = check_bm(bm, "kv_bm_allocate_batch");
    if (st != KV_OK) return st;
    if (n < 0 || (n > 0 && (!rows || !num_new_tokens)))
        return pkv::record_error(KV_ERR_INVALID_ARG, "kv_bm_allocate_batch: null arrays or n %d", n);
    kv_status first = KV_OK;
    for (int32_t i = 0; i < n; ++i) {
        const kv_status s = kv_bm_allocate(bm, rows[i], num_new_tokens[i]);
        if (status_out) status_out[i] = s;
        if (s != KV_OK && first == KV_OK) first = s;
    }
    return first;
}

kv_status kv_bm_free(kv_block_manager *bm, int32_t row) {
    kv_status st = check_bm(bm, "kv_bm_free");
    if (st == KV_OK) st = check_row(bm, row, "kv_bm_free");
    if (st != KV_OK) return st;
    const int32_t *e = bm->row_entries(row);
    for (int32_t j = bm->first_live[row]; j < bm->nblk[row]; ++j) bm->drop(e[j]);
    bm->nblk[row] = 0;
    bm->first_live[row] = 0;
    bm->tokens[row] = 0;
    return KV_OK;
}

kv_status kv_bm_share_prefix(kv_block_manager *bm, int32_t dst_row, int32_t src_row, int32_t num_blocks) {
    kv_status st = check_bm(bm, "kv_bm_share_prefix");
    if (st == KV_OK) st = check_row(bm, dst_row, "kv_bm_share_prefix");
    if (st == KV_OK) st = check_row(bm, src_row, "kv_bm_share_prefix");
    if (st != KV_OK) return st;
    if (dst_row == src_row || num_blocks < 0)
        return pkv::record_error(KV_ERR_INVALID_ARG, "kv_bm_share_prefix: rows %d -> %d, %d blocks",
                                 src_row, dst_row, num_blocks);
    if (bm->nblk[dst_row] != 0 || bm->tokens[dst_row] != 0)
        return pkv::record_error(KV_ERR_INVALID_ARG, "kv_bm_share_prefix: row %d is not empty", dst_row);
    if (num_blocks > bm->nblk[src_row] ||
        bm->tokens[src_row] < static_cast<int64_t>(num_blocks) * bm->block_size)
        return pkv::record_error(KV_ERR_INVALID_ARG,
                                 "kv_bm_share_prefix: row %d has no %d full blocks", src_row, num_blocks);
    if (num_blocks > 0 && bm->first_live[src_row] > 0)
        return pkv::record_error(KV_ERR_INVALID_ARG,
                                 "kv_bm_share_prefix: row %d released its first blocks", src_row);
    const int32_t *s = bm->row_entries(src_row);
    for (int32_t j = 0; j < num_blocks; ++j) {
        const int32_t b = s[j];
        ++bm->ref[b];
        bm->stage(dst_row, j, b);
    }
    bm->nblk[dst_row] = num_blocks;
    bm->first_live[dst_row] = 0;
    bm->tokens[dst_row] = static_cast<int64_t>(num_blocks) * bm->block_size;
    return KV_OK;
}

int32_t kv_bm_num_free_blocks(const kv_block_manager *bm) { return bm ? bm->num_free : -1; }

int32_t kv_bm_ref_count(const kv_block_manager *bm, int32_t block) {
    if (!bm || block < 0 || block >= bm->num_blocks) return -1;
    return bm->ref[block];
}

kv_status kv_bm_row(const kv_block_manager *bm, int32_t row, int32_t *num_tokens, int32_t *num_blocks,
                    int32_t *blocks, int32_t capacity) {
    kv_status st = check_bm(bm, "kv_bm_row");
    if (st == KV_OK) st = check_row(bm, row, "kv_bm_row");
    if (st != KV_OK) return st;
    if (num_tokens) *num_tokens = static_cast<int32_t>(bm->tokens[row]);
    if (num_blocks) *num_blocks = bm->nblk[row];
    if (blocks) {
        if (capacity < bm->nblk[row])
            return pkv::record_error(KV_ERR_WORKSPACE, "kv_bm_row: %d entries, capacity %d",
                                     bm->nblk[row], capacity);
        const int32_t *e = bm->row_entries(row);
        std::copy(e, e + bm->nblk[row], blocks);
    }
    return KV_OK;
}

kv_status kv_bm_pending(const kv_block_manager *bm, int32_t *num_updates, int32_t *num_zero) {
    kv_status st = check_bm(bm, "kv_bm_pending");
    if (st != KV_OK) return st;
    if (num_updates) *num_updates = static_cast<int32_t>(bm->dirty_list.size());
    if (num_zero) *num_zero = bm->pending_zero();
    return KV_OK;
}

kv_status kv_bm_flush(kv_block_manager *bm, int32_t *updates, int32_t max_updates, int32_t *num_updates,
                      int32_t *zero_ids, int32_t max_zero, int32_t *num_zero) {
    kv_status st = check_bm(bm, "kv_bm_flush");
    if (st != KV_OK) return st;
    const int64_t nu = static_cast<int64_t>(bm->dirty_list.size());
    const int32_t nz = bm->pending_zero();
    if ((nu > 0 && !updates) || (nz > 0 && !zero_ids) || nu > max_updates || nz > max_zero)
        return pkv::record_error(KV_ERR_WORKSPACE,
                                 "kv_bm_flush: %lld updates and %d zero-fill ids pending, room for %d and %d",
                                 static_cast<long long>(nu), nz, max_updates, max_zero);
    std::sort(bm->dirty_list.begin(), bm->dirty_list.end());
    for (int64_t i = 0; i < nu; ++i) {
        const int64_t e = bm->dirty_list[i];
        updates[3 * i + 0] = static_cast<int32_t>(e / bm->max_blocks);
        updates[3 * i + 1] = static_cast<int32_t>(e % bm->max_blocks);
        updates[3 * i + 2] = bm->table[e];
        bm->dirty[e] = 0;
    }
    bm->dirty_list.clear();
    int32_t z = 0;
    if (bm->zero_fill) {
        for (int32_t b : bm->fresh_list)
            if (bm->ref[b] > 0) zero_ids[z++] = b;
        std::sort(zero_ids, zero_ids + z);
    }
    for (int32_t b : bm->fresh_list) bm->fresh[b] = 0;
    bm->fresh_list.clear();
    if (num_updates) *num_updates = static_cast<int32_t>(nu);
    if (num_zero) *num_zero = z;
    return KV_OK;
}

}  // extern "C"
