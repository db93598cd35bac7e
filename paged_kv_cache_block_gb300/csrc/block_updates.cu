// Worker-side application of the block manager's staged writes: block-table entries and the
// zero fill of newly assigned blocks ("vLLM의 KV cache 연결 흐름", section "GPU worker가 하는 일":
// append the new block ids to the request's row of the block table, zero-fill new blocks).
//
// One launch does both.  The table writes are a handful of scattered int32 stores.  The zero
// fill is the bandwidth part: every listed block of every cache (K and V of each layer) is a
// contiguous region of block_bytes, written from a zeroed 16 KB shared-memory tile by bulk
// asynchronous copies (cp.async.bulk shared -> global, the tensor-memory-access engine), a few
// instructions per 16 KB instead of a thousand vector stores.  Work units are (zero id, cache,
// 16 KB chunk) in that order, so one CTA's contiguous range of units is a contiguous stretch of
// memory; the grid is at most two CTAs per SM.
#include "common.cuh"
#include "kernels.h"

namespace pkv {
namespace {

constexpr int kZeroChunk = 16384;  // bytes per bulk store and size of the zero tile
constexpr int kUpdThreads = 128;   // 4 warps; lane 0 of each issues bulk stores

struct ZeroArgs {
    void *caches[KV_MAX_ZERO_CACHES];
    int32_t num_caches;
    int32_t chunks_per_block;  // ceil(block_bytes / kZeroChunk)
    int64_t block_bytes;
    int64_t num_units;         // num_zero * num_caches * chunks_per_block
};

__device__ __forceinline__ void bulk_store_s2g(void *gdst, uint32_t ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(gdst), "r"(ssrc), "r"(bytes) : "memory");
}

__global__ void __launch_bounds__(kUpdThreads)
apply_block_updates_kernel(const int32_t *__restrict__ updates, int32_t num_updates,
                           int32_t *__restrict__ block_table, int64_t bt_stride, int32_t num_rows,
                           int32_t max_blocks, const int32_t *__restrict__ zero_ids,
                           int32_t num_blocks, int32_t *d_err, const __grid_constant__ ZeroArgs z) {
    // ---- table writes: one thread per (row, column, id)
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < num_updates;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t r = updates[3 * i], c = updates[3 * i + 1], v = updates[3 * i + 2];
        if (r >= 0 && r < num_rows && c >= 0 && c < max_blocks && v >= -1 && v < num_blocks)
            block_table[static_cast<int64_t>(r) * bt_stride + c] = v;
        else
            report(d_err, KV_DERR_BAD_UPDATE);
    }
    if (z.num_units == 0) return;

    // ---- zero fill: this CTA's contiguous range of units
    const int64_t per = (z.num_units + gridDim.x - 1) / gridDim.x;
    const int64_t u0 = per * blockIdx.x;
    const int64_t u1 = u0 + per < z.num_units ? u0 + per : z.num_units;
    if (u0 >= u1) return;

    __shared__ __align__(128) uint4 tile[kZeroChunk / 16];
    for (int i = threadIdx.x; i < kZeroChunk / 16; i += blockDim.x) tile[i] = make_uint4(0, 0, 0, 0);
    // the zeros, written through the generic proxy, must be visible to the bulk copies
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    if (lane != 0) return;
    const uint32_t src = static_cast<uint32_t>(__cvta_generic_to_shared(tile));
    const int64_t per_id = static_cast<int64_t>(z.num_caches) * z.chunks_per_block;
    for (int64_t u = u0 + warp; u < u1; u += nwarps) {
        const int64_t zi = u / per_id;
        const int64_t rem = u - zi * per_id;
        const int cache = static_cast<int>(rem / z.chunks_per_block);
        const int chunk = static_cast<int>(rem - static_cast<int64_t>(cache) * z.chunks_per_block);
        const int32_t b = zero_ids[zi];
        if (b < 0 || b >= num_blocks) {
            if (cache == 0 && chunk == 0) report(d_err, KV_DERR_BAD_UPDATE);
            continue;
        }
        const int64_t off = static_cast<int64_t>(chunk) * kZeroChunk;
        const int64_t left = z.block_bytes - off;
        const uint32_t bytes = static_cast<uint32_t>(left < kZeroChunk ? left : kZeroChunk);
        char *dst = static_cast<char *>(z.caches[cache]) + static_cast<int64_t>(b) * z.block_bytes + off;
        bulk_store_s2g(dst, src, bytes);
    }
    // every store complete (not only its shared-memory reads) before the CTA retires
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

}  // namespace

cudaError_t launch_block_updates(const int32_t *updates, int32_t num_updates, int32_t *block_table,
                                 int64_t bt_stride, int32_t num_rows, int32_t max_blocks,
                                 const int32_t *zero_ids, int32_t num_zero, void *const *caches,
                                 int32_t num_caches, int64_t block_bytes, int32_t num_blocks,
                                 int32_t *d_err, int sm_count, cudaStream_t stream) {
    ZeroArgs z{};
    z.num_caches = num_zero > 0 ? num_caches : 0;
    for (int i = 0; i < z.num_caches; ++i) z.caches[i] = caches[i];
    z.block_bytes = block_bytes;
    z.chunks_per_block = static_cast<int32_t>((block_bytes + kZeroChunk - 1) / kZeroChunk);
    z.num_units = static_cast<int64_t>(num_zero) * z.num_caches * z.chunks_per_block;
    const int64_t upd_ctas = (static_cast<int64_t>(num_updates) + kUpdThreads - 1) / kUpdThreads;
    int64_t grid = z.num_units > upd_ctas ? z.num_units : upd_ctas;
    const int64_t cap = 2 * static_cast<int64_t>(sm_count);
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    apply_block_updates_kernel<<<static_cast<unsigned>(grid), kUpdThreads, 0, stream>>>(
        updates, num_updates, block_table, bt_stride, num_rows, max_blocks, zero_ids, num_blocks, d_err, z);
    return cudaGetLastError();
}

}  // namespace pkv
