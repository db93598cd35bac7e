// C ABI of libpagedkv.so: host-side argument checks, launch planning and TMA descriptor encoding.
// Every entry point validates what the host can see, then enqueues kernels on the caller's
// stream.  Nothing here allocates device memory or synchronises.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

thread_local char g_last_error[512] = "";

kv_status fail(kv_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
kv_status fail(kv_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

kv_status ok() {
    g_last_error[0] = '\0';
    return KV_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device of the stream, made current for this runtime instance so attribute queries and
// launches agree with the caller's context.  The legacy stream, and a stream that is being
// captured into a graph (where the query is not permitted), use the thread's current device,
// which an earlier uncaptured call on that stream has selected.
cudaError_t bind_device(cudaStream_t stream, int *dev) {
    if (stream) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t e = cudaStreamIsCapturing(stream, &cs);
        if (e != cudaSuccess) return e;
        if (cs == cudaStreamCaptureStatusNone) {
            e = cudaStreamGetDevice(stream, dev);
            if (e != cudaSuccess) return e;
            return cudaSetDevice(*dev);
        }
    }
    return cudaGetDevice(dev);
}

struct DeviceInfo {
    int sm_count;
    int smem_optin;
};

// SM count and opt-in shared memory of a device, queried once per device and then reused (the
// only state the library keeps: immutable device properties).
cudaError_t device_info(int dev, DeviceInfo *info) {
    constexpr int kMaxDevices = 64;
    static DeviceInfo cache[kMaxDevices];
    static std::once_flag once[kMaxDevices];
    static cudaError_t status[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [dev] {
        DeviceInfo d;
        cudaError_t e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cache[dev] = d;
        status[dev] = e;
    });
    *info = cache[dev];
    return status[dev];
}

int round_up(int x, int m) { return (x + m - 1) / m * m; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Launch geometry of the decode kernel.  Deterministic in its arguments and the device's SM
// count / shared-memory limit, so the workspace query and the decode call always agree.
kv_status plan_decode(int32_t num_seqs, int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, int32_t max_seq_len, int32_t window,
                      int32_t num_workers, kv_dtype cache_dtype, const DeviceInfo &dev,
                      pkv::DecodePlan *p, bool fused = false) {
    const bool fp8 = cache_dtype == KV_FP8_E4M3, int4 = cache_dtype == KV_INT4;
    // the fused step has the same geometry and workspace, plus a writer warp
    if (num_seqs < 0 || q_len < 1 || num_q_heads < 1 || num_kv_heads < 1 || max_seq_len < 1 ||
        window < 0 || num_workers < 0)
        return fail(KV_ERR_INVALID_ARG, "negative or zero size argument");
    if (num_q_heads % num_kv_heads)
        return fail(KV_ERR_INVALID_ARG, "num_q_heads (%d) is not a multiple of num_kv_heads (%d)",
                    num_q_heads, num_kv_heads);
    if (head_dim != 64 && head_dim != 128)
        return fail(KV_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
    if ((fp8 || int4) && head_dim != 128)
        return fail(KV_ERR_UNSUPPORTED, "E4M3 and INT4 caches need head_dim 128");
    if (block_size != 4 && block_size != 8 && block_size != 16 && block_size != 32)
        return fail(KV_ERR_UNSUPPORTED, "block_size %d (supported: 4, 8, 16, 32)", block_size);
    if (q_len > 8) return fail(KV_ERR_UNSUPPORTED, "q_len %d (supported: 1..8)", q_len);
    const int g = num_q_heads / num_kv_heads;
    const int rows = g * q_len;
    if (rows > 64)
        return fail(KV_ERR_UNSUPPORTED, "group size x q_len = %d query rows per kv head (max 64)", rows);
    // bytes of one key row of one head in a TMA box, and boxes per row
    const int row_bytes = int4 ? head_dim / 2 : 128;
    const int ndb = int4 ? 1 : head_dim * (fp8 ? 1 : 2) / 128;
    p->rows_per_warp = rows <= 8 ? 8 : 16;
    p->warps_per_head = (rows + p->rows_per_warp - 1) / p->rows_per_warp;
    const int max_warps = p->rows_per_warp == 8 ? pkv::DecodeLaunch<8>::kMaxConsumers
                                                : pkv::DecodeLaunch<16>::kMaxConsumers;
    p->blocks_per_stage = block_size >= 16 ? 1 : 16 / block_size;
    p->stage_tokens = p->blocks_per_stage * block_size;

    // kv heads per CTA: the largest divisor of num_kv_heads whose warps and stage fit
    int hg = 0;
    for (int c = num_kv_heads; c >= 1; --c) {
        if (num_kv_heads % c) continue;
        if (c * p->warps_per_head > max_warps) continue;
        const int box = round_up(c * block_size * row_bytes, 1024);
        if (2 * p->blocks_per_stage * ndb * box > 64 * 1024) continue;
        hg = c;
        break;
    }
    if (hg == 0) return fail(KV_ERR_UNSUPPORTED, "no head grouping fits one CTA");
    p->heads_per_cta = hg;
    p->box_bytes = hg * block_size * row_bytes;
    p->box_stride = round_up(p->box_bytes, 1024);
    p->threads = (hg * p->warps_per_head + 1 + (fused ? 1 : 0)) * 32;
    p->num_items = (num_kv_heads / hg) * num_seqs;
    p->rows_per_item = hg * rows;
    const size_t stage = static_cast<size_t>(2) * p->blocks_per_stage * ndb * p->box_stride;
    p->num_ctas = num_workers > 0 ? num_workers : dev.sm_count;
    if (p->num_ctas > 65535) return fail(KV_ERR_UNSUPPORTED, "num_workers > 65535");
    p->sets_per_cta = 1;
    p->num_workers = p->num_ctas;
    // alignment slack, barriers (2 per stage and the fused step's written-item word) and stage
    // masks, the stage prefix, plus the kernel's static shared memory; the length table joins
    // them when that costs the ring no stage (else the kernel reads lengths from seq_lens)
    const size_t fixed = 1024 + 21 * 8 + 8 + 4 * (static_cast<size_t>(p->num_items) + 1) + 256;
    const size_t lens = 4 * static_cast<size_t>(num_seqs);
    if (static_cast<size_t>(dev.smem_optin) < fixed + 2 * stage)
        return fail(KV_ERR_UNSUPPORTED, "batch too large for the shared-memory stage table");
    auto stages_with = [&](size_t extra) {
        const size_t avail = static_cast<size_t>(dev.smem_optin) - fixed;
        const int n = avail >= extra ? static_cast<int>((avail - extra) / stage) : 0;
        return n > 8 ? 8 : n;
    };
    const int ns = stages_with(0);
    p->lens_smem = stages_with(lens) == ns ? 1 : 0;
    p->num_stages = ns;
    p->smem_bytes = p->num_stages * stage + fixed - 128 + (p->lens_smem ? lens : 0);
    const size_t slots = static_cast<size_t>(p->num_items) + p->num_ctas;
    p->ws_prefix_off = 0;
    p->ws_pieces_off = align256(4 * (static_cast<size_t>(p->num_items) + 1));
    p->ws_lse_off = p->ws_pieces_off + align256(8 * static_cast<size_t>(p->num_items));
    p->ws_o_off = p->ws_lse_off + align256(4 * slots * p->rows_per_item);
    // a piece's fixed cost (the q rows, the output and the masked boundary units of a new item),
    // in quarter stages: about 6 stages for 16-row warps and 2 for 8-row warps over 128-dim
    // heads; with 64-dim heads equal stage counts measured no slower
    p->item_cost = p->rows_per_warp == 16 ? 24 : (head_dim == 128 ? 8 : 0);
    // partial O: one fragment tile (rows_per_warp x head_dim floats) per consumer warp and slot when
    // every row of a warp's tile is a query row, else one row per query row
    const size_t tile_rows = static_cast<size_t>(hg) * p->warps_per_head * p->rows_per_warp;
    p->tile_ws = tile_rows == static_cast<size_t>(p->rows_per_item) ? 1 : 0;
    p->workspace_bytes = p->ws_o_off + 4 * slots * p->rows_per_item * head_dim;
    (void)max_seq_len;
    return KV_OK;
}

// Launch geometry of the INT4 decode kernel (paged_decode_int4.cu): CTAs of 16 warps (8 with
// 16-row tiles), each warp with its own ring of NS stages of one head's K and V boxes; the warps
// form sets of heads_per_cta * warps_per_head, one stream-K worker each.
kv_status plan_decode_int4(int32_t num_seqs, int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_dim, int32_t block_size, int32_t max_seq_len, int32_t window,
                           int32_t num_workers, const DeviceInfo &dev, pkv::DecodePlan *p) {
    if (num_seqs < 0 || q_len < 1 || num_q_heads < 1 || num_kv_heads < 1 || max_seq_len < 1 ||
        window < 0 || num_workers < 0)
        return fail(KV_ERR_INVALID_ARG, "negative or zero size argument");
    if (num_q_heads % num_kv_heads)
        return fail(KV_ERR_INVALID_ARG, "num_q_heads (%d) is not a multiple of num_kv_heads (%d)",
                    num_q_heads, num_kv_heads);
    if (head_dim != 128) return fail(KV_ERR_UNSUPPORTED, "INT4 caches need head_dim 128");
    if (block_size != 4 && block_size != 8 && block_size != 16 && block_size != 32)
        return fail(KV_ERR_UNSUPPORTED, "block_size %d (supported: 4, 8, 16, 32)", block_size);
    if (q_len > 8) return fail(KV_ERR_UNSUPPORTED, "q_len %d (supported: 1..8)", q_len);
    const int g = num_q_heads / num_kv_heads;
    const int rows = g * q_len;
    if (rows > 64)
        return fail(KV_ERR_UNSUPPORTED, "group size x q_len = %d query rows per kv head (max 64)", rows);
    p->rows_per_warp = rows <= 8 ? 8 : 16;
    p->warps_per_head = (rows + p->rows_per_warp - 1) / p->rows_per_warp;
    const int warps = pkv::int4_decode_warps(p->rows_per_warp);
    // kv heads per set: the divisor of num_kv_heads that keeps the most warps busy (the larger
    // one on a tie)
    int hg = 0, best = 0;
    for (int c = num_kv_heads; c >= 1; --c) {
        if (num_kv_heads % c || c * p->warps_per_head > warps) continue;
        const int used = warps / (c * p->warps_per_head) * c * p->warps_per_head;
        if (used > best) {
            best = used;
            hg = c;
        }
    }
    if (hg == 0) return fail(KV_ERR_UNSUPPORTED, "no head grouping fits one CTA");
    p->heads_per_cta = hg;
    p->sets_per_cta = warps / (hg * p->warps_per_head);
    // 32-key stages (16 keys with 4-token blocks): half the per-stage work of 16-key stages
    p->blocks_per_stage = block_size >= 32 ? 1 : (block_size == 4 ? 4 : 32 / block_size);
    p->stage_tokens = p->blocks_per_stage * block_size;
    p->box_bytes = block_size * head_dim / 2;          // one block of one head
    p->box_stride = round_up(p->box_bytes, 512);       // the 64B swizzle repeats every 512 bytes
    p->threads = warps * 32;
    p->num_items = (num_kv_heads / hg) * num_seqs;
    p->rows_per_item = hg * rows;
    p->tile_ws = 0;
    p->lens_smem = 1;
    p->num_workers = num_workers > 0 ? num_workers : p->sets_per_cta * dev.sm_count;
    p->num_ctas = (p->num_workers + p->sets_per_cta - 1) / p->sets_per_cta;
    if (p->num_ctas > 65535) return fail(KV_ERR_UNSUPPORTED, "num_workers too large");
    // per warp and stage: the K and V boxes, a barrier and a mask; plus alignment slack, the
    // stage prefix and the length table; the kernel's static shared memory is 128 bytes
    const size_t stage = static_cast<size_t>(2) * p->blocks_per_stage * p->box_stride;
    const size_t per_stage = static_cast<size_t>(warps) * (stage + 8 + 4);
    const size_t fixed = 1024 + 4 * (static_cast<size_t>(p->num_items) + 1) + 4 * static_cast<size_t>(num_seqs);
    if (static_cast<size_t>(dev.smem_optin) < fixed + 128 + 2 * per_stage)
        return fail(KV_ERR_UNSUPPORTED, "batch too large for the shared-memory stage table");
    const int ns = static_cast<int>((dev.smem_optin - 128 - fixed) / per_stage);
    p->num_stages = ns > 8 ? 8 : ns;
    p->smem_bytes = p->num_stages * per_stage + fixed;
    const size_t slots = static_cast<size_t>(p->num_items) + p->num_workers;
    p->ws_prefix_off = 0;
    p->ws_lse_off = align256(4 * (static_cast<size_t>(p->num_items) + 1));
    p->ws_o_off = p->ws_lse_off + align256(4 * slots * p->rows_per_item);
    p->workspace_bytes = p->ws_o_off + 4 * slots * p->rows_per_item * head_dim;
    (void)max_seq_len;
    return KV_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// The cache viewed as (dim, token-in-block, head, block); one box = one block's rows for a
// group of heads, 128 bytes of head_dim, swizzled 128B (INT4: the whole 64-byte row, as bytes,
// swizzled 64B).  Dims past the pool read as zeros.
kv_status encode_cache_map(CUtensorMap *m, const void *base, kv_dtype cache_dtype, int32_t num_blocks,
                           int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                           int32_t heads_per_cta) {
    auto fn = encode_fn();
    if (!fn) return fail(KV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const bool int4 = cache_dtype == KV_INT4;
    const bool bytes = int4 || cache_dtype == KV_FP8_E4M3;
    const uint64_t eb = bytes ? 1 : 2;
    const uint64_t row = int4 ? head_dim / 2 : head_dim;  // elements of the tensor map per head row
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(row), static_cast<cuuint64_t>(block_size),
                                static_cast<cuuint64_t>(num_kv_heads),
                                static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t strides[3] = {eb * num_kv_heads * row, eb * row, eb * block_size * num_kv_heads * row};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(int4 ? row : 128 / eb), static_cast<cuuint32_t>(block_size),
                               static_cast<cuuint32_t>(heads_per_cta), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 4,
                    const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, int4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KV_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return KV_OK;
}

// Queries [num_tokens, num_q_heads, head_dim] viewed as (dim, head, token); one box = the 64
// dims (128 bytes) of `group` heads of `tokens` tokens, swizzled 128B.
kv_status encode_query_map(CUtensorMap *m, const void *base, int32_t num_tokens, int32_t num_q_heads,
                           int32_t head_dim, int32_t group, int32_t tokens) {
    auto fn = encode_fn();
    if (!fn) return fail(KV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_q_heads),
                                static_cast<cuuint64_t>(num_tokens)};
    const cuuint64_t strides[2] = {2ull * head_dim, 2ull * num_q_heads * head_dim};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(tokens)};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void *>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KV_ERR_CUDA, "cuTensorMapEncodeTiled (queries) failed (CUresult %d)", (int)r);
    return KV_OK;
}

kv_status cuda_fail(cudaError_t e, const char *what) {
    return fail(KV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace

namespace pkv {
kv_status record_error(kv_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}
}  // namespace pkv

extern "C" {

const char *kv_status_string(kv_status s) {
    switch (s) {
        case KV_OK: return "KV_OK";
        case KV_ERR_INVALID_ARG: return "KV_ERR_INVALID_ARG";
        case KV_ERR_UNSUPPORTED: return "KV_ERR_UNSUPPORTED";
        case KV_ERR_CUDA: return "KV_ERR_CUDA";
        case KV_ERR_WORKSPACE: return "KV_ERR_WORKSPACE";
        case KV_ERR_OUT_OF_BLOCKS: return "KV_ERR_OUT_OF_BLOCKS";
    }
    return "KV_ERR_UNKNOWN";
}

const char *kv_last_error(void) { return g_last_error; }

kv_status kv_compute_slot_mapping(const int32_t *block_table, int64_t bt_stride,
                                  int32_t num_seqs, int32_t max_blocks_per_seq,
                                  const int32_t *query_start_loc, const int32_t *positions,
                                  int32_t num_tokens, int32_t block_size, int32_t num_blocks,
                                  int64_t *slot_mapping, int32_t *d_err, void *stream) {
    if (num_tokens < 0 || num_seqs < 0 || max_blocks_per_seq < 0 || block_size < 1 || num_blocks < 0 ||
        bt_stride < max_blocks_per_seq)
        return fail(KV_ERR_INVALID_ARG, "invalid size argument");
    if (num_tokens == 0) return ok();
    if (!query_start_loc || !positions || !slot_mapping || (num_seqs > 0 && !block_table))
        return fail(KV_ERR_INVALID_ARG, "null pointer");
    int dev;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = bind_device(s, &dev);
    if (e != cudaSuccess) return cuda_fail(e, "device of stream");
    e = pkv::launch_slot_mapping(block_table, bt_stride, num_seqs, max_blocks_per_seq,
                                 query_start_loc, positions, num_tokens, block_size, num_blocks,
                                 slot_mapping, d_err, s);
    if (e != cudaSuccess) return cuda_fail(e, "slot mapping launch");
    return ok();
}

kv_status kv_reshape_and_cache(const void *key, const void *value, kv_dtype src_dtype,
                               int64_t key_row_stride, int64_t value_row_stride,
                               int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                               const int64_t *slot_mapping, void *k_cache, void *v_cache,
                               kv_dtype cache_dtype, int32_t num_blocks, int32_t block_size,
                               float k_scale, float v_scale, int32_t *d_err, void *stream) {
    if (num_tokens < 0 || num_kv_heads < 1 || head_dim < 8 || num_blocks < 0 || block_size < 1)
        return fail(KV_ERR_INVALID_ARG, "invalid size argument");
    if (num_tokens == 0) return ok();
    if (!key || !value || !slot_mapping || !k_cache || !v_cache)
        return fail(KV_ERR_INVALID_ARG, "null pointer");
    if (src_dtype != KV_F16 && src_dtype != KV_BF16)
        return fail(KV_ERR_UNSUPPORTED, "source dtype must be fp16 or bf16");
    if (cache_dtype == KV_INT4)
        return fail(KV_ERR_UNSUPPORTED, "INT4 caches are written by kv_reshape_and_cache_int4");
    if (cache_dtype != src_dtype && cache_dtype != KV_FP8_E4M3)
        return fail(KV_ERR_UNSUPPORTED, "cache dtype must equal the source dtype or be E4M3");
    if (head_dim % 8)
        return fail(KV_ERR_UNSUPPORTED, "head_dim must be a multiple of 8");
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
    if (key_row_stride < row || value_row_stride < row || key_row_stride % 8 || value_row_stride % 8)
        return fail(KV_ERR_INVALID_ARG, "row strides must be >= num_kv_heads*head_dim and multiples of 8");
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return fail(KV_ERR_INVALID_ARG, "key, value and caches must be 16-byte aligned");
    if (cache_dtype == KV_FP8_E4M3 && !(k_scale > 0.f && v_scale > 0.f && std::isfinite(k_scale) &&
                                        std::isfinite(v_scale)))
        return fail(KV_ERR_INVALID_ARG, "E4M3 scales must be finite and > 0");
    int dev;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = bind_device(s, &dev);
    if (e != cudaSuccess) return cuda_fail(e, "device of stream");
    DeviceInfo info;
    if ((e = device_info(dev, &info)) != cudaSuccess) return cuda_fail(e, "device attributes");
    e = pkv::launch_reshape_and_cache(key, value, src_dtype, key_row_stride, value_row_stride,
                                      num_tokens, num_kv_heads, head_dim, slot_mapping, k_cache,
                                      v_cache, cache_dtype,
                                      static_cast<int64_t>(num_blocks) * block_size, k_scale,
                                      v_scale, d_err, info.sm_count, s);
    if (e != cudaSuccess) return cuda_fail(e, "cache write launch");
    return ok();
}

size_t kv_paged_attention_workspace_size(int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
                                         int32_t num_kv_heads, int32_t head_dim,
                                         int32_t block_size, kv_dtype cache_dtype,
                                         int32_t max_seq_len, int32_t window,
                                         int32_t num_workers) {
    int dev;
    if (cudaGetDevice(&dev) != cudaSuccess) return SIZE_MAX;
    DeviceInfo info;
    if (device_info(dev, &info) != cudaSuccess) return SIZE_MAX;
    pkv::DecodePlan p{};
    const kv_status st =
        cache_dtype == KV_INT4
            ? plan_decode_int4(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                               max_seq_len, window, num_workers, info, &p)
            : plan_decode(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, max_seq_len,
                          window, num_workers, cache_dtype, info, &p);
    if (st != KV_OK) return SIZE_MAX;
    return p.workspace_bytes;
}

kv_status kv_paged_attention_plan_info(int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                       kv_dtype cache_dtype, int32_t max_seq_len, int32_t window,
                                       int32_t num_workers, int64_t *info) {
    if (!info) return fail(KV_ERR_INVALID_ARG, "null info");
    int dev;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "current device");
    DeviceInfo di;
    if ((e = device_info(dev, &di)) != cudaSuccess) return cuda_fail(e, "device attributes");
    pkv::DecodePlan p{};
    const bool int4 = cache_dtype == KV_INT4;
    const kv_status st =
        int4 ? plan_decode_int4(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, max_seq_len,
                                window, num_workers, di, &p)
             : plan_decode(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, max_seq_len,
                           window, num_workers, cache_dtype, di, &p);
    if (st != KV_OK) return st;
    const int ndb = int4 ? 1 : head_dim * (cache_dtype == KV_FP8_E4M3 ? 1 : 2) / 128;
    info[0] = p.num_stages;
    info[1] = static_cast<int64_t>(2) * p.blocks_per_stage * ndb * p.box_stride;
    info[2] = p.heads_per_cta;
    info[3] = p.num_ctas;
    info[4] = p.threads;
    info[5] = p.rows_per_warp;
    info[6] = p.num_items;
    info[7] = static_cast<int64_t>(p.workspace_bytes);
    return ok();
}

kv_status kv_paged_attention_decode(const void *q, kv_dtype q_dtype, int32_t num_seqs,
                                    int32_t q_len, int32_t num_q_heads, const void *k_cache,
                                    const void *v_cache, kv_dtype cache_dtype,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                    int32_t num_blocks, const int32_t *block_table,
                                    int64_t bt_stride, int32_t max_blocks_per_seq,
                                    const int32_t *seq_lens, int32_t max_seq_len, float scale,
                                    int32_t window, float k_scale, float v_scale,
                                    int32_t num_workers, void *workspace,
                                    size_t workspace_bytes, void *out, float *lse_out,
                                    int32_t *d_err, void *stream) {
    if (q_dtype != KV_F16 && q_dtype != KV_BF16)
        return fail(KV_ERR_UNSUPPORTED, "q dtype must be fp16 or bf16");
    if (cache_dtype != q_dtype && cache_dtype != KV_FP8_E4M3)
        return fail(KV_ERR_UNSUPPORTED, "a 16-bit cache must have the q dtype");
    const bool fp8 = cache_dtype == KV_FP8_E4M3;
    if (fp8 && !(k_scale > 0.f && v_scale > 0.f && std::isfinite(k_scale) && std::isfinite(v_scale)))
        return fail(KV_ERR_INVALID_ARG, "E4M3 scales must be finite and > 0");
    if (!std::isfinite(scale)) return fail(KV_ERR_INVALID_ARG, "scale must be finite");
    if (num_blocks < 1 || max_blocks_per_seq < 1 || bt_stride < max_blocks_per_seq)
        return fail(KV_ERR_INVALID_ARG, "invalid pool or block-table size");
    if (num_seqs == 0) return ok();
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out)
        return fail(KV_ERR_INVALID_ARG, "null pointer");
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        (lse_out && !aligned(lse_out, 4)) || !aligned(block_table, 4) || !aligned(seq_lens, 4))
        return fail(KV_ERR_INVALID_ARG, "q, out and caches must be 16-byte aligned");
    int dev;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = bind_device(s, &dev);
    if (e != cudaSuccess) return cuda_fail(e, "device of stream");
    DeviceInfo info;
    if ((e = device_info(dev, &info)) != cudaSuccess) return cuda_fail(e, "device attributes");
    pkv::DecodePlan plan{};
    kv_status st = plan_decode(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                               max_seq_len, window, num_workers, cache_dtype, info, &plan);
    if (st != KV_OK) return st;
    pkv::DecodeArgs a;
    std::memset(&a, 0, sizeof a);
    if (!workspace || workspace_bytes < plan.workspace_bytes)
        return fail(KV_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", plan.workspace_bytes,
                    workspace ? workspace_bytes : 0);
    if (!aligned(workspace, 256)) return fail(KV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    a.ws_prefix = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + plan.ws_prefix_off);
    a.ws_pieces = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + plan.ws_pieces_off);
    a.ws_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + plan.ws_lse_off);
    a.ws_o = reinterpret_cast<float *>(static_cast<char *>(workspace) + plan.ws_o_off);
    CUtensorMap tk, tv;
    if ((st = encode_cache_map(&tk, k_cache, cache_dtype, num_blocks, block_size, num_kv_heads, head_dim,
                               plan.heads_per_cta)) != KV_OK)
        return st;
    if ((st = encode_cache_map(&tv, v_cache, cache_dtype, num_blocks, block_size, num_kv_heads, head_dim,
                               plan.heads_per_cta)) != KV_OK)
        return st;
    a.q = q;
    a.out = out;
    a.lse_out = lse_out;
    a.block_table = block_table;
    a.bt_stride = bt_stride;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.seq_lens = seq_lens;
    a.max_seq_len = max_seq_len;
    a.d_err = d_err;
    a.num_seqs = num_seqs;
    a.q_len = q_len;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.window = window;
    a.scale_log2 = scale * (fp8 ? k_scale : 1.0f) * 1.4426950408889634f;
    a.v_scale = fp8 ? v_scale : 1.0f;
    e = pkv::launch_paged_decode(tk, tv, a, plan, q_dtype, cache_dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "paged decode launch");
    return ok();
}

kv_status kv_selftest_bounded_wait(int32_t limit_us, int32_t *d_err, int32_t *d_waited_us, void *stream) {
    if (limit_us < 1 || limit_us > 1000000) return fail(KV_ERR_INVALID_ARG, "limit_us must be in 1 .. 1000000");
    if (!d_err) return fail(KV_ERR_INVALID_ARG, "null d_err");
    if (!aligned(d_err, 4) || (d_waited_us && !aligned(d_waited_us, 4)))
        return fail(KV_ERR_INVALID_ARG, "d_err and d_waited_us must be 4-byte aligned");
    int dev;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = bind_device(s, &dev);
    if (e != cudaSuccess) return cuda_fail(e, "device of stream");
    e = pkv::launch_selftest_bounded_wait(limit_us, d_err, d_waited_us, s);
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    return ok();
}

// ---------------------------------------------------------------- INT4 caches (pagedkv_int4.h)

static kv_status check_int4_layout(int32_t head_dim, int32_t group_size, const float *k_scales,
                                   const float *v_scales) {
    if (head_dim != 128) return fail(KV_ERR_UNSUPPORTED, "INT4 caches need head_dim 128");
    if (group_size < 8 || group_size > head_dim || (group_size & (group_size - 1)))
        return fail(KV_ERR_UNSUPPORTED, "group_size %d (supported: 8, 16, 32, 64, 128)", group_size);
    if (!k_scales || !v_scales) return fail(KV_ERR_INVALID_ARG, "null scale array");
    if (!aligned(k_scales, 4) || !aligned(v_scales, 4))
        return fail(KV_ERR_INVALID_ARG, "scale arrays must be 4-byte aligned");
    return KV_OK;
}

kv_status kv_reshape_and_cache_int4(const void *key, const void *value, kv_dtype src_dtype,
                                    int64_t key_row_stride, int64_t value_row_stride,
                                    int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                    const int64_t *slot_mapping, void *k_cache, void *v_cache,
                                    int32_t num_blocks, int32_t block_size, const float *k_scales,
                                    const float *v_scales, int32_t group_size, int32_t *d_err,
                                    void *stream) {
    if (num_tokens < 0 || num_kv_heads < 1 || head_dim < 8 || num_blocks < 0 || block_size < 1)
        return fail(KV_ERR_INVALID_ARG, "invalid size argument");
    if (num_tokens == 0) return ok();
    if (!key || !value || !slot_mapping || !k_cache || !v_cache)
        return fail(KV_ERR_INVALID_ARG, "null pointer");
    if (src_dtype != KV_F16 && src_dtype != KV_BF16)
        return fail(KV_ERR_UNSUPPORTED, "source dtype must be fp16 or bf16");
    kv_status st = check_int4_layout(head_dim, group_size, k_scales, v_scales);
    if (st != KV_OK) return st;
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
    if (key_row_stride < row || value_row_stride < row || key_row_stride % 8 || value_row_stride % 8)
        return fail(KV_ERR_INVALID_ARG, "row strides must be >= num_kv_heads*head_dim and multiples of 8");
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return fail(KV_ERR_INVALID_ARG, "key, value and caches must be 16-byte aligned");
    int dev;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = bind_device(s, &dev);
    if (e != cudaSuccess) return cuda_fail(e, "device of stream");
    DeviceInfo info;
    if ((e = device_info(dev, &info)) != cudaSuccess) return cuda_fail(e, "device attributes");
    e = pkv::launch_reshape_and_cache_int4(key, value, src_dtype, key_row_stride, value_row_stride,
                                           num_tokens, num_kv_heads, head_dim, slot_mapping, k_cache,
                                           v_cache, static_cast<int64_t>(num_blocks) * block_size,
                                           k_scales, v_scales, group_size, d_err, info.sm_count, s);
    if (e != cudaSuccess) return cuda_fail(e, "INT4 cache write launch");
    return ok();
}

kv_status kv_paged_attention_decode_int4(
    const void *q, kv_dtype q_dtype, int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
    const void *k_cache, const void *v_cache, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int32_t num_blocks, const int32_t *block_table, int64_t bt_stride,
    int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t max_seq_len, float scale,
    int32_t window, const float *k_scales, const float *v_scales, int32_t group_size,
    int32_t num_workers, void *workspace, size_t workspace_bytes, void *out, float *lse_out,
    int32_t *d_err, void *stream) {
    if (q_dtype != KV_F16 && q_dtype != KV_BF16)
        return fail(KV_ERR_UNSUPPORTED, "q dtype must be fp16 or bf16");
    if (!std::isfinite(scale)) return fail(KV_ERR_INVALID_ARG, "scale must be finite");
    if (num_blocks < 1 || max_blocks_per_seq < 1 || bt_stride < max_blocks_per_seq)
        return fail(KV_ERR_INVALID_ARG, "invalid pool or block-table size");
    if (num_seqs == 0) return ok();
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out)
        return fail(KV_ERR_INVALID_ARG, "null pointer");
    kv_status st = check_int4_layout(head_dim, group_size, k_scales, v_scales);
    if (st != KV_OK) return st;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        (lse_out && !aligned(lse_out, 4)) || !aligned(block_table, 4) || !aligned(seq_lens, 4))
        return fail(KV_ERR_INVALID_ARG, "q, out and caches must be 16-byte aligned");
    int dev;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = bind_device(s, &dev);
    if (e != cudaSuccess) return cuda_fail(e, "device of stream");
    DeviceInfo info;
    if ((e = device_info(dev, &info)) != cudaSuccess) return cuda_fail(e, "device attributes");
    pkv::DecodePlan plan{};
    st = plan_decode_int4(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                          max_seq_len, window, num_workers, info, &plan);
    if (st != KV_OK) return st;
    if (!workspace || workspace_bytes < plan.workspace_bytes)
        return fail(KV_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", plan.workspace_bytes,
                    workspace ? workspace_bytes : 0);
    if (!aligned(workspace, 256)) return fail(KV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    pkv::DecodeArgs a;
    std::memset(&a, 0, sizeof a);
    a.ws_prefix = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + plan.ws_prefix_off);
    a.ws_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + plan.ws_lse_off);
    a.ws_o = reinterpret_cast<float *>(static_cast<char *>(workspace) + plan.ws_o_off);
    CUtensorMap tk, tv;
    // boxes of one head: every warp loads its own head's rows
    if ((st = encode_cache_map(&tk, k_cache, KV_INT4, num_blocks, block_size, num_kv_heads, head_dim, 1)) != KV_OK)
        return st;
    if ((st = encode_cache_map(&tv, v_cache, KV_INT4, num_blocks, block_size, num_kv_heads, head_dim, 1)) != KV_OK)
        return st;
    a.q = q;
    a.out = out;
    a.lse_out = lse_out;
    a.block_table = block_table;
    a.bt_stride = bt_stride;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.seq_lens = seq_lens;
    a.max_seq_len = max_seq_len;
    a.d_err = d_err;
    a.num_seqs = num_seqs;
    a.q_len = q_len;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.window = window;
    // the MMAs see codes in units of 2^-24 (q carries the remaining factors)
    a.scale_log2 = scale * 1.4426950408889634f * 16777216.f;
    a.v_scale = 1.0f;
    a.k_gscales = k_scales;
    a.v_gscales = v_scales;
    int shift = 0;
    while ((1 << shift) < group_size) ++shift;
    a.group_shift = shift;
    a.lse_offset_scale = 8.f * scale;
    e = pkv::launch_paged_decode_int4(tk, tv, a, plan, q_dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "INT4 paged decode launch");
    return ok();
}

kv_status kv_decode_step_int4(
    const int32_t *block_table, int64_t bt_stride, int32_t max_blocks_per_seq,
    const int32_t *query_start_loc, const int32_t *positions, int64_t *slot_mapping, const void *key,
    const void *value, int64_t key_row_stride, int64_t value_row_stride, const void *q, kv_dtype q_dtype,
    int32_t num_seqs, int32_t q_len, int32_t num_q_heads, void *k_cache, void *v_cache,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
    const int32_t *seq_lens, int32_t max_seq_len, float scale, int32_t window, const float *k_scales,
    const float *v_scales, int32_t group_size, int32_t num_workers, void *workspace,
    size_t workspace_bytes, void *out, float *lse_out, int32_t *d_err, void *stream) {
    if (q_dtype != KV_F16 && q_dtype != KV_BF16)
        return fail(KV_ERR_UNSUPPORTED, "q dtype must be fp16 or bf16");
    if (!std::isfinite(scale)) return fail(KV_ERR_INVALID_ARG, "scale must be finite");
    if (num_blocks < 1 || max_blocks_per_seq < 1 || bt_stride < max_blocks_per_seq)
        return fail(KV_ERR_INVALID_ARG, "invalid pool or block-table size");
    if (num_seqs < 0 || q_len < 1) return fail(KV_ERR_INVALID_ARG, "invalid batch size");
    if (num_seqs == 0) return ok();
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out || !query_start_loc ||
        !positions || !key || !value)
        return fail(KV_ERR_INVALID_ARG, "null pointer");
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
    if (key_row_stride < row || value_row_stride < row || key_row_stride % 8 || value_row_stride % 8)
        return fail(KV_ERR_INVALID_ARG, "row strides must be >= num_kv_heads*head_dim and multiples of 8");
    if (!aligned(key, 16) || !aligned(value, 16) || (slot_mapping && !aligned(slot_mapping, 8)))
        return fail(KV_ERR_INVALID_ARG, "key and value must be 16-byte aligned");
    kv_status st = check_int4_layout(head_dim, group_size, k_scales, v_scales);
    if (st != KV_OK) return st;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        (lse_out && !aligned(lse_out, 4)) || !aligned(block_table, 4) || !aligned(seq_lens, 4))
        return fail(KV_ERR_INVALID_ARG, "q, out and caches must be 16-byte aligned");
    int dev;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = bind_device(s, &dev);
    if (e != cudaSuccess) return cuda_fail(e, "device of stream");
    DeviceInfo info;
    if ((e = device_info(dev, &info)) != cudaSuccess) return cuda_fail(e, "device attributes");
    pkv::DecodePlan plan{};
    st = plan_decode_int4(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                          max_seq_len, window, num_workers, info, &plan);
    if (st != KV_OK) return st;
    if (!workspace || workspace_bytes < plan.workspace_bytes)
        return fail(KV_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", plan.workspace_bytes,
                    workspace ? workspace_bytes : 0);
    if (!aligned(workspace, 256)) return fail(KV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    pkv::DecodeArgs a;
    std::memset(&a, 0, sizeof a);
    a.ws_prefix = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + plan.ws_prefix_off);
    a.ws_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + plan.ws_lse_off);
    a.ws_o = reinterpret_cast<float *>(static_cast<char *>(workspace) + plan.ws_o_off);
    CUtensorMap tk, tv;
    // boxes of one head: every warp loads its own head's rows
    if ((st = encode_cache_map(&tk, k_cache, KV_INT4, num_blocks, block_size, num_kv_heads, head_dim, 1)) != KV_OK)
        return st;
    if ((st = encode_cache_map(&tv, v_cache, KV_INT4, num_blocks, block_size, num_kv_heads, head_dim, 1)) != KV_OK)
        return st;
    a.q = q;
    a.out = out;
    a.lse_out = lse_out;
    a.block_table = block_table;
    a.bt_stride = bt_stride;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.seq_lens = seq_lens;
    a.max_seq_len = max_seq_len;
    a.d_err = d_err;
    a.num_seqs = num_seqs;
    a.q_len = q_len;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.window = window;
    // the MMAs see codes in units of 2^-24 (q carries the remaining factors)
    a.scale_log2 = scale * 1.4426950408889634f * 16777216.f;
    a.v_scale = 1.0f;
    a.k_gscales = k_scales;
    a.v_gscales = v_scales;
    int shift = 0;
    while ((1 << shift) < group_size) ++shift;
    a.group_shift = shift;
    a.lse_offset_scale = 8.f * scale;
    pkv::StepArgs f;
    f.query_start_loc = query_start_loc;
    f.positions = positions;
    f.num_tokens = num_seqs * q_len;
    f.key = key;
    f.value = value;
    f.key_row_stride = key_row_stride;
    f.value_row_stride = value_row_stride;
    f.k_cache = k_cache;
    f.v_cache = v_cache;
    f.total_slots = static_cast<int64_t>(num_blocks) * block_size;
    f.k_scale = 1.0f;
    f.v_scale = 1.0f;
    f.slot_mapping = slot_mapping;
    e = pkv::launch_decode_step_int4(tk, tv, a, f, plan, q_dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "INT4 decode step launch");
    return ok();
}

kv_status kv_decode_step(const int32_t *block_table, int64_t bt_stride, int32_t max_blocks_per_seq,
                         const int32_t *query_start_loc, const int32_t *positions,
                         int64_t *slot_mapping, const void *key, const void *value,
                         int64_t key_row_stride, int64_t value_row_stride, const void *q,
                         kv_dtype q_dtype, int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
                         void *k_cache, void *v_cache, kv_dtype cache_dtype, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, int32_t num_blocks,
                         const int32_t *seq_lens, int32_t max_seq_len, float scale, int32_t window,
                         float k_scale, float v_scale, int32_t num_workers, void *workspace,
                         size_t workspace_bytes, void *out, float *lse_out, int32_t *d_err,
                         void *stream) {
    if (q_dtype != KV_F16 && q_dtype != KV_BF16)
        return fail(KV_ERR_UNSUPPORTED, "q and new K/V dtype must be fp16 or bf16");
    if (cache_dtype != q_dtype && cache_dtype != KV_FP8_E4M3)
        return fail(KV_ERR_UNSUPPORTED, "a 16-bit cache must have the q dtype");
    const bool fp8 = cache_dtype == KV_FP8_E4M3;
    if (fp8 && !(k_scale > 0.f && v_scale > 0.f && std::isfinite(k_scale) && std::isfinite(v_scale)))
        return fail(KV_ERR_INVALID_ARG, "E4M3 scales must be finite and > 0");
    if (!std::isfinite(scale)) return fail(KV_ERR_INVALID_ARG, "scale must be finite");
    if (num_blocks < 1 || max_blocks_per_seq < 1 || bt_stride < max_blocks_per_seq || num_seqs < 0 ||
        q_len < 1)
        return fail(KV_ERR_INVALID_ARG, "invalid pool, block-table or batch size");
    if (num_seqs == 0) return ok();
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out || !query_start_loc ||
        !positions || !key || !value)
        return fail(KV_ERR_INVALID_ARG, "null pointer");
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
    if (key_row_stride < row || value_row_stride < row || key_row_stride % 8 || value_row_stride % 8)
        return fail(KV_ERR_INVALID_ARG, "row strides must be >= num_kv_heads*head_dim and multiples of 8");
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(key, 16) || !aligned(value, 16) || (lse_out && !aligned(lse_out, 4)) ||
        (slot_mapping && !aligned(slot_mapping, 8)))
        return fail(KV_ERR_INVALID_ARG, "q, out, key, value and caches must be 16-byte aligned");
    int dev;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = bind_device(s, &dev);
    if (e != cudaSuccess) return cuda_fail(e, "device of stream");
    DeviceInfo info;
    if ((e = device_info(dev, &info)) != cudaSuccess) return cuda_fail(e, "device attributes");
    pkv::DecodePlan plan{};
    kv_status st = plan_decode(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                               max_seq_len, window, num_workers, cache_dtype, info, &plan, true);
    if (st != KV_OK) return st;
    if (!workspace || workspace_bytes < plan.workspace_bytes)
        return fail(KV_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", plan.workspace_bytes,
                    workspace ? workspace_bytes : 0);
    if (!aligned(workspace, 256)) return fail(KV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    CUtensorMap tk, tv;
    if ((st = encode_cache_map(&tk, k_cache, cache_dtype, num_blocks, block_size, num_kv_heads, head_dim,
                               plan.heads_per_cta)) != KV_OK)
        return st;
    if ((st = encode_cache_map(&tv, v_cache, cache_dtype, num_blocks, block_size, num_kv_heads, head_dim,
                               plan.heads_per_cta)) != KV_OK)
        return st;
    pkv::DecodeArgs a;
    std::memset(&a, 0, sizeof a);
    char *ws = static_cast<char *>(workspace);
    a.ws_prefix = reinterpret_cast<int32_t *>(ws + plan.ws_prefix_off);
    a.ws_pieces = reinterpret_cast<int32_t *>(ws + plan.ws_pieces_off);
    a.ws_lse = reinterpret_cast<float *>(ws + plan.ws_lse_off);
    a.ws_o = reinterpret_cast<float *>(ws + plan.ws_o_off);
    a.q = q;
    a.out = out;
    a.lse_out = lse_out;
    a.block_table = block_table;
    a.bt_stride = bt_stride;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.seq_lens = seq_lens;
    a.max_seq_len = max_seq_len;
    a.d_err = d_err;
    a.num_seqs = num_seqs;
    a.q_len = q_len;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.window = window;
    a.scale_log2 = scale * (fp8 ? k_scale : 1.0f) * 1.4426950408889634f;
    a.v_scale = fp8 ? v_scale : 1.0f;
    pkv::StepArgs f;
    f.query_start_loc = query_start_loc;
    f.positions = positions;
    f.num_tokens = num_seqs * q_len;
    f.key = key;
    f.value = value;
    f.key_row_stride = key_row_stride;
    f.value_row_stride = value_row_stride;
    f.k_cache = k_cache;
    f.v_cache = v_cache;
    f.total_slots = static_cast<int64_t>(num_blocks) * block_size;
    f.k_scale = k_scale;
    f.v_scale = v_scale;
    f.slot_mapping = slot_mapping;
    e = pkv::launch_decode_step(tk, tv, a, f, plan, q_dtype, cache_dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode step launch");
    return ok();
}

kv_status kv_apply_block_updates(const int32_t *updates, int32_t num_updates, int32_t *block_table,
                                 int64_t bt_stride, int32_t num_rows, int32_t max_blocks_per_row,
                                 const int32_t *zero_ids, int32_t num_zero, void *const *caches,
                                 int32_t num_caches, int64_t block_bytes, int32_t num_blocks,
                                 int32_t *d_err, void *stream) {
    if (num_updates < 0 || num_zero < 0 || num_rows < 0 || max_blocks_per_row < 0 || num_blocks < 0 ||
        bt_stride < max_blocks_per_row)
        return fail(KV_ERR_INVALID_ARG, "invalid size argument");
    if (num_updates > 0 && (!updates || !block_table))
        return fail(KV_ERR_INVALID_ARG, "null updates or block table");
    if (num_zero > 0) {
        if (!zero_ids || !caches) return fail(KV_ERR_INVALID_ARG, "null zero-fill ids or cache array");
        if (num_caches < 1 || num_caches > KV_MAX_ZERO_CACHES)
            return fail(KV_ERR_INVALID_ARG, "num_caches %d outside [1, %d]", num_caches, KV_MAX_ZERO_CACHES);
        if (block_bytes <= 0 || block_bytes % 16)
            return fail(KV_ERR_INVALID_ARG, "block_bytes %lld must be a positive multiple of 16",
                        static_cast<long long>(block_bytes));
        for (int i = 0; i < num_caches; ++i)
            if (!caches[i] || !aligned(caches[i], 16))
                return fail(KV_ERR_INVALID_ARG, "cache %d is null or not 16-byte aligned", i);
    }
    if (num_updates == 0 && num_zero == 0) return ok();
    int dev;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = bind_device(s, &dev);
    if (e != cudaSuccess) return cuda_fail(e, "device of stream");
    DeviceInfo info;
    if ((e = device_info(dev, &info)) != cudaSuccess) return cuda_fail(e, "device attributes");
    e = pkv::launch_block_updates(updates, num_updates, block_table, bt_stride, num_rows,
                                  max_blocks_per_row, zero_ids, num_zero, caches, num_caches,
                                  block_bytes, num_blocks, d_err, info.sm_count, s);
    if (e != cudaSuccess) return cuda_fail(e, "block update launch");
    return ok();
}

kv_status kv_paged_attention_prefill(const void *q, kv_dtype q_dtype, const int32_t *query_start_loc,
                                     int32_t num_seqs, int32_t num_tokens, int32_t max_query_len,
                                     int32_t num_q_heads, const void *k_cache, const void *v_cache,
                                     kv_dtype cache_dtype, int32_t num_kv_heads, int32_t head_dim,
                                     int32_t block_size, int32_t num_blocks, const int32_t *block_table,
                                     int64_t bt_stride, int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                     int32_t max_seq_len, float scale, int32_t window, void *out,
                                     float *lse_out, int32_t *d_err, void *stream) {
    if (num_seqs < 0 || num_tokens < 0 || max_query_len < 0 || num_q_heads < 1 || num_kv_heads < 1 ||
        num_blocks < 1 || block_size < 1 || max_blocks_per_seq < 0 || bt_stride < max_blocks_per_seq ||
        max_seq_len < 0 || window < 0)
        return fail(KV_ERR_INVALID_ARG, "invalid size argument");
    if (num_seqs == 0 || num_tokens == 0 || max_query_len == 0) return ok();
    if (!q || !query_start_loc || !k_cache || !v_cache || !block_table || !seq_lens || !out)
        return fail(KV_ERR_INVALID_ARG, "null pointer");
    if (num_q_heads % num_kv_heads)
        return fail(KV_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads");
    const int32_t g = num_q_heads / num_kv_heads;
    if (q_dtype != KV_F16 && q_dtype != KV_BF16)
        return fail(KV_ERR_UNSUPPORTED, "prefill: q must be fp16 or bf16");
    if (cache_dtype != q_dtype) return fail(KV_ERR_UNSUPPORTED, "prefill: the cache dtype must equal the q dtype");
    if (head_dim != 128) return fail(KV_ERR_UNSUPPORTED, "prefill: head_dim must be 128");
    if (block_size != 8 && block_size != 16 && block_size != 32)
        return fail(KV_ERR_UNSUPPORTED, "prefill: block_size must be 8, 16 or 32");
    if (g > 128 || (g & (g - 1)))
        return fail(KV_ERR_UNSUPPORTED, "prefill: num_q_heads / num_kv_heads must be a power of two <= 128");
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
        return fail(KV_ERR_INVALID_ARG, "q, caches and out must be 16-byte aligned");
    if (!(scale >= 0.f) || !std::isfinite(scale)) return fail(KV_ERR_INVALID_ARG, "scale must be finite and >= 0");
    const int64_t tiles = static_cast<int64_t>(num_seqs) * ((max_query_len + 128 / g - 1) / (128 / g));
    if (tiles > 0x7fffffff) return fail(KV_ERR_UNSUPPORTED, "prefill: too many query tiles");
    int dev;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = bind_device(s, &dev);
    if (e != cudaSuccess) return cuda_fail(e, "device of stream");
    DeviceInfo info;
    if ((e = device_info(dev, &info)) != cudaSuccess) return cuda_fail(e, "device attributes");
    if (static_cast<size_t>(info.smem_optin) < pkv::prefill_smem_bytes())
        return fail(KV_ERR_UNSUPPORTED, "prefill: needs %zu bytes of shared memory per block, the device has %d",
                    pkv::prefill_smem_bytes(), info.smem_optin);
    CUtensorMap tq, tk, tv;
    kv_status st = encode_query_map(&tq, q, num_tokens, num_q_heads, head_dim, g, 128 / g);
    if (st == KV_OK) st = encode_cache_map(&tk, k_cache, cache_dtype, num_blocks, block_size, num_kv_heads, head_dim, 1);
    if (st == KV_OK) st = encode_cache_map(&tv, v_cache, cache_dtype, num_blocks, block_size, num_kv_heads, head_dim, 1);
    if (st != KV_OK) return st;
    pkv::PrefillArgs a;
    a.query_start_loc = query_start_loc;
    a.seq_lens = seq_lens;
    a.block_table = block_table;
    a.bt_stride = bt_stride;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_seqs = num_seqs;
    a.num_tokens = num_tokens;
    a.max_query_len = max_query_len;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.max_seq_len = max_seq_len;
    a.window = window;
    a.scale = scale;
    a.out = out;
    a.lse_out = lse_out;
    a.d_err = d_err;
    e = pkv::launch_prefill(tq, tk, tv, a, q_dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return ok();
}

}  // extern "C"
