// kv_paged_attention_decode_noalloc: paged decode attention whose scratch lives in a file-scope
// device array, for callers that cannot allocate device memory themselves.
//
// Who needs it: code that runs where calling cudaMalloc is not an option - a plugin inside a
// host framework that owns every device allocation and hands out none, a real-time decode loop
// where an allocation could synchronise the device or fail under fragmentation, or a C caller
// with no allocator of its own.  They pass inputs and outputs only; the library supplies the
// log-sum-exp workspace from g_decode_scratch.
//
// Set-up: the first call on a device (with that device current) looks up the device address of
// g_decode_scratch with cudaGetSymbolAddress and checks the result; the address is kept per device
// once a lookup succeeds (a failed lookup is retried by the next call).  Make that first call
// before any stream capture.  Nothing here allocates: no cudaMalloc, no cudaFree,
// no allocating library routine.
//
// Sharing: every call on a device uses the same array, and it keeps the previous call's contents.
// The kernels write every byte they later read within one call (the stage prefix and each
// partial result are written before they are read), so no clearing is needed between calls.
// Two calls whose work overlaps on the GPU (for example on two streams without ordering between
// them) race on the array: order them on one stream, or use kv_paged_attention_decode with a
// workspace per stream.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

// Maximum scratch: KV_NOALLOC_SCRATCH_BYTES (32 MiB), held by every GPU that loads the library
// until the process exits.  In host code this name is only a stand-in for the symbol, never a
// device address: the kernels get the address from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[KV_NOALLOC_SCRATCH_BYTES];

static constexpr int kMaxDevices = 64;

extern "C" kv_status kv_paged_attention_decode_noalloc(
    const void *q, kv_dtype q_dtype, int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
    const void *k_cache, const void *v_cache, kv_dtype cache_dtype, int32_t num_kv_heads,
    int32_t head_dim, int32_t block_size, int32_t num_blocks, const int32_t *block_table,
    int64_t bt_stride, int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t max_seq_len,
    float scale, int32_t window, float k_scale, float v_scale, int32_t num_workers, void *out,
    float *lse_out, int32_t *d_err, void *stream) {
    // the device whose copy of the array this call uses: the stream's, as for the other entry
    // points (the current device while the stream is being captured)
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    cudaError_t e = cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (s) e = cudaStreamIsCapturing(s, &cs);
    if (e == cudaSuccess) e = (s && cs == cudaStreamCaptureStatusNone) ? cudaStreamGetDevice(s, &dev)
                                                                       : cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);
    if (e != cudaSuccess) return pkv::record_error(KV_ERR_CUDA, "device of stream: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return pkv::record_error(KV_ERR_UNSUPPORTED, "device %d", dev);

    // once per device, with that device current: the device address of the scratch array.  Only
    // a successful lookup is kept, so a call that failed here (for example one made during stream
    // capture) leaves the next call free to try again.
    static std::atomic<void *> scratch[kMaxDevices];
    static std::mutex setup_mu[kMaxDevices];
    void *base = scratch[dev].load(std::memory_order_acquire);
    if (base == nullptr) {
        std::lock_guard<std::mutex> lock(setup_mu[dev]);
        base = scratch[dev].load(std::memory_order_relaxed);
        if (base == nullptr) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_decode_scratch);
            if (e != cudaSuccess || p == nullptr)
                return pkv::record_error(KV_ERR_CUDA, "cudaGetSymbolAddress of the scratch: %s",
                                         cudaGetErrorString(e));
            scratch[dev].store(p, std::memory_order_release);
            base = p;
        }
    }

    // an empty batch still gets the full call's argument checks (it launches nothing)
    if (num_seqs == 0)
        return kv_paged_attention_decode(q, q_dtype, num_seqs, q_len, num_q_heads, k_cache, v_cache,
                                         cache_dtype, num_kv_heads, head_dim, block_size, num_blocks,
                                         block_table, bt_stride, max_blocks_per_seq, seq_lens,
                                         max_seq_len, scale, window, k_scale, v_scale, num_workers,
                                         nullptr, 0, out, lse_out, d_err, stream);
    const size_t need = kv_paged_attention_workspace_size(num_seqs, q_len, num_q_heads, num_kv_heads,
                                                          head_dim, block_size, cache_dtype,
                                                          max_seq_len, window, num_workers);
    if (need == SIZE_MAX)  // invalid or unsupported sizes: let the full call report which
        return kv_paged_attention_decode(q, q_dtype, num_seqs, q_len, num_q_heads, k_cache, v_cache,
                                         cache_dtype, num_kv_heads, head_dim, block_size, num_blocks,
                                         block_table, bt_stride, max_blocks_per_seq, seq_lens,
                                         max_seq_len, scale, window, k_scale, v_scale, num_workers,
                                         nullptr, 0, out, lse_out, d_err, stream);
    if (need > static_cast<size_t>(KV_NOALLOC_SCRATCH_BYTES))
        return pkv::record_error(KV_ERR_WORKSPACE,
                                 "these sizes need %zu bytes of scratch; the static scratch holds %zu "
                                 "(use kv_paged_attention_decode with a caller workspace)",
                                 need, static_cast<size_t>(KV_NOALLOC_SCRATCH_BYTES));
    return kv_paged_attention_decode(q, q_dtype, num_seqs, q_len, num_q_heads, k_cache, v_cache,
                                     cache_dtype, num_kv_heads, head_dim, block_size, num_blocks,
                                     block_table, bt_stride, max_blocks_per_seq, seq_lens,
                                     max_seq_len, scale, window, k_scale, v_scale, num_workers,
                                     base, KV_NOALLOC_SCRATCH_BYTES, out, lse_out, d_err,
                                     stream);
}
