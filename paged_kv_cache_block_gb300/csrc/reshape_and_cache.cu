// Cache write: scatter this step's new K/V rows into their slots of the paged cache
// [num_blocks, block_size, num_kv_heads, head_dim] ("vLLM의 KV cache 연결 흐름", section
// "Slot mapping은 왜 필요한가"; layout from "vLLM Worker侧GPU KV Cache初始化流程深度解析", section
// "Worker与ModelRunner的协作"; FP8 E4M3 and INT4 caches from its section "KV Cache技术背景").
#include "common.cuh"
#include "kernels.h"

namespace pkv {

// One thread per 16-byte chunk (8 elements) of a source row, for K and V together.  A slot
// row is num_kv_heads * head_dim contiguous elements, so chunk c of token t lands at element
// slot * row + 8c whatever head it belongs to.
template <typename ST>
__global__ void copy_rows_kernel(const ST *__restrict__ key, const ST *__restrict__ value,
                                 int64_t key_row_stride, int64_t value_row_stride,
                                 int32_t num_tokens, int32_t chunks_per_row,
                                 const int64_t *__restrict__ slot_mapping, ST *__restrict__ k_cache,
                                 ST *__restrict__ v_cache, int64_t total_slots, int32_t *d_err) {
    const int64_t n = static_cast<int64_t>(num_tokens) * chunks_per_row;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t t = static_cast<int32_t>(i / chunks_per_row);
        const int32_t c = static_cast<int32_t>(i - static_cast<int64_t>(t) * chunks_per_row);
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= total_slots) {
            if (c == 0) report(d_err, KV_DERR_BAD_SLOT);
            continue;
        }
        const uint4 kx = *reinterpret_cast<const uint4 *>(key + t * key_row_stride + 8 * c);
        const uint4 vx = *reinterpret_cast<const uint4 *>(value + t * value_row_stride + 8 * c);
        const int64_t dst = (slot * chunks_per_row + c) * 8;
        *reinterpret_cast<uint4 *>(k_cache + dst) = kx;
        *reinterpret_cast<uint4 *>(v_cache + dst) = vx;
    }
}

template <typename ST>
__global__ void quantise_rows_kernel(const ST *__restrict__ key, const ST *__restrict__ value,
                                     int64_t key_row_stride, int64_t value_row_stride,
                                     int32_t num_tokens, int32_t chunks_per_row,
                                     const int64_t *__restrict__ slot_mapping,
                                     uint8_t *__restrict__ k_cache, uint8_t *__restrict__ v_cache,
                                     int64_t total_slots, float k_scale, float v_scale,
                                     int32_t *d_err) {
    const int64_t n = static_cast<int64_t>(num_tokens) * chunks_per_row;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t t = static_cast<int32_t>(i / chunks_per_row);
        const int32_t c = static_cast<int32_t>(i - static_cast<int64_t>(t) * chunks_per_row);
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= total_slots) {
            if (c == 0) report(d_err, KV_DERR_BAD_SLOT);
            continue;
        }
        const uint4 kx = *reinterpret_cast<const uint4 *>(key + t * key_row_stride + 8 * c);
        const uint4 vx = *reinterpret_cast<const uint4 *>(value + t * value_row_stride + 8 * c);
        const int64_t dst = (slot * chunks_per_row + c) * 8;
        *reinterpret_cast<uint2 *>(k_cache + dst) = quantise8<ST>(kx, k_scale);
        *reinterpret_cast<uint2 *>(v_cache + dst) = quantise8<ST>(vx, v_scale);
    }
}

// INT4 with group scales: one thread per 16-byte chunk (8 elements) of a source row, giving 4
// bytes of cache (quantise_int4x8 in common.cuh).  The chunk's 8 dims lie in one scale group
// (group_size is a multiple of 8).
template <typename ST>
__global__ void quantise_int4_rows_kernel(const ST *__restrict__ key, const ST *__restrict__ value,
                                          int64_t key_row_stride, int64_t value_row_stride,
                                          int32_t num_tokens, int32_t chunks_per_row,
                                          int32_t chunks_per_head, int32_t group_shift,
                                          int32_t groups_per_head,
                                          const int64_t *__restrict__ slot_mapping,
                                          uint32_t *__restrict__ k_cache, uint32_t *__restrict__ v_cache,
                                          int64_t total_slots, const float *__restrict__ k_scales,
                                          const float *__restrict__ v_scales, int32_t *d_err) {
    const int64_t n = static_cast<int64_t>(num_tokens) * chunks_per_row;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t t = static_cast<int32_t>(i / chunks_per_row);
        const int32_t c = static_cast<int32_t>(i - static_cast<int64_t>(t) * chunks_per_row);
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= total_slots) {
            if (c == 0) report(d_err, KV_DERR_BAD_SLOT);
            continue;
        }
        const int32_t h = c / chunks_per_head;
        const int32_t sidx = h * groups_per_head + (((c - h * chunks_per_head) * 8) >> group_shift);
        const uint4 kx = *reinterpret_cast<const uint4 *>(key + t * key_row_stride + 8 * c);
        const uint4 vx = *reinterpret_cast<const uint4 *>(value + t * value_row_stride + 8 * c);
        const int64_t dst = slot * chunks_per_row + c;
        k_cache[dst] = quantise_int4x8<ST>(kx, k_scales[sidx]);
        v_cache[dst] = quantise_int4x8<ST>(vx, v_scales[sidx]);
    }
}

cudaError_t launch_reshape_and_cache_int4(const void *key, const void *value, int src_dtype,
                                          int64_t key_row_stride, int64_t value_row_stride,
                                          int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                          const int64_t *slot_mapping, void *k_cache, void *v_cache,
                                          int64_t total_slots, const float *k_scales,
                                          const float *v_scales, int32_t group_size, int32_t *d_err,
                                          int sm_count, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int32_t chunks = num_kv_heads * head_dim / 8;
    const int64_t n = static_cast<int64_t>(num_tokens) * chunks;
    const int threads = 256;
    int64_t blocks = (n + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sm_count) * 16;
    if (blocks > cap) blocks = cap;
    int shift = 0;
    while ((1 << shift) < group_size) ++shift;
    const dim3 grid(static_cast<unsigned>(blocks));
    if (src_dtype == KV_F16)
        quantise_int4_rows_kernel<__half><<<grid, threads, 0, stream>>>(
            static_cast<const __half *>(key), static_cast<const __half *>(value), key_row_stride,
            value_row_stride, num_tokens, chunks, head_dim / 8, shift, head_dim / group_size,
            slot_mapping, static_cast<uint32_t *>(k_cache), static_cast<uint32_t *>(v_cache),
            total_slots, k_scales, v_scales, d_err);
    else
        quantise_int4_rows_kernel<__nv_bfloat16><<<grid, threads, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(key), static_cast<const __nv_bfloat16 *>(value),
            key_row_stride, value_row_stride, num_tokens, chunks, head_dim / 8, shift,
            head_dim / group_size, slot_mapping, static_cast<uint32_t *>(k_cache),
            static_cast<uint32_t *>(v_cache), total_slots, k_scales, v_scales, d_err);
    return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache(const void *key, const void *value, int src_dtype,
                                     int64_t key_row_stride, int64_t value_row_stride,
                                     int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                     const int64_t *slot_mapping, void *k_cache, void *v_cache,
                                     int cache_dtype, int64_t total_slots, float k_scale,
                                     float v_scale, int32_t *d_err, int sm_count,
                                     cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int32_t chunks = num_kv_heads * head_dim / 8;
    const int64_t n = static_cast<int64_t>(num_tokens) * chunks;
    const int threads = 256;
    int64_t blocks = (n + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sm_count) * 16;
    if (blocks > cap) blocks = cap;
    const dim3 grid(static_cast<unsigned>(blocks));
    if (cache_dtype == KV_FP8_E4M3) {
        if (src_dtype == KV_F16)
            quantise_rows_kernel<__half><<<grid, threads, 0, stream>>>(
                static_cast<const __half *>(key), static_cast<const __half *>(value),
                key_row_stride, value_row_stride, num_tokens, chunks, slot_mapping,
                static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache), total_slots,
                k_scale, v_scale, d_err);
        else
            quantise_rows_kernel<__nv_bfloat16><<<grid, threads, 0, stream>>>(
                static_cast<const __nv_bfloat16 *>(key), static_cast<const __nv_bfloat16 *>(value),
                key_row_stride, value_row_stride, num_tokens, chunks, slot_mapping,
                static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache), total_slots,
                k_scale, v_scale, d_err);
    } else {
        copy_rows_kernel<uint16_t><<<grid, threads, 0, stream>>>(
            static_cast<const uint16_t *>(key), static_cast<const uint16_t *>(value),
            key_row_stride, value_row_stride, num_tokens, chunks, slot_mapping,
            static_cast<uint16_t *>(k_cache), static_cast<uint16_t *>(v_cache), total_slots, d_err);
    }
    return cudaGetLastError();
}

}  // namespace pkv
