// Slot mapping: token position -> (logical block, offset) -> physical block -> cache slot.
// "Deep Dive into vLLM Worker-Side GPU KV Cache Initialization", section "Pinpointing the
// Token Slot"; "vLLM의 KV cache 연결 흐름", section "Slot mapping은 왜 필요한가".
#include "common.cuh"
#include "kernels.h"

namespace pkv {

// One thread per token.  The token's request row is the last r with query_start_loc[r] <= t,
// found by binary search over query_start_loc (non-decreasing), staged in shared memory when it
// fits so the search costs no dependent global loads.
constexpr int kQslSmem = 8192;

__global__ void slot_mapping_kernel(const int32_t *__restrict__ block_table, int64_t bt_stride,
                                    int32_t num_seqs, int32_t max_blocks_per_seq,
                                    const int32_t *__restrict__ query_start_loc,
                                    const int32_t *__restrict__ positions, int32_t num_tokens,
                                    int32_t block_size, int32_t num_blocks,
                                    int64_t *__restrict__ slot_mapping, int32_t *d_err) {
    __shared__ int32_t qsl_s[kQslSmem];
    const bool staged = num_seqs + 1 <= kQslSmem;
    if (staged)
        for (int i = threadIdx.x; i <= num_seqs; i += blockDim.x) qsl_s[i] = query_start_loc[i];
    __syncthreads();
    const int32_t *qsl = staged ? qsl_s : query_start_loc;
    for (int32_t t = blockIdx.x * blockDim.x + threadIdx.x; t < num_tokens;
         t += gridDim.x * blockDim.x)
        slot_mapping[t] = slot_of_token(t, qsl, num_seqs, positions, block_table, bt_stride,
                                        max_blocks_per_seq, block_size, num_blocks, d_err);
}

cudaError_t launch_slot_mapping(const int32_t *block_table, int64_t bt_stride, int32_t num_seqs,
                                int32_t max_blocks_per_seq, const int32_t *query_start_loc,
                                const int32_t *positions, int32_t num_tokens, int32_t block_size,
                                int32_t num_blocks, int64_t *slot_mapping, int32_t *d_err,
                                cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int threads = 256;
    const int blocks = (num_tokens + threads - 1) / threads;
    slot_mapping_kernel<<<blocks < 65535 ? blocks : 65535, threads, 0, stream>>>(
        block_table, bt_stride, num_seqs, max_blocks_per_seq, query_start_loc, positions,
        num_tokens, block_size, num_blocks, slot_mapping, d_err);
    return cudaGetLastError();
}

}  // namespace pkv
