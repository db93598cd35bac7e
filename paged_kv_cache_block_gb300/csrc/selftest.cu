// kv_selftest_bounded_wait: the bounded mbarrier wait of every kernel, made to run out.
#include "common.cuh"
#include "kernels.h"

namespace pkv {
namespace {

__global__ void bounded_wait_kernel(unsigned long long limit_ns, int32_t *d_err, int32_t *d_waited_us) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);  // one arrival expected; none comes
    fence_barrier_init();
    const unsigned long long t0 = globaltimer_ns();
    const bool done = mbar_wait_limit(b, 0, limit_ns);
    const unsigned long long t1 = globaltimer_ns();
    if (!done) report(d_err, KV_DERR_TIMEOUT);
    if (d_waited_us) *d_waited_us = static_cast<int32_t>((t1 - t0) / 1000ull);
}

}  // namespace

cudaError_t launch_selftest_bounded_wait(int32_t limit_us, int32_t *d_err, int32_t *d_waited_us,
                                         cudaStream_t stream) {
    bounded_wait_kernel<<<1, 1, 0, stream>>>(static_cast<unsigned long long>(limit_us) * 1000ull, d_err,
                                             d_waited_us);
    return cudaGetLastError();
}

}  // namespace pkv
