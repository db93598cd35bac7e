/*
 * pagedkv_selftest.h - a check of the library's failure path on the GPU (part of libpagedkv.so).
 *
 * Every wait inside the library's kernels (on a TMA transfer, on another warp's release) is a
 * bounded mbarrier wait: after its limit the warp reports KV_DERR_TIMEOUT in *d_err, stops, lets
 * its copies in flight land and returns, so the device context stays usable.  No correct input
 * makes a wait run out, so this call provides one that does: a kernel whose single thread waits,
 * with the same bounded-wait code, on an mbarrier phase that nothing completes.
 */
#ifndef PAGEDKV_SELFTEST_H
#define PAGEDKV_SELFTEST_H

#include "pagedkv.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * kv_selftest_bounded_wait - enqueue one kernel (one CTA, one thread) that initialises an
 * mbarrier expecting one arrival, waits on its first phase for limit_us microseconds (nothing
 * arrives), then sets KV_DERR_TIMEOUT in *d_err (a device int32; atomicOr) and writes the waited
 * time in microseconds to *d_waited_us (device int32, may be NULL).  No memory is touched but
 * these two words and the kernel's own shared memory.
 *   limit_us  1 .. 1,000,000 (KV_ERR_INVALID_ARG otherwise)
 * Returns KV_OK once the kernel is enqueued; the caller synchronises and reads *d_err.
 */
KV_API kv_status kv_selftest_bounded_wait(int32_t limit_us, int32_t *d_err, int32_t *d_waited_us,
                                          void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_SELFTEST_H */
