// Device helpers for the paged KV cache kernels (sm_103a): inline PTX for mbarriers, TMA tensor
// copies, ldmatrix and mma.sync, plus the bounded waits and error reporting every kernel uses.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedkv.h"

namespace pkv {

// A wait that has not completed after this long gives up, reports KV_DERR_TIMEOUT and returns.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ void report(int32_t *d_err, int32_t bits) {
    if (d_err) atomicOr(d_err, bits);
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete; false once limit_ns have passed.
__device__ __forceinline__ bool mbar_wait_limit(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t n = 0;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 255u) == 255u && globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// The waits of the library's kernels: false after the 2 s limit.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    return mbar_wait_limit(bar, parity, kWaitLimitNs);
}

// Wait for an mbarrier phase with the thread suspended in hardware between checks (a hint of
// up to 0.5 ms a check; it resumes as soon as the phase completes), so that waiting warps do
// not take issue slots from the warps sharing their scheduler.  False after the 2 s limit.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(500000u)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// Release store / acquire load of a shared-memory word, between the threads of a CTA.
__device__ __forceinline__ void st_release_cta(int32_t *p, int32_t v) {
    asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int32_t ld_acquire_cta(const int32_t *p) {
    int32_t v;
    asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}

// Wait until the shared word *p is at least v (a thread of the same CTA raises it with
// st_release_cta); false after the 2 s limit.
__device__ __forceinline__ bool wait_at_least_bounded(const int32_t *p, int32_t v) {
    if (ld_acquire_cta(p) >= v) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        __nanosleep(64);
        if (ld_acquire_cta(p) >= v) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// Prefetch of the L2 line holding p.
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)) : "memory");
}

// 4-D tiled tensor copy global -> shared, completion signalled on an mbarrier (tx bytes).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2, int32_t c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// ------------------------------------------------------------------ tensor-core fragments
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

template <typename T> struct MmaOp;

template <> struct MmaOp<__nv_bfloat16> {
    __device__ __forceinline__ static void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};

template <> struct MmaOp<__half> {
    __device__ __forceinline__ static void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};

// Pack two floats into the 16-bit type T (round to nearest even), low half = a.
template <typename T> __device__ __forceinline__ uint32_t pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
template <> __device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// The two values of a packed pair of T, widened to float (low half first).
template <typename T> __device__ __forceinline__ float2 unpack2(uint32_t v);
template <> __device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t v) {
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}
template <> __device__ __forceinline__ float2 unpack2<__half>(uint32_t v) {
    return __half22float2(*reinterpret_cast<__half2 *>(&v));
}

template <typename T> __device__ __forceinline__ float to_float(T x);
template <> __device__ __forceinline__ float to_float<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <> __device__ __forceinline__ float to_float<__half>(__half x) { return __half2float(x); }

template <typename T> __device__ __forceinline__ T from_float(float x);
template <> __device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}
template <> __device__ __forceinline__ __half from_float<__half>(float x) {
    return __float2half_rn(x);
}

// The row (sequence) of token t: the last r with query_start_loc[r] <= t, or -1.  Decode batches
// give every sequence q_len tokens, so row t / q_len is tried first (one round trip); other
// offsets fall back to a binary search.
__device__ __forceinline__ int token_row(int32_t t, const int32_t *qsl, int32_t num_seqs, int32_t q_len) {
    const int guess = q_len > 0 ? t / q_len : 0;
    if (guess < num_seqs) {
        const int lo_t = qsl[guess], hi_t = qsl[guess + 1];
        if (lo_t <= t && t < hi_t) return guess;
    }
    int lo = 0, hi = num_seqs + 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (qsl[mid] <= t) lo = mid + 1;
        else hi = mid;
    }
    return lo - 1;
}

// ------------------------------------------------------------------ cache write helpers
// Slot of token t ("Pinpointing the Token Slot": logical block pos / bs, offset pos % bs, slot =
// physical * bs + offset), or -1 for padding, tokens in no request's range and invalid entries
// (which also set their error bit).  qsl is non-decreasing; the row is the last r with
// qsl[r] <= t.
__device__ __forceinline__ int64_t slot_of_token(int32_t t, const int32_t *qsl, int32_t num_seqs,
                                                 const int32_t *__restrict__ positions,
                                                 const int32_t *__restrict__ block_table,
                                                 int64_t bt_stride, int32_t max_blocks_per_seq,
                                                 int32_t block_size, int32_t num_blocks,
                                                 int32_t *d_err) {
    const int32_t pos = positions[t];
    int32_t lo = 0, hi = num_seqs + 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi) >> 1;
        if (qsl[mid] <= t) lo = mid + 1;
        else hi = mid;
    }
    const int32_t row = lo - 1;
    if (row < 0 || row >= num_seqs || t >= qsl[row + 1] || pos < 0) return -1;
    const int32_t logical = pos / block_size;
    const int32_t offset = pos - logical * block_size;
    if (logical >= max_blocks_per_seq) {
        report(d_err, KV_DERR_PAST_TABLE);
        return -1;
    }
    const int32_t physical = block_table[row * bt_stride + logical];
    if (physical < 0 || physical >= num_blocks) {
        report(d_err, KV_DERR_BAD_BLOCK);
        return -1;
    }
    return static_cast<int64_t>(physical) * block_size + offset;
}

// Eight 16-bit source values -> eight E4M3 bytes: x / scale in IEEE float32 (correctly rounded
// division), then E4M3 with round-to-nearest-even and saturation to the largest finite value
// (CUDA's own conversion).
template <typename ST>
__device__ __forceinline__ uint2 quantise8(uint4 raw, float scale) {
    const ST *e = reinterpret_cast<const ST *>(&raw);
    uint32_t w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t word = 0;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const float a = __fdiv_rn(to_float<ST>(e[4 * h + 2 * p]), scale);
            const float b = __fdiv_rn(to_float<ST>(e[4 * h + 2 * p + 1]), scale);
            const __nv_fp8x2_storage_t q =
                __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
            word |= static_cast<uint32_t>(q) << (16 * p);
        }
        w[h] = word;
    }
    return make_uint2(w[0], w[1]);
}

// INT4 codes of eight 16-bit source values with one scale: each value divided by the scale in
// float32 (correctly rounded), converted to the nearest integer with ties to even (NaN gives 0,
// overflow saturates), clamped to [-8, 7]; code i in bits 4i .. 4i+3.
__device__ __forceinline__ uint32_t int4_code(float x, float scale) {
    int q = __float2int_rn(__fdiv_rn(x, scale));
    q = q < -8 ? -8 : (q > 7 ? 7 : q);
    return static_cast<uint32_t>(q) & 0xFu;
}

template <typename ST>
__device__ __forceinline__ uint32_t quantise_int4x8(uint4 raw, float scale) {
    const ST *e = reinterpret_cast<const ST *>(&raw);
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) w |= int4_code(to_float<ST>(e[i]), scale) << (4 * i);
    return w;
}


// ------------------------------------------------------------------ grid-wide ordering
// Make this thread's earlier generic-proxy global writes visible to later async-proxy (TMA)
// reads, and the reverse.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Transpose of an 8x8 matrix of 16-bit elements held one row per lane quad (mma fragments).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Eight INT4 codes (one 32-bit word, code i in bits 4i..4i+3) -> four fp16x2 pairs of their
// offset-binary values u = code ^ 8 as subnormals: p[0] = codes (0, 4) * 2^-24,
// p[1] = codes (1, 5) * 2^-20, p[2] = codes (2, 6) * 2^-24, p[3] = codes (3, 7) * 2^-20.
// A pair's low half holds the code from the word's low 16 bits.
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t mask, uint32_t x) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(r) : "r"(a), "r"(mask), "r"(x));  // (a & mask) ^ x
    return r;
}
__device__ __forceinline__ void int4x8_to_h2x4(uint32_t w, uint32_t (&p)[4]) {
    const uint32_t w8 = w >> 8;
    p[0] = and_xor(w, 0x000f000fu, 0x00080008u);
    p[1] = and_xor(w, 0x00f000f0u, 0x00800080u);
    p[2] = and_xor(w8, 0x000f000fu, 0x00080008u);
    p[3] = and_xor(w8, 0x00f000f0u, 0x00800080u);
}

// 2^x on the SFU (ex2.approx); -inf -> +0.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace pkv
