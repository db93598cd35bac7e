// Chunked-prefill paged attention on the fifth-generation tensor cores (tcgen05, TMEM, TMA).
//
// A prefill step ("vLLM의 KV cache 연결 흐름", section "EngineCore가 하는 일": a step computes a
// request's tokens that are not yet in the cache, num_new_tokens of them) attends each new token
// to the sequence's cached keys and to the earlier new tokens, through the block table
// (section "Slot mapping은 왜 필요한가").  Sequence b's n_b query rows are those of
// query_start_loc, at positions L_b - n_b .. L_b - 1; row i sees keys j <= its position (and
// j > position - W with a window), GQA maps q head hq to kv head hq / (Hq / Hkv).  Unlike decode,
// this is a dense contraction: 128 query rows x 128 keys x 128 dims per tile pair.
//
// One CTA computes one tile of 128 query rows of one (sequence, kv head): 128 / g tokens x the
// g query heads of the group (row r = token r / g, head r % g), so each K/V tile read from HBM
// serves all g heads.  Per 128-key tile j:
//   S_j = Q K_j^T      tcgen05.mma kind::f16, M 128, N 128, K 16 x 8, A and B K-major in shared
//                      memory (128B swizzle, as the TMA writes them), fp32 accumulator in TMEM
//   P_j = exp2(S_j * scale * log2 e - m)   softmax warps: one thread per row reads its row of
//                      S_j from TMEM (tcgen05.ld), masks, updates the running max and sum, and
//                      writes P_j (16-bit) to shared memory in the same swizzled K-major layout
//   O += P_j V_j       tcgen05.mma, A = P_j (K-major), B = V_j (MN-major: V rows are keys),
//                      accumulated in TMEM across tiles
// The running max is only moved when a row's new maximum exceeds the one in use by more than
// 2^8 (exp2 values stay below 256, exact enough in fp32 and 16-bit); only then is that row of
// O rescaled in TMEM.  Both the sum and O use the same reference, so the result is unchanged.
//
// Warp roles (192 threads): warps 0-3 softmax and epilogue (thread = TMEM lane = query row),
// warp 4 TMA producer (Q once, then K and V tiles into a 4-entry ring: K0 V0 K1 V1 ...), warp 5
// TMEM allocation and the single thread that issues every MMA.  S is double-buffered in TMEM
// (columns 0-127, 128-255; O in 256-383) so S_{j+1} runs on the tensor cores while the softmax
// warps work on S_j.  Every wait is bounded (2 s): on expiry the CTA reports KV_DERR_TIMEOUT,
// drains what it issued, frees TMEM and returns.
#include "common.cuh"
#include "kernels.h"

namespace pkv {
namespace {

constexpr int kBM = 128;                    // query rows per tile = TMEM lanes
constexpr int kBN = 128;                    // keys per K/V tile
constexpr int kHalfBytes = 128 * 128;       // 128 rows x 64 16-bit elements (one swizzle column)
constexpr int kTileBytes = 2 * kHalfBytes;  // a Q, K, V or P tile: two 64-column halves
constexpr int kStages = 4;                  // K/V ring entries
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;         // S0, S1, O (128 columns each), rounded to a power of 2
constexpr uint32_t kColO = 256;
constexpr float kRescaleLog2 = 8.0f;

constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kTileBytes;
constexpr int kOffP = kOffKV + kStages * kTileBytes;
constexpr int kOffBar = kOffP + 2 * kTileBytes;
constexpr int kNumBars = 16;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;  // + TMEM address, abort flag, alignment

// mbarrier indices
constexpr int kBarQ = 0, kBarKvFull = 1, kBarKvEmpty = 5, kBarS = 9, kBarP = 11, kBarPv = 13,
              kBarDrain = 15;

struct PrefillParams {
    const int32_t *qsl;
    const int32_t *seq_lens;
    const int32_t *block_table;
    int64_t bt_stride;
    int32_t max_blocks_per_seq;
    int32_t num_tokens, num_q_heads, group, tokens_per_tile, qtiles;
    int32_t block_size, num_blocks, max_seq_len, max_query_len, window;
    float scale_log2;
    void *out;
    float *lse_out;
    int32_t *d_err;
};

// ---------------------------------------------------------------- tcgen05 helpers

// Shared-memory matrix descriptor: start address, leading and stride byte offsets (16-byte
// units), the fixed version bit 46, 128B swizzle (mode 2 in bits 61-63).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
           (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A and B type (bits 7-9,
// 10-12: 0 fp16, 1 bf16), B major-ness (bit 16: 0 K-major, 1 MN-major), N / 8 (bits 17-22),
// M / 16 (bits 24-28).
__host__ __device__ constexpr uint32_t mma_idesc(uint32_t ab, bool b_mn_major, int M, int N) {
    return (1u << 4) | (ab << 7) | (ab << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

template <typename T> struct AbFormat;
template <> struct AbFormat<__half> { static constexpr uint32_t value = 0; };
template <> struct AbFormat<__nv_bfloat16> { static constexpr uint32_t value = 1; };

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on an mbarrier when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// ---------------------------------------------------------------- the kernel

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
prefill_attention_kernel(const __grid_constant__ CUtensorMap tmap_q,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x / p.qtiles;
    const int qt = p.qtiles - 1 - static_cast<int>(blockIdx.x % p.qtiles);  // longest tiles first
    const int h = blockIdx.y;
    const int g = p.group, TQ = p.tokens_per_tile, bs = p.block_size;
    const int q0 = p.qsl[b];
    const int n = p.qsl[b + 1] - q0;
    const int L = p.seq_lens[b];
    const int t0 = qt * TQ;
    if (t0 >= n) return;  // the whole CTA: no query row here

    const bool len_ok = n <= p.max_query_len && q0 >= 0 && q0 + n <= p.num_tokens && L >= n &&
                        L <= p.max_seq_len && (L + bs - 1) / bs <= p.max_blocks_per_seq;
    if (!len_ok) {
        // rows of a rejected sequence are written as zeros (lse -inf)
        if (threadIdx.x == 0) report(p.d_err, KV_DERR_BAD_LEN);
        const int rows = q0 < 0 ? 0 : max(0, min(n, p.num_tokens - q0) - t0);
        T *out = static_cast<T *>(p.out);
        for (int r = threadIdx.x; r < kBM; r += blockDim.x) {
            const int tl = r / g;
            if (tl >= min(TQ, rows)) continue;
            const int64_t row = static_cast<int64_t>(q0 + t0 + tl) * p.num_q_heads + h * g + r % g;
            uint4 *o = reinterpret_cast<uint4 *>(out + row * 128);
            for (int c = 0; c < 16; ++c) o[c] = make_uint4(0, 0, 0, 0);
            if (p.lse_out) p.lse_out[row] = -INFINITY;
        }
        return;
    }

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + kOffBar + kNumBars * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffBar + kNumBars * 8 + 4);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    if (threadIdx.x == 0) {
        mbar_init(bar(kBarQ), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(kBarKvFull + s), 1);
            mbar_init(bar(kBarKvEmpty + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(kBarS + s), 1);
            mbar_init(bar(kBarP + s), 128);
            mbar_init(bar(kBarPv + s), 1);
        }
        mbar_init(bar(kBarDrain), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    // keys this tile needs: from the window start of its first query to its last query
    const int n_tile = min(TQ, n - t0);
    const int p_first = L - n + t0;
    const int p_last = p_first + n_tile - 1;
    const int kv_lo = p.window > 0 ? max(0, p_first - p.window + 1) : 0;
    const int kt0 = kv_lo / kBN;
    const int ntiles = p_last / kBN + 1 - kt0;

    if (warp == 4) {
        // ============================================================ TMA producer
        const int bpt = kBN / bs;                  // blocks per K/V tile
        const int nblk_seq = (L + bs - 1) / bs;
        const int first_blk = kv_lo / bs;          // blocks before it are never read
        if (lane == 0) {
            prefetch_tensormap(&tmap_q);
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
            mbar_arrive_expect_tx(bar(kBarQ), kTileBytes);
            tma_load_3d(smem_u32(smem + kOffQ), &tmap_q, bar(kBarQ), 0, h * g, q0 + t0);
            tma_load_3d(smem_u32(smem + kOffQ + kHalfBytes), &tmap_q, bar(kBarQ), 64, h * g, q0 + t0);
        }
        int my_id = p.num_blocks;
        int issued = 0;
        for (int i = 0; i < 2 * ntiles; ++i) {
            const int t = i >> 1;
            const bool is_v = i & 1;
            if (!is_v) {
                const int lb = (kt0 + t) * bpt + lane;
                my_id = p.num_blocks;  // one past the pool: the copy reads zeros
                if (lane < bpt && lb >= first_blk && lb < nblk_seq) {
                    const int e = p.block_table[static_cast<int64_t>(b) * p.bt_stride + lb];
                    if (e >= 0 && e < p.num_blocks) my_id = e;
                    else report(p.d_err, KV_DERR_BAD_BLOCK);
                }
            }
            const int slot = i % kStages;
            int stop = 0;
            if (lane == 0) {
                if (i >= kStages && !mbar_wait_bounded(bar(kBarKvEmpty + slot), ((i / kStages) - 1) & 1)) {
                    stop = 1;
                    report(p.d_err, KV_DERR_TIMEOUT);
                    *abort_flag = 1;
                } else if (*abort_flag) {
                    stop = 1;
                }
                if (!stop) mbar_arrive_expect_tx(bar(kBarKvFull + slot), kTileBytes);
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
            const CUtensorMap *m = is_v ? &tmap_v : &tmap_k;
            uint8_t *dst = smem + kOffKV + slot * kTileBytes;
            for (int j = 0; j < bpt; ++j) {
                const int id = __shfl_sync(0xffffffffu, my_id, j);
                if (lane == 0) {
                    tma_load_4d(smem_u32(dst + j * bs * 128), m, bar(kBarKvFull + slot), 0, 0, h, id);
                    tma_load_4d(smem_u32(dst + kHalfBytes + j * bs * 128), m, bar(kBarKvFull + slot), 64, 0, h, id);
                }
            }
            issued = i + 1;
        }
        // never leave with copies in flight into this CTA's shared memory
        if (lane == 0) {
            if (!mbar_wait_bounded(bar(kBarQ), 0)) report(p.d_err, KV_DERR_TIMEOUT);
            for (int i = max(0, issued - kStages); i < issued; ++i)
                if (!mbar_wait_bounded(bar(kBarKvFull + i % kStages), (i / kStages) & 1))
                    report(p.d_err, KV_DERR_TIMEOUT);
        }
    } else if (warp == 5) {
        // ============================================================ MMA issue (one thread)
        if (lane == 0) {
            constexpr uint32_t ab = AbFormat<T>::value;
            constexpr uint32_t idesc_s = mma_idesc(ab, false, kBM, kBN);
            constexpr uint32_t idesc_pv = mma_idesc(ab, true, kBM, 128);
            const uint32_t sq = smem_u32(smem + kOffQ);
            bool dead = !mbar_wait_bounded(bar(kBarQ), 0);
            tc_fence_after();
            for (int t = 0; t <= ntiles && !dead; ++t) {
                if (*abort_flag) break;
                if (t < ntiles) {
                    // S_t = Q K_t^T into S buffer t % 2
                    const int i = 2 * t, slot = i % kStages;
                    if (!mbar_wait_bounded(bar(kBarKvFull + slot), (i / kStages) & 1)) {
                        dead = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sk = smem_u32(smem + kOffKV + slot * kTileBytes);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t off = (k >> 2) * kHalfBytes + (k & 3) * 32;
                        mma_f16(tmem + (t & 1) * 128, smem_desc(sq + off, 16, 1024),
                                smem_desc(sk + off, 16, 1024), idesc_s, k > 0);
                    }
                    mma_commit(bar(kBarKvEmpty + slot));
                    mma_commit(bar(kBarS + (t & 1)));
                }
                if (t >= 1) {
                    // O += P_u V_u
                    const int u = t - 1;
                    if (!mbar_wait_bounded(bar(kBarP + (u & 1)), (u >> 1) & 1)) {
                        dead = true;
                        break;
                    }
                    const int i = 2 * u + 1, slot = i % kStages;
                    if (!mbar_wait_bounded(bar(kBarKvFull + slot), (i / kStages) & 1)) {
                        dead = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sp = smem_u32(smem + kOffP + (u & 1) * kTileBytes);
                    const uint32_t sv = smem_u32(smem + kOffKV + slot * kTileBytes);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t off_p = (k >> 2) * kHalfBytes + (k & 3) * 32;
                        mma_f16(tmem + kColO, smem_desc(sp + off_p, 16, 1024),
                                smem_desc(sv + k * 2048, kHalfBytes, 1024), idesc_pv, (u > 0 || k > 0));
                    }
                    mma_commit(bar(kBarKvEmpty + slot));
                    mma_commit(bar(kBarPv + (u & 1)));
                }
            }
            if (dead) {
                report(p.d_err, KV_DERR_TIMEOUT);
                *abort_flag = 1;
            }
            // every MMA issued has completed before TMEM is freed
            mma_commit(bar(kBarDrain));
            if (!mbar_wait_bounded(bar(kBarDrain), 0)) report(p.d_err, KV_DERR_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ============================================================ softmax + epilogue
        const int r = threadIdx.x;                 // query row = TMEM lane
        const int tl = r / g;
        const bool valid = tl < n_tile;
        const int pos = p_first + tl;              // this row's query position
        const int klo = p.window > 0 ? pos - p.window + 1 : 0;
        const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        float m_used = -INFINITY, l = 0.f;
        bool dead = false;
        int t = 0;
        // waits are decided for the whole warp: its lanes take the warp-collective TMEM
        // loads and stores together
        auto wait_all = [&](int i, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait_bounded(bar(i), parity));
        };
        for (; t < ntiles; ++t) {
            if (!wait_all(kBarS + (t & 1), (t >> 1) & 1)) {
                dead = true;
                break;
            }
            tc_fence_after();
            float s[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(trow + (t & 1) * 128 + c * 32, s + c * 32);
            tmem_wait_ld();
            const int kbase = (kt0 + t) * kBN;
            float mt = -INFINITY;
#pragma unroll
            for (int c = 0; c < 128; ++c) {
                const int k = kbase + c;
                const bool vis = valid && k <= pos && k >= klo;
                s[c] = vis ? s[c] * p.scale_log2 : -INFINITY;
                mt = fmaxf(mt, s[c]);
            }
            float factor = 1.f;
            bool rescale = false;
            if (mt > m_used + kRescaleLog2) {  // also the first finite maximum (-inf + 8 = -inf)
                factor = fast_exp2(m_used - mt);
                rescale = l > 0.f;
                l *= factor;
                m_used = mt;
            }
            const float ref = m_used == -INFINITY ? 0.f : m_used;
            // P buffer t % 2 is free once PV_{t-2} has completed
            if (t >= 2 && !wait_all(kBarPv + (t & 1), ((t - 2) >> 1) & 1)) {
                dead = true;
                break;
            }
            uint8_t *pb = smem + kOffP + (t & 1) * kTileBytes;
            float sum = 0.f;
#pragma unroll
            for (int c8 = 0; c8 < 16; ++c8) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    w[e] = pack2<T>(fast_exp2(s[c8 * 8 + 2 * e] - ref), fast_exp2(s[c8 * 8 + 2 * e + 1] - ref));
                    const float2 u = unpack2<T>(w[e]);
                    sum += u.x + u.y;
                }
                const int c = c8 & 7;
                *reinterpret_cast<uint4 *>(pb + (c8 >> 3) * kHalfBytes + r * 128 + ((c ^ (r & 7)) << 4)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
            l += sum;
            if (__any_sync(0xffffffffu, rescale)) {
                // O holds PV_0 .. PV_{t-1}: wait for the last of them, then scale the rows that
                // moved their maximum (the warp loads and stores together; others scale by 1)
                if (!wait_all(kBarPv + ((t - 1) & 1), ((t - 1) >> 1) & 1)) {
                    dead = true;
                    break;
                }
                tc_fence_after();
                const float f = rescale ? factor : 1.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float o[32];
                    tmem_ld32(trow + kColO + c * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= f;
                    tmem_st32(trow + kColO + c * 32, o);
                }
                tmem_wait_st();
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // P for the tensor cores
            tc_fence_before();
            mbar_arrive(bar(kBarP + (t & 1)));
        }
        if (dead) {
            if (r == 0) report(p.d_err, KV_DERR_TIMEOUT);
            *abort_flag = 1;
        } else {
            // the last PV has landed: O / l, rounded to T, and the log-sum-exp
            const int u = ntiles - 1;
            const bool ok = wait_all(kBarPv + (u & 1), (u >> 1) & 1);
            if (!ok) {
                if (r == 0) report(p.d_err, KV_DERR_TIMEOUT);
                *abort_flag = 1;
            }
            tc_fence_after();
            const int64_t row = static_cast<int64_t>(q0 + t0 + tl) * p.num_q_heads + h * g + r % g;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            T *out = static_cast<T *>(p.out) + row * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float o[32];
                tmem_ld32(trow + kColO + c * 32, o);
                tmem_wait_ld();
                if (valid && ok) {
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) w[i] = pack2<T>(o[2 * i] * inv, o[2 * i + 1] * inv);
                    uint4 *dst = reinterpret_cast<uint4 *>(out + c * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                }
            }
            if (valid && ok && p.lse_out)
                p.lse_out[row] = l > 0.f ? (m_used + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

template <typename T>
cudaError_t launch_typed(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         const PrefillParams &p, int num_seqs, int num_kv_heads, cudaStream_t stream) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_attention_kernel<T>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const dim3 grid(static_cast<unsigned>(num_seqs) * p.qtiles, num_kv_heads);
    prefill_attention_kernel<T><<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

size_t prefill_smem_bytes() { return kSmemBytes; }

cudaError_t launch_prefill(const CUtensorMap &tmap_q, const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                           const PrefillArgs &a, int q_dtype, cudaStream_t stream) {
    PrefillParams p;
    p.qsl = a.query_start_loc;
    p.seq_lens = a.seq_lens;
    p.block_table = a.block_table;
    p.bt_stride = a.bt_stride;
    p.max_blocks_per_seq = a.max_blocks_per_seq;
    p.num_tokens = a.num_tokens;
    p.num_q_heads = a.num_q_heads;
    p.group = a.num_q_heads / a.num_kv_heads;
    p.tokens_per_tile = kBM / p.group;
    p.qtiles = (a.max_query_len + p.tokens_per_tile - 1) / p.tokens_per_tile;
    p.block_size = a.block_size;
    p.num_blocks = a.num_blocks;
    p.max_seq_len = a.max_seq_len;
    p.max_query_len = a.max_query_len;
    p.window = a.window;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.out = a.out;
    p.lse_out = a.lse_out;
    p.d_err = a.d_err;
    if (q_dtype == KV_BF16)
        return launch_typed<__nv_bfloat16>(tmap_q, tmap_k, tmap_v, p, a.num_seqs, a.num_kv_heads, stream);
    return launch_typed<__half>(tmap_q, tmap_k, tmap_v, p, a.num_seqs, a.num_kv_heads, stream);
}

}  // namespace pkv
