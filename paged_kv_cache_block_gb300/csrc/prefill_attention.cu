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
// One CTA computes two consecutive tiles of 128 query rows (A and B) of one (sequence, kv
// head); a tile is 128 / g tokens x the g query heads of the group (row r = token r / g, head
// r % g), so each K/V tile read serves 2 x 128 rows.  Per 128-key tile j and Q tile x:
//   S_x,j = Q_x K_j^T    tcgen05.mma kind::f16, M 128, N 128, K 16 x 8; A and B K-major in shared
//                        memory (128B swizzle, as the TMA writes them); fp32 accumulator in TMEM
//   P_x,j = exp2(S_x,j * scale * log2 e - m)   one thread per row reads its row of S from TMEM
//                        (tcgen05.ld), masks (only tiles that hold a hidden key), tracks the
//                        maximum, and writes P (16-bit pairs) back into TMEM over the S columns it
//                        has read; the normaliser sums the rounded weights
//   O_x += P_x,j V_j     tcgen05.mma with A in TMEM (P) and B = V_j (MN-major: V rows are keys),
//                        fp32 in TMEM across tiles; once it has completed, S_x,j+1 may overwrite
//                        the P columns
// The weights are computed against the reference maximum already in use; only when a row's
// maximum exceeds it by more than 2^8 (its first visible tile, or a rare jump) are that row's O
// and sum rescaled and the tile's weights computed again, so the exponentials stay below 256.
//
// Warp roles (352 threads): warps 0-3 softmax for Q tile A, 4-7 for Q tile B (thread = TMEM
// lane = query row), warp 8 TMA producer (Q once, then K and V tiles into a 5-entry ring: K0 V0
// K1 V1 ..., block ids read a tile ahead), warps 9 and 10 issue the MMAs of tile A and of tile B
// (one lane each; warp 9 also allocates TMEM).  The two softmax warpgroups take turns, so one
// tile's softmax overlaps the other tile's products.  TMEM: S_A / P_A in columns 0-127, S_B / P_B
// 128-255, O_A 256-383, O_B 384-511.  Every wait is bounded (2 s): on expiry the CTA reports
// KV_DERR_TIMEOUT, drains what it issued, frees TMEM and returns.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace pkv {
namespace {

constexpr int kBM = 128;                    // query rows per Q tile = TMEM lanes
constexpr int kBN = 128;                    // keys per K/V tile
constexpr int kQHalf = 128 * 128;           // 128 rows x 64 16-bit elements (one swizzle column)
constexpr int kQBytes = 2 * kQHalf;         // a Q tile: 128 rows x 128 dims
constexpr int kKVHalf = kBN * 128;          // 128 keys x 64 dims
constexpr int kKVBytes = 2 * kKVHalf;       // a K or V tile: 128 keys x 128 dims
constexpr int kStages = 5;                  // K/V ring entries
constexpr int kThreads = 352;               // 2 softmax warpgroups, a TMA warp, an MMA warp per Q tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr float kRescaleLog2 = 8.0f;

constexpr int kOffQ = 0;                               // Q_A, Q_B
constexpr int kOffKV = kOffQ + 2 * kQBytes;
constexpr int kOffBar = kOffKV + kStages * kKVBytes;
constexpr int kNumBars = 24;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;  // + TMEM address, abort flag, alignment

// mbarrier indices; S, P, Pv (last PV of a tile) and Pd (every PV) are per Q tile x: + x
constexpr int kBarQ = 0, kBarKvFull = 1, kBarKvEmpty = 1 + kStages, kBarS = 1 + 2 * kStages,
              kBarP = kBarS + 2, kBarPv = kBarP + 2, kBarPd = kBarPv + 2, kBarDrain = kBarPd + 2,  // Drain + x
              kBarTurn = kBarDrain + 2;  // Turn + x: the other Q tile's softmax has finished a pass
static_assert(kBarTurn + 1 < kNumBars, "mbarrier slots");

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

// The same product with A read from TMEM (lane = row of A, 32-bit column c = elements 2c and
// 2c + 1 of the row, low half first).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
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

// Asynchronous 32-column load (registers valid only after tmem_wait_regs on the same array).
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
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
}

// Wait for this thread's TMEM loads; the registers pass through the wait so that no use of
// them can be scheduled before it.
__device__ __forceinline__ void tmem_wait_regs(uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
          "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
          "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
          "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
          "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
        :
        : "memory");
}

__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
        "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
        "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
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

// Packed fp32 pair helpers (sm_100 f32x2 instructions): one instruction for two elements; the
// pairs are formed and split with register moves only.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
prefill_attention_kernel(const __grid_constant__ CUtensorMap tmap_q,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x / p.qtiles;
    const int qt = p.qtiles - 1 - static_cast<int>(blockIdx.x % p.qtiles);  // longest pairs first
    const int h = blockIdx.y;
    const int g = p.group, TQ = p.tokens_per_tile, bs = p.block_size;
    const int q0 = p.qsl[b];
    const int n = p.qsl[b + 1] - q0;
    const int L = p.seq_lens[b];
    const int t0 = qt * 2 * TQ;  // first token of Q tile A; Q tile B follows it
    if (t0 >= n) return;         // the whole CTA: no query row here

    const bool len_ok = n <= p.max_query_len && q0 >= 0 && q0 + n <= p.num_tokens && L >= n &&
                        L <= p.max_seq_len && (L + bs - 1) / bs <= p.max_blocks_per_seq;
    if (!len_ok) {
        // rows of a rejected sequence are written as zeros (lse -inf)
        if (threadIdx.x == 0) report(p.d_err, KV_DERR_BAD_LEN);
        const int rows = q0 < 0 ? 0 : max(0, min(n, p.num_tokens - q0) - t0);
        T *out = static_cast<T *>(p.out);
        for (int r = threadIdx.x; r < 2 * kBM; r += blockDim.x) {
            const int tl = r / g;
            if (tl >= min(2 * TQ, rows)) continue;
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

    // the two Q tiles: rows [0,128) = A, [128,256) = B; tokens, positions and key-tile ranges
    int nq[2], pf[2], pl[2], j0[2], j1[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        nq[x] = max(0, min(TQ, n - (t0 + x * TQ)));
        pf[x] = L - n + t0 + x * TQ;
        pl[x] = pf[x] + nq[x] - 1;
        const int lo = p.window > 0 ? max(0, pf[x] - p.window + 1) : 0;
        j0[x] = lo / kBN;
        j1[x] = nq[x] > 0 ? pl[x] / kBN + 1 : j0[x];
    }
    const bool has_b = nq[1] > 0;
    const int J0 = j0[0];                        // tile A's window starts first
    const int J1 = has_b ? j1[1] : j1[0];        // tile B's keys end last
    const int kv_lo = p.window > 0 ? max(0, pf[0] - p.window + 1) : 0;

    if (threadIdx.x == 0) {
        mbar_init(bar(kBarQ), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(kBarKvFull + s), 1);
            mbar_init(bar(kBarKvEmpty + s), has_b ? 2 : 1);  // one release per Q tile's MMA warp
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(kBarS + x), 1);
            mbar_init(bar(kBarP + x), 128);
            mbar_init(bar(kBarPv + x), 1);
            mbar_init(bar(kBarPd + x), 1);
        }
        mbar_init(bar(kBarDrain), 1);
        mbar_init(bar(kBarDrain + 1), 1);
        mbar_init(bar(kBarTurn), 128);
        mbar_init(bar(kBarTurn + 1), 128);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 9) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 8) {
        // ============================================================ TMA producer
        const int bpt = kBN / bs;                  // blocks per K/V tile
        const int nblk_seq = (L + bs - 1) / bs;
        const int first_blk = kv_lo / bs;          // blocks before it are never read
        if (lane == 0) {
            prefetch_tensormap(&tmap_q);
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
            mbar_arrive_expect_tx(bar(kBarQ), (has_b ? 2 : 1) * kQBytes);
            for (int x = 0; x < (has_b ? 2 : 1); ++x) {
                const uint32_t dq = smem_u32(smem + kOffQ + x * kQBytes);
                tma_load_3d(dq, &tmap_q, bar(kBarQ), 0, h * g, q0 + t0 + x * TQ);
                tma_load_3d(dq + kQHalf, &tmap_q, bar(kBarQ), 64, h * g, q0 + t0 + x * TQ);
            }
        }
        // block ids of key tile j: lane l holds block j * bpt + l; the next tile's ids are read
        // while this tile's copies are issued, so their latency is off the critical path
        auto block_id = [&](int j) {
            const int lb = j * bpt + lane;
            int id = p.num_blocks;  // one past the pool: the copy reads zeros
            if (lane < bpt && lb >= first_blk && lb < nblk_seq) {
                const int e = p.block_table[static_cast<int64_t>(b) * p.bt_stride + lb];
                if (e >= 0 && e < p.num_blocks) id = e;
                else report(p.d_err, KV_DERR_BAD_BLOCK);
            }
            return id;
        };
        int my_id = p.num_blocks, next_id = J0 < J1 ? block_id(J0) : p.num_blocks;
        int issued = 0;
        for (int i = 0; i < 2 * (J1 - J0); ++i) {
            const int j = J0 + (i >> 1);
            const bool is_v = i & 1;
            if (!is_v) {
                my_id = next_id;
                if (j + 1 < J1) next_id = block_id(j + 1);
            }
            const int slot = i % kStages;
            int stop = 0;
            if (lane == 0) {
                if (i >= kStages && !mbar_wait_sleep(bar(kBarKvEmpty + slot), ((i / kStages) - 1) & 1)) {
                    stop = 1;
                    report(p.d_err, KV_DERR_TIMEOUT);
                    *abort_flag = 1;
                } else if (*abort_flag) {
                    stop = 1;
                }
                if (!stop) mbar_arrive_expect_tx(bar(kBarKvFull + slot), kKVBytes);
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
            const CUtensorMap *m = is_v ? &tmap_v : &tmap_k;
            uint8_t *dst = smem + kOffKV + slot * kKVBytes;
            for (int jb = 0; jb < bpt; ++jb) {
                const int id = __shfl_sync(0xffffffffu, my_id, jb);
                if (lane == 0) {
                    tma_load_4d(smem_u32(dst + jb * bs * 128), m, bar(kBarKvFull + slot), 0, 0, h, id);
                    tma_load_4d(smem_u32(dst + kKVHalf + jb * bs * 128), m, bar(kBarKvFull + slot), 64, 0, h, id);
                }
            }
            issued = i + 1;
        }
        // never leave with copies in flight into this CTA's shared memory
        if (lane == 0) {
            if (!mbar_wait_sleep(bar(kBarQ), 0)) report(p.d_err, KV_DERR_TIMEOUT);
            for (int i = max(0, issued - kStages); i < issued; ++i)
                if (!mbar_wait_sleep(bar(kBarKvFull + i % kStages), (i / kStages) & 1))
                    report(p.d_err, KV_DERR_TIMEOUT);
        }
    } else if (warp == 9 || (warp == 10 && has_b)) {
        // ============================================================ MMA issue
        // One warp per Q tile x (warp 9: A, warp 10: B), so the two tiles' chains advance
        // independently and share the tensor core.  Over the key tiles j in order:
        //   - once the softmax has written P_x(i - 1) into TMEM (over the S_x columns it read):
        //     O_x += P_x(i - 1) V_{j-1} (A from TMEM), which releases V_{j-1};
        //   - once that product has completed (its A reads the columns S_x(i) overwrites):
        //     S_x(i) = Q_x K_j^T, which releases K_j;
        //   - key tiles x does not read are released as soon as they have landed, so that every
        //     ring entry gets one release per Q tile.
        // S_x(i) completing implies PV_x(i - 1) has too, which leaves O_x settled for a rescale.
        // The whole warp runs the schedule and forms the descriptors (warp-uniform values); one
        // lane issues the tcgen05 instructions.  Shared-memory descriptors are built once and
        // advanced by adding (byte offset >> 4) to their start-address field.
        const int x = warp - 9;
        constexpr uint32_t ab = AbFormat<T>::value;
        constexpr uint32_t idesc_s = mma_idesc(ab, false, kBM, kBN);
        constexpr uint32_t idesc_pv = mma_idesc(ab, true, kBM, 128);
        const uint64_t dq = smem_desc(smem_u32(smem + kOffQ + x * kQBytes), 16, 1024);
        const uint64_t dk0 = smem_desc(smem_u32(smem + kOffKV), 16, 1024);
        const uint64_t dv0 = smem_desc(smem_u32(smem + kOffKV), kKVHalf, 1024);
        const uint32_t t_sx = tmem + x * 128, t_ox = tmem + kColO + x * 128;
        const int xj0 = j0[x], xj1 = j1[x];
        const bool leader = lane == 0;
        // the MMA warps poll (no suspension hint): they react to a softmax hand-over or a
        // finished product within a few cycles, which is the latency that paces each tile
        auto wait_warp = [&](int i, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait_bounded(bar(i), parity));
        };
        int npd = 0;  // PV products committed to kBarPd + x so far
        bool dead = !wait_warp(kBarQ, 0);
        tc_fence_after();
        for (int j = J0; j <= J1 && !dead; ++j) {
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;  // decided for the whole warp
            const int ik = 2 * (j - J0), iv = ik - 1;
            const int sk_slot = ik % kStages, sv_slot = (iv + kStages) % kStages;
            const bool pv = j - 1 >= xj0 && j - 1 < xj1;   // PV_x of key tile j - 1
            const bool sx = j < J1 && j >= xj0 && j < xj1;  // S_x of key tile j
            if (pv) {
                const int u = j - 1 - xj0;
                if (!wait_warp(kBarP + x, u & 1) || !wait_warp(kBarKvFull + sv_slot, (iv / kStages) & 1)) {
                    dead = true;
                    break;
                }
                tc_fence_after();
                const uint64_t dv = dv0 + static_cast<uint64_t>((sv_slot * kKVBytes) >> 4);
                uint64_t db[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) db[k] = dv + ((k * 2048) >> 4);
                if (leader) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) mma_f16_ts(t_ox, t_sx + k * 8, db[k], idesc_pv, (u > 0 || k > 0));
                    mma_commit(bar(kBarKvEmpty + sv_slot));           // V_{j-1}: this tile is done with it
                    mma_commit(bar(sx ? kBarPd + x : kBarPv + x));    // S_x(u + 1) waits, or x is done
                }
                __syncwarp();
            }
            if (j == J1) break;
            if (sx) {
                if (pv) {
                    if (!wait_warp(kBarPd + x, npd & 1)) {
                        dead = true;
                        break;
                    }
                    ++npd;
                }
                if (!wait_warp(kBarKvFull + sk_slot, (ik / kStages) & 1)) {
                    dead = true;
                    break;
                }
                tc_fence_after();
                const uint64_t dk = dk0 + static_cast<uint64_t>((sk_slot * kKVBytes) >> 4);
                uint64_t da[8], db[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    da[k] = dq + (((k >> 2) * kQHalf + (k & 3) * 32) >> 4);
                    db[k] = dk + (((k >> 2) * kKVHalf + (k & 3) * 32) >> 4);
                }
                if (leader) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) mma_f16(t_sx, da[k], db[k], idesc_s, k > 0);
                    mma_commit(bar(kBarS + x));
                    mma_commit(bar(kBarKvEmpty + sk_slot));  // K_j: this tile is done with it
                }
                __syncwarp();
            } else {
                // a key tile this Q tile does not read: release its K and V entries once landed
                const int ivj = ik + 1, vj_slot = ivj % kStages;
                if (!wait_warp(kBarKvFull + sk_slot, (ik / kStages) & 1)) {
                    dead = true;
                    break;
                }
                if (leader) mbar_arrive(bar(kBarKvEmpty + sk_slot));
                if (!wait_warp(kBarKvFull + vj_slot, (ivj / kStages) & 1)) {
                    dead = true;
                    break;
                }
                if (leader) mbar_arrive(bar(kBarKvEmpty + vj_slot));
                __syncwarp();
            }
        }
        if (dead && leader) {
            report(p.d_err, KV_DERR_TIMEOUT);
            *abort_flag = 1;
        }
        // every MMA this warp issued has completed before TMEM is freed
        if (leader) mma_commit(bar(kBarDrain + x));
        __syncwarp();
        if (!wait_warp(kBarDrain + x, 0) && leader) report(p.d_err, KV_DERR_TIMEOUT);
    } else if (warp < 4 || has_b) {
        // ============================================================ softmax + epilogue
        const int x = warp >> 2;                   // Q tile
        const int r = threadIdx.x & 127;           // query row in the tile = TMEM lane
        const int tl = r / g;
        const bool valid = tl < nq[x];
        const int pos = pf[x] + tl;                // this row's query position
        const int klo = p.window > 0 ? pos - p.window + 1 : 0;
        const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t t_o = trow + kColO + x * 128;
        const float c2 = p.scale_log2;
        const int xp_first = pf[x], xp_last = pl[x], xj0 = j0[x];
        float m_used = -INFINITY;  // the reference maximum of O and l, in log2 units
        float2 lsum = make_float2(0.f, 0.f);
        bool dead = false;
        // waits are decided for the whole warp: its lanes take the warp-collective TMEM
        // loads and stores together
        auto wait_all = [&](int i, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait_sleep(bar(i), parity));
        };
        const int ntiles = j1[x] - j0[x];
        // One pass over the tile's S in the common case (weights against the reference in use,
        // the tile maximum tracked alongside), 32 columns at a time with the next load in
        // flight.  The weights stay in registers until the pass (and a redo, if the maximum
        // moved) is over, then go to TMEM over the first 64 columns of S_x, as the A operand of
        // the next PV product.
        const float2 cc = make_float2(c2, c2);
        const uint32_t t_s = trow + x * 128;
        uint32_t w[64];
        auto weights = [&](auto masked_tag, int kbase, float nref, float &mraw, float2 &tsum) {
            constexpr bool masked = decltype(masked_tag)::value;
            const float2 rr = make_float2(nref, nref);
            uint32_t ra[32], rb[32];
            auto chunk = [&](const uint32_t (&v)[32], int c) {
                const int k0 = kbase + c * 32;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float s0 = __uint_as_float(v[2 * k]), s1 = __uint_as_float(v[2 * k + 1]);
                    const float2 e = fma2(make_float2(s0, s1), cc, rr);
                    float e0 = fast_exp2(e.x), e1 = fast_exp2(e.y);
                    if constexpr (masked) {
                        const int kk = k0 + 2 * k;
                        const bool v0 = valid && kk <= pos && kk >= klo;
                        const bool v1 = valid && kk + 1 <= pos && kk + 1 >= klo;
                        e0 = v0 ? e0 : 0.f;
                        e1 = v1 ? e1 : 0.f;
                        mraw = fmaxf(mraw, fmaxf(v0 ? s0 : -INFINITY, v1 ? s1 : -INFINITY));
                    } else {
                        mraw = fmaxf(mraw, fmaxf(s0, s1));
                    }
                    w[c * 16 + k] = pack2<T>(e0, e1);
                    tsum = add2(tsum, unpack2<T>(w[c * 16 + k]));
                }
            };
            mraw = -INFINITY;
            tsum = make_float2(0.f, 0.f);
            tmem_ld32_async(t_s, ra);
            tmem_wait_regs(ra);
            tmem_ld32_async(t_s + 32, rb);
            chunk(ra, 0);
            tmem_wait_regs(rb);
            tmem_ld32_async(t_s + 64, ra);
            chunk(rb, 1);
            tmem_wait_regs(ra);
            tmem_ld32_async(t_s + 96, rb);
            chunk(ra, 2);
            tmem_wait_regs(rb);
            chunk(rb, 3);
        };
        // The two softmax warpgroups take turns (A's pass k, then B's pass k, then A's pass k+1
        // ...): they share the schedulers and the exponential units, and alternating them keeps
        // one tile's softmax overlapped with the other tile's products instead of both at once.
        const int n_other = has_b ? j1[x ^ 1] - j0[x ^ 1] : 0;
        for (int i = 0; i < ntiles; ++i) {
            if (!wait_all(kBarS + x, i & 1)) {
                dead = true;
                break;
            }
            // A's pass i waits for B's pass i - 1; B's pass i for A's pass i
            const int turn = x == 0 ? i - 1 : i;
            if (turn >= 0 && turn < n_other && !wait_all(kBarTurn + x, turn & 1)) {
                dead = true;
                break;
            }
            tc_fence_after();
            // a tile whose keys every row sees needs no mask (rows past the chunk compute
            // garbage that is never stored)
            const int kbase = (xj0 + i) * kBN;
            const bool masked = kbase + kBN - 1 > xp_first || (p.window > 0 && kbase < xp_last - p.window + 1);
            float mraw;
            float2 tsum;
            auto run_weights = [&](float nref, float &mx) {
                if (masked) weights(std::true_type{}, kbase, nref, mx, tsum);
                else weights(std::false_type{}, kbase, nref, mx, tsum);
            };
            run_weights(m_used == -INFINITY ? 0.f : -m_used, mraw);
            // scale >= 0, so the scaled maximum is the maximum of the scaled scores
            const float mt = mraw == -INFINITY ? -INFINITY : mraw * c2;
            const bool moved = mt > m_used + kRescaleLog2;  // also the first finite maximum
            if (__any_sync(0xffffffffu, moved)) {
                const bool rescale = moved && m_used != -INFINITY;  // O and l hold earlier tiles
                const float f = moved ? fast_exp2(m_used - mt) : 1.f;
                if (moved) {
                    m_used = mt;
                    lsum.x *= f;
                    lsum.y *= f;
                }
                if (__any_sync(0xffffffffu, rescale)) {
                    // the warp loads and stores O together; rows that keep their maximum scale by 1
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        float o[32];
                        tmem_ld32(t_o + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] *= f;
                        tmem_st32(t_o + c * 32, o);
                    }
                    tmem_wait_st();
                }
                float m2;
                run_weights(m_used == -INFINITY ? 0.f : -m_used, m2);
            }
            lsum = add2(lsum, tsum);
            // P_x into TMEM: 128 keys of 16-bit weights = 64 columns over the S_x just read
            tmem_st32u(t_s, w);
            tmem_st32u(t_s + 32, w + 32);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(kBarP + x));
            if (has_b) mbar_arrive(bar(kBarTurn + (x ^ 1)));  // the other tile's next pass may start
        }
        if (dead) {
            if (r == 0) report(p.d_err, KV_DERR_TIMEOUT);
            *abort_flag = 1;
        } else {
            // the last PV has landed (committed once, after x's last product): O / l, rounded,
            // and the log-sum-exp
            const bool ok = wait_all(kBarPv + x, 0);
            if (!ok) {
                if (r == 0) report(p.d_err, KV_DERR_TIMEOUT);
                *abort_flag = 1;
            }
            tc_fence_after();
            const float l = lsum.x + lsum.y;
            const int64_t row = static_cast<int64_t>(q0 + t0 + x * TQ + tl) * p.num_q_heads + h * g + r % g;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            T *out = static_cast<T *>(p.out) + row * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float o[32];
                tmem_ld32(t_o + c * 32, o);
                tmem_wait_ld();
                if (valid && ok) {
                    uint32_t ow[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) ow[k] = pack2<T>(o[2 * k] * inv, o[2 * k + 1] * inv);
                    uint4 *dst = reinterpret_cast<uint4 *>(out + c * 32);
#pragma unroll
                    for (int k = 0; k < 4; ++k) dst[k] = make_uint4(ow[4 * k], ow[4 * k + 1], ow[4 * k + 2], ow[4 * k + 3]);
                }
            }
            if (valid && ok && p.lse_out)
                p.lse_out[row] = l > 0.f ? (m_used + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9)
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
    // a CTA takes two consecutive Q tiles (2 * tokens_per_tile tokens)
    p.qtiles = (a.max_query_len + 2 * p.tokens_per_tile - 1) / (2 * p.tokens_per_tile);
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
