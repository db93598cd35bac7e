// Paged decode attention: persistent stream-K schedule, TMA-fed tensor-core MMAs, online softmax,
// log-sum-exp merge of the pieces of sequences that straddle CTAs.
//
// What it computes: "vLLM의 KV cache 연결 흐름", sections "Slot mapping은 왜 필요한가" and
// "Forward 직전의 metadata" (attention reads past K/V through the block table);
// "Understanding PageAttention Memory Optimization", section "Handling Softmax Across Blocks"
// (the softmax needs every block: an online softmax carries a running max and sum across
// blocks); GQA from "Deep Dive into vLLM Worker-Side GPU KV Cache Initialization", section
// "Hybrid Attention Mechanisms"; sliding windows from "vLLM Worker侧GPU KV Cache初始化流程深度解析",
// section "混合注意力机制"; speculative query tokens from "vLLM의 KV cache 연결 흐름", section
// "EngineCore가 하는 일".
//
// How (GB300):
//   * Work is the flat list of (kv-head group, sequence, stage) triples, a stage being 16 or 32
//     consecutive keys of one sequence (whole cache blocks).  Each resident CTA takes one
//     contiguous, equal share of that list (stream-K), so every SM streams the same number of
//     bytes whatever the length mix.  A CTA writes the output of a sequence it covers whole;
//     pieces of a sequence split between CTAs go to the workspace as (o/l, lse) and the merge
//     kernel combines them: LSE = log sum_s exp(lse_s), out = sum_s exp(lse_s - LSE) o_s.
//   * One producer warp reads block-table entries 32 at a time (one coalesced load) and issues
//     TMA tensor copies of whole (block, head group) tiles of K and V into a ring of shared-memory
//     stages guarded by mbarriers (expect-tx on "full", one arrival per consumer warp on
//     "empty").  The tensor map views the cache as (dim, token-in-block, head, block), so a copy
//     lands a block's rows head-major with the 128-byte swizzle: ldmatrix reads of 8 key rows
//     hit 8 different bank groups.
//   * Each consumer warp owns one kv head and 8 or 16 of its query rows (rows are (query
//     token, q head) pairs of the GQA group).  Scores are computed transposed, S^T = K q^T, as
//     m16n8k16 MMAs with keys as M and query rows as N, so a group of 4 queries costs no padded
//     rows; movmatrix turns the rounded probabilities into the B operand of O^T = V^T P^T.
//     Softmax statistics are float32 with exp2; the rescale of O is skipped while the running
//     max does not move.
//   * E4M3 caches are widened in registers: ldmatrix moves the bytes, cvt.f16x2.e4m3x2 widens
//     them, and the head-dim order this produces is folded into the q fragments (for K) and
//     into the output index (for V); k_scale folds into the score scale, v_scale into the output.
//   * INT4 caches (rows of 64 bytes, TMA boxes swizzled 64B) are widened by bit operations into
//     fp16 subnormals: a nibble n is stored two's complement, n ^ 8 = n + 8 is its offset-binary
//     value u in [0, 15], and the fp16 whose bits are u (or u << 4) is exactly u * 2^-24 (or
//     u * 2^-20).  One AND-XOR per pair of elements, no conversion instruction.  The offset 8
//     comes back out exactly: for K it shifts every score of a query row by the same amount
//     (8 * scale * sum_d q_d), which the softmax ignores and the log-sum-exp subtracts; for V
//     out_d = vscale_d * (sum_j p_j u_jd / l - 8), since the normaliser l is the sum of the same
//     rounded weights.  The per-dim K scales and the 2^-20 / 2^-24 units fold into q, the V
//     scales into the output.
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace pkv {

struct Fp8E4M3 {};    // tag for an E4M3 cache
struct Int4Group {};  // tag for an INT4 cache with group scales

template <typename CT> struct CacheTraits {
    static constexpr int kBytes = 2;
    static constexpr bool kFp8 = false;
    static constexpr bool kInt4 = false;
};
template <> struct CacheTraits<Fp8E4M3> {
    static constexpr int kBytes = 1;
    static constexpr bool kFp8 = true;
    static constexpr bool kInt4 = false;
};
template <> struct CacheTraits<Int4Group> {
    static constexpr int kBytes = 1;  // per two elements
    static constexpr bool kFp8 = false;
    static constexpr bool kInt4 = true;
};

struct KernelParams {
    DecodeArgs a;
    StepArgs f;            // fused decode step only: the slot mapping and cache write inputs
    int heads_per_cta;     // HG
    int warps_per_head;    // ceil(group * q_len / rows_per_warp)
    int blocks_per_stage;  // BPS
    int num_stages;        // NS
    int box_bytes, box_stride;
    int num_items;         // (num_kv_heads / HG) * num_seqs
    int rows_per_item;     // HG * group * q_len
};

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Four E4M3 bytes -> two packed fp16 pairs (bytes 0,1 -> lo; bytes 2,3 -> hi), exact.
__device__ __forceinline__ void e4m3x4_to_h2x2(uint32_t four, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(four));
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

// The CTA that owns flat stage s when S stages are split into G equal shares
// (CTA c owns [c*S/G, (c+1)*S/G)).
__host__ __device__ __forceinline__ int owner_cta(long long s, long long S, int G) {
    return static_cast<int>(((s + 1) * G - 1) / S);
}

// One 16-byte chunk c of token t's K and V rows (row = chunks 16-byte chunks) into its slot:
// a bit copy, or E4M3 quantisation with the per-tensor scales.
template <typename QT, typename CT>
__device__ __forceinline__ void write_row_chunk(const StepArgs &f, int64_t t, int64_t slot, int chunks, int c) {
    const uint4 kx = *reinterpret_cast<const uint4 *>(static_cast<const QT *>(f.key) + t * f.key_row_stride + 8 * c);
    const uint4 vx = *reinterpret_cast<const uint4 *>(static_cast<const QT *>(f.value) + t * f.value_row_stride + 8 * c);
    const int64_t dst = (slot * chunks + c) * 8;
    if constexpr (CacheTraits<CT>::kFp8) {
        *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(f.k_cache) + dst) = quantise8<QT>(kx, f.k_scale);
        *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(f.v_cache) + dst) = quantise8<QT>(vx, f.v_scale);
    } else {
        *reinterpret_cast<uint4 *>(static_cast<QT *>(f.k_cache) + dst) = kx;
        *reinterpret_cast<uint4 *>(static_cast<QT *>(f.v_cache) + dst) = vx;
    }
}

// One warp per (item, row): combine the pieces of a sequence that several CTAs shared, and
// write zeros (lse -inf) for sequences whose length was rejected.  P is the stage prefix.
template <typename QT, int D>
__device__ __forceinline__ void merge_row(const KernelParams &kp, const int32_t *P, int num_ctas,
                                          int64_t w, int lane) {
    const DecodeArgs &a = kp.a;
    const int item = static_cast<int>(w / kp.rows_per_item);
    const int rr = static_cast<int>(w - static_cast<int64_t>(item) * kp.rows_per_item);
    const int B = a.num_seqs;
    const int g = a.num_q_heads / a.num_kv_heads;
    const int R = g * a.q_len;
    const int seq = item % B, grp = item / B;
    const int h_loc = rr / R, r = rr % R;
    const int64_t tokq = static_cast<int64_t>(seq) * a.q_len + r / g;
    const int64_t rowid = tokq * a.num_q_heads + (grp * kp.heads_per_cta + h_loc) * g + r % g;
    const long long p0 = P[item], p1 = P[item + 1], S = P[kp.num_items];
    constexpr int kPer = D / 32;
    QT *orow = static_cast<QT *>(a.out) + rowid * D + lane * kPer;
    if (p1 == p0) {  // rejected length: defined output
#pragma unroll
        for (int e = 0; e < kPer; ++e) orow[e] = from_float<QT>(0.f);
        if (a.lse_out && lane == 0) a.lse_out[rowid] = -INFINITY;
        return;
    }
    const int c_lo = owner_cta(p0, S, num_ctas), c_hi = owner_cta(p1 - 1, S, num_ctas);
    if (c_lo == c_hi) return;  // one CTA covered it and wrote the output
    // with more CTAs than stages some shares are empty and wrote nothing
    auto empty_share = [&](int c) { return S * c / num_ctas == S * (c + 1) / num_ctas; };
    float mx = -INFINITY;
    for (int c = c_lo + lane; c <= c_hi; c += 32)
        if (!empty_share(c)) mx = fmaxf(mx, __ldcg(a.ws_lse + static_cast<int64_t>(item + c) * kp.rows_per_item + rr));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    if (mx != -INFINITY) {
        for (int c = c_lo; c <= c_hi; ++c) {
            if (empty_share(c)) continue;
            const int64_t wrow = static_cast<int64_t>(item + c) * kp.rows_per_item + rr;
            const float wgt = expf(__ldcg(a.ws_lse + wrow) - mx);
            wsum += wgt;
            const float *src = a.ws_o + wrow * D + lane * kPer;  // written by other CTAs: via L2
#pragma unroll
            for (int e = 0; e < kPer; ++e) acc[e] += wgt * __ldcg(src + e);
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
    for (int e = 0; e < kPer; e += 2)
        *reinterpret_cast<uint32_t *>(orow + e) = pack2<QT>(acc[e] * inv, acc[e + 1] * inv);
    if (a.lse_out && lane == 0) a.lse_out[rowid] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

// Where one 16-key chunk of a stage sits in shared memory, for the lane that addresses it.
struct ChunkRef {
    uint32_t kbase, vbase;  // shared addresses of this lane's K and V rows (segment 0)
    int kk, vk;             // their swizzle keys
    int c0;                 // index of the chunk's first key in the sequence
    int tok0;               // index of the first key of the chunk's stage
    uint32_t mask;          // valid blocks of that stage
};

template <typename QT, typename CT, int D, int RN, bool kFused>
__global__ void __maxnreg__(DecodeLaunch<RN>::kMaxRegs)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v,
                        const __grid_constant__ KernelParams kp) {
    constexpr bool kFp8 = CacheTraits<CT>::kFp8;
    constexpr bool kInt4 = CacheTraits<CT>::kInt4;
    static_assert(!kInt4 || (D == 128 && !kFused), "INT4 caches: head_dim 128, attention only");
    using MT = typename std::conditional<kFp8 || kInt4, __half, QT>::type;  // MMA operand type
    constexpr int kEB = CacheTraits<CT>::kBytes;
    constexpr int kNDB = kInt4 ? 1 : D * kEB / 128;  // row segments (TMA boxes) per head row
    constexpr int kRow = kInt4 ? 64 : 128;           // bytes of one key row in a box
    constexpr int kKS = D / 16;          // k-steps of K q^T (16 dims each)
    constexpr int kMT = D / 16;          // m-tiles of V^T P^T (16 dims each)
    constexpr int kNR = RN / 8;          // n-tiles of query rows

    const DecodeArgs &a = kp.a;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int HG = kp.heads_per_cta, MW = kp.warps_per_head;
    const int ncw = HG * MW;
    const int bs = a.block_size, BPS = kp.blocks_per_stage, ST = BPS * bs, NS = kp.num_stages;
    const int B = a.num_seqs, NI = kp.num_items;
    const int g = a.num_q_heads / a.num_kv_heads;
    const int R = g * a.q_len;
    const int q_len = a.q_len;

    // ---------------------------------------------------------------- shared memory
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int stage_bytes = 2 * BPS * kNDB * kp.box_stride;
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + NS * stage_bytes);
    uint64_t *empty_bar = full_bar + NS;
    uint32_t *stage_mask = reinterpret_cast<uint32_t *>(empty_bar + NS);
    volatile uint32_t *abort_flag = stage_mask + NS;
    int32_t *P = reinterpret_cast<int32_t *>(stage_mask + NS + 1);  // [NI + 1] stage prefix
    int32_t *Ls = P + NI + 1;                                       // [B] lengths (-1: rejected)
    __shared__ int32_t warp_sums[32];

    // ---------------------------------------------------------------- prologue
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), ncw);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    const int G = gridDim.x, cta = blockIdx.x;
    for (int i = threadIdx.x; i < B; i += blockDim.x) {
        const int L = a.seq_lens[i];
        const bool ok = L >= q_len && L <= a.max_seq_len && (L + bs - 1) / bs <= a.max_blocks_per_seq;
        if (!ok && blockIdx.x == 0) report(a.d_err, KV_DERR_BAD_LEN);
        Ls[i] = ok ? L : -1;
    }
    __syncthreads();
    // stage counts of the items (group-major, then sequence), inclusive scan into P[1..NI]
    {
        const int T = blockDim.x;
        const int per = (NI + T - 1) / T;
        const int lo = min(NI, static_cast<int>(threadIdx.x) * per), hi = min(NI, lo + per);
        auto stages_of = [&](int it) {
            const int L = Ls[it % B];
            if (L < 0) return 0;
            const int lo_key = a.window > 0 ? max(0, L - q_len - a.window + 1) : 0;
            const int nb = (L + bs - 1) / bs - lo_key / bs;
            return (nb + BPS - 1) / BPS;
        };
        int sum = 0;
        for (int i = lo; i < hi; ++i) sum += stages_of(i);
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) warp_sums[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int nw = (T + 31) >> 5;
            int w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += v;
            }
            if (lane < nw) warp_sums[lane] = w;
        }
        __syncthreads();
        int run = incl - sum + (warp > 0 ? warp_sums[warp - 1] : 0);
        if (threadIdx.x == 0) P[0] = 0;
        for (int i = lo; i < hi; ++i) {
            run += stages_of(i);
            P[i + 1] = run;
        }
    }
    __syncthreads();
    if (blockIdx.x == 0)  // the merge kernel reads the same prefix
        for (int i = threadIdx.x; i <= NI; i += blockDim.x) a.ws_prefix[i] = P[i];

    const long long S = P[NI];
    const long long s_begin = S * cta / G, s_end = S * (cta + 1) / G;
    int item0 = 0;
    {
        int lo = 0, hi = NI;  // first item i with P[i+1] > s_begin
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (P[mid + 1] > s_begin) hi = mid;
            else lo = mid + 1;
        }
        item0 = lo;
    }
    if constexpr (kFused) {
        // ---- fused step, part 1: before this CTA reads any cache block, it writes the new-token
        // rows its own stages will read: the head group's part of every new token whose position
        // falls in one of its stages (each such row has exactly one reader).  Rows no stage reads
        // (padding, rejected lengths, positions outside the attended range) are written by CTA 0.
        const StepArgs &f = kp.f;
        const int chunks_g = HG * D / 8;             // 16-byte source chunks of a head group's part
        for (int item = item0; s_begin < s_end && item < NI && P[item] < s_end; ++item) {
            if (P[item + 1] == P[item]) continue;
            const int seq = item % B, grp = item / B;
            const int L = Ls[seq];
            const int nblk = (L + bs - 1) / bs;
            const int b0 = (a.window > 0 ? max(0, L - q_len - a.window + 1) : 0) / bs;
            const long long ka = max(s_begin, static_cast<long long>(P[item])) - P[item];
            const long long kb = min(s_end, static_cast<long long>(P[item + 1])) - P[item];
            const int plo = (b0 + static_cast<int>(ka) * BPS) * bs;
            const int phi = min((b0 + static_cast<int>(kb) * BPS) * bs, nblk * bs);
            const int r0 = f.query_start_loc[seq], r1 = f.query_start_loc[seq + 1];
            for (int i = threadIdx.x; i < (r1 - r0) * chunks_g; i += blockDim.x) {
                const int t = r0 + i / chunks_g, c = i % chunks_g;
                const int p = f.positions[t];
                if (p < plo || p >= phi) continue;
                const int physical = a.block_table[static_cast<int64_t>(seq) * a.bt_stride + p / bs];
                const bool ok = physical >= 0 && physical < a.num_blocks;
                const int64_t slot = ok ? static_cast<int64_t>(physical) * bs + p % bs : -1;
                if (grp == 0 && c == 0 && f.slot_mapping) f.slot_mapping[t] = slot;
                if (!ok) continue;  // the attention reports and masks this block
                write_row_chunk<QT, CT>(f, t, slot, a.num_kv_heads * D / 8, grp * chunks_g + c);
            }
        }
        {   // rows no stage reads: each CTA takes an equal share of the tokens
            const int T = f.num_tokens;
            const int t0 = static_cast<int>(static_cast<long long>(T) * cta / G);
            const int t1 = static_cast<int>(static_cast<long long>(T) * (cta + 1) / G);
            for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
                int lo = 0, hi = B + 1;  // the token's row: last r with query_start_loc[r] <= t
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (f.query_start_loc[mid] <= t) lo = mid + 1;
                    else hi = mid;
                }
                const int row = lo - 1;
                const int p = f.positions[t];
                bool read = false;
                if (row >= 0 && row < B && t < f.query_start_loc[row + 1] && p >= 0 && Ls[row] >= 0) {
                    const int L = Ls[row];
                    const int b0 = (a.window > 0 ? max(0, L - q_len - a.window + 1) : 0) / bs;
                    read = p >= b0 * bs && p < (L + bs - 1) / bs * bs;
                }
                if (read) continue;
                const int64_t slot = slot_of_token(t, f.query_start_loc, B, f.positions, a.block_table,
                                                   a.bt_stride, a.max_blocks_per_seq, bs, a.num_blocks,
                                                   a.d_err);
                if (f.slot_mapping) f.slot_mapping[t] = slot;
                if (slot < 0) continue;
                if (slot >= f.total_slots) {
                    report(a.d_err, KV_DERR_BAD_SLOT);
                    continue;
                }
                const int chunks = a.num_kv_heads * D / 8;
                for (int c = 0; c < chunks; ++c) write_row_chunk<QT, CT>(f, t, slot, chunks, c);
            }
        }
        fence_proxy_async_global();  // this CTA's TMA copies below read these rows
        __syncthreads();
        fence_proxy_async_global();
    }

    if (s_begin < s_end) {
    // ================================================================ producer warp
    if (warp == ncw) {
        const uint32_t tx = 2u * BPS * kNDB * kp.box_bytes;
        int item = item0;
        int cache_base = 0, cache_item = -1;  // lanes hold block ids [cache_base, +32) of cache_item
        int my_id = a.num_blocks;
        bool my_ok = false;
        int issued = 0, pslot = 0;
        uint32_t pround = 0;  // completed passes over the ring
        for (long long s = s_begin; s < s_end; ++s) {
            while (P[item + 1] <= s) ++item;
            const int k = static_cast<int>(s - P[item]);
            const int seq = item % B, grp = item / B;
            const int L = Ls[seq];
            const int nblk = (L + bs - 1) / bs;
            const int lb0 = (a.window > 0 ? max(0, L - q_len - a.window + 1) : 0) / bs + k * BPS;
            if (cache_item != item || lb0 + BPS > cache_base + 32) {
                cache_item = item;
                cache_base = lb0;
                const int lb = cache_base + lane;
                my_ok = false;
                my_id = a.num_blocks;  // one past the pool: a copy from there reads zeros
                if (lb < nblk) {
                    const int e = a.block_table[static_cast<int64_t>(seq) * a.bt_stride + lb];
                    if (e >= 0 && e < a.num_blocks) {
                        my_id = e;
                        my_ok = true;
                    } else {
                        report(a.d_err, KV_DERR_BAD_BLOCK);
                    }
                }
            }
            const int slot = pslot;
            // lane 0 waits for the slot and decides for the whole warp: 0 go, 1 stop (a consumer
            // gave up), 2 stop (this wait timed out)
            int stop = 0;
            if (lane == 0) {
                if (pround > 0 && !mbar_wait_bounded(smem_u32(&empty_bar[slot]), (pround + 1) & 1))
                    stop = 2;
                else if (*abort_flag)
                    stop = 1;
                if (stop == 2) {
                    report(a.d_err, KV_DERR_TIMEOUT);
                    *abort_flag = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
            uint32_t mask = 0;
            int ids[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int src = lb0 - cache_base + (j < BPS ? j : 0);
                ids[j] = __shfl_sync(0xffffffffu, my_id, src);
                const int okj = __shfl_sync(0xffffffffu, my_ok ? 1 : 0, src);
                if (j < BPS && okj) mask |= 1u << j;
            }
            if (lane == 0) {
                uint8_t *stage = smem + slot * stage_bytes;
                stage_mask[slot] = mask;
                const uint32_t bar = smem_u32(&full_bar[slot]);
                mbar_arrive_expect_tx(bar, tx);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (j >= BPS) break;
                    const int id = ((mask >> j) & 1u) ? ids[j] : a.num_blocks;
#pragma unroll
                    for (int db = 0; db < kNDB; ++db) {
                        const uint32_t dk = smem_u32(stage + ((0 * BPS + j) * kNDB + db) * kp.box_stride);
                        const uint32_t dv = smem_u32(stage + ((1 * BPS + j) * kNDB + db) * kp.box_stride);
                        tma_load_4d(dk, &tmap_k, bar, db * (128 / kEB), 0, grp * HG, id);
                        tma_load_4d(dv, &tmap_v, bar, db * (128 / kEB), 0, grp * HG, id);
                    }
                }
            }
            ++issued;
            if (++pslot == NS) {
                pslot = 0;
                ++pround;
            }
        }
        // never leave with copies in flight into this CTA's shared memory
        if (lane == 0)
            for (int i = max(0, issued - NS); i < issued; ++i)
                if (!mbar_wait_bounded(smem_u32(&full_bar[i % NS]), (i / NS) & 1))
                    report(a.d_err, KV_DERR_TIMEOUT);
    } else {

    // ================================================================ consumer warps
    const int h_loc = warp / MW, rt = warp % MW;
    const int c4 = lane & 3, l4 = lane >> 2;

    // shared-memory rows this lane addresses for ldmatrix, per 16-key chunk of a stage (a stage
    // holds one or two chunks): K rows key (lane>>3 & 1)*8 + lane&7; V rows (16-bit caches)
    // key (lane>>4)*8 + lane&7, (E4M3 caches) the same keys as K
    // (the second chunk of a stage exists only for 32-key blocks: it lies 16 rows further down
    // the same box, with the same swizzle keys)
    uint32_t koff, voff;
    int kkey, vkey;
    {
        const int tk = ((lane >> 3) & 1) * 8 + (lane & 7);
        const int tv = (kFp8 || kInt4) ? tk : (lane >> 4) * 8 + (lane & 7);
        const int jk = tk / bs, rk = h_loc * bs + (tk - jk * bs);
        const int jv = tv / bs, rv = h_loc * bs + (tv - jv * bs);
        koff = (jk * kNDB) * kp.box_stride + rk * kRow;
        voff = ((BPS + jv) * kNDB) * kp.box_stride + rv * kRow;
        // 16-byte chunk c of row r sits at chunk c ^ key: 128B swizzle key r & 7, 64B (r >> 1) & 3
        kkey = kInt4 ? (rk >> 1) & 3 : rk & 7;
        vkey = kInt4 ? (rv >> 1) & 3 : rv & 7;
    }
    const int n_chunks = ST / 16;
    const bool pair_stages = NS >= 5;

    float o[kMT][kNR][4];
    float m_run[kNR][2], l_run[kNR][2];
    uint32_t qb[kNR][kKS][2];
    int pos_hi[kNR][2];  // position of each of this lane's rows (-1: padding row)
    float q_sum[kNR][2];  // INT4: sum_d q_d of each of this lane's rows, as the MMAs see q
    const float sl2 = a.scale_log2;
    const int W = a.window;

    int item = item0, seg_k0 = 0;
    int seq = 0, grp = 0, L = 0, b0 = 0, key_lo = 0, lo_last = 0, hi_first = 0, n_item = 0;
    int slot = 0;
    uint32_t phase = 0;
    const int s0 = static_cast<int>(s_begin), s1 = static_cast<int>(s_end);

    // NCH 16-key chunks processed together; kMasked: some chunk holds keys a row must not see, or
    // keys whose V rows may hold anything (past the sequence, before the window, failed validation)
    auto unit = [&](const ChunkRef (&cr)[2], auto nch_tag, auto masked_tag) {
        constexpr int NCH = decltype(nch_tag)::value;
        constexpr bool kMasked = decltype(masked_tag)::value;
        // independent accumulation chains: one per chunk; with a single chunk and a single row
        // tile the k-steps alternate between two
        constexpr bool kSplitK = NCH == 1 && kNR == 1;

        // ---- S^T = K q^T: 16 keys x RN query rows per chunk
        float sa[NCH][kNR][4], sb[kNR][4];
#pragma unroll
        for (int nt = 0; nt < kNR; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sb[nt][e] = 0.f;
#pragma unroll
                for (int j = 0; j < NCH; ++j) sa[j][nt][e] = 0.f;
            }
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
            if constexpr (kInt4) {
                // a 16-byte chunk holds 32 dims; one ldmatrix.x4 takes two chunks of 16 keys
                // (r[2h]: keys l4, r[2h+1]: keys l4 + 8, of chunk 2cp + h).  Each register holds
                // dims 8c4 .. 8c4+7 of its key: k-step 2*chunk + t takes the pairs of dims
                // (8c4+2t, 8c4+2t+4) and (8c4+2t+1, 8c4+2t+5), the order the q fragments follow.
#pragma unroll
                for (int cp = 0; cp < D / 64; ++cp) {
                    const int cch = 2 * cp + (lane >> 4);
                    uint32_t r[4];
                    ldsm_x4(cr[j].kbase + ((cch ^ cr[j].kk) << 4), r[0], r[1], r[2], r[3]);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t ua[4], ub[4];
                        int4x8_to_h2x4(r[2 * h], ua);
                        int4x8_to_h2x4(r[2 * h + 1], ub);
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            const int ks = 2 * (2 * cp + h) + t;
                            uint32_t af[4] = {ua[2 * t], ub[2 * t], ua[2 * t + 1], ub[2 * t + 1]};
#pragma unroll
                            for (int nt = 0; nt < kNR; ++nt)
                                MmaOp<MT>::run((kSplitK && (ks & 1)) ? sb[nt] : sa[j][nt], af, qb[nt][ks][0],
                                               qb[nt][ks][1]);
                        }
                    }
                }
            } else if constexpr (kFp8) {
#pragma unroll
                for (int p2 = 0; p2 < kKS; p2 += 2) {
                    const int cch = p2 + (lane >> 4);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(cr[j].kbase + ((cch ^ cr[j].kk) << 4), r0, r1, r2, r3);
                    // each register: 4 bytes = dims 4*c4 .. 4*c4+3 of one key
                    uint32_t a0[4], a1[4];
                    e4m3x4_to_h2x2(r0, a0[0], a0[2]);
                    e4m3x4_to_h2x2(r1, a0[1], a0[3]);
                    e4m3x4_to_h2x2(r2, a1[0], a1[2]);
                    e4m3x4_to_h2x2(r3, a1[1], a1[3]);
#pragma unroll
                    for (int nt = 0; nt < kNR; ++nt) {
                        MmaOp<MT>::run(sa[j][nt], a0, qb[nt][p2][0], qb[nt][p2][1]);
                        MmaOp<MT>::run(kSplitK ? sb[nt] : sa[j][nt], a1, qb[nt][p2 + 1][0], qb[nt][p2 + 1][1]);
                    }
                }
            } else {
#pragma unroll
                for (int ks = 0; ks < kKS; ++ks) {
                    const int q8 = 2 * ks + (lane >> 4);  // 16-byte chunk along the row
                    const int seg = q8 >> 3, cch = q8 & 7;
                    uint32_t af[4];
                    ldsm_x4(cr[j].kbase + seg * kp.box_stride + ((cch ^ cr[j].kk) << 4), af[0], af[1], af[2], af[3]);
#pragma unroll
                    for (int nt = 0; nt < kNR; ++nt)
                        MmaOp<MT>::run((kSplitK && (ks & 1)) ? sb[nt] : sa[j][nt], af, qb[nt][ks][0], qb[nt][ks][1]);
                }
            }
        }

        // ---- scale, mask, online softmax over the unit (lane: keys l4, l4+8 of each chunk;
        // rows 2*c4, 2*c4+1)
        bool moved = false;
        float alpha[kNR][2];
#pragma unroll
        for (int nt = 0; nt < kNR; ++nt) {
#pragma unroll
            for (int j = 0; j < NCH; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float v = (kSplitK ? sa[j][nt][e] + sb[nt][e] : sa[j][nt][e]) * sl2;
                    if constexpr (kMasked) {
                        const int tok = cr[j].c0 + l4 + (e >> 1) * 8;
                        const bool blk_ok = (cr[j].mask >> ((tok - cr[j].tok0) / bs)) & 1u;
                        const int ph = pos_hi[nt][e & 1];
                        const bool okk = blk_ok && tok <= ph && (W <= 0 || tok > ph - W);
                        v = okk ? v : -INFINITY;
                    }
                    sa[j][nt][e] = v;
                }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float mx = fmaxf(sa[0][nt][e], sa[0][nt][e + 2]);
#pragma unroll
                for (int j = 1; j < NCH; ++j) mx = fmaxf(mx, fmaxf(sa[j][nt][e], sa[j][nt][e + 2]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float m_new = fmaxf(m_run[nt][e], mx);
                moved |= m_new != m_run[nt][e];
                const float ref = m_new == -INFINITY ? 0.f : m_new;
                alpha[nt][e] = fast_exp2(m_run[nt][e] - ref);
                m_run[nt][e] = m_new;
#pragma unroll
                for (int j = 0; j < NCH; ++j) {
                    sa[j][nt][e] = fast_exp2(sa[j][nt][e] - ref);
                    sa[j][nt][e + 2] = fast_exp2(sa[j][nt][e + 2] - ref);
                }
            }
        }
        // P^T as the B operand: rounded pairs (key l4 or l4+8; rows 2c4, 2c4+1), transposed
        uint32_t pb[NCH][kNR][2];
#pragma unroll
        for (int nt = 0; nt < kNR; ++nt) {
            float add0 = 0.f, add1 = 0.f;
#pragma unroll
            for (int j = 0; j < NCH; ++j) {
                const uint32_t lo = pack2<MT>(sa[j][nt][0], sa[j][nt][1]);
                const uint32_t hi = pack2<MT>(sa[j][nt][2], sa[j][nt][3]);
                // the normaliser sums the rounded weights the MMA uses
                const float2 ul = unpack2<MT>(lo), uh = unpack2<MT>(hi);
                add0 += ul.x + uh.x;
                add1 += ul.y + uh.y;
                pb[j][nt][0] = movmatrix_t(lo);
                pb[j][nt][1] = movmatrix_t(hi);
            }
            l_run[nt][0] = l_run[nt][0] * alpha[nt][0] + add0;
            l_run[nt][1] = l_run[nt][1] * alpha[nt][1] + add1;
        }
        if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
                for (int nt = 0; nt < kNR; ++nt) {
                    o[mt][nt][0] *= alpha[nt][0];
                    o[mt][nt][1] *= alpha[nt][1];
                    o[mt][nt][2] *= alpha[nt][0];
                    o[mt][nt][3] *= alpha[nt][1];
                }
        }

        // ---- O^T += V^T P^T, chunk by chunk.  V^T fragments hold keys 2c4, 2c4+1 (regs 0,1) and
        // +8 (regs 2,3); in a masked unit the V elements of keys outside [key_lo, L) or in an
        // invalid block are zeroed, so 0 * NaN never reaches the accumulators
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
            uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;
            if constexpr (kMasked && !kInt4) {
                uint32_t keep[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = cr[j].c0 + 2 * c4 + (e >> 1) * 8 + (e & 1);
                    const bool blk_ok = (cr[j].mask >> ((tok - cr[j].tok0) / bs)) & 1u;
                    keep[e] = (blk_ok && tok >= key_lo && tok < L) ? 0xffffu : 0u;
                }
                keep_lo = keep[0] | (keep[1] << 16);
                keep_hi = keep[2] | (keep[3] << 16);
            }
            if constexpr (kInt4) {
                // V^T fragments straight from the transposed load: a register holds keys
                // (2c4, 2c4+1) x dims 4l4 .. 4l4+3 of one chunk, so its four pairs are key pairs at
                // four dims.  m-tile 2*chunk + h2 takes dims 4l4+2h2 (accumulator rows l4) and
                // 4l4+2h2+1 (rows l4+8).  Codes decode to finite values, so keys outside the
                // attended range need no masking here: their weights are exactly 0.
#pragma unroll
                for (int cp = 0; cp < D / 64; ++cp) {
                    const int cch = 2 * cp + (lane >> 4);
                    uint32_t r[4];
                    ldsm_x4_t(cr[j].vbase + ((cch ^ cr[j].vk) << 4), r[0], r[1], r[2], r[3]);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t ua[4], ub[4];
                        int4x8_to_h2x4(r[2 * h], ua);
                        int4x8_to_h2x4(r[2 * h + 1], ub);
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const int mt = 2 * (2 * cp + h) + h2;
                            uint32_t af[4] = {ua[2 * h2], ua[2 * h2 + 1], ub[2 * h2], ub[2 * h2 + 1]};
#pragma unroll
                            for (int nt = 0; nt < kNR; ++nt) MmaOp<MT>::run(o[mt][nt], af, pb[j][nt][0], pb[j][nt][1]);
                        }
                    }
                }
            } else if constexpr (kFp8) {
#pragma unroll
                for (int mt2 = 0; mt2 < kMT; mt2 += 2) {
                    const int cch = mt2 + (lane >> 4);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4_t(cr[j].vbase + ((cch ^ cr[j].vk) << 4), r0, r1, r2, r3);
                    // each register: keys (2c4, 2c4+1) x dims (2*l4, 2*l4+1) of one 16-dim chunk;
                    // regroup into (key pair at dim 2*l4) and (key pair at dim 2*l4+1)
                    uint32_t af0[4], af1[4];
                    e4m3x4_to_h2x2(__byte_perm(r0, 0, 0x3120), af0[0], af0[1]);
                    e4m3x4_to_h2x2(__byte_perm(r1, 0, 0x3120), af0[2], af0[3]);
                    e4m3x4_to_h2x2(__byte_perm(r2, 0, 0x3120), af1[0], af1[1]);
                    e4m3x4_to_h2x2(__byte_perm(r3, 0, 0x3120), af1[2], af1[3]);
                    if constexpr (kMasked) {
                        af0[0] &= keep_lo; af0[1] &= keep_lo; af0[2] &= keep_hi; af0[3] &= keep_hi;
                        af1[0] &= keep_lo; af1[1] &= keep_lo; af1[2] &= keep_hi; af1[3] &= keep_hi;
                    }
#pragma unroll
                    for (int nt = 0; nt < kNR; ++nt) {
                        MmaOp<MT>::run(o[mt2][nt], af0, pb[j][nt][0], pb[j][nt][1]);
                        MmaOp<MT>::run(o[mt2 + 1][nt], af1, pb[j][nt][0], pb[j][nt][1]);
                    }
                }
            } else {
#pragma unroll
                for (int mt = 0; mt < kMT; ++mt) {
                    const int q8 = 2 * mt + ((lane >> 3) & 1);
                    const int seg = q8 >> 3, cch = q8 & 7;
                    uint32_t af[4];
                    ldsm_x4_t(cr[j].vbase + seg * kp.box_stride + ((cch ^ cr[j].vk) << 4), af[0], af[1], af[2], af[3]);
                    if constexpr (kMasked) {
                        af[0] &= keep_lo;
                        af[1] &= keep_lo;
                        af[2] &= keep_hi;
                        af[3] &= keep_hi;
                    }
#pragma unroll
                    for (int nt = 0; nt < kNR; ++nt) MmaOp<MT>::run(o[mt][nt], af, pb[j][nt][0], pb[j][nt][1]);
                }
            }
        }
    };

    for (int s = s0; s < s1; ++s) {
        while (P[item + 1] <= s) ++item;
        const int k = s - P[item];
        if (s == s0 || k == 0) {
            // ------------------------------------------------ a new piece of a sequence
            seg_k0 = k;
            seq = item % B;
            grp = item / B;
            L = Ls[seq];
            n_item = P[item + 1] - P[item];
            key_lo = a.window > 0 ? max(0, L - q_len - a.window + 1) : 0;
            b0 = key_lo / bs;
            lo_last = a.window > 0 ? max(0, L - a.window) : 0;
            hi_first = L - q_len;
            const int hkv = grp * HG + h_loc;
#pragma unroll
            for (int nt = 0; nt < kNR; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = rt * RN + nt * 8 + 2 * c4 + e;
                    pos_hi[nt][e] = r < R ? L - q_len + r / g : -1;
                    m_run[nt][e] = -INFINITY;
                    l_run[nt][e] = 0.f;
                }
                // q as the B operand (column = query row l4), dims in the order the K operand
                // delivers them
                const int rq = rt * RN + nt * 8 + l4;
                const QT *qrow = nullptr;
                if (rq < R) {
                    const int64_t tok = static_cast<int64_t>(seq) * q_len + rq / g;
                    qrow = static_cast<const QT *>(a.q) + (tok * a.num_q_heads + hkv * g + rq % g) * D;
                }
                if constexpr (kInt4) {
                    // dims (d, d + 4) with d = 32*(ks/2) + 8c4 + 2(ks&1) + hf, times their K
                    // scales; odd dims (hf 1) meet codes in units of 2^-20, so they take 1/16
                    const float *ksc = a.k_gscales + static_cast<int64_t>(hkv) * (D >> a.group_shift);
                    float qs = 0.f;
#pragma unroll
                    for (int ks = 0; ks < kKS; ++ks) {
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const int d = 32 * (ks >> 1) + 8 * c4 + 2 * (ks & 1) + hf;
                            const float f = hf ? 0.0625f : 1.f;
                            uint32_t v = 0;
                            if (qrow)
                                v = pack2<MT>(to_float<QT>(qrow[d]) * ksc[d >> a.group_shift] * f,
                                              to_float<QT>(qrow[d + 4]) * ksc[(d + 4) >> a.group_shift] * f);
                            qb[nt][ks][hf] = v;
                            const float2 u = unpack2<MT>(v);
                            qs += (u.x + u.y) * (hf ? 16.f : 1.f);
                        }
                    }
                    qs += __shfl_xor_sync(0xffffffffu, qs, 1);
                    qs += __shfl_xor_sync(0xffffffffu, qs, 2);
                    // row l4 of the tile now has its sum in lanes 4*l4 ..; this lane's rows are 2c4+e
                    q_sum[nt][0] = __shfl_sync(0xffffffffu, qs, 8 * c4);
                    q_sum[nt][1] = __shfl_sync(0xffffffffu, qs, 8 * c4 + 4);
                } else {
#pragma unroll
                    for (int ks = 0; ks < kKS; ++ks) {
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const int d = kFp8 ? ks * 16 + 4 * c4 + 2 * hf : ks * 16 + hf * 8 + 2 * c4;
                            uint32_t v = 0;
                            if (qrow) v = pack2<MT>(to_float<QT>(qrow[d]), to_float<QT>(qrow[d + 1]));
                            qb[nt][ks][hf] = v;
                        }
                    }
                }
#pragma unroll
                for (int mt = 0; mt < kMT; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
            }
        }

        // a unit of work is 32 keys when possible: the next stage of the same piece joins this
        // one when a stage holds a single 16-key chunk and the ring is deep enough that holding
        // two stages still leaves three in flight; a 32-key stage is a unit by itself
        const bool two = pair_stages && n_chunks == 1 && s + 1 < s1 && k + 1 < n_item;
        const int slot2 = slot + 1 == NS ? 0 : slot + 1;
        const uint32_t phase2 = slot + 1 == NS ? phase ^ 1u : phase;
        bool landed = mbar_wait_bounded(smem_u32(&full_bar[slot]), phase);
        if (two) landed = landed && mbar_wait_bounded(smem_u32(&full_bar[slot2]), phase2);
        if (!__all_sync(0xffffffffu, landed)) {  // the warp gives up together
            if (lane == 0) {
                report(a.d_err, KV_DERR_TIMEOUT);
                *abort_flag = 1;
            }
            break;
        }
        const uint32_t full_mask = (1u << BPS) - 1u;
        ChunkRef cr[2];
        {
            const uint32_t st0 = smem_u32(smem + slot * stage_bytes);
            const int tok0 = (b0 + k * BPS) * bs;
            cr[0] = ChunkRef{st0 + koff, st0 + voff, kkey, vkey, tok0, tok0, stage_mask[slot]};
            if (two) {
                const uint32_t st1 = smem_u32(smem + slot2 * stage_bytes);
                const int tok1 = (b0 + (k + 1) * BPS) * bs;
                cr[1] = ChunkRef{st1 + koff, st1 + voff, kkey, vkey, tok1, tok1, stage_mask[slot2]};
            } else {
                cr[1] = ChunkRef{st0 + koff + 16 * kRow, st0 + voff + 16 * kRow, kkey, vkey, tok0 + 16, tok0,
                                 stage_mask[slot]};
            }
        }
        const bool pair = two || n_chunks == 2;
        bool need_mask = (cr[0].c0 < lo_last) || (cr[0].c0 + 15 > hi_first) || (cr[0].mask != full_mask);
        if (pair)
            need_mask = need_mask || (cr[1].c0 < lo_last) || (cr[1].c0 + 15 > hi_first) ||
                        (cr[1].mask != full_mask);
        if (pair) {
            if (need_mask) unit(cr, std::integral_constant<int, 2>{}, std::true_type{});
            else unit(cr, std::integral_constant<int, 2>{}, std::false_type{});
        } else {
            if (need_mask) unit(cr, std::integral_constant<int, 1>{}, std::true_type{});
            else unit(cr, std::integral_constant<int, 1>{}, std::false_type{});
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(smem_u32(&empty_bar[slot]));
            if (two) mbar_arrive(smem_u32(&empty_bar[slot2]));
        }
        const int used = two ? 2 : 1;
        for (int u = 0; u < used; ++u)
            if (++slot == NS) {
                slot = 0;
                phase ^= 1u;
            }
        const int k_last = k + used - 1;
        s += used - 1;  // the loop's ++s moves past the unit

        // ------------------------------------------------ end of a piece: write it out
        if (k_last == n_item - 1 || s == s1 - 1) {
            const bool whole = seg_k0 == 0 && k_last == n_item - 1;
            const int hkv = grp * HG + h_loc;
#pragma unroll
            for (int nt = 0; nt < kNR; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float l = l_run[nt][e];
                    l += __shfl_xor_sync(0xffffffffu, l, 4);
                    l += __shfl_xor_sync(0xffffffffu, l, 8);
                    l += __shfl_xor_sync(0xffffffffu, l, 16);
                    const int r = rt * RN + nt * 8 + 2 * c4 + e;
                    if (r >= R) continue;
                    const float inv = l > 0.f ? (kInt4 ? 1.f : a.v_scale) / l : 0.f;
                    float lse = l > 0.f ? (m_run[nt][e] + log2f(l)) * 0.69314718055994531f : -INFINITY;
                    if constexpr (kInt4) lse -= a.lse_offset_scale * q_sum[nt][e];
                    const int64_t tokq = static_cast<int64_t>(seq) * q_len + r / g;
                    const int64_t rowid = tokq * a.num_q_heads + hkv * g + r % g;
                    const int64_t wrow = static_cast<int64_t>(item + cta) * kp.rows_per_item + h_loc * R + r;
#pragma unroll
                    for (int mt = 0; mt < kMT; ++mt) {
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            // dim of accumulator row l4 (hf 0) / l4+8 (hf 1) of m-tile mt
                            int d;
                            float v;
                            if constexpr (kInt4) {
                                d = (mt >> 1) * 32 + 4 * l4 + 2 * (mt & 1) + hf;
                                const float unit = hf ? 1048576.f : 16777216.f;  // 2^20, 2^24
                                const float vsc = a.v_gscales[static_cast<int64_t>(hkv) * (D >> a.group_shift) +
                                                              (d >> a.group_shift)];
                                v = l > 0.f ? vsc * fmaf(o[mt][nt][2 * hf + e] * unit, inv, -8.f) : 0.f;
                            } else {
                                d = kFp8 ? mt * 16 + 2 * l4 + hf : mt * 16 + l4 + 8 * hf;
                                v = o[mt][nt][2 * hf + e] * inv;
                            }
                            if (whole) static_cast<QT *>(a.out)[rowid * D + d] = from_float<QT>(v);
                            else a.ws_o[wrow * D + d] = v;
                        }
                    }
                    if (l4 == 0) {
                        if (whole) {
                            if (a.lse_out) a.lse_out[rowid] = lse;
                        } else {
                            a.ws_lse[wrow] = lse;
                        }
                    }
                }
            }
        }
    }
    }  // consumer warps
    }  // s_begin < s_end

}

template <typename QT, int D>
__global__ void lse_merge_kernel(const __grid_constant__ KernelParams kp, int num_ctas) {
    const int64_t rows = static_cast<int64_t>(kp.num_items) * kp.rows_per_item;
    const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (w >= rows) return;
    merge_row<QT, D>(kp, kp.a.ws_prefix, num_ctas, w, threadIdx.x & 31);
}

template <typename QT, typename CT, int D, int RN, bool kFused>
static cudaError_t launch_typed(const CUtensorMap &tk, const CUtensorMap &tv, const KernelParams &kp,
                                const DecodePlan &plan, cudaStream_t stream) {
    auto kern = paged_decode_kernel<QT, CT, D, RN, kFused>;
    // raise the kernel's dynamic shared-memory limit to the device maximum once per device
    constexpr int kMaxDevices = 64;
    static std::once_flag once[kMaxDevices];
    static cudaError_t attr_status[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev >= kMaxDevices) return e != cudaSuccess ? e : cudaErrorInvalidDevice;
    std::call_once(once[dev], [&] {
        int optin = 0;
        cudaFuncAttributes fa;
        cudaError_t r = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (r == cudaSuccess) r = cudaFuncGetAttributes(&fa, kern);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     optin - static_cast<int>(fa.sharedSizeBytes));
        if (r != cudaSuccess) (void)cudaGetLastError();  // keep the failure out of later checks
        attr_status[dev] = r;
    });
    if (attr_status[dev] != cudaSuccess) return attr_status[dev];
    {
        kern<<<plan.num_ctas, plan.threads, plan.smem_bytes, stream>>>(tk, tv, kp);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        const int64_t rows = static_cast<int64_t>(kp.num_items) * kp.rows_per_item;
        const int threads = 256;
        const int64_t blocks = (rows * 32 + threads - 1) / threads;
        lse_merge_kernel<QT, D><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(kp, plan.num_ctas);
        return cudaGetLastError();
    }
}

template <typename QT, typename CT, int D, bool kFused>
static cudaError_t launch_rows(const CUtensorMap &tk, const CUtensorMap &tv, const KernelParams &kp,
                               const DecodePlan &plan, cudaStream_t stream) {
    return plan.rows_per_warp == 8 ? launch_typed<QT, CT, D, 8, kFused>(tk, tv, kp, plan, stream)
                                   : launch_typed<QT, CT, D, 16, kFused>(tk, tv, kp, plan, stream);
}

template <bool kFused>
static cudaError_t launch_any(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                              const KernelParams &kp, const DecodePlan &plan, int q_dtype,
                              int cache_dtype, cudaStream_t stream) {
    const bool f16 = q_dtype == KV_F16;
    if constexpr (!kFused) {
        if (cache_dtype == KV_INT4)
            return f16 ? launch_rows<__half, Int4Group, 128, false>(tmap_k, tmap_v, kp, plan, stream)
                       : launch_rows<__nv_bfloat16, Int4Group, 128, false>(tmap_k, tmap_v, kp, plan, stream);
    }
    if (cache_dtype == KV_FP8_E4M3)
        return f16 ? launch_rows<__half, Fp8E4M3, 128, kFused>(tmap_k, tmap_v, kp, plan, stream)
                   : launch_rows<__nv_bfloat16, Fp8E4M3, 128, kFused>(tmap_k, tmap_v, kp, plan, stream);
    if (kp.a.head_dim == 64)
        return f16 ? launch_rows<__half, __half, 64, kFused>(tmap_k, tmap_v, kp, plan, stream)
                   : launch_rows<__nv_bfloat16, __nv_bfloat16, 64, kFused>(tmap_k, tmap_v, kp, plan, stream);
    return f16 ? launch_rows<__half, __half, 128, kFused>(tmap_k, tmap_v, kp, plan, stream)
               : launch_rows<__nv_bfloat16, __nv_bfloat16, 128, kFused>(tmap_k, tmap_v, kp, plan, stream);
}

static KernelParams make_params(const DecodeArgs &a, const DecodePlan &plan) {
    KernelParams kp;
    kp.a = a;
    kp.f = StepArgs{};
    kp.heads_per_cta = plan.heads_per_cta;
    kp.warps_per_head = plan.warps_per_head;
    kp.blocks_per_stage = plan.blocks_per_stage;
    kp.num_stages = plan.num_stages;
    kp.box_bytes = plan.box_bytes;
    kp.box_stride = plan.box_stride;
    kp.num_items = plan.num_items;
    kp.rows_per_item = plan.rows_per_item;
    return kp;
}

cudaError_t launch_paged_decode(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                                const DecodeArgs &a, const DecodePlan &plan, int q_dtype,
                                int cache_dtype, cudaStream_t stream) {
    if (a.num_seqs == 0) return cudaSuccess;
    return launch_any<false>(tmap_k, tmap_v, make_params(a, plan), plan, q_dtype, cache_dtype, stream);
}

cudaError_t launch_decode_step(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                               const DecodeArgs &a, const StepArgs &f, const DecodePlan &plan,
                               int q_dtype, int cache_dtype, cudaStream_t stream) {
    if (a.num_seqs == 0) return cudaSuccess;
    KernelParams kp = make_params(a, plan);
    kp.f = f;
    return launch_any<true>(tmap_k, tmap_v, kp, plan, q_dtype, cache_dtype, stream);
}

}  // namespace pkv
