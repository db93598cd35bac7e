// Paged decode attention over 16-bit and E4M3 caches: persistent stream-K schedule, TMA-fed
// tensor-core MMAs, online softmax, log-sum-exp merge of the pieces of sequences that straddle
// CTAs.  This header holds the kernel template and its typed launcher; paged_attention.cu
// instantiates it for 16-bit caches and paged_attention_fp8.cu for E4M3 caches, two translation
// units that compile in parallel.
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
//   * INT4 caches have their own kernel (paged_decode_int4.cu) on the same schedule and merge.
#pragma once

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "decode_common.cuh"
#include "kernels.h"

namespace pkv {

struct Fp8E4M3 {};  // tag for an E4M3 cache

template <typename CT> struct CacheTraits {
    static constexpr int kBytes = 2;
    static constexpr bool kFp8 = false;
};
template <> struct CacheTraits<Fp8E4M3> {
    static constexpr int kBytes = 1;
    static constexpr bool kFp8 = true;
};

// Four E4M3 bytes -> two packed fp16 pairs (bytes 0,1 -> lo; bytes 2,3 -> hi), exact.
__device__ __forceinline__ void e4m3x4_to_h2x2(uint32_t four, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(four));
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

// Where one 16-key chunk of a stage sits in shared memory, for the lane that addresses it.
struct ChunkRef {
    uint32_t kbase, vbase;  // shared addresses of this lane's K and V rows (segment 0)
    int kk, vk;             // their swizzle keys
    int c0;                 // index of the chunk's first key in the sequence
    int tok0;               // index of the first key of the chunk's stage
    uint32_t mask;          // valid blocks of that stage
};

template <typename QT, typename CT, int D, int RN, bool kFused, int kBS>
__global__ void __maxnreg__(DecodeLaunch<RN>::kMaxRegs)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v,
                        const __grid_constant__ KernelParams kp) {
    constexpr bool kFp8 = CacheTraits<CT>::kFp8;
    using MT = typename std::conditional<kFp8, __half, QT>::type;  // MMA operand type
    constexpr int kEB = CacheTraits<CT>::kBytes;
    constexpr int kNDB = D * kEB / 128;  // 128-byte row segments (TMA boxes) per head row
    constexpr int kKS = D / 16;          // k-steps of K q^T (16 dims each)
    constexpr int kMT = D / 16;          // m-tiles of V^T P^T (16 dims each)
    constexpr int kNR = RN / 8;          // n-tiles of query rows

    const DecodeArgs &a = kp.a;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int HG = kp.heads_per_cta, MW = kp.warps_per_head;
    const int ncw = HG * MW;
    // kBS > 0: the block size (one block per stage) is a compile-time constant, so the slot and
    // stage arithmetic folds; 0 reads both from the arguments
    const int bs = kBS ? kBS : a.block_size, BPS = kBS ? 1 : kp.blocks_per_stage;
    const int ST = BPS * bs, NS = kp.num_stages;
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
    if (threadIdx.x == 32) {  // the descriptors' fetch overlaps the schedule
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), ncw);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    const int G = gridDim.x, cta = blockIdx.x;
    build_schedule(a, NI, BPS, Ls, P, warp_sums);
    if (blockIdx.x == 0)  // the merge kernel reads the same prefix
        for (int i = threadIdx.x; i <= NI; i += blockDim.x) a.ws_prefix[i] = P[i];

    const long long S = P[NI];
    const int A = active_shares(S, G);
    const long long s_begin = share_begin(S, A, cta), s_end = share_begin(S, A, cta + 1);
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
        const int tv = kFp8 ? tk : (lane >> 4) * 8 + (lane & 7);
        const int jk = tk / bs, rk = h_loc * bs + (tk - jk * bs);
        const int jv = tv / bs, rv = h_loc * bs + (tv - jv * bs);
        koff = (jk * kNDB) * kp.box_stride + rk * 128;
        voff = ((BPS + jv) * kNDB) * kp.box_stride + rv * 128;
        kkey = rk & 7;
        vkey = rv & 7;
    }
    const int n_chunks = ST / 16;
    const bool pair_stages = NS >= 5;

    float o[kMT][kNR][4];
    float m_run[kNR][2], l_run[kNR][2];
    uint32_t qb[kNR][kKS][2];
    int pos_hi[kNR][2];  // position of each of this lane's rows (-1: padding row)
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
            if constexpr (kFp8) {
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
            if constexpr (kMasked) {
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
            if constexpr (kFp8) {
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
                cr[1] = ChunkRef{st0 + koff + 16 * 128, st0 + voff + 16 * 128, kkey, vkey, tok0 + 16, tok0,
                                 stage_mask[slot]};
            }
        }
        const bool pair = two || n_chunks == 2;
        auto chunk_masked = [&](const ChunkRef &c) {
            return (c.c0 < lo_last) || (c.c0 + 15 > hi_first) || (c.mask != full_mask);
        };
        if constexpr (kNR == 1) {
            const bool need_mask = chunk_masked(cr[0]) || (pair && chunk_masked(cr[1]));
            if (pair) {
                if (need_mask) unit(cr, std::integral_constant<int, 2>{}, std::true_type{});
                else unit(cr, std::integral_constant<int, 2>{}, std::false_type{});
            } else {
                if (need_mask) unit(cr, std::integral_constant<int, 1>{}, std::true_type{});
                else unit(cr, std::integral_constant<int, 1>{}, std::false_type{});
            }
        } else {
            // 16-row warps hold twice the accumulators: their 32-key units run as two 16-key
            // units in turn, which keeps the registers of a second chunk's scores free (no spills)
            const ChunkRef one[2][2] = {{cr[0], cr[0]}, {cr[1], cr[1]}};
            for (int j = 0; j < (pair ? 2 : 1); ++j) {
                if (chunk_masked(one[j][0])) unit(one[j], std::integral_constant<int, 1>{}, std::true_type{});
                else unit(one[j], std::integral_constant<int, 1>{}, std::false_type{});
            }
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
                    const float inv = l > 0.f ? a.v_scale / l : 0.f;
                    const float lse = l > 0.f ? (m_run[nt][e] + log2f(l)) * 0.69314718055994531f : -INFINITY;
                    const int64_t tokq = static_cast<int64_t>(seq) * q_len + r / g;
                    const int64_t rowid = tokq * a.num_q_heads + hkv * g + r % g;
                    const int64_t wrow = static_cast<int64_t>(item + cta) * kp.rows_per_item + h_loc * R + r;
#pragma unroll
                    for (int mt = 0; mt < kMT; ++mt) {
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            // dim of accumulator row l4 (hf 0) / l4+8 (hf 1) of m-tile mt
                            const int d = kFp8 ? mt * 16 + 2 * l4 + hf : mt * 16 + l4 + 8 * hf;
                            const float v = o[mt][nt][2 * hf + e] * inv;
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
static cudaError_t merge_typed(const KernelParams &kp, int num_workers, cudaStream_t stream) {
    const int64_t rows = static_cast<int64_t>(kp.num_items) * kp.rows_per_item;
    const int threads = 256;
    const int64_t blocks = (rows * 32 + threads - 1) / threads;
    lse_merge_kernel<QT, D><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(kp, num_workers);
    return cudaGetLastError();
}

template <typename QT, typename CT, int D, int RN, bool kFused, int kBS>
static cudaError_t launch_typed(const CUtensorMap &tk, const CUtensorMap &tv, const KernelParams &kp,
                                const DecodePlan &plan, cudaStream_t stream) {
    auto kern = paged_decode_kernel<QT, CT, D, RN, kFused, kBS>;
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
        return merge_typed<QT, D>(kp, plan.num_ctas, stream);
    }
}

template <typename QT, typename CT, int D, bool kFused>
static cudaError_t launch_rows(const CUtensorMap &tk, const CUtensorMap &tv, const KernelParams &kp,
                               const DecodePlan &plan, cudaStream_t stream) {
    // the FP8 cache with 16-token blocks (one block per stage) runs a kernel with that block size
    // built in; measured 6% faster on a 32-sequence Llama-70B-shaped batch (16-bit caches gain ~1%)
    if constexpr (CacheTraits<CT>::kFp8) {
        if (kp.a.block_size == 16 && kp.blocks_per_stage == 1)
            return plan.rows_per_warp == 8 ? launch_typed<QT, CT, D, 8, kFused, 16>(tk, tv, kp, plan, stream)
                                           : launch_typed<QT, CT, D, 16, kFused, 16>(tk, tv, kp, plan, stream);
    }
    return plan.rows_per_warp == 8 ? launch_typed<QT, CT, D, 8, kFused, 0>(tk, tv, kp, plan, stream)
                                   : launch_typed<QT, CT, D, 16, kFused, 0>(tk, tv, kp, plan, stream);
}

// E4M3 caches (paged_attention_fp8.cu): launch_rows over (f16 or bf16 queries, head dim 128)
template <bool kFused>
cudaError_t launch_rows_fp8(const CUtensorMap &tk, const CUtensorMap &tv, const KernelParams &kp,
                            const DecodePlan &plan, bool f16, cudaStream_t stream);

}  // namespace pkv
