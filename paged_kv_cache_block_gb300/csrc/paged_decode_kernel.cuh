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

// One 16-byte chunk c of token t's K and V rows, loaded ahead of the slot it goes to.
template <typename QT> struct RowChunk {
    uint4 k, v;
    __device__ __forceinline__ void load(const StepArgs &f, int64_t t, int c) {
        k = *reinterpret_cast<const uint4 *>(static_cast<const QT *>(f.key) + t * f.key_row_stride + 8 * c);
        v = *reinterpret_cast<const uint4 *>(static_cast<const QT *>(f.value) + t * f.value_row_stride + 8 * c);
    }
    template <typename CT>
    __device__ __forceinline__ void store(const StepArgs &f, int64_t slot, int chunks, int c) const {
        const int64_t dst = (slot * chunks + c) * 8;
        if constexpr (CacheTraits<CT>::kFp8) {
            *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(f.k_cache) + dst) = quantise8<QT>(k, f.k_scale);
            *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(f.v_cache) + dst) = quantise8<QT>(v, f.v_scale);
        } else {
            *reinterpret_cast<uint4 *>(static_cast<QT *>(f.k_cache) + dst) = k;
            *reinterpret_cast<uint4 *>(static_cast<QT *>(f.v_cache) + dst) = v;
        }
    }
};

// Fused step, writer warp: the head group grp's part of the new-token rows of sequence seq
// (query rows r0 .. r1, lane holding the position of row r0 + lane) whose positions lie in
// [plo, phi), the range this CTA's stages of the item read; with their slot mapping entries
// (written by head group 0).  The source chunks load beside the table entries and go out in
// batches.
template <typename QT, typename CT, int D, int kWB>
__device__ __forceinline__ void write_item_rows(const StepArgs &f, const DecodeArgs &a, int seq, int grp, int HG,
                                             int r0, int r1, int pl, int plo, int phi, int lane) {
    // kWB: 16-byte chunks a lane has in flight (a decode item's rows are one batch: q_len tokens
    // of its head group's part)
    const int bs = a.block_size;
    const int chunks_g = HG * D / 8, chunks = a.num_kv_heads * D / 8;
    const int n = r1 - r0;
    for (int jb = 0; jb < n; jb += 32) {
        const int j = jb + lane;
        const int p = j < n ? (jb == 0 ? pl : f.positions[r0 + j]) : -1;
        const bool in = j < n && p >= plo && p < phi;
        const int phys = in ? a.block_table[static_cast<int64_t>(seq) * a.bt_stride + p / bs] : -1;
        const int npairs = min(32, n - jb) * chunks_g;
        long long slot = -2;  // not yet known
        for (int base = 0; base < npairs; base += 32 * kWB) {
            RowChunk<QT> src[kWB];
#pragma unroll
            for (int u = 0; u < kWB; ++u) {
                const int i = base + u * 32 + lane;
                if (i < npairs) src[u].load(f, r0 + jb + i / chunks_g, grp * chunks_g + i % chunks_g);
            }
            if (slot == -2) {
                const bool ok = in && phys >= 0 && phys < a.num_blocks;
                slot = ok ? static_cast<long long>(phys) * bs + p % bs : -1;
                // an invalid block is reported and masked by the attention itself
                if (in && grp == 0 && f.slot_mapping) f.slot_mapping[r0 + j] = slot;
            }
#pragma unroll
            for (int u = 0; u < kWB; ++u) {
                const int i = base + u * 32 + lane;
                const long long sl = __shfl_sync(0xffffffffu, slot, i < npairs ? (i / chunks_g) & 31 : 0);
                if (i < npairs && sl >= 0) src[u].template store<CT>(f, sl, chunks, grp * chunks_g + i % chunks_g);
            }
        }
    }
}

// Fused step, writer warp: CTA cta's equal share of the tokens whose rows no stage of any CTA
// reads (padding, rejected lengths, positions outside the attended range): slot mapping entry
// and, for a valid slot, the whole row.
template <typename QT, typename CT, int D, bool kLens>
__device__ __forceinline__ void write_unread_rows(const StepArgs &f, const DecodeArgs &a, const int32_t *Ls,
                                               int cta, int G, int lane) {
    const int B = a.num_seqs, bs = a.block_size, q_len = a.q_len;
    const int T = f.num_tokens;
    const int t0 = static_cast<int>(static_cast<long long>(T) * cta / G);
    const int t1 = static_cast<int>(static_cast<long long>(T) * (cta + 1) / G);
    const int chunks = a.num_kv_heads * D / 8;
    for (int t = t0; t < t1; ++t) {
        const int row = token_row(t, f.query_start_loc, B, q_len);
        const int p = f.positions[t];
        bool read = false;
        int L = -1;
        if (row >= 0 && row < B) {
            if constexpr (kLens) L = Ls[row];
            else L = checked_len(a, row);
        }
        if (L >= 0 && t < f.query_start_loc[row + 1] && p >= 0) {
            const int b0 = (a.window > 0 ? max(0, L - q_len - a.window + 1) : 0) / bs;
            read = p >= b0 * bs && p < (L + bs - 1) / bs * bs;
        }
        if (read) continue;
        const int64_t slot = slot_of_token(t, f.query_start_loc, B, f.positions, a.block_table, a.bt_stride,
                                           a.max_blocks_per_seq, bs, a.num_blocks, a.d_err);
        if (lane == 0 && f.slot_mapping) f.slot_mapping[t] = slot;
        if (slot < 0) continue;
        if (slot >= f.total_slots) {
            if (lane == 0) report(a.d_err, KV_DERR_BAD_SLOT);
            continue;
        }
        for (int c = lane; c < chunks; c += 32) write_row_chunk<QT, CT>(f, t, slot, chunks, c);
    }
}

// The out rows [T, Hq, D] of a consumer warp's tile: query row r (0 .. R-1, (token, head of the
// GQA group) pairs of one kv head) of sequence seq.
struct TileRows {
    int64_t tok0;  // seq * q_len
    int hq0;       // first q head of the kv head: hkv * g
    int g, R, Hq;
    __device__ __forceinline__ int64_t row(int r) const { return (tok0 + r / g) * Hq + hq0 + r % g; }
};

// A warp's normalised O tile (RN query rows x D dims, in the accumulator fragments of the
// O^T = V^T P^T products, row scale inv) into out.  The fragments hold one dim for two rows
// (16-bit caches) or two dims of one row (E4M3 caches); a movmatrix transpose, or the pairing of
// neighbouring lanes, gives every lane four adjacent dims of one row, stored at once.
template <typename QT, bool kFp8, int D, int RN, int kMT = D / 16>
__device__ __forceinline__ void store_out_tile(const float (&o)[kMT][RN / 8][4], const float (&inv)[RN / 8][2],
                                               int rbase, const TileRows &tr, QT *out, int lane, int mt0 = 0) {
    // o holds m-tiles mt0 .. mt0 + kMT - 1 of the tile
    constexpr int kNR = RN / 8;
    const int c4 = lane & 3, l4 = lane >> 2;
#pragma unroll
    for (int nt = 0; nt < kNR; ++nt) {
        if constexpr (!kFp8) {
            // fragment: dim l4 (or l4 + 8) of rows 2c4, 2c4+1; transposed: row l4, dims 2c4, 2c4+1
            const int r = rbase + nt * 8 + l4;
            QT *orow = r < tr.R ? out + tr.row(r) * D : nullptr;
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt) {
                uint32_t lo = pack2<QT>(o[mt][nt][0] * inv[nt][0], o[mt][nt][1] * inv[nt][1]);
                uint32_t hi = pack2<QT>(o[mt][nt][2] * inv[nt][0], o[mt][nt][3] * inv[nt][1]);
                lo = movmatrix_t(lo);
                hi = movmatrix_t(hi);
                // lanes c4 and c4^1 swap halves: the even one holds dims 2c4 .. 2c4+3, the odd one
                // dims 6+2c4 .. 9+2c4 (the upper eight of the m-tile)
                const uint32_t got = __shfl_xor_sync(0xffffffffu, (c4 & 1) ? lo : hi, 1);
                const uint2 v = (c4 & 1) ? make_uint2(got, hi) : make_uint2(lo, got);
                const int d = (mt0 + mt) * 16 + ((c4 & 1) ? 6 + 2 * c4 : 2 * c4);
                if (orow) *reinterpret_cast<uint2 *>(orow + d) = v;
            }
        } else {
            // fragment: dims 2l4, 2l4+1 of rows 2c4 (e 0) and 2c4+1 (e 1); lanes l4 and l4^1
            // swap rows, the even one keeping row 2c4, the odd one row 2c4+1
            const int e = l4 & 1;
            const int r = rbase + nt * 8 + 2 * c4 + e;
            QT *orow = r < tr.R ? out + tr.row(r) * D : nullptr;
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt) {
                const uint32_t p0 = pack2<QT>(o[mt][nt][0] * inv[nt][0], o[mt][nt][2] * inv[nt][0]);
                const uint32_t p1 = pack2<QT>(o[mt][nt][1] * inv[nt][1], o[mt][nt][3] * inv[nt][1]);
                const uint32_t got = __shfl_xor_sync(0xffffffffu, e ? p0 : p1, 4);
                const uint2 v = e ? make_uint2(got, p1) : make_uint2(p0, got);
                if (orow) *reinterpret_cast<uint2 *>(orow + (mt0 + mt) * 16 + 2 * (l4 & ~1)) = v;
            }
        }
    }
}

// A warp's partial O tile (normalised, rows scaled by inv) into its workspace tile, in fragment
// order: one float4 a lane per (n-tile, m-tile), so a warp's stores are whole 512-byte runs.
template <int D, int RN>
__device__ __forceinline__ void store_ws_tile(const float (&o)[D / 16][RN / 8][4], const float (&inv)[RN / 8][2],
                                              float4 *tile, int lane) {
    constexpr int kMT = D / 16, kNR = RN / 8;
#pragma unroll
    for (int nt = 0; nt < kNR; ++nt)
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt)
            tile[(nt * kMT + mt) * 32 + lane] = make_float4(o[mt][nt][0] * inv[nt][0], o[mt][nt][1] * inv[nt][1],
                                                            o[mt][nt][2] * inv[nt][0], o[mt][nt][3] * inv[nt][1]);
}

// Where one 16-key chunk of a stage sits in shared memory, for the lane that addresses it.
struct ChunkRef {
    uint32_t kbase, vbase;  // shared addresses of this lane's K and V rows (segment 0)
    int kk, vk;             // their swizzle keys
    int c0;                 // index of the chunk's first key in the sequence
    int tok0;               // index of the first key of the chunk's stage
    uint32_t mask;          // valid blocks of that stage
};

template <typename QT, typename CT, int D, int RN, bool kFused, int kBS, bool kLens>
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
    // fused step: the last item whose new-token rows the writer warp has put in (monotonic)
    int32_t *written_upto = reinterpret_cast<int32_t *>(empty_bar + NS);
    uint32_t *stage_mask = reinterpret_cast<uint32_t *>(empty_bar + NS + 1);
    volatile uint32_t *abort_flag = stage_mask + NS;
    int32_t *P = reinterpret_cast<int32_t *>(stage_mask + NS + 1);  // [NI + 1] stage prefix

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
        *written_upto = -1;
        *abort_flag = 0;
        fence_barrier_init();
    }
    const int G = gridDim.x, cta = blockIdx.x;
    // the length table, when the plan kept it in shared memory (else lengths are read from
    // seq_lens where they are needed, so that large batches keep the ring's stages)
    // (kLens: the plan kept the length table in shared memory)
    int32_t *Ls = kLens ? P + NI + 1 : nullptr;
    const bool any_empty = build_schedule<kLens>(a, NI, BPS, Ls, P, warp_sums);
    // an item with stages has an accepted length
    auto len_of = [&](int seq) {
        if constexpr (kLens) return Ls[seq];
        else return a.seq_lens[seq];
    };
    if (blockIdx.x == 0)  // the merge kernel reads the same prefix
        for (int i = threadIdx.x; i <= NI; i += blockDim.x) a.ws_prefix[i] = P[i];

    // this CTA's share of the stages: equal costs, a piece costing its stages plus a fixed part
    long long s_begin, s_end;
    share_of(cta, G, P, NI, kp.item_cost, any_empty, &s_begin, &s_end);
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
    if (threadIdx.x == 0) {
        // for the merge: this CTA holds the first stage of the items it starts, the last of those
        // it ends
        for (int i = item0; i < NI && P[i] < s_end; ++i) {
            if (P[i + 1] == P[i]) continue;
            if (P[i] >= s_begin) a.ws_pieces[2 * i] = cta;
            if (P[i + 1] - 1 < s_end) a.ws_pieces[2 * i + 1] = cta;
        }
    }
    if (warp == ncw) {
    // ================================================================ producer warp
    // In the fused step the writer warp puts in the new-token rows this CTA's stages read; the
    // copy of the first stage of an item that holds one of them waits for that item's writes,
    // every other copy goes at once.
    if (s_begin < s_end) {
        const uint32_t tx = 2u * BPS * kNDB * kp.box_bytes;
        int item = item0;
        int cache_base = 0, cache_item = -1;  // lanes hold block ids [cache_base, +32) of cache_item
        int my_id = a.num_blocks;
        bool my_ok = false;
        int issued = 0, pslot = 0;
        uint32_t pround = 0;  // completed passes over the ring
        constexpr int kTablePrefetchStages = 4;
        // fused step: of item guard_item, the first stage holding a row the writer puts in
        // (guard_k)
        int guard_item = -1, guard_k = 0x7fffffff;
        int len_item = -1, len_cur = 0;  // the length of the sequence of item len_item
        for (long long s = s_begin; s < s_end; ++s) {
            while (P[item + 1] <= s) ++item;
            const int k = static_cast<int>(s - P[item]);
            const int seq = item % B, grp = item / B;
            int L;
            if constexpr (kLens) {
                L = Ls[seq];
            } else {
                if (len_item != item) {  // read once an item
                    len_item = item;
                    len_cur = len_of(seq);
                }
                L = len_cur;
            }
            const int nblk = (L + bs - 1) / bs;
            const int lb0 = (a.window > 0 ? max(0, L - q_len - a.window + 1) : 0) / bs + k * BPS;
            // fused step: a new item's query offsets load beside its block ids (below), then its
            // positions
            const bool new_item = kFused && guard_item != item;
            int r0 = 0, r1 = 0, pg = -1;
            if (new_item) {
                r0 = kp.f.query_start_loc[seq];
                r1 = kp.f.query_start_loc[seq + 1];
                // the positions of rows seq * q_len .. (where a decode batch puts this sequence's
                // tokens), loaded beside the offsets; reloaded below if the offsets differ
                const int tg = seq * q_len + lane;
                if (lane < q_len && tg < kp.f.num_tokens) pg = kp.f.positions[tg];
            }
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
            if (new_item) {
                // the first stage of this item holding a row the writer puts in: positions in
                // the range this CTA's stages of the item read
                guard_item = item;
                const int b0i = lb0 - k * BPS;
                const long long ka = max(s_begin, static_cast<long long>(P[item])) - P[item];
                const long long kb = min(s_end, static_cast<long long>(P[item + 1])) - P[item];
                const int plo = (b0i + static_cast<int>(ka) * BPS) * bs;
                const int phi = min((b0i + static_cast<int>(kb) * BPS) * bs, nblk * bs);
                const bool guessed = r0 == seq * q_len && r1 - r0 == q_len;
                int my_k = 0x7fffffff;
                for (int j = lane; j < r1 - r0; j += 32) {
                    const int p = guessed ? pg : kp.f.positions[r0 + j];
                    if (p >= plo && p < phi) my_k = min(my_k, (p / bs - b0i) / BPS);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) my_k = min(my_k, __shfl_xor_sync(0xffffffffu, my_k, o));
                guard_k = my_k;
            }
            if (lane == 0 && s + kTablePrefetchStages == P[item + 1] && P[item + 1] < s_end) {
                // the next item's first block ids: into L2 ahead of its first copies
                int nx = item + 1;
                while (P[nx + 1] == P[nx]) ++nx;
                const int nseq = nx % B, nL = len_of(nseq);
                const int nb0 = (a.window > 0 ? max(0, nL - q_len - a.window + 1) : 0) / bs;
                prefetch_l2(a.block_table + static_cast<int64_t>(nseq) * a.bt_stride + nb0);
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
            if constexpr (kFused) {
                if (item == guard_item && k >= guard_k) {
                    int late = 0;
                    if (lane == 0) {
                        if (!wait_at_least_bounded(written_upto, item)) {
                            late = 1;
                            report(a.d_err, KV_DERR_TIMEOUT);
                            *abort_flag = 1;
                        } else {
                            fence_proxy_async_global();
                        }
                    }
                    if (__shfl_sync(0xffffffffu, late, 0)) break;
                    guard_k = 0x7fffffff;  // this item's rows are in
                }
            }
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
    }
    } else if (kFused && warp == ncw + 1) {
    // ================================================================ writer warp (fused step)
    // The head group's part of every new token whose position lies in one of this CTA's stages
    // (each such row has exactly one reader: this CTA), item by item, each followed by a proxy
    // fence that orders the rows before the producer's copies and a signal (the item's index);
    // then this CTA's share of the rows no stage reads.
        for (int item = item0; s_begin < s_end && item < NI && P[item] < s_end; ++item) {
            if (P[item + 1] == P[item]) continue;
            const int seq = item % B, grp = item / B;
            const int L = len_of(seq);
            const int nblk = (L + bs - 1) / bs;
            const int b0 = (a.window > 0 ? max(0, L - q_len - a.window + 1) : 0) / bs;
            const long long ka = max(s_begin, static_cast<long long>(P[item])) - P[item];
            const long long kb = min(s_end, static_cast<long long>(P[item + 1])) - P[item];
            const int plo = (b0 + static_cast<int>(ka) * BPS) * bs;
            const int phi = min((b0 + static_cast<int>(kb) * BPS) * bs, nblk * bs);
            const int r0 = kp.f.query_start_loc[seq], r1 = kp.f.query_start_loc[seq + 1];
            const int pl = lane < r1 - r0 ? kp.f.positions[r0 + lane] : -1;
            write_item_rows<QT, CT, D, RN == 16 ? 16 : 8>(kp.f, a, seq, grp, HG, r0, r1, pl, plo, phi, lane);
            // this item's rows are in: the producer may copy its stages that hold them
            fence_proxy_async_global();
            __syncwarp();
            if (lane == 0) st_release_cta(written_upto, item);
        }
        // rows nobody reads, after the signals (nothing waits for them)
        write_unread_rows<QT, CT, D, kLens>(kp.f, a, Ls, cta, G, lane);
    } else if (warp < ncw && s_begin < s_end) {

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
            L = len_of(seq);
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
                        if (qrow) {
                            // an aligned pair of q elements in one load (the MMA operand itself
                            // for 16-bit caches)
                            const uint32_t w = *reinterpret_cast<const uint32_t *>(qrow + d);
                            if constexpr (std::is_same<MT, QT>::value) {
                                v = w;
                            } else {
                                const float2 f2 = unpack2<QT>(w);
                                v = pack2<MT>(f2.x, f2.y);
                            }
                        }
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
            const TileRows tr{static_cast<int64_t>(seq) * q_len, hkv * g, g, R, a.num_q_heads};
            float inv[kNR][2];
#pragma unroll
            for (int nt = 0; nt < kNR; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float l = l_run[nt][e];
                    l += __shfl_xor_sync(0xffffffffu, l, 4);
                    l += __shfl_xor_sync(0xffffffffu, l, 8);
                    l += __shfl_xor_sync(0xffffffffu, l, 16);
                    inv[nt][e] = l > 0.f ? a.v_scale / l : 0.f;
                    const int r = rt * RN + nt * 8 + 2 * c4 + e;
                    if (l4 == 0 && r < R) {
                        const float lse = l > 0.f ? (m_run[nt][e] + log2f(l)) * 0.69314718055994531f : -INFINITY;
                        if (whole) {
                            if (a.lse_out) a.lse_out[tr.row(r)] = lse;
                        } else {
                            a.ws_lse[static_cast<int64_t>(item + cta) * kp.rows_per_item + h_loc * R + r] = lse;
                        }
                    }
                }
            }
            if (whole) {
                store_out_tile<QT, kFp8, D, RN>(o, inv, rt * RN, tr, static_cast<QT *>(a.out), lane);
            } else if (kp.tile_ws) {
                store_ws_tile<D, RN>(o, inv,
                                     reinterpret_cast<float4 *>(a.ws_o) +
                                         (static_cast<int64_t>(item + cta) * ncw + warp) * (RN * D / 4),
                                     lane);
            } else {
                // warps with rows past the group (padding): the real rows only, one per workspace row
#pragma unroll
                for (int nt = 0; nt < kNR; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int r = rt * RN + nt * 8 + 2 * c4 + e;
                        if (r >= R) continue;
                        float *wrow = a.ws_o + (static_cast<int64_t>(item + cta) * kp.rows_per_item + h_loc * R + r) * D;
#pragma unroll
                        for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf)
                                wrow[kFp8 ? mt * 16 + 2 * l4 + hf : mt * 16 + l4 + 8 * hf] = o[mt][nt][2 * hf + e] * inv[nt][e];
                    }
            }
        }
    }
    }  // consumer warps

}

// The merge of split sequences for this kernel: one warp per (consumer-warp tile of an item, run
// of kMW m-tiles).  A tile one CTA covered whole was written by that CTA; a split tile's pieces
// are combined, LSE = log sum_c exp(lse_c), out = sum_c exp(lse_c - LSE) o_c, and written like a
// whole tile.  A rejected length gives zero rows and lse -inf.  Pieces go eight (16-row tiles:
// four) at a time, every load of a group issued before the sums use it: two round trips through
// L2 (the stage range with the piece owners, then the pieces) for a tile with up to that many
// pieces.
template <typename QT, bool kFp8, int D, int RN>
struct TileMerge {
    static constexpr int kMW = 1;  // m-tiles a warp merges
    static constexpr int kRuns = D / 16 / kMW;
};

template <typename QT, bool kFp8, int D, int RN>
__global__ void __launch_bounds__(128) tile_merge_kernel(const __grid_constant__ KernelParams kp, int num_ctas) {
    constexpr int kNR = RN / 8, kMW = TileMerge<QT, kFp8, D, RN>::kMW, kRuns = TileMerge<QT, kFp8, D, RN>::kRuns;
    constexpr int kMT = D / 16, kG = RN == 8 ? 8 : 4;  // pieces a group
    const DecodeArgs &a = kp.a;
    const int ncw = kp.heads_per_cta * kp.warps_per_head;
    const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (w >= static_cast<int64_t>(kp.num_items) * ncw * kRuns) return;
    const int lane = threadIdx.x & 31, c4 = lane & 3;
    const int run = static_cast<int>(w % kRuns);
    const int64_t tw = w / kRuns;
    const int item = static_cast<int>(tw / ncw), t = static_cast<int>(tw - static_cast<int64_t>(item) * ncw);
    const int MW = kp.warps_per_head, h_loc = t / MW, rt = t - h_loc * MW;
    const int B = a.num_seqs, g = a.num_q_heads / a.num_kv_heads, R = g * a.q_len;
    const int seq = item % B, grp = item / B;
    const TileRows tr{static_cast<int64_t>(seq) * a.q_len, (grp * kp.heads_per_cta + h_loc) * g, g, R, a.num_q_heads};
    // the item's stage range and the shares holding its first and last stage, in one round trip
    // (the owners are read even for an empty item, whose entries may hold anything, and used only
    // for a non-empty one)
    const int32_t *P = a.ws_prefix;
    const int32_t p0 = P[item], p1 = P[item + 1];
    const int c_lo = a.ws_pieces[2 * item], c_hi = a.ws_pieces[2 * item + 1];
    float acc[kMW][kNR][4];
#pragma unroll
    for (int m = 0; m < kMW; ++m)
#pragma unroll
        for (int nt = 0; nt < kNR; ++nt) acc[m][nt][0] = acc[m][nt][1] = acc[m][nt][2] = acc[m][nt][3] = 0.f;
    float inv[kNR][2], mx[kNR][2], wsum[kNR][2];
#pragma unroll
    for (int nt = 0; nt < kNR; ++nt) {
        inv[nt][0] = inv[nt][1] = 0.f;
        mx[nt][0] = mx[nt][1] = -INFINITY;
        wsum[nt][0] = wsum[nt][1] = 0.f;
    }
    if (p1 > p0) {
        if (c_lo == c_hi) return;  // one CTA covered it and wrote the output
        auto has = [&](int c) { return c <= c_hi; };
        const float *lse_base = a.ws_lse + static_cast<int64_t>(item) * kp.rows_per_item + h_loc * R;
        auto lse_of = [&](int c, int nt, int e) {
            const int r = rt * RN + nt * 8 + 2 * c4 + e;
            return has(c) && r < R ? __ldcg(lse_base + static_cast<int64_t>(c) * kp.rows_per_item + r) : -INFINITY;
        };
        // A group of pieces at a time, all of its loads issued before any is used (one round trip
        // through L2 for a tile of up to kG pieces).  The reference maximum is the largest lse seen
        // so far; a later group with a larger one rescales the sums (exp(old - new)).
        for (int base = c_lo; base <= c_hi; base += kG) {
            float4 v[kG][kNR][kMW];
            float wl[kG][kNR][2];
#pragma unroll
            for (int u = 0; u < kG; ++u) {
                const bool ok = has(base + u);
                const float4 *tile = reinterpret_cast<const float4 *>(a.ws_o) +
                                     (static_cast<int64_t>(item + base + u) * ncw + t) * (RN * D / 4);
#pragma unroll
                for (int nt = 0; nt < kNR; ++nt)
#pragma unroll
                    for (int m = 0; m < kMW; ++m)
                        v[u][nt][m] = ok ? __ldcg(tile + (nt * kMT + run * kMW + m) * 32 + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int nt = 0; nt < kNR; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) wl[u][nt][e] = lse_of(base + u, nt, e);
            }
#pragma unroll
            for (int nt = 0; nt < kNR; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float gm = -INFINITY;
#pragma unroll
                    for (int u = 0; u < kG; ++u) gm = fmaxf(gm, wl[u][nt][e]);
                    if (gm > mx[nt][e]) {
                        // earlier groups' sums against the new maximum (none in the first group)
                        const float f = mx[nt][e] != -INFINITY ? expf(mx[nt][e] - gm) : 0.f;
                        wsum[nt][e] *= f;
#pragma unroll
                        for (int m = 0; m < kMW; ++m) {
                            acc[m][nt][e] *= f;
                            acc[m][nt][2 + e] *= f;
                        }
                        mx[nt][e] = gm;
                    }
                }
#pragma unroll
            for (int u = 0; u < kG; ++u)
#pragma unroll
                for (int nt = 0; nt < kNR; ++nt) {
                    float w0 = wl[u][nt][0], w1 = wl[u][nt][1];
                    w0 = (w0 != -INFINITY && mx[nt][0] != -INFINITY) ? expf(w0 - mx[nt][0]) : 0.f;
                    w1 = (w1 != -INFINITY && mx[nt][1] != -INFINITY) ? expf(w1 - mx[nt][1]) : 0.f;
                    wsum[nt][0] += w0;
                    wsum[nt][1] += w1;
                    // pieces of weight 0 (empty rows) may hold anything: selected away, never multiplied
#pragma unroll
                    for (int m = 0; m < kMW; ++m) {
                        acc[m][nt][0] += w0 > 0.f ? w0 * v[u][nt][m].x : 0.f;
                        acc[m][nt][1] += w1 > 0.f ? w1 * v[u][nt][m].y : 0.f;
                        acc[m][nt][2] += w0 > 0.f ? w0 * v[u][nt][m].z : 0.f;
                        acc[m][nt][3] += w1 > 0.f ? w1 * v[u][nt][m].w : 0.f;
                    }
                }
        }
#pragma unroll
        for (int nt = 0; nt < kNR; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) inv[nt][e] = wsum[nt][e] > 0.f ? 1.f / wsum[nt][e] : 0.f;
    }
    store_out_tile<QT, kFp8, D, RN, kMW>(acc, inv, rt * RN, tr, static_cast<QT *>(a.out), lane, run * kMW);
    if (run == 0 && a.lse_out && (lane >> 2) == 0) {
#pragma unroll
        for (int nt = 0; nt < kNR; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = rt * RN + nt * 8 + 2 * c4 + e;
                if (r < R) a.lse_out[tr.row(r)] = wsum[nt][e] > 0.f ? mx[nt][e] + logf(wsum[nt][e]) : -INFINITY;
            }
    }
}

template <typename QT, bool kFp8, int D, int RN>
static cudaError_t tile_merge(const KernelParams &kp, int num_workers, cudaStream_t stream) {
    const int64_t warps = static_cast<int64_t>(kp.num_items) * kp.heads_per_cta * kp.warps_per_head *
                          TileMerge<QT, kFp8, D, RN>::kRuns;
    const int threads = 128;
    const int64_t blocks = (warps * 32 + threads - 1) / threads;
    tile_merge_kernel<QT, kFp8, D, RN><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(kp, num_workers);
    return cudaGetLastError();
}

template <typename QT, typename CT, int D, int RN, bool kFused, int kBS, bool kLens>
static cudaError_t launch_typed(const CUtensorMap &tk, const CUtensorMap &tv, const KernelParams &kp,
                                const DecodePlan &plan, cudaStream_t stream) {
    auto kern = paged_decode_kernel<QT, CT, D, RN, kFused, kBS, kLens>;
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
        return kp.tile_ws ? tile_merge<QT, CacheTraits<CT>::kFp8, D, RN>(kp, plan.num_ctas, stream)
                          : row_merge<QT, D>(kp, plan.num_ctas, stream);
    }
}

template <typename QT, typename CT, int D, bool kFused>
static cudaError_t launch_rows(const CUtensorMap &tk, const CUtensorMap &tv, const KernelParams &kp,
                               const DecodePlan &plan, cudaStream_t stream) {
    // the FP8 cache with 16-token blocks (one block per stage) runs a kernel with that block size
    // built in; measured 6% faster on a 32-sequence Llama-70B-shaped batch (16-bit caches gain ~1%)
    if (!plan.lens_smem)  // a batch whose length table would cost the ring a stage
        return plan.rows_per_warp == 8 ? launch_typed<QT, CT, D, 8, kFused, 0, false>(tk, tv, kp, plan, stream)
                                       : launch_typed<QT, CT, D, 16, kFused, 0, false>(tk, tv, kp, plan, stream);
    if constexpr (CacheTraits<CT>::kFp8) {
        if (kp.a.block_size == 16 && kp.blocks_per_stage == 1)
            return plan.rows_per_warp == 8 ? launch_typed<QT, CT, D, 8, kFused, 16, true>(tk, tv, kp, plan, stream)
                                           : launch_typed<QT, CT, D, 16, kFused, 16, true>(tk, tv, kp, plan, stream);
    }
    return plan.rows_per_warp == 8 ? launch_typed<QT, CT, D, 8, kFused, 0, true>(tk, tv, kp, plan, stream)
                                   : launch_typed<QT, CT, D, 16, kFused, 0, true>(tk, tv, kp, plan, stream);
}

// E4M3 caches (paged_attention_fp8.cu): launch_rows over (f16 or bf16 queries, head dim 128)
template <bool kFused>
cudaError_t launch_rows_fp8(const CUtensorMap &tk, const CUtensorMap &tv, const KernelParams &kp,
                            const DecodePlan &plan, bool f16, cudaStream_t stream);

}  // namespace pkv
