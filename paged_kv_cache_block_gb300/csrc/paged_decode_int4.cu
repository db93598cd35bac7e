// Paged decode attention over INT4 caches with group scales (kv_paged_attention_decode_int4).
//
// What it computes: the decode attention of paged_decode_kernel.cuh ("vLLM의 KV cache 연결 흐름",
// sections "Slot mapping은 왜 필요한가" and "Forward 직전의 metadata"; "Understanding
// PageAttention Memory Optimization", section "Handling Softmax Across Blocks"; GQA, windows and
// speculative tokens as there) over the INT4 cache of "vLLM Worker侧GPU KV Cache初始化流程深度解析",
// section "KV Cache技术背景": element = code * scale[head][dim / group_size].
//
// How (GB300).  INT4 moves a quarter of the bf16 bytes, so per byte the kernel does four times the
// instruction work (widening, MMAs, softmax) and needs more warps to hide its latencies than the
// 16-bit kernel's one producer + eight consumers.  Here every warp is its own pipeline:
//   * A CTA holds 16 warps (8 with 16-row tiles) in independent sets; a set is one stream-K worker
//     with one warp per (kv head of its group, row tile), taking an equal contiguous share of the
//     flat (head group, sequence, stage) list.  Pieces of a sequence split between workers are
//     merged by the log-sum-exp merge kernel, as in the 16-bit path.
//   * Each warp owns a ring of shared-memory stages and fills it itself: lane 0 issues the TMA
//     copies of its own head's rows (a box of one block x one head: block_size rows of 64 bytes,
//     swizzled 64B) NS stages ahead of what the warp consumes, refilling a slot as soon as the warp
//     has read it.  No producer warp and no cross-warp barrier: 16 warps fit the 128 registers a
//     thread that four warps per SM sub-partition leave.
//   * The block-table entries are read by the warp, 32 at a time (one coalesced load).
//   * Scores are S^T = K q^T on m16n8k16 MMAs (keys as M), nibbles widened to fp16 subnormals by
//     one AND-XOR per pair (u = code ^ 8 is the offset-binary value; the fp16 with bits u or u << 4
//     is u * 2^-24 or u * 2^-20).  The offset 8 comes back out exactly: a per-row shift of every
//     score for K (the softmax ignores it, the log-sum-exp subtracts 8 * scale * sum_d q_d), and
//     out_d = vscale_d * (sum_j p_j u_jd / l - 8) for V.  K scales and the 2^-20 / 2^-24 units fold
//     into q before it is rounded to fp16; V scales multiply the float32 output.
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "decode_common.cuh"
#include "kernels.h"

namespace pkv {
namespace {

constexpr int kD = 128;         // head_dim
constexpr int kRowBytes = 64;   // one head's row of a slot

template <int RN> struct Int4Launch {
    static constexpr int kWarps = RN == 8 ? 16 : 8;
    static constexpr int kThreads = kWarps * 32;
};

__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Where one 16-key chunk of a stage sits in this warp's ring, for the lane that addresses it.
struct Int4Chunk {
    uint32_t kbase, vbase;  // shared addresses of this lane's K and V rows
    int key;                // their 64B-swizzle key
    int c0;                 // index of the chunk's first key in the sequence
    int tok0;               // index of the first key of the chunk's stage
    uint32_t mask;          // valid blocks of that stage
};

// One 16-byte chunk c (8 elements) of token t's K and V rows, as INT4 codes, into its slot: 4 bytes
// of each cache (the layout and rounding of kv_reshape_and_cache_int4).
template <typename QT>
__device__ __forceinline__ void write_int4_chunk(const DecodeArgs &a, const StepArgs &f, int64_t t, int64_t slot,
                                                 int chunks, int c) {
    const uint4 kx = *reinterpret_cast<const uint4 *>(static_cast<const QT *>(f.key) + t * f.key_row_stride + 8 * c);
    const uint4 vx = *reinterpret_cast<const uint4 *>(static_cast<const QT *>(f.value) + t * f.value_row_stride + 8 * c);
    const int per_head = kD / 8;
    const int h = c / per_head;
    const int sidx = h * (kD >> a.group_shift) + (((c - h * per_head) * 8) >> a.group_shift);
    static_cast<uint32_t *>(f.k_cache)[slot * chunks + c] = quantise_int4x8<QT>(kx, a.k_gscales[sidx]);
    static_cast<uint32_t *>(f.v_cache)[slot * chunks + c] = quantise_int4x8<QT>(vx, a.v_gscales[sidx]);
}

// kBS: the block size when it is fixed at compile time (8, 16 or 32: stages of 32 keys whose
// geometry is then constant), 0 when it is read from the arguments (4, and 16-row tiles)
template <typename QT, int RN, bool kFused, int kBS>
__global__ void __launch_bounds__(Int4Launch<RN>::kThreads, 1)
    paged_decode_int4_kernel(const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v,
                             const __grid_constant__ KernelParams kp) {
    using MT = __half;  // MMA operand type
    constexpr int kWarps = Int4Launch<RN>::kWarps;
    constexpr int kKS = kD / 16;  // k-steps of K q^T
    constexpr int kMT = kD / 16;  // m-tiles of V^T P^T
    constexpr int kNR = RN / 8;   // n-tiles of query rows

    const DecodeArgs &a = kp.a;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int HG = kp.heads_per_cta, MW = kp.warps_per_head;
    const int wps = HG * MW;  // warps per set
    const int set = warp / wps, wi = warp - set * wps;
    const int h_loc = wi / MW, rt = wi - h_loc * MW;
    static_assert(kBS == 0 || kBS == 8 || kBS == 16 || kBS == 32, "compile-time block sizes give 32-key stages");
    const int bs = kBS ? kBS : a.block_size;
    const int BPS = kBS ? 32 / kBS : kp.blocks_per_stage;
    const int ST = BPS * bs, NS = kp.num_stages;
    const int B = a.num_seqs, NI = kp.num_items;
    const int g = a.num_q_heads / a.num_kv_heads;
    const int R = g * a.q_len;
    const int q_len = a.q_len;
    const int gshift = a.group_shift;

    // ---------------------------------------------------------------- shared memory
    // [kWarps][NS] stages of (K boxes, V boxes), [kWarps][NS] full barriers, [kWarps][NS] stage
    // masks, the stage prefix [NI + 1] and the length table [B]
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int stage_bytes = 2 * BPS * kp.box_stride;
    uint8_t *ring = smem + static_cast<size_t>(warp) * NS * stage_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(kWarps) * NS * stage_bytes);
    uint64_t *full_bar = bars + warp * NS;
    uint32_t *masks = reinterpret_cast<uint32_t *>(bars + kWarps * NS);
    uint32_t *smask = masks + warp * NS;
    int32_t *P = reinterpret_cast<int32_t *>(masks + kWarps * NS);
    int32_t *Ls = P + NI + 1;
    __shared__ int32_t warp_sums[32];

    if (threadIdx.x == 32) {  // the descriptors' fetch overlaps the schedule
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    if (lane == 0) {
        for (int i = 0; i < NS; ++i) mbar_init(smem_u32(&full_bar[i]), 1);
        fence_barrier_init();
    }
    (void)build_schedule(a, NI, BPS, Ls, P, warp_sums);
    if (blockIdx.x == 0)  // the merge kernel reads the same prefix
        for (int i = threadIdx.x; i <= NI; i += blockDim.x) a.ws_prefix[i] = P[i];

    // ---------------------------------------------------------------- this warp's share
    const int G = kp.num_workers;
    const int vc = blockIdx.x * kp.sets_per_cta + set;
    if (set >= kp.sets_per_cta || vc >= G) return;
    const long long S = P[NI];
    const int A = active_shares(S, G);
    const long long s_begin = share_begin(S, A, vc), s_end = share_begin(S, A, vc + 1);
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
        // ---- the one-launch step: before this worker reads any cache block, its warps write the
        // new-token rows its own stages will read (the head group's part of every new token whose
        // position falls in one of its stages: each such row has exactly one reader), and an equal
        // share of the tokens whose rows no stage reads; then the slot mapping is complete too
        const StepArgs &f = kp.f;
        const int st = wi * 32 + lane, nst = wps * 32;  // this thread among the worker's
        const int chunks = a.num_kv_heads * kD / 8;     // 16-byte source chunks of a token row
        const int chunks_g = HG * kD / 8;               // ... of a head group's part
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
            for (int i = st; i < (r1 - r0) * chunks_g; i += nst) {
                const int t = r0 + i / chunks_g, c = i % chunks_g;
                const int p = f.positions[t];
                if (p < plo || p >= phi) continue;
                const int physical = a.block_table[static_cast<int64_t>(seq) * a.bt_stride + p / bs];
                const bool ok = physical >= 0 && physical < a.num_blocks;
                const int64_t slot = ok ? static_cast<int64_t>(physical) * bs + p % bs : -1;
                if (grp == 0 && c == 0 && f.slot_mapping) f.slot_mapping[t] = slot;
                if (!ok) continue;  // the attention reports and masks this block
                write_int4_chunk<QT>(a, f, t, slot, chunks, grp * chunks_g + c);
            }
        }
        {   // rows no stage reads: each worker takes an equal share of the tokens
            const int T = f.num_tokens;
            const int t0 = static_cast<int>(static_cast<long long>(T) * vc / G);
            const int t1 = static_cast<int>(static_cast<long long>(T) * (vc + 1) / G);
            for (int t = t0 + st; t < t1; t += nst) {
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
                for (int c = 0; c < chunks; ++c) write_int4_chunk<QT>(a, f, t, slot, chunks, c);
            }
        }
        // the worker's TMA copies below read these rows: generic-proxy writes ordered before
        // async-proxy reads, across the worker's warps
        fence_proxy_async_global();
        if (wps == 1) {
            __syncwarp();
        } else {
            asm volatile("bar.sync %0, %1;" ::"r"(1 + set), "r"(nst) : "memory");
        }
        fence_proxy_async_global();
    }
    if (s_begin >= s_end) return;
    const int s0 = static_cast<int>(s_begin), s1 = static_cast<int>(s_end);

    // ---------------------------------------------------------------- the warp's own producer
    // Issues stage ps into slot p_slot: one K and one V box per block of the stage.  Per-item
    // values are recomputed only when the item changes; lanes hold the block ids of 32
    // consecutive logical blocks of the current item.
    const uint32_t stage_tx = 2u * BPS * kp.box_bytes;
    int ps = s0, p_slot = 0, p_item = item0 - 1, p_end = s0;  // p_end: first stage past p_item
    int p_row = 0, p_head = 0, p_nblk = 0, p_lb = 0;          // table row, kv head, blocks, next block
    int cache_base = 0, my_id = a.num_blocks;
    bool my_ok = false;
    auto refresh_ids = [&](int base) {
        cache_base = base;
        const int lb = base + lane;
        my_ok = false;
        my_id = a.num_blocks;  // one past the pool: a copy from there reads zeros
        if (lb < p_nblk) {
            const int e = a.block_table[static_cast<int64_t>(p_row) * a.bt_stride + lb];
            if (e >= 0 && e < a.num_blocks) {
                my_id = e;
                my_ok = true;
            } else if (wi == 0) {
                report(a.d_err, KV_DERR_BAD_BLOCK);
            }
        }
    };
    auto issue = [&]() {
        if (ps >= p_end) {  // the next item with stages
            do {
                ++p_item;
                p_end = P[p_item + 1];
            } while (p_end <= ps);
            const int seq = p_item % B, grp = p_item / B;
            const int L = Ls[seq];
            p_row = seq;
            p_head = grp * HG + h_loc;
            p_nblk = (L + bs - 1) / bs;
            p_lb = (a.window > 0 ? max(0, L - q_len - a.window + 1) : 0) / bs + (ps - P[p_item]) * BPS;
            refresh_ids(p_lb);
        } else if (p_lb + BPS > cache_base + 32) {
            refresh_ids(p_lb);
        }
        const int src0 = p_lb - cache_base;
        uint32_t mask = 0;
        int ids[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j < BPS) {
                ids[j] = __shfl_sync(0xffffffffu, my_id, src0 + j);
                if (__shfl_sync(0xffffffffu, my_ok ? 1 : 0, src0 + j)) mask |= 1u << j;
            }
        }
        if (lane == 0) {
            const uint32_t st = smem_u32(ring + static_cast<size_t>(p_slot) * stage_bytes);
            smask[p_slot] = mask;
            const uint32_t bar = smem_u32(&full_bar[p_slot]);
            mbar_arrive_expect_tx(bar, stage_tx);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (j < BPS) {
                    const int id = ((mask >> j) & 1u) ? ids[j] : a.num_blocks;
                    tma_load_4d(st + j * kp.box_stride, &tmap_k, bar, 0, 0, p_head, id);
                    tma_load_4d(st + (BPS + j) * kp.box_stride, &tmap_v, bar, 0, 0, p_head, id);
                }
            }
        }
        p_lb += BPS;
        ++ps;
        if (++p_slot == NS) p_slot = 0;
    };
    for (int i = 0; i < NS && ps < s1; ++i) issue();
    __syncwarp();

    // ---------------------------------------------------------------- consumer state
    const int c4 = lane & 3, l4 = lane >> 2;
    // ldmatrix rows of this lane in a stage: key (lane>>3 & 1)*8 + lane&7 of each 16-key chunk
    // (the same keys for K and, through the transposed load, for V)
    uint32_t koff, voff;
    int rkey;
    {
        const int tk = ((lane >> 3) & 1) * 8 + (lane & 7);
        const int jk = tk / bs, rk = tk - jk * bs;
        koff = jk * kp.box_stride + rk * kRowBytes;
        voff = (BPS + jk) * kp.box_stride + rk * kRowBytes;
        rkey = (rk >> 1) & 3;  // 64B swizzle: 16-byte chunk c of row r sits at c ^ ((r >> 1) & 3)
    }
    const int n_chunks = ST / 16;
    // the second 16-key chunk of a 32-key stage: 16 rows further down a 32-token block, or the
    // same rows of the block 16 / block_size boxes further on
    const int off16 = bs >= 32 ? 16 * kRowBytes : (16 / bs) * kp.box_stride;

    float o[kMT][kNR][4];
    float m_run[kNR][2], l_run[kNR][2];
    float q_sum[kNR][2];  // sum_d q_d of each of this lane's rows, as the MMAs see q
    uint32_t qb[kNR][kKS][2];
    int pos_hi[kNR][2];  // position of each of this lane's rows (-1: padding row)
    const float sl2 = a.scale_log2;
    const int W = a.window;

    int item = item0, seg_k0 = 0;
    int seq = 0, grp = 0, L = 0, b0 = 0, lo_last = 0, hi_first = 0, n_item = 0;
    int slot = 0;
    uint32_t phase = 0;
    bool failed = false;
    int consumed = 0;  // stages waited for and read

    auto unit = [&](const Int4Chunk (&cr)[2], auto nch_tag, auto masked_tag) {
        constexpr int NCH = decltype(nch_tag)::value;
        constexpr bool kMasked = decltype(masked_tag)::value;
        constexpr bool kSplitK = NCH == 1 && kNR == 1;

        // ---- S^T = K q^T: 16 keys x RN query rows per chunk.  One ldmatrix.x4 takes two 16-byte
        // chunks (32 dims each) of 16 keys: r[2h] keys l4, r[2h+1] keys l4 + 8, of chunk 2cp + h;
        // a register holds dims 8c4 .. 8c4+7 of its key, and k-step 2*chunk + t takes the dim
        // pairs (8c4+2t, 8c4+2t+4) and (8c4+2t+1, 8c4+2t+5), the order the q fragments follow
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
#pragma unroll
            for (int cp = 0; cp < kD / 64; ++cp) {
                const int cch = 2 * cp + (lane >> 4);
                uint32_t r[4];
                ldsm_x4(cr[j].kbase + ((cch ^ cr[j].key) << 4), r[0], r[1], r[2], r[3]);
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
        }

        // ---- scale, mask, online softmax (lane: keys l4, l4+8 of each chunk; rows 2c4, 2c4+1)
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

        // ---- O^T += V^T P^T.  A transposed-load register holds keys (2c4, 2c4+1) x dims
        // 4l4 .. 4l4+3 of one chunk, so its four pairs are key pairs at four dims; m-tile
        // 2*chunk + h2 takes dims 4l4+2h2 (accumulator rows l4) and 4l4+2h2+1 (rows l4+8).
        // Codes decode to finite values, so keys outside the attended range need no masking
        // here: their weights are exactly 0.
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
#pragma unroll
            for (int cp = 0; cp < kD / 64; ++cp) {
                const int cch = 2 * cp + (lane >> 4);
                uint32_t r[4];
                ldsm_x4_t(cr[j].vbase + ((cch ^ cr[j].key) << 4), r[0], r[1], r[2], r[3]);
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
        }
    };

    int item_begin = P[item0], item_end = P[item0 + 1];
    for (int s = s0; s < s1; ++s) {
        if (s >= item_end) {
            do {
                ++item;
                item_begin = item_end;
                item_end = P[item + 1];
            } while (item_end <= s);
        }
        const int k = s - item_begin;
        if (s == s0 || k == 0) {
            // ------------------------------------------------ a new piece of a sequence
            seg_k0 = k;
            seq = item % B;
            grp = item / B;
            L = Ls[seq];
            n_item = item_end - item_begin;
            const int key_lo = a.window > 0 ? max(0, L - q_len - a.window + 1) : 0;
            b0 = key_lo / bs;
            lo_last = a.window > 0 ? max(0, L - a.window) : 0;
            hi_first = L - q_len;
            const int hkv = grp * HG + h_loc;
            const float *ksc = a.k_gscales + static_cast<int64_t>(hkv) * (kD >> gshift);
#pragma unroll
            for (int nt = 0; nt < kNR; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = rt * RN + nt * 8 + 2 * c4 + e;
                    pos_hi[nt][e] = r < R ? L - q_len + r / g : -1;
                    m_run[nt][e] = -INFINITY;
                    l_run[nt][e] = 0.f;
                }
                // q as the B operand (column = query row l4): dims (d, d + 4) with
                // d = 32*(ks/2) + 8c4 + 2(ks&1) + hf, times their K scales; odd dims (hf 1) meet
                // codes in units of 2^-20, so they take 1/16
                const int rq = rt * RN + nt * 8 + l4;
                const QT *qrow = nullptr;
                if (rq < R) {
                    const int64_t tok = static_cast<int64_t>(seq) * q_len + rq / g;
                    qrow = static_cast<const QT *>(a.q) + (tok * a.num_q_heads + hkv * g + rq % g) * kD;
                }
                float qs = 0.f;
#pragma unroll
                for (int ks = 0; ks < kKS; ++ks) {
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int d = 32 * (ks >> 1) + 8 * c4 + 2 * (ks & 1) + hf;
                        const float f = hf ? 0.0625f : 1.f;
                        uint32_t v = 0;
                        if (qrow)
                            v = pack2<MT>(to_float<QT>(qrow[d]) * ksc[d >> gshift] * f,
                                          to_float<QT>(qrow[d + 4]) * ksc[(d + 4) >> gshift] * f);
                        qb[nt][ks][hf] = v;
                        const float2 u = unpack2<MT>(v);
                        qs += (u.x + u.y) * (hf ? 16.f : 1.f);
                    }
                }
                qs += __shfl_xor_sync(0xffffffffu, qs, 1);
                qs += __shfl_xor_sync(0xffffffffu, qs, 2);
                // row l4 of the tile has its sum in lanes 4*l4 ..; this lane's rows are 2c4 + e
                q_sum[nt][0] = __shfl_sync(0xffffffffu, qs, 8 * c4);
                q_sum[nt][1] = __shfl_sync(0xffffffffu, qs, 8 * c4 + 4);
#pragma unroll
                for (int mt = 0; mt < kMT; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
            }
        }

        // a unit is 32 keys when possible: the next stage of the same piece joins a 16-key one
        const bool two = n_chunks == 1 && NS >= 2 && s + 1 < s1 && k + 1 < n_item;
        const int slot2 = slot + 1 == NS ? 0 : slot + 1;
        const uint32_t phase2 = slot + 1 == NS ? phase ^ 1u : phase;
        bool landed = mbar_wait_sleep(smem_u32(&full_bar[slot]), phase);
        if (two) landed = landed && mbar_wait_sleep(smem_u32(&full_bar[slot2]), phase2);
        if (!__all_sync(0xffffffffu, landed)) {  // the warp gives up together
            if (lane == 0) report(a.d_err, KV_DERR_TIMEOUT);
            failed = true;
            break;
        }
        const uint32_t full_mask = (1u << BPS) - 1u;
        Int4Chunk cr[2];
        {
            const uint32_t st0 = smem_u32(ring + static_cast<size_t>(slot) * stage_bytes);
            const int tok0 = (b0 + k * BPS) * bs;
            cr[0] = Int4Chunk{st0 + koff, st0 + voff, rkey, tok0, tok0, smask[slot]};
            if (two) {
                const uint32_t st1 = smem_u32(ring + static_cast<size_t>(slot2) * stage_bytes);
                const int tok1 = (b0 + (k + 1) * BPS) * bs;
                cr[1] = Int4Chunk{st1 + koff, st1 + voff, rkey, tok1, tok1, smask[slot2]};
            } else {  // a 32-key stage
                cr[1] = Int4Chunk{st0 + koff + off16, st0 + voff + off16, rkey, tok0 + 16, tok0, smask[slot]};
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
        // every lane's reads of the consumed slots are done: order them before the copies that
        // refill those slots
        fence_proxy_async_shared();
        __syncwarp();
        const int used = two ? 2 : 1;
        consumed += used;
        for (int u = 0; u < used; ++u) {
            if (ps < s1) issue();
            if (++slot == NS) {
                slot = 0;
                phase ^= 1u;
            }
        }
        __syncwarp();
        const int k_last = k + used - 1;
        s += used - 1;  // the loop's ++s moves past the unit

        // ------------------------------------------------ end of a piece: write it out
        if (k_last == n_item - 1 || s == s1 - 1) {
            const bool whole = seg_k0 == 0 && k_last == n_item - 1;
            const int hkv = grp * HG + h_loc;
            const float *vsc = a.v_gscales + static_cast<int64_t>(hkv) * (kD >> gshift);
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
                    const float inv = l > 0.f ? 1.f / l : 0.f;
                    const float lse = l > 0.f ? (m_run[nt][e] + log2f(l)) * 0.69314718055994531f -
                                                    a.lse_offset_scale * q_sum[nt][e]
                                              : -INFINITY;
                    const int64_t tokq = static_cast<int64_t>(seq) * q_len + r / g;
                    const int64_t rowid = tokq * a.num_q_heads + hkv * g + r % g;
                    const int64_t wrow = static_cast<int64_t>(item + vc) * kp.rows_per_item + h_loc * R + r;
#pragma unroll
                    for (int mt = 0; mt < kMT; ++mt) {
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            // dim of accumulator row l4 (hf 0) / l4+8 (hf 1) of m-tile mt
                            const int d = (mt >> 1) * 32 + 4 * l4 + 2 * (mt & 1) + hf;
                            const float unit_scale = hf ? 1048576.f : 16777216.f;  // 2^20, 2^24
                            const float v =
                                l > 0.f ? vsc[d >> gshift] * fmaf(o[mt][nt][2 * hf + e] * unit_scale, inv, -8.f) : 0.f;
                            if (whole) static_cast<QT *>(a.out)[rowid * kD + d] = from_float<QT>(v);
                            else a.ws_o[wrow * kD + d] = v;
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
    // never leave with copies in flight into this warp's ring (only after a timed-out wait): the
    // stages issued but not consumed sit in the slots from the current one on, one phase each
    if (failed && lane == 0) {
        int sl = slot;
        uint32_t ph = phase;
        for (int i = 0; i < (ps - s0) - consumed; ++i) {
            (void)mbar_wait_bounded(smem_u32(&full_bar[sl]), ph);
            if (++sl == NS) {
                sl = 0;
                ph ^= 1u;
            }
        }
    }
}

template <typename QT, int RN, bool kFused, int kBS>
cudaError_t launch_int4_typed(const CUtensorMap &tk, const CUtensorMap &tv, const KernelParams &kp,
                              const DecodePlan &plan, int q_dtype, cudaStream_t stream) {
    auto kern = paged_decode_int4_kernel<QT, RN, kFused, kBS>;
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
        if (r != cudaSuccess) (void)cudaGetLastError();
        attr_status[dev] = r;
    });
    if (attr_status[dev] != cudaSuccess) return attr_status[dev];
    kern<<<plan.num_ctas, Int4Launch<RN>::kThreads, plan.smem_bytes, stream>>>(tk, tv, kp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_lse_merge(kp, kp.num_workers, q_dtype, stream);
}

}  // namespace

int int4_decode_warps(int rows_per_warp) {
    return rows_per_warp == 8 ? Int4Launch<8>::kWarps : Int4Launch<16>::kWarps;
}

template <bool kFused>
static cudaError_t launch_int4_any(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v, const DecodeArgs &a,
                                   const StepArgs &f, const DecodePlan &plan, int q_dtype, cudaStream_t stream) {
    if (a.num_seqs == 0) return cudaSuccess;
    KernelParams kp;
    kp.a = a;
    kp.f = f;
    kp.heads_per_cta = plan.heads_per_cta;
    kp.warps_per_head = plan.warps_per_head;
    kp.blocks_per_stage = plan.blocks_per_stage;
    kp.num_stages = plan.num_stages;
    kp.box_bytes = plan.box_bytes;
    kp.box_stride = plan.box_stride;
    kp.num_items = plan.num_items;
    kp.rows_per_item = plan.rows_per_item;
    kp.sets_per_cta = plan.sets_per_cta;
    kp.num_workers = plan.num_workers;
    kp.tile_ws = 0;
    kp.item_cost = 0;
    kp.lens_smem = 1;
    const bool f16 = q_dtype == KV_F16;
    if (plan.rows_per_warp == 8) {
        // 8-row tiles: the block size as a compile-time constant where stages hold 32 keys
        switch (a.block_size) {
            case 8:
                return f16 ? launch_int4_typed<__half, 8, kFused, 8>(tmap_k, tmap_v, kp, plan, q_dtype, stream)
                           : launch_int4_typed<__nv_bfloat16, 8, kFused, 8>(tmap_k, tmap_v, kp, plan, q_dtype, stream);
            case 16:
                return f16 ? launch_int4_typed<__half, 8, kFused, 16>(tmap_k, tmap_v, kp, plan, q_dtype, stream)
                           : launch_int4_typed<__nv_bfloat16, 8, kFused, 16>(tmap_k, tmap_v, kp, plan, q_dtype, stream);
            case 32:
                return f16 ? launch_int4_typed<__half, 8, kFused, 32>(tmap_k, tmap_v, kp, plan, q_dtype, stream)
                           : launch_int4_typed<__nv_bfloat16, 8, kFused, 32>(tmap_k, tmap_v, kp, plan, q_dtype, stream);
            default:
                return f16 ? launch_int4_typed<__half, 8, kFused, 0>(tmap_k, tmap_v, kp, plan, q_dtype, stream)
                           : launch_int4_typed<__nv_bfloat16, 8, kFused, 0>(tmap_k, tmap_v, kp, plan, q_dtype, stream);
        }
    }
    return f16 ? launch_int4_typed<__half, 16, kFused, 0>(tmap_k, tmap_v, kp, plan, q_dtype, stream)
               : launch_int4_typed<__nv_bfloat16, 16, kFused, 0>(tmap_k, tmap_v, kp, plan, q_dtype, stream);
}

cudaError_t launch_paged_decode_int4(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                                     const DecodeArgs &a, const DecodePlan &plan, int q_dtype,
                                     cudaStream_t stream) {
    return launch_int4_any<false>(tmap_k, tmap_v, a, StepArgs{}, plan, q_dtype, stream);
}

cudaError_t launch_decode_step_int4(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                                    const DecodeArgs &a, const StepArgs &f, const DecodePlan &plan,
                                    int q_dtype, cudaStream_t stream) {
    return launch_int4_any<true>(tmap_k, tmap_v, a, f, plan, q_dtype, stream);
}

}  // namespace pkv
