// Paged decode attention with split-KV and a log-sum-exp merge.
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
//   * one CTA = (partition of one sequence's keys, group of kv heads); a partition is a run of
//     whole cache blocks, and a pipeline stage is 16 or 32 tokens of it;
//   * one producer warp walks the block table and issues TMA tensor copies of whole
//     (block, head group) tiles, K and V, into a ring of shared-memory stages guarded by
//     mbarriers (expect-tx on "full", one arrival per consumer warp on "empty").  The tensor map
//     views the cache as (dim, token-in-block, head, block), so one copy lands a block's rows
//     head-major in shared memory with the 128-byte swizzle: the ldmatrix reads below are free
//     of bank conflicts;
//   * each consumer warp owns one kv head and 16 query rows of its GQA group (rows are
//     (query token, q head) pairs; q_len speculative tokens x group size); q.K^T and p.V run as
//     m16n8k16 tensor-core MMAs with float32 accumulators, softmax statistics in float32 with
//     exp2, warp-shuffle max/sum across the 4 lanes that share a row;
//   * E4M3 caches are converted to fp16 per warp in shared memory (exact), k_scale folds into
//     the score scale and v_scale into the output;
//   * sequences with one partition write the output directly; others write (o/l, lse) partials
//     to the workspace and a second kernel merges them: LSE = log sum_s exp(lse_s),
//     out = sum_s exp(lse_s - LSE) o_s.
#include <type_traits>

#include "common.cuh"
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

// Keys a sequence's queries can see start at the window of its first query token; partitions
// start at the cache block holding that key.
__host__ __device__ __forceinline__ int first_key(int L, int q_len, int window) {
    const int lo = L - q_len - window + 1;
    return window > 0 ? (lo > 0 ? lo : 0) : 0;
}

__host__ __device__ __forceinline__ bool seq_len_ok(int L, int q_len, int max_seq_len, int bs,
                                                    int max_blocks_per_seq) {
    return L >= q_len && L <= max_seq_len && (L + bs - 1) / bs <= max_blocks_per_seq;
}

__host__ __device__ __forceinline__ int seq_parts(int L, int q_len, int window, int bs,
                                                  int part_tokens) {
    const int nblk = (L + bs - 1) / bs;
    const int b0 = first_key(L, q_len, window) / bs;
    return ((nblk - b0) * bs + part_tokens - 1) / part_tokens;
}

struct KernelParams {
    DecodeArgs a;
    int heads_per_cta, m_tiles, blocks_per_stage, part_tokens, max_parts, num_stages;
    int box_bytes, box_stride;
};

template <int D> struct MaxWarps {
    static constexpr int value = D == 128 ? 8 : 12;  // consumer warps per CTA
};

template <typename QT, typename CT, int D>
__global__ void __launch_bounds__((MaxWarps<D>::value + 1) * 32, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v,
                        const __grid_constant__ KernelParams kp) {
    constexpr bool kFp8 = CacheTraits<CT>::kFp8;
    using MT = typename std::conditional<kFp8, __half, QT>::type;  // MMA operand type
    constexpr int kEB = CacheTraits<CT>::kBytes;
    constexpr int kNDB = D * kEB / 128;   // TMA boxes along head_dim per block
    constexpr int kNDB16 = D * 2 / 128;   // 128-byte row segments of a 16-bit row
    constexpr int kKS = D / 16;           // k-steps of q.K^T
    constexpr int kNT = D / 8;            // n-tiles of p.V

    const DecodeArgs &a = kp.a;
    const int part = blockIdx.x, b = blockIdx.y, hgrp = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int HG = kp.heads_per_cta, MTL = kp.m_tiles;
    const int ncw = HG * MTL;
    const int bs = a.block_size, BPS = kp.blocks_per_stage, ST = BPS * bs, NS = kp.num_stages;
    const int g = a.num_q_heads / a.num_kv_heads;
    const int R = g * a.q_len;

    const int L = a.seq_lens[b];
    const bool len_ok = seq_len_ok(L, a.q_len, a.max_seq_len, bs, a.max_blocks_per_seq);
    int nparts = 1, blk_begin = 0, blk_end = 0;
    if (len_ok) {
        nparts = seq_parts(L, a.q_len, a.window, bs, kp.part_tokens);
        const int b0 = first_key(L, a.q_len, a.window) / bs;
        const int nblk = (L + bs - 1) / bs;
        blk_begin = b0 + part * (kp.part_tokens / bs);
        blk_end = min(nblk, blk_begin + kp.part_tokens / bs);
    } else if (part == 0 && hgrp == 0 && threadIdx.x == 0) {
        report(a.d_err, KV_DERR_BAD_LEN);
    }
    if (part >= nparts) return;
    const int n_stages = len_ok ? (blk_end - blk_begin + BPS - 1) / BPS : 0;

    // ---------------------------------------------------------------- shared memory carve-up
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int stage_bytes = 2 * BPS * kNDB * kp.box_stride;
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + NS * stage_bytes);
    uint64_t *empty_bar = full_bar + NS;
    uint32_t *stage_mask = reinterpret_cast<uint32_t *>(empty_bar + NS);
    volatile uint32_t *abort_flag = stage_mask + NS;
    uint8_t *scratch = smem + ((NS * stage_bytes + 16 * NS + 4 * NS + 4 + 1023) & ~1023);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), ncw);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    // ================================================================ producer warp
    if (warp == ncw) {
        if (lane == 0 && n_stages > 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
            const int32_t *row = a.block_table + static_cast<int64_t>(b) * a.bt_stride;
            const uint32_t tx = 2u * BPS * kNDB * kp.box_bytes;
            int issued = 0;
            for (int i = 0; i < n_stages; ++i) {
                const int slot = i % NS;
                if (i >= NS) {
                    if (!mbar_wait_bounded(smem_u32(&empty_bar[slot]), ((i / NS) + 1) & 1)) {
                        report(a.d_err, KV_DERR_TIMEOUT);
                        *abort_flag = 1;
                        break;
                    }
                }
                if (*abort_flag) break;
                uint8_t *stage = smem + slot * stage_bytes;
                // validate this stage's block ids first: the mask must be stored before the
                // arrival that publishes the stage
                uint32_t mask = 0;
                for (int j = 0; j < BPS; ++j) {
                    const int lb = blk_begin + i * BPS + j;
                    if (lb < blk_end) {
                        const int e = row[lb];
                        if (e >= 0 && e < a.num_blocks) mask |= 1u << j;
                        else report(a.d_err, KV_DERR_BAD_BLOCK);
                    }
                }
                stage_mask[slot] = mask;
                const uint32_t bar = smem_u32(&full_bar[slot]);
                mbar_arrive_expect_tx(bar, tx);
                for (int j = 0; j < BPS; ++j) {
                    // invalid or past-the-end blocks copy from one past the pool: zeros
                    const int id = ((mask >> j) & 1u) ? row[blk_begin + i * BPS + j] : a.num_blocks;
                    for (int db = 0; db < kNDB; ++db) {
                        const uint32_t dk = smem_u32(stage + ((0 * BPS + j) * kNDB + db) * kp.box_stride);
                        const uint32_t dv = smem_u32(stage + ((1 * BPS + j) * kNDB + db) * kp.box_stride);
                        tma_load_4d(dk, &tmap_k, bar, db * (128 / kEB), 0, hgrp * HG, id);
                        tma_load_4d(dv, &tmap_v, bar, db * (128 / kEB), 0, hgrp * HG, id);
                    }
                }
                ++issued;
            }
            // never leave with copies in flight into this CTA's shared memory
            for (int i = max(0, issued - NS); i < issued; ++i)
                if (!mbar_wait_bounded(smem_u32(&full_bar[i % NS]), (i / NS) & 1))
                    report(a.d_err, KV_DERR_TIMEOUT);
        }
        return;
    }

    // ================================================================ consumer warps
    const int h_loc = warp / MTL, mt = warp % MTL;
    const int hkv = hgrp * HG + h_loc;
    const int q_len = a.q_len;
    const int r0 = mt * 16 + (lane >> 2), r1 = r0 + 8;

    // query rows of this lane: row r = (query token r / g, q head hkv*g + r % g)
    int pos_hi[2], pos_lo[2];
    const QT *qrow[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int r = k ? r1 : r0;
        if (r < R && len_ok) {
            const int qi = r / g;
            const int p = L - q_len + qi;
            pos_hi[k] = p;
            pos_lo[k] = a.window > 0 ? max(0, p - a.window + 1) : 0;
            const int64_t tok = static_cast<int64_t>(b) * q_len + qi;
            qrow[k] = static_cast<const QT *>(a.q) + (tok * a.num_q_heads + hkv * g + r % g) * D;
        } else {
            pos_hi[k] = -1;
            pos_lo[k] = 0;
            qrow[k] = nullptr;
        }
    }
    const int key_lo = len_ok ? first_key(L, q_len, a.window) : 0;  // first key any row sees
    const int lo_last = len_ok ? (a.window > 0 ? max(0, L - a.window) : 0) : 0;
    const int hi_first = L - q_len;  // every row sees keys <= this one

    // Q as A fragments (rows r0, r1; k = 2*(lane%4) + {0,1} and + 8)
    uint32_t qa[kKS][4];
#pragma unroll
    for (int ks = 0; ks < kKS; ++ks) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int d = ks * 16 + half * 8 + 2 * (lane & 3);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                uint32_t v = 0;
                if (qrow[k]) {
                    const float x0 = to_float<QT>(qrow[k][d]);
                    const float x1 = to_float<QT>(qrow[k][d + 1]);
                    v = pack2<MT>(x0, x1);
                }
                qa[ks][half * 2 + k] = v;
            }
        }
    }

    float o[kNT][4];
#pragma unroll
    for (int n = 0; n < kNT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    const float sl2 = a.scale_log2;

    uint8_t *my_scratch = scratch + warp * (2 * kNDB16 * ST * 128);

    for (int i = 0; i < n_stages; ++i) {
        const int slot = i % NS;
        if (!mbar_wait_bounded(smem_u32(&full_bar[slot]), (i / NS) & 1)) {
            if (lane == 0) report(a.d_err, KV_DERR_TIMEOUT);
            *abort_flag = 1;
            break;
        }
        const uint32_t mask = stage_mask[slot];
        const int stage_tok0 = (blk_begin + i * BPS) * bs;
        const uint8_t *stage = smem + slot * stage_bytes;

        // 16-bit view of this head's K and V rows: base of (tensor, segment) and row index of
        // stage token tt.  Native 16-bit caches read the TMA boxes in place; E4M3 caches are
        // first widened to fp16 into this warp's scratch, laid out as one box per segment.
        if constexpr (kFp8) {
#pragma unroll
            for (int tn = 0; tn < 2; ++tn) {
                for (int item = lane; item < ST * 2; item += 32) {
                    const int tt = item >> 1, hf = item & 1;
                    const int j = tt / bs, t = tt - j * bs;
                    const int srow = h_loc * bs + t;
                    const uint8_t *src = stage + ((tn * BPS + j) * kNDB) * kp.box_stride + srow * 128;
                    uint8_t *dst = my_scratch + (tn * kNDB16 + hf) * ST * 128 + tt * 128;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int sc = hf * 4 + c;
                        const uint4 raw = *reinterpret_cast<const uint4 *>(src + ((sc ^ (srow & 7)) << 4));
                        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
                        uint32_t hv[8];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(
                                static_cast<__nv_fp8x2_storage_t>(w[u] & 0xffffu), __NV_E4M3);
                            const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(
                                static_cast<__nv_fp8x2_storage_t>(w[u] >> 16), __NV_E4M3);
                            hv[2 * u] = static_cast<uint32_t>(lo.x) | (static_cast<uint32_t>(lo.y) << 16);
                            hv[2 * u + 1] = static_cast<uint32_t>(hi.x) | (static_cast<uint32_t>(hi.y) << 16);
                        }
                        *reinterpret_cast<uint4 *>(dst + (((2 * c) ^ (tt & 7)) << 4)) =
                            make_uint4(hv[0], hv[1], hv[2], hv[3]);
                        *reinterpret_cast<uint4 *>(dst + (((2 * c + 1) ^ (tt & 7)) << 4)) =
                            make_uint4(hv[4], hv[5], hv[6], hv[7]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
        }

        for (int ck = 0; ck < ST / 16; ++ck) {
            const int c0 = stage_tok0 + ck * 16;  // absolute index of the chunk's first key
            // rows (within the 16-bit view) that this lane addresses in ldmatrix
            const int ttk = ck * 16 + ((lane >> 4) << 3) + (lane & 7);
            const int ttv = ck * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
            uint32_t kbase, vbase;
            int kkey, vkey, seg_stride;
            if constexpr (kFp8) {
                kbase = smem_u32(my_scratch) + ttk * 128;
                vbase = smem_u32(my_scratch + kNDB16 * ST * 128) + ttv * 128;
                kkey = ttk & 7;
                vkey = ttv & 7;
                seg_stride = ST * 128;
            } else {
                const int jk = ttk / bs, tk = ttk - jk * bs;
                const int jv = ttv / bs, tv = ttv - jv * bs;
                kbase = smem_u32(stage + (jk * kNDB) * kp.box_stride) + (h_loc * bs + tk) * 128;
                vbase = smem_u32(stage + ((BPS + jv) * kNDB) * kp.box_stride) + (h_loc * bs + tv) * 128;
                kkey = (h_loc * bs + tk) & 7;
                vkey = (h_loc * bs + tv) & 7;
                seg_stride = kp.box_stride;
            }

            // ---- s = q . K^T for 16 keys (two n-tiles of 8)
            float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int ks = 0; ks < kKS; ++ks) {
                const int seg = ks >> 2;
                const int chunk = ((ks & 3) << 1) + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kbase + seg * seg_stride + ((chunk ^ kkey) << 4), b0, b1, b2, b3);
                MmaOp<MT>::run(s[0], qa[ks], b0, b1);
                MmaOp<MT>::run(s[1], qa[ks], b2, b3);
            }

            // ---- scale, mask, online softmax
            const uint32_t full_mask = (1u << BPS) - 1u;
            const bool need_mask = (c0 < lo_last) || (c0 + 15 > hi_first) || (mask != full_mask);
            float x[2][4];
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float v = s[n][e] * sl2;
                    if (need_mask) {
                        const int tok = c0 + n * 8 + 2 * (lane & 3) + (e & 1);
                        const int k = e >> 1;
                        const bool blk_ok = (mask >> ((tok - stage_tok0) / bs)) & 1u;
                        const bool ok = blk_ok && tok >= pos_lo[k] && tok <= pos_hi[k];
                        v = ok ? v : -INFINITY;
                    }
                    x[n][e] = v;
                }
            float alpha[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                float mx = fmaxf(fmaxf(x[0][2 * k], x[0][2 * k + 1]), fmaxf(x[1][2 * k], x[1][2 * k + 1]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(m_run[k], mx);
                const float ref = m_new == -INFINITY ? 0.f : m_new;
                alpha[k] = fast_exp2(m_run[k] - ref);
                m_run[k] = m_new;
#pragma unroll
                for (int n = 0; n < 2; ++n) {
                    x[n][2 * k] = fast_exp2(x[n][2 * k] - ref);
                    x[n][2 * k + 1] = fast_exp2(x[n][2 * k + 1] - ref);
                }
            }
            // p as the A fragment of p.V (keys of n-tile 0 then n-tile 1)
            uint32_t pa[4];
            pa[0] = pack2<MT>(x[0][0], x[0][1]);
            pa[1] = pack2<MT>(x[0][2], x[0][3]);
            pa[2] = pack2<MT>(x[1][0], x[1][1]);
            pa[3] = pack2<MT>(x[1][2], x[1][3]);
            // the normaliser sums the rounded weights the MMA actually uses, so the output is
            // an exact weighted average of V up to the accumulation order
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const float2 u = unpack2<MT>(pa[k]), w = unpack2<MT>(pa[k + 2]);
                l_run[k] = l_run[k] * alpha[k] + ((u.x + u.y) + (w.x + w.y));
            }
#pragma unroll
            for (int n = 0; n < kNT; ++n) {
                o[n][0] *= alpha[0];
                o[n][1] *= alpha[0];
                o[n][2] *= alpha[1];
                o[n][3] *= alpha[1];
            }

            // keys whose V rows may hold anything (past the sequence, before the window, or in
            // a block that failed validation) get their V elements zeroed, so 0 * NaN never
            // reaches the accumulators
            uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;
            if (need_mask) {
                const int tk0 = c0 + 2 * (lane & 3);
                uint32_t keep[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = tk0 + (e >> 1) * 8 + (e & 1);
                    const bool blk_ok = (mask >> ((tok - stage_tok0) / bs)) & 1u;
                    keep[e] = (blk_ok && tok >= key_lo && tok < L) ? 0xffffu : 0u;
                }
                keep_lo = keep[0] | (keep[1] << 16);
                keep_hi = keep[2] | (keep[3] << 16);
            }

            // ---- o += p . V (V rows are keys, columns are head_dim)
#pragma unroll
            for (int np = 0; np < kNT / 2; ++np) {
                const int seg = np >> 2;
                const int chunk = ((np & 3) << 1) + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vbase + seg * seg_stride + ((chunk ^ vkey) << 4), b0, b1, b2, b3);
                b0 &= keep_lo;
                b1 &= keep_hi;
                b2 &= keep_lo;
                b3 &= keep_hi;
                MmaOp<MT>::run(o[2 * np], pa, b0, b1);
                MmaOp<MT>::run(o[2 * np + 1], pa, b2, b3);
            }
        }
        if constexpr (!kFp8) {
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
        }
    }

    // ---------------------------------------------------------------- epilogue
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        l_run[k] += __shfl_xor_sync(0xffffffffu, l_run[k], 1);
        l_run[k] += __shfl_xor_sync(0xffffffffu, l_run[k], 2);
    }
    const bool single = nparts == 1;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int r = k ? r1 : r0;
        if (r >= R) continue;
        const int qi = r / g;
        const int64_t tok = static_cast<int64_t>(b) * q_len + qi;
        const int64_t rowid = tok * a.num_q_heads + hkv * g + r % g;
        const float l = l_run[k];
        const float inv = l > 0.f ? a.v_scale / l : 0.f;
        const float lse = l > 0.f ? (m_run[k] + log2f(l)) * 0.69314718055994531f : -INFINITY;
        if (single) {
            QT *orow = static_cast<QT *>(a.out) + rowid * D;
#pragma unroll
            for (int n = 0; n < kNT; ++n) {
                const int d = n * 8 + 2 * (lane & 3);
                const float v0 = o[n][2 * k] * inv, v1 = o[n][2 * k + 1] * inv;
                *reinterpret_cast<uint32_t *>(orow + d) = pack2<QT>(v0, v1);
            }
            if (a.lse_out && (lane & 3) == 0) a.lse_out[rowid] = lse;
        } else {
            float *wrow = a.ws_o + (rowid * kp.max_parts + part) * D;
#pragma unroll
            for (int n = 0; n < kNT; ++n) {
                const int d = n * 8 + 2 * (lane & 3);
                *reinterpret_cast<float2 *>(wrow + d) = make_float2(o[n][2 * k] * inv, o[n][2 * k + 1] * inv);
            }
            if ((lane & 3) == 0) a.ws_lse[rowid * kp.max_parts + part] = lse;
        }
    }
}

// One warp per query row (token, q head) of a split sequence: merge the partitions' (o_s, lse_s)
// by log-sum-exp.
template <typename QT, int D>
__global__ void lse_merge_kernel(const __grid_constant__ KernelParams kp) {
    const DecodeArgs &a = kp.a;
    const int64_t rows = static_cast<int64_t>(a.num_seqs) * a.q_len * a.num_q_heads;
    const int64_t rowid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (rowid >= rows) return;
    const int b = static_cast<int>(rowid / (static_cast<int64_t>(a.q_len) * a.num_q_heads));
    const int L = a.seq_lens[b];
    if (!seq_len_ok(L, a.q_len, a.max_seq_len, a.block_size, a.max_blocks_per_seq)) return;
    const int nparts = seq_parts(L, a.q_len, a.window, a.block_size, kp.part_tokens);
    if (nparts <= 1) return;
    const float *lse_s = a.ws_lse + rowid * kp.max_parts;
    float mx = -INFINITY;
    for (int s = lane; s < nparts; s += 32) mx = fmaxf(mx, lse_s[s]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    constexpr int kPer = D / 32;  // dims per lane
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    if (mx != -INFINITY) {
        for (int s = 0; s < nparts; ++s) {
            const float w = expf(lse_s[s] - mx);
            wsum += w;
            const float *src = a.ws_o + (rowid * kp.max_parts + s) * D + lane * kPer;
#pragma unroll
            for (int e = 0; e < kPer; ++e) acc[e] += w * src[e];
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    QT *orow = static_cast<QT *>(a.out) + rowid * D + lane * kPer;
#pragma unroll
    for (int e = 0; e < kPer; e += 2)
        *reinterpret_cast<uint32_t *>(orow + e) = pack2<QT>(acc[e] * inv, acc[e + 1] * inv);
    if (a.lse_out && lane == 0) a.lse_out[rowid] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

template <typename QT, typename CT, int D>
static cudaError_t launch_typed(const CUtensorMap &tk, const CUtensorMap &tv, const KernelParams &kp,
                                const DecodePlan &plan, cudaStream_t stream) {
    auto kern = paged_decode_kernel<QT, CT, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(plan.smem_bytes));
    if (e != cudaSuccess) return e;
    const int groups = kp.a.num_kv_heads / plan.heads_per_cta;
    dim3 grid(plan.max_parts, kp.a.num_seqs, groups);
    kern<<<grid, plan.threads, plan.smem_bytes, stream>>>(tk, tv, kp);
    e = cudaGetLastError();
    if (e != cudaSuccess || plan.max_parts <= 1) return e;
    const int64_t rows = static_cast<int64_t>(kp.a.num_seqs) * kp.a.q_len * kp.a.num_q_heads;
    const int threads = 256;
    const int64_t blocks = (rows * 32 + threads - 1) / threads;
    lse_merge_kernel<QT, D><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(kp);
    return cudaGetLastError();
}

cudaError_t launch_paged_decode(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                                const DecodeArgs &a, const DecodePlan &plan, int q_dtype,
                                int cache_dtype, cudaStream_t stream) {
    if (a.num_seqs == 0) return cudaSuccess;
    KernelParams kp;
    kp.a = a;
    kp.heads_per_cta = plan.heads_per_cta;
    kp.m_tiles = plan.m_tiles;
    kp.blocks_per_stage = plan.blocks_per_stage;
    kp.part_tokens = plan.part_tokens;
    kp.max_parts = plan.max_parts;
    kp.num_stages = plan.num_stages;
    kp.box_bytes = plan.box_bytes;
    kp.box_stride = plan.box_stride;
    const bool f16 = q_dtype == KV_F16;
    if (cache_dtype == KV_FP8_E4M3) {
        return f16 ? launch_typed<__half, Fp8E4M3, 128>(tmap_k, tmap_v, kp, plan, stream)
                   : launch_typed<__nv_bfloat16, Fp8E4M3, 128>(tmap_k, tmap_v, kp, plan, stream);
    }
    if (a.head_dim == 64)
        return f16 ? launch_typed<__half, __half, 64>(tmap_k, tmap_v, kp, plan, stream)
                   : launch_typed<__nv_bfloat16, __nv_bfloat16, 64>(tmap_k, tmap_v, kp, plan, stream);
    return f16 ? launch_typed<__half, __half, 128>(tmap_k, tmap_v, kp, plan, stream)
               : launch_typed<__nv_bfloat16, __nv_bfloat16, 128>(tmap_k, tmap_v, kp, plan, stream);
}

}  // namespace pkv
