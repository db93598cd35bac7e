// Pieces shared by the decode kernels (paged_decode_kernel.cuh, paged_decode_int4.cu): launch
// parameters, the stream-K schedule over (head group, sequence, stage) and the log-sum-exp merge
// of sequences whose stages were split between workers ("Understanding PageAttention Memory
// Optimization", section "Handling Softmax Across Blocks": the softmax needs every block, so
// partial results carry their own maximum and sum and are combined exactly).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace pkv {

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
    int sets_per_cta;      // INT4 kernel: independent warp sets (stream-K workers) per CTA
    int num_workers;       // INT4 kernel: stream-K workers in all (the shares the stages are cut in)
    int tile_ws;           // 16-bit / E4M3 kernel: partial results as fragment tiles (every row of a
                           // consumer warp's tile is a query row); else one workspace row per query row
    int item_cost;         // 16-bit / E4M3 kernel: a piece's fixed cost in quarter stages (shares are cut
                           // by stages plus this per item); 0: equal stage counts
    int lens_smem;         // 16-bit / E4M3 kernel: the length table is in shared memory (it fits
                           // without costing the ring a stage); else lengths are read from seq_lens
};

// The CTA that owns flat stage s when S stages are split into G equal shares
// (CTA c owns [c*S/G, (c+1)*S/G)).
__host__ __device__ __forceinline__ int owner_cta(long long s, long long S, int G) {
    return static_cast<int>(((s + 1) * G - 1) / S);
}

// Shares actually cut from S stages by G workers: at most G, and few enough that a share holds
// at least kMinShareStages stages (one when S is smaller).  Small batches are then cut into a few
// pieces of several stages rather than one per stage (each piece costs its own output and a
// place in the merge), no share is empty and the merge never walks empty shares.
constexpr int kMinShareStages = 4;
__host__ __device__ __forceinline__ int active_shares(long long S, int G) {
    const long long by_work = S >= kMinShareStages ? S / kMinShareStages : (S > 0 ? 1 : 0);
    return by_work < G ? static_cast<int>(by_work) : G;
}

// First stage of worker w's share (S for a worker without one); its share ends where worker
// w + 1's begins.
__host__ __device__ __forceinline__ long long share_begin(long long S, int A, int w) {
    return w < A ? S * w / A : S;
}

// The first stage at or past cost position x when item i costs h quarter stages of fixed cost
// followed by its stages at 4 quarters each (item i starts at cost 4 * P[i] + h * i): the number
// of stages whose start cost lies below x.  P is the stage prefix of NI items.
__device__ __forceinline__ long long stage_at_cost(long long x, const int32_t *P, int NI, int h) {
    int lo = 0, hi = NI;  // the last item starting at or before x
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (4LL * P[mid] + static_cast<long long>(h) * mid <= x) lo = mid;
        else hi = mid - 1;
    }
    if (lo == NI) return P[NI];
    const long long past = x - (4LL * P[lo] + static_cast<long long>(h) * lo) - h;
    const long long k = past <= 0 ? 0 : (past + 3) / 4;
    const long long n = P[lo + 1] - P[lo];
    return P[lo] + (k < n ? k : n);
}

// The share [*b, *e) of worker w of G over the S stages of the NI items: equal costs of stages
// plus item_cost quarter stages a piece (no share empty), or, when shares that small could be
// empty (or an item has no stages), min(G, S) equal stage counts.
__device__ __forceinline__ void share_of(int w, int G, const int32_t *P, int NI, int item_cost, bool any_empty,
                                         long long *b, long long *e) {
    const long long S = P[NI];
    const long long C = 4 * S + static_cast<long long>(item_cost) * NI;
    if (item_cost > 0 && !any_empty && C / G >= item_cost + 8) {
        *b = stage_at_cost(C * w / G, P, NI, item_cost);
        *e = stage_at_cost(C * (w + 1) / G, P, NI, item_cost);
    } else {
        const int A = active_shares(S, G);
        *b = share_begin(S, A, w);
        *e = share_begin(S, A, w + 1);
    }
}

// The length of sequence b when it is accepted (at least q_len, at most max_seq_len, within the
// block table), else -1.
__device__ __forceinline__ int checked_len(const DecodeArgs &a, int b) {
    const int L = a.seq_lens[b];
    const bool ok = L >= a.q_len && L <= a.max_seq_len &&
                    (L + a.block_size - 1) / a.block_size <= a.max_blocks_per_seq;
    return ok ? L : -1;
}

// Per-CTA schedule, computed by every thread of the block (it contains __syncthreads):
//   Ls[b]  the length of sequence b, or -1 when it is rejected (KV_DERR_BAD_LEN, reported once);
//          without kLens there is no table: lengths are read from seq_lens (checked_len);
//   (returns whether some length was rejected)
//   P[i]   the number of stages of items 0 .. i-1 (an item is (head group, sequence), group-major;
//          a stage is BPS consecutive cache blocks of the attended range), P[0] = 0.
template <bool kLens = true>
__device__ __forceinline__ bool build_schedule(const DecodeArgs &a, int NI, int BPS, int32_t *Ls,
                                               int32_t *P, int32_t *warp_sums) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = a.num_seqs, q_len = a.q_len, bs = a.block_size;
    int rejected = 0;
    for (int i = threadIdx.x; i < B; i += blockDim.x) {
        const int L = checked_len(a, i);
        if (L < 0 && blockIdx.x == 0) report(a.d_err, KV_DERR_BAD_LEN);
        rejected |= L < 0 ? 1 : 0;
        if constexpr (kLens) Ls[i] = L;
    }
    const bool any_rejected = __syncthreads_or(rejected) != 0;
    // stage counts of the items (group-major, then sequence), inclusive scan into P[1..NI]
    {
        const int T = blockDim.x;
        const int per = (NI + T - 1) / T;
        const int lo = min(NI, static_cast<int>(threadIdx.x) * per), hi = min(NI, lo + per);
        // block_size and BPS are powers of two: shifts, not divisions
        const int bs_shift = __ffs(bs) - 1, bps_shift = __ffs(BPS) - 1;
        auto stages_of = [&](int seq) {  // of an item of sequence seq
            int L;
            if constexpr (kLens) L = Ls[seq];
            else L = checked_len(a, seq);
            if (L < 0) return 0;
            const int lo_key = a.window > 0 ? max(0, L - q_len - a.window + 1) : 0;
            const int nb = ((L + bs - 1) >> bs_shift) - (lo_key >> bs_shift);
            return (nb + BPS - 1) >> bps_shift;
        };
        int sum = 0;
        const int seq_lo = lo % B;
        for (int i = lo, sq = seq_lo; i < hi; ++i, sq = sq + 1 == B ? 0 : sq + 1) sum += stages_of(sq);
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
        for (int i = lo, sq = seq_lo; i < hi; ++i, sq = sq + 1 == B ? 0 : sq + 1) {
            run += stages_of(sq);
            P[i + 1] = run;
        }
    }
    __syncthreads();
    return any_rejected;  // (an item without stages is one of a rejected length)
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
    num_ctas = active_shares(S, num_ctas);
    constexpr int kPer = D / 32;
    constexpr int kFewPieces = 8;  // rows split into at most this many pieces take the short path
    QT *orow = static_cast<QT *>(a.out) + rowid * D + lane * kPer;
    if (p1 == p0) {  // rejected length: defined output
#pragma unroll
        for (int e = 0; e < kPer; ++e) orow[e] = from_float<QT>(0.f);
        if (a.lse_out && lane == 0) a.lse_out[rowid] = -INFINITY;
        return;
    }
    // the shares holding the item's first and last stage: written by the kernel, or (equal
    // stage counts) computed
    const bool owners = a.ws_pieces != nullptr;
    const int c_lo = owners ? a.ws_pieces[2 * item] : owner_cta(p0, S, num_ctas);
    const int c_hi = owners ? a.ws_pieces[2 * item + 1] : owner_cta(p1 - 1, S, num_ctas);
    if (c_lo == c_hi) return;  // one CTA covered it and wrote the output
    // with min(workers, stages) shares none is empty; kept as a guard for equal stage counts
    auto empty_share = [&](int c) { return !owners && S * c / num_ctas == S * (c + 1) / num_ctas; };
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
    float wsum = 0.f, mx = -INFINITY;
    const int n = c_hi - c_lo + 1;
    if (n <= kFewPieces) {
        // the common case: the pieces' lse (lane u holds piece u) and partial rows are all loaded
        // at once, before the weights are known, so a row costs two round trips through L2 (the
        // prefix, then everything else).  Empty shares wrote nothing and rows of weight 0 may
        // hold anything: they are selected away, never multiplied.
        const bool has = lane < n && !empty_share(c_lo + lane);
        const float lv = has ? __ldcg(a.ws_lse + static_cast<int64_t>(item + c_lo + lane) * kp.rows_per_item + rr)
                             : -INFINITY;
        float v[kFewPieces][kPer];
#pragma unroll
        for (int u = 0; u < kFewPieces; ++u) {
            const float *src = a.ws_o + (static_cast<int64_t>(item + c_lo + u) * kp.rows_per_item + rr) * D + lane * kPer;
#pragma unroll
            for (int e = 0; e < kPer; ++e) v[u][e] = u < n ? __ldcg(src + e) : 0.f;
        }
        mx = lv;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float wl = has && mx != -INFINITY ? expf(lv - mx) : 0.f;
        wsum = wl;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
#pragma unroll
        for (int u = 0; u < kFewPieces; ++u) {
            const float wu = __shfl_sync(0xffffffffu, wl, u);
#pragma unroll
            for (int e = 0; e < kPer; ++e) acc[e] += wu > 0.f ? wu * v[u][e] : 0.f;
        }
    } else {
        for (int c = c_lo + lane; c <= c_hi; c += 32)
            if (!empty_share(c)) mx = fmaxf(mx, __ldcg(a.ws_lse + static_cast<int64_t>(item + c) * kp.rows_per_item + rr));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (mx != -INFINITY) {
            // pieces 32 at a time: lane i weighs piece base + i; the partial rows are then loaded
            // four pieces at a time, every load issued before the sums use them
            for (int base = c_lo; base <= c_hi; base += 32) {
                const int c = base + lane;
                float wl = 0.f;
                if (c <= c_hi && !empty_share(c))
                    wl = expf(__ldcg(a.ws_lse + static_cast<int64_t>(item + c) * kp.rows_per_item + rr) - mx);
                float wsb = wl;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) wsb += __shfl_xor_sync(0xffffffffu, wsb, o);
                wsum += wsb;
                const int nb = min(32, c_hi - base + 1);
                for (int u0 = 0; u0 < nb; u0 += 4) {
                    float w[4], vv[4][kPer];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        w[u] = __shfl_sync(0xffffffffu, wl, (u0 + u) & 31);
                        const bool ok = u0 + u < nb && w[u] > 0.f;  // a piece of weight 0 adds nothing
                        const float *src =
                            a.ws_o + (static_cast<int64_t>(item + base + u0 + u) * kp.rows_per_item + rr) * D + lane * kPer;
#pragma unroll
                        for (int e = 0; e < kPer; ++e) vv[u][e] = ok ? __ldcg(src + e) : 0.f;
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int e = 0; e < kPer; ++e) acc[e] += w[u] * vv[u][e];
                }
            }
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
    for (int e = 0; e < kPer; e += 2)
        *reinterpret_cast<uint32_t *>(orow + e) = pack2<QT>(acc[e] * inv, acc[e + 1] * inv);
    if (a.lse_out && lane == 0) a.lse_out[rowid] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

template <typename QT, int D>
__global__ void lse_merge_kernel(const __grid_constant__ KernelParams kp, int num_ctas) {
    const int64_t rows = static_cast<int64_t>(kp.num_items) * kp.rows_per_item;
    const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (w >= rows) return;
    merge_row<QT, D>(kp, kp.a.ws_prefix, num_ctas, w, threadIdx.x & 31);
}

template <typename QT, int D>
static cudaError_t row_merge(const KernelParams &kp, int num_workers, cudaStream_t stream) {
    const int64_t rows = static_cast<int64_t>(kp.num_items) * kp.rows_per_item;
    const int threads = 256;
    const int64_t blocks = (rows * 32 + threads - 1) / threads;
    lse_merge_kernel<QT, D><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(kp, num_workers);
    return cudaGetLastError();
}

// The row merge for a finished INT4 decode launch (defined in paged_attention.cu): one warp per
// (item, row) over num_items * rows_per_item rows, num_workers the shares the stages were cut in.
// (The 16-bit and E4M3 decode kernels write their partial results as fragment tiles and have
// their own tile merge, in paged_decode_kernel.cuh.)
cudaError_t launch_lse_merge(const KernelParams &kp, int num_workers, int q_dtype, cudaStream_t stream);

}  // namespace pkv
