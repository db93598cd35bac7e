// Host side of the paged decode over 16-bit and E4M3 caches: parameters, the 16-bit
// instantiations of the kernel (paged_decode_kernel.cuh) and the row merge launcher of the INT4
// kernel.  The E4M3 instantiations are in paged_attention_fp8.cu.
#include "paged_decode_kernel.cuh"

namespace pkv {

cudaError_t launch_lse_merge(const KernelParams &kp, int num_workers, int q_dtype, cudaStream_t stream) {
    const bool d64 = kp.a.head_dim == 64;
    if (q_dtype == KV_F16)
        return d64 ? row_merge<__half, 64>(kp, num_workers, stream) : row_merge<__half, 128>(kp, num_workers, stream);
    return d64 ? row_merge<__nv_bfloat16, 64>(kp, num_workers, stream)
               : row_merge<__nv_bfloat16, 128>(kp, num_workers, stream);
}

template <bool kFused>
static cudaError_t launch_any(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                              const KernelParams &kp, const DecodePlan &plan, int q_dtype,
                              int cache_dtype, cudaStream_t stream) {
    const bool f16 = q_dtype == KV_F16;
    if (cache_dtype == KV_FP8_E4M3) return launch_rows_fp8<kFused>(tmap_k, tmap_v, kp, plan, f16, stream);
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
    kp.sets_per_cta = 1;
    kp.num_workers = plan.num_ctas;
    kp.tile_ws = plan.tile_ws;
    kp.item_cost = plan.item_cost;
    kp.lens_smem = plan.lens_smem;
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
