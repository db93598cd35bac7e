// The E4M3-cache instantiations of the paged decode kernel (paged_decode_kernel.cuh), in a
// translation unit of their own so that they compile in parallel with the 16-bit ones.
#include "paged_decode_kernel.cuh"

namespace pkv {

template <bool kFused>
cudaError_t launch_rows_fp8(const CUtensorMap &tk, const CUtensorMap &tv, const KernelParams &kp,
                            const DecodePlan &plan, bool f16, cudaStream_t stream) {
    return f16 ? launch_rows<__half, Fp8E4M3, 128, kFused>(tk, tv, kp, plan, stream)
               : launch_rows<__nv_bfloat16, Fp8E4M3, 128, kFused>(tk, tv, kp, plan, stream);
}

template cudaError_t launch_rows_fp8<false>(const CUtensorMap &, const CUtensorMap &, const KernelParams &,
                                            const DecodePlan &, bool, cudaStream_t);
template cudaError_t launch_rows_fp8<true>(const CUtensorMap &, const CUtensorMap &, const KernelParams &,
                                           const DecodePlan &, bool, cudaStream_t);

}  // namespace pkv
