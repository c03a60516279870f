// Quantised GEMV instantiations for 4-bit affine weights, groups of 32 and 64
// (kernel in k_gemv.cuh).
#include "k_gemv.cuh"

namespace sd {

cudaError_t launch_gemv_a4(const GemvArgs& a, int sm_count, cudaStream_t st) {
    cudaError_t e = gemv_detail::check_gemv(a);
    if (e != cudaSuccess) return e;
    if (a.W.kind == SD_A4G32)
        return a.nb == 1 ? gemv_detail::launch_t<SD_A4G32, 1>(a, sm_count, st) : gemv_detail::launch_t<SD_A4G32, 2>(a, sm_count, st);
    if (a.W.kind == SD_A4G64)
        return a.nb == 1 ? gemv_detail::launch_t<SD_A4G64, 1>(a, sm_count, st) : gemv_detail::launch_t<SD_A4G64, 2>(a, sm_count, st);
    return cudaErrorInvalidValue;
}

}  // namespace sd
