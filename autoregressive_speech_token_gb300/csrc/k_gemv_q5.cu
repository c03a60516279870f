// Quantised GEMV instantiations for Q5_0 weights (kernel in k_gemv.cuh).
#include "k_gemv.cuh"

namespace sd {

cudaError_t launch_gemv_q5(const GemvArgs& a, int sm_count, cudaStream_t st) {
    cudaError_t e = gemv_detail::check_gemv(a);
    if (e != cudaSuccess) return e;
    return a.nb == 1 ? gemv_detail::launch_t<SD_Q5_0, 1>(a, sm_count, st) : gemv_detail::launch_t<SD_Q5_0, 2>(a, sm_count, st);
}

}  // namespace sd
