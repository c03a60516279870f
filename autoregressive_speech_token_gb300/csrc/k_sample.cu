// On-device sampler kernel: one 512-thread CTA per row around sample_block()
// (sample_dev.cuh), logits staged in shared memory, token written to device
// memory -- no host round trip.
#include "sample_dev.cuh"

namespace sd {
namespace {

constexpr int kST = 512;

__global__ void __launch_bounds__(kST, 1) k_sample(const SampleArgs a) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ __align__(16) unsigned char smraw[];
    __shared__ sample_detail::SampleScratch ss;
    const int b = blockIdx.x;
    const float* up = (a.u_seq && *a.u_seq) ? (*a.u_seq) + (size_t)(*a.step_idx) * gridDim.x + b
                                            : a.u + (size_t)b * a.u_stride + a.u_off;
    const int tok = sample_detail::sample_block(a.logits + (size_t)b * a.ld, a.V, *a.sp, up, smraw, ss, a.err,
                                                a.seen ? a.seen + (size_t)b * a.seen_ld : nullptr);
    if (threadIdx.x == 0) {
        a.out[(size_t)b * a.out_stride + a.out_off] = tok;
        if (a.out_seq && *a.out_seq) (*a.out_seq)[(size_t)(*a.step_idx) * gridDim.x + b] = tok;
    }
}

}  // namespace

size_t sample_smem_bytes(int V) { return sample_smem_bytes_dev(V, kST); }

cudaError_t launch_sample(const SampleArgs& a, int rows, cudaStream_t st) {
    if (a.V < 1 || a.V > sample_detail::kMaxV) return cudaErrorInvalidValue;
    const size_t smem = sample_smem_bytes(a.V);
    cudaError_t e = cudaFuncSetAttribute(k_sample, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_k(k_sample, dim3(rows), dim3(kST), smem, st, a);
}

}  // namespace sd
