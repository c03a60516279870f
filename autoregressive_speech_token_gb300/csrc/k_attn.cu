// Split-KV decode attention kernel: one CTA per work item of attn_item()
// (attn_dev.cuh), grid (nsplit, kv heads, rows).
#include "attn_dev.cuh"

namespace sd {
namespace {

constexpr int kAttnThreads = 128;

__global__ void __launch_bounds__(kAttnThreads) k_attn_decode(const AttnArgs a) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ __align__(16) float sm[];
    __shared__ attn_detail::AttnScratch ss;
    attn_detail::attn_item(a, blockIdx.x, blockIdx.y, blockIdx.z, sm, ss);
}

}  // namespace

size_t attention_smem_bytes(const AttnArgs& a) { return attention_smem_bytes_dev(a); }

cudaError_t launch_attention(const AttnArgs& a, int B, cudaStream_t st) {
    const int G = a.n_head / a.n_kv;
    if ((a.hd != 64 && a.hd != 128) || a.n_head % a.n_kv || G > attn_detail::kMaxGroup || a.nsplit < 1 ||
        a.nsplit > 128 || !a.counters || !a.out)
        return cudaErrorInvalidValue;
    const size_t smem = attention_smem_bytes(a);
    if (smem > 220 * 1024) return cudaErrorInvalidValue;
    if (smem > 32 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_attn_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_k(k_attn_decode, dim3(a.nsplit, a.n_kv, B), dim3(kAttnThreads), smem, st, a);
}

}  // namespace sd
