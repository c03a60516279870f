// Split-KV decode attention over an fp16 cache laid out [row][layer*kv_head][pos][dim].
//
// "Chatterbox -> ggml Port: Development Journal", section 3.13: the cache is
// stored the way flash attention reads it ([HD, n_ctx, n_head] per layer), the
// step writes its new K/V at n_past, and a one-token step needs no mask.  The
// Llama-style T3 and the Qwen Talker rotate q and k with NEOX (half-split)
// RoPE first (journal section 3.19).
//
// Grid (nsplit, n_kv, B): each CTA takes one contiguous chunk of the
// positions [0, pos] for one (row, kv head) and every query head of that kv
// head's group, and emits an unnormalised partial (o, running max m, sum l).
// The CTA whose chunk holds `pos` rotates and rounds the new key/value to fp16,
// stores them in the cache and then reads them back like every other position.
// The combine (log-sum-exp over chunks) runs in the consumer's prologue (the
// O projection) or in k_attn_combine for the op-level entry.
#include "sd_internal.cuh"

namespace sd {
namespace {

constexpr int kAttnThreads = 128;
constexpr int kMaxGroup = 4;  // query heads per kv head

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void __launch_bounds__(kAttnThreads) k_attn_decode(const AttnArgs a) {
    pdl_trigger();
    pdl_wait();
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int hd = a.hd, half = hd >> 1, G = a.n_head / a.n_kv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
    const int pos = *a.pos_ptr + a.pos_add;
    const int ps = part_stride(hd);

    extern __shared__ float sm[];
    float* q_s = sm;                      // [G][hd]
    float* sc = sm + kMaxGroup * 128;     // [G][chunk]
    __shared__ float s_red[kMaxGroup][4];

    if (pos < 0 || pos >= a.n_ctx) {
        if (tid == 0 && a.err) atomicExch(a.err, 1);
        return;
    }
    const int n = pos + 1;
    const int chunk = (n + a.nsplit - 1) / a.nsplit;
    const int s0 = split * chunk;
    const int s1 = min(n, s0 + chunk);
    float* part_base = a.part + ((size_t)(b * a.n_head + g * G) * a.nsplit + split) * ps;
    if (s0 >= s1) {  // empty chunk: neutral partial
        for (int i = tid; i < G * ps; i += blockDim.x) {
            const int gq = i / ps, d = i - gq * ps;
            part_base[(size_t)gq * a.nsplit * ps + d] = (d == hd) ? -INFINITY : 0.f;
        }
        return;
    }

    const size_t head_base = ((size_t)(b * a.row_heads + a.head_off + g) * a.n_ctx) * hd;
    __half* kc = a.kc + head_base;
    __half* vc = a.vc + head_base;
    const float scale = rsqrtf((float)hd);

    // queries of the group, rotated, pre-scaled by 1/sqrt(hd)
    for (int i = tid; i < G * half; i += blockDim.x) {
        const int gq = i / half, d = i - gq * half;
        const float* qh = a.q + (size_t)b * a.q_stride + (size_t)(g * G + gq) * hd;
        float x0 = qh[d], x1 = qh[d + half];
        if (a.rope_cos) {
            const float c = a.rope_cos[(size_t)pos * half + d], s = a.rope_sin[(size_t)pos * half + d];
            const float y0 = x0 * c - x1 * s, y1 = x0 * s + x1 * c;
            x0 = y0;
            x1 = y1;
        }
        q_s[gq * hd + d] = x0 * scale;
        q_s[gq * hd + d + half] = x1 * scale;
    }
    // append the new key/value if this chunk holds `pos`
    if (a.knew && s0 <= pos && pos < s1) {
        const float* kh = a.knew + (size_t)b * a.q_stride + (size_t)g * hd;
        const float* vh = a.vnew + (size_t)b * a.q_stride + (size_t)g * hd;
        for (int d = tid; d < half; d += blockDim.x) {
            float x0 = kh[d], x1 = kh[d + half];
            if (a.rope_cos) {
                const float c = a.rope_cos[(size_t)pos * half + d], s = a.rope_sin[(size_t)pos * half + d];
                const float y0 = x0 * c - x1 * s, y1 = x0 * s + x1 * c;
                x0 = y0;
                x1 = y1;
            }
            kc[(size_t)pos * hd + d] = __float2half_rn(x0);
            kc[(size_t)pos * hd + d + half] = __float2half_rn(x1);
            vc[(size_t)pos * hd + d] = __float2half_rn(vh[d]);
            vc[(size_t)pos * hd + d + half] = __float2half_rn(vh[d + half]);
        }
    }
    __syncthreads();

    // scores: one position per warp iteration; lanes split the head dimension
    const int dpl = hd / 32;  // 2 (hd 64) or 4 (hd 128)
    for (int j = s0 + warp; j < s1; j += nw) {
        const __half* kr = kc + (size_t)j * hd + lane * dpl;
        float kv[4];
        if (dpl == 2) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(kr));
            kv[0] = f.x; kv[1] = f.y;
        } else {
            const float2 f0 = __half22float2(reinterpret_cast<const __half2*>(kr)[0]);
            const float2 f1 = __half22float2(reinterpret_cast<const __half2*>(kr)[1]);
            kv[0] = f0.x; kv[1] = f0.y; kv[2] = f1.x; kv[3] = f1.y;
        }
        for (int gq = 0; gq < G; ++gq) {
            float s = 0.f;
            for (int d = 0; d < dpl; ++d) s = fmaf(q_s[gq * hd + lane * dpl + d], kv[d], s);
            s = warp_sum(s);
            if (lane == 0) sc[gq * chunk + (j - s0)] = s;
        }
    }
    __syncthreads();

    // softmax statistics of the chunk, per query head
    const int len = s1 - s0;
    float m[kMaxGroup], l[kMaxGroup];
    for (int gq = 0; gq < G; ++gq) {
        float mx = -INFINITY;
        for (int j = tid; j < len; j += blockDim.x) mx = fmaxf(mx, sc[gq * chunk + j]);
        mx = warp_max(mx);
        if (lane == 0) s_red[gq][warp] = mx;
    }
    __syncthreads();
    for (int gq = 0; gq < G; ++gq) {
        float mx = s_red[gq][0];
        for (int w = 1; w < nw; ++w) mx = fmaxf(mx, s_red[gq][w]);
        m[gq] = mx;
    }
    __syncthreads();
    for (int gq = 0; gq < G; ++gq) {
        float s = 0.f;
        for (int j = tid; j < len; j += blockDim.x) {
            const float p = expf(sc[gq * chunk + j] - m[gq]);
            sc[gq * chunk + j] = p;
            s += p;
        }
        s = warp_sum(s);
        if (lane == 0) s_red[gq][warp] = s;
    }
    __syncthreads();
    for (int gq = 0; gq < G; ++gq) {
        float s = 0.f;
        for (int w = 0; w < nw; ++w) s += s_red[gq][w];
        l[gq] = s;
    }

    // o = sum_j p_j V_j: thread owns one dimension, positions split in `reps` interleaved groups
    const int reps = blockDim.x / hd;  // 2 (hd 64) or 1 (hd 128)
    const int d = tid % hd, rgp = tid / hd;
    float acc[kMaxGroup] = {0.f, 0.f, 0.f, 0.f};
    if (rgp < reps) {
        for (int j = rgp; j < len; j += reps) {
            const float vv = __half2float(vc[(size_t)(s0 + j) * hd + d]);
            for (int gq = 0; gq < G; ++gq) acc[gq] = fmaf(sc[gq * chunk + j], vv, acc[gq]);
        }
    }
    __syncthreads();
    // reduce the position groups through shared memory (reuse q_s)
    for (int gq = 0; gq < G; ++gq) {
        if (rgp < reps) q_s[rgp * hd + d] = acc[gq];
        __syncthreads();
        if (tid < hd) {
            float o = 0.f;
            for (int r = 0; r < reps; ++r) o += q_s[r * hd + tid];
            float* dst = part_base + (size_t)gq * a.nsplit * ps;
            dst[tid] = o;
            if (tid == 0) {
                dst[hd] = m[gq];
                dst[hd + 1] = l[gq];
            }
        }
        __syncthreads();
    }
}

__global__ void k_attn_combine(const float* __restrict__ part, int H, int hd, int nsplit, float* __restrict__ out) {
    const int bh = blockIdx.x;
    const int ps = part_stride(hd);
    const float* p = part + (size_t)bh * nsplit * ps;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, p[s * ps + hd]);
    float L = 0.f;
    for (int s = 0; s < nsplit; ++s)
        if (p[s * ps + hd + 1] > 0.f) L = fmaf(expf(p[s * ps + hd] - M), p[s * ps + hd + 1], L);
    for (int d = threadIdx.x; d < hd; d += blockDim.x) {
        float o = 0.f;
        for (int s = 0; s < nsplit; ++s)
            if (p[s * ps + hd + 1] > 0.f) o = fmaf(expf(p[s * ps + hd] - M), p[s * ps + d], o);
        out[(size_t)bh * hd + d] = o / L;
    }
}

}  // namespace

cudaError_t launch_attention(const AttnArgs& a, int B, cudaStream_t st) {
    const int G = a.n_head / a.n_kv;
    if ((a.hd != 64 && a.hd != 128) || a.n_head % a.n_kv || G > kMaxGroup || a.nsplit < 1) return cudaErrorInvalidValue;
    const int chunk_max = (a.n_ctx + a.nsplit - 1) / a.nsplit;
    const size_t smem = (size_t)(kMaxGroup * 128 + G * chunk_max) * sizeof(float);
    if (smem > 200 * 1024) return cudaErrorInvalidValue;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_attn_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_k(k_attn_decode, dim3(a.nsplit, a.n_kv, B), dim3(kAttnThreads), smem, st, a);
}

cudaError_t launch_attn_combine(const float* part, int B, int H, int hd, int nsplit, float* out, cudaStream_t st) {
    k_attn_combine<<<B * H, 128, 0, st>>>(part, H, hd, nsplit, out);
    return cudaGetLastError();
}

}  // namespace sd
