// Split-KV decode attention over an fp16 cache laid out [row][layer*kv_head][pos][dim].
//
// "Chatterbox -> ggml Port: Development Journal", section 3.13: the cache is
// stored the way flash attention reads it ([HD, n_ctx, n_head] per layer), the
// step writes its new K/V at n_past, and a one-token step needs no mask.  The
// Llama-style T3 and the Qwen Talker rotate q and k with NEOX (half-split)
// RoPE first (journal section 3.19).
//
// A work item is one contiguous chunk of the positions [0, pos] for one
// (row, kv head) and every query head of that kv head's group.  It stages the
// chunk's K and V rows in shared memory with all loads issued at once, then
// computes an unnormalised partial (o, running max m, sum l).  The item whose
// chunk holds `pos` rotates and rounds the new key/value to fp16 and writes
// them to the cache (and to its staged copy).  The last item of a (row, kv
// head) to finish -- counted with an atomic, no waiting -- combines the
// partials by log-sum-exp in chunk order and writes the attention output
// o[row][head*hd + d]; it then resets the counter.
#pragma once
#include "sd_internal.cuh"

namespace sd {
namespace attn_detail {

constexpr int kMaxGroup = 4;  // query heads per kv head

struct AttnScratch {
    float red[kMaxGroup][32];
    float w[kMaxGroup * 128];  // combine weights [G][nsplit]
    int last;
};


static __device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
static __device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

static __device__ __forceinline__ void rope_pair(float& x0, float& x1, const float* cs, const float* sn, int pos, int half,
                                          int d) {
    if (!cs) return;
    const float c = cs[(size_t)pos * half + d], s = sn[(size_t)pos * half + d];
    const float y0 = x0 * c - x1 * s, y1 = x0 * s + x1 * c;
    x0 = y0;
    x1 = y1;
}

// One work item: chunk `split` of (row b, kv head g).  `sm` is the dynamic
// shared memory (attention_smem_bytes), `ss` the small scratch.  Block size: a
// multiple of 32, at most kMaxGroup * 128 threads.  Loads of buffers written
// by other CTAs of a persistent kernel go through L2 (ld.global.cg).
static __device__ void attn_item(const AttnArgs& a, int split, int g, int b, float* sm, AttnScratch& ss) {
    const int hd = a.hd, half = hd >> 1, G = a.n_head / a.n_kv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
    const int pos = __ldcg(a.pos_ptr) + a.pos_add;
    const int ps = part_stride(hd);
    const int span = a.max_len > 0 ? a.max_len : a.n_ctx;
    const int chunk_max = (span + a.nsplit - 1) / a.nsplit;

    float* q_s = sm;                                 // [G][hd]
    float* sc = q_s + kMaxGroup * 128;               // [G][chunk_max]
    __half* ks = reinterpret_cast<__half*>(sc + kMaxGroup * chunk_max);  // [chunk_max][hd]
    __half* vs = ks + (size_t)chunk_max * hd;                           // [chunk_max][hd]
    auto& s_red = ss.red;
    float* s_w = ss.w;
    int& s_last = ss.last;

    if (pos < 0 || pos >= a.n_ctx || pos >= span) {
        if (tid == 0 && a.err) atomicExch(a.err, 1);
        __syncthreads();
        return;
    }
    const int n = pos + 1;
    const int chunk = (n + a.nsplit - 1) / a.nsplit;
    const int s0 = split * chunk;
    const int s1 = min(n, s0 + chunk);
    const int len = s1 > s0 ? s1 - s0 : 0;
    float* part_base = a.part + ((size_t)(b * a.n_head + g * G) * a.nsplit + split) * ps;
    const size_t head_base = ((size_t)(b * a.row_heads + a.head_off + g) * a.n_ctx) * hd;
    __half* kc = a.kc + head_base;
    __half* vc = a.vc + head_base;

    if (len > 0) {
        // stage the chunk's cached rows (positions < pos) with 16-byte loads, all in flight together
        const int vpr = hd / 8;                        // uint4 per row
        const int old_rows = min(s1, pos) - s0;        // rows already in the cache
        const int nvec = (old_rows > 0 ? old_rows : 0) * vpr;
        const uint4* kg = reinterpret_cast<const uint4*>(kc + (size_t)s0 * hd);
        const uint4* vg = reinterpret_cast<const uint4*>(vc + (size_t)s0 * hd);
        uint4* k4 = reinterpret_cast<uint4*>(ks);
        uint4* v4 = reinterpret_cast<uint4*>(vs);
#pragma unroll 4
        for (int i = tid; i < nvec; i += blockDim.x) {
            const uint4 kk = __ldcg(kg + i), vv = __ldcg(vg + i);
            k4[i] = kk;
            v4[i] = vv;
        }
        // queries of the group, rotated, pre-scaled by 1/sqrt(hd)
        const float scale = rsqrtf((float)hd);
        for (int i = tid; i < G * half; i += blockDim.x) {
            const int gq = i / half, d = i - gq * half;
            const float* qh = a.q + (size_t)b * a.q_stride + (size_t)(g * G + gq) * hd;
            float x0 = __ldcg(qh + d), x1 = __ldcg(qh + d + half);
            rope_pair(x0, x1, a.rope_cos, a.rope_sin, pos, half, d);
            q_s[gq * hd + d] = x0 * scale;
            q_s[gq * hd + d + half] = x1 * scale;
        }
        // the new key/value: rotate, round to fp16, write to the cache and the staged chunk
        if (s0 <= pos && pos < s1 && a.knew) {
            const float* kh = a.knew + (size_t)b * a.q_stride + (size_t)g * hd;
            const float* vh = a.vnew + (size_t)b * a.q_stride + (size_t)g * hd;
            const int r = pos - s0;
            for (int d = tid; d < half; d += blockDim.x) {
                float x0 = __ldcg(kh + d), x1 = __ldcg(kh + d + half);
                rope_pair(x0, x1, a.rope_cos, a.rope_sin, pos, half, d);
                const __half k0 = __float2half_rn(x0), k1 = __float2half_rn(x1);
                const __half v0 = __float2half_rn(__ldcg(vh + d)), v1 = __float2half_rn(__ldcg(vh + d + half));
                kc[(size_t)pos * hd + d] = k0; kc[(size_t)pos * hd + d + half] = k1;
                vc[(size_t)pos * hd + d] = v0; vc[(size_t)pos * hd + d + half] = v1;
                ks[(size_t)r * hd + d] = k0; ks[(size_t)r * hd + d + half] = k1;
                vs[(size_t)r * hd + d] = v0; vs[(size_t)r * hd + d + half] = v1;
            }
        } else if (s0 <= pos && pos < s1) {
            // op-level use: the cache already holds position pos
            const uint4* kp = reinterpret_cast<const uint4*>(kc + (size_t)pos * hd);
            const uint4* vp = reinterpret_cast<const uint4*>(vc + (size_t)pos * hd);
            for (int i = tid; i < vpr; i += blockDim.x) {
                k4[(pos - s0) * vpr + i] = __ldcg(kp + i);
                v4[(pos - s0) * vpr + i] = __ldcg(vp + i);
            }
        }
        __syncthreads();

        // scores: one position per warp iteration; lanes split the head dimension
        const int dpl = hd / 32;  // 2 (hd 64) or 4 (hd 128)
        for (int j = warp; j < len; j += nw) {
            const __half* kr = ks + (size_t)j * hd + lane * dpl;
            float kv[4];
            const float2 f0 = __half22float2(reinterpret_cast<const __half2*>(kr)[0]);
            kv[0] = f0.x; kv[1] = f0.y;
            if (dpl == 4) {
                const float2 f1 = __half22float2(reinterpret_cast<const __half2*>(kr)[1]);
                kv[2] = f1.x; kv[3] = f1.y;
            }
            for (int gq = 0; gq < G; ++gq) {
                float s = 0.f;
                for (int d = 0; d < dpl; ++d) s = fmaf(q_s[gq * hd + lane * dpl + d], kv[d], s);
                s = warp_sum(s);
                if (lane == 0) sc[gq * chunk_max + j] = s;
            }
        }
        __syncthreads();

        // softmax statistics of the chunk, per query head
        float m[kMaxGroup], l[kMaxGroup];
        for (int gq = 0; gq < G; ++gq) {
            float mx = -INFINITY;
            for (int j = tid; j < len; j += blockDim.x) mx = fmaxf(mx, sc[gq * chunk_max + j]);
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
                const float p = expf(sc[gq * chunk_max + j] - m[gq]);
                sc[gq * chunk_max + j] = p;
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

        // o = sum_j p_j V_j: thread owns one dimension, positions in `reps` interleaved groups
        const int reps = blockDim.x / hd;  // 2 (hd 64) or 1 (hd 128)
        const int d = tid % hd, rgp = tid / hd;
        float acc[kMaxGroup] = {0.f, 0.f, 0.f, 0.f};
        if (rgp < reps) {
            for (int j = rgp; j < len; j += reps) {
                const float vv = __half2float(vs[(size_t)j * hd + d]);
                for (int gq = 0; gq < G; ++gq) acc[gq] = fmaf(sc[gq * chunk_max + j], vv, acc[gq]);
            }
        }
        __syncthreads();
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
    } else {
        // empty chunk: neutral partial
        for (int i = tid; i < G * ps; i += blockDim.x) {
            const int gq = i / ps, d = i - gq * ps;
            part_base[(size_t)gq * a.nsplit * ps + d] = (d == hd) ? -INFINITY : 0.f;
        }
        __syncthreads();
    }

    // ---- the last CTA of this (row, kv head) combines the chunks
    if (tid == 0) {
        __threadfence();
        const int prev = atomicAdd(&a.counters[b * a.n_kv + g], 1);
        s_last = (prev == a.nsplit - 1);
    }
    __syncthreads();
    const bool last = s_last;
    __syncthreads();
    if (!last) return;
    __threadfence();
    const int S = a.nsplit;
    float* w = s_w;
    if (tid < G) {
        const float* p = a.part + ((size_t)(b * a.n_head + g * G + tid) * S) * ps;
        float M = -INFINITY;
        for (int s = 0; s < S; ++s) M = fmaxf(M, __ldcg(p + s * ps + hd));
        float L = 0.f;
        for (int s = 0; s < S; ++s) {
            const float ls = __ldcg(p + s * ps + hd + 1);
            const float e = ls > 0.f ? expf(__ldcg(p + s * ps + hd) - M) : 0.f;
            w[tid * S + s] = e;
            L = fmaf(e, ls, L);
        }
        const float inv = 1.0f / L;
        for (int s = 0; s < S; ++s) w[tid * S + s] *= inv;
    }
    __syncthreads();
    for (int i = tid; i < G * hd; i += blockDim.x) {
        const int gq = i / hd, d = i - gq * hd;
        const float* p = a.part + ((size_t)(b * a.n_head + g * G + gq) * S) * ps + d;
        float o = 0.f;
        for (int s = 0; s < S; ++s) o = fmaf(w[gq * S + s], __ldcg(p + s * ps), o);
        a.out[(size_t)b * a.out_stride + (size_t)(g * G + gq) * hd + d] = o;
    }
    if (tid == 0) a.counters[b * a.n_kv + g] = 0;
    __syncthreads();
}


}  // namespace attn_detail

inline size_t attention_smem_bytes_dev(const AttnArgs& a) {
    const int span = a.max_len > 0 ? a.max_len : a.n_ctx;
    const int chunk_max = (span + a.nsplit - 1) / a.nsplit;
    return sizeof(float) * (size_t)(attn_detail::kMaxGroup * 128 + attn_detail::kMaxGroup * chunk_max) +
           2 * sizeof(__half) * (size_t)chunk_max * a.hd;
}

}  // namespace sd
