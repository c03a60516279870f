// Prompt prefill around the tensor-core GEMM: embeddings of all prompt
// positions, per-row norms, RoPE + fp16 KV append for a block of positions,
// and causal attention over the cached prefix.
//
// "Chatterbox -> ggml Port: Development Journal", section 3.2: the prompt
// runs as one graph over all prompt positions and fills the KV cache that the
// step graph then extends; section 3.13: the cache is laid out [head][pos][dim]
// and written at n_past (here: positions 0..n-1 at once); the prompt graph uses
// a causal mask (journal section 3.12: position j is visible to query i when
// j <= i).
#include "sd_internal.cuh"

namespace sd {
namespace {

// X[b*np + p] = table[tok[b*ld + p0 + p]] (+ pos_table[p0 + p]) for p < np
__global__ void k_embed_rows(const float* __restrict__ table, const float* __restrict__ pos_table,
                             const int32_t* __restrict__ tok, int ld, int p0, int np, int d, int V,
                             float* __restrict__ X, int* err) {
    const int m = blockIdx.x, b = m / np, p = m - b * np;
    int t = tok[(size_t)b * ld + p0 + p];
    if (t < 0 || t >= V) {
        if (threadIdx.x == 0 && err) atomicExch(err, 3);
        t = 0;
    }
    const float4* e = reinterpret_cast<const float4*>(table + (size_t)t * d);
    const float4* q = pos_table ? reinterpret_cast<const float4*>(pos_table + (size_t)(p0 + p) * d) : nullptr;
    float4* x = reinterpret_cast<float4*>(X + (size_t)m * d);
    for (int i = threadIdx.x; i < d / 4; i += blockDim.x) {
        float4 v = e[i];
        if (q) {
            const float4 w = q[i];
            v.x += w.x; v.y += w.y; v.z += w.z; v.w += w.w;
        }
        x[i] = v;
    }
}

// H[m] = norm(X[m]) * g (+ b): LayerNorm (biased variance) or RMSNorm, one CTA
// per row; X rows ldx apart, H rows d apart.
__global__ void __launch_bounds__(256) k_rownorm(const float* __restrict__ X, int ldx, int d, int ln,
                                                 const float* __restrict__ g, const float* __restrict__ bta, float eps,
                                                 float* __restrict__ H) {
    const int m = blockIdx.x, tid = threadIdx.x;
    const float* x = X + (size_t)m * ldx;
    __shared__ float red[32];
    __shared__ float stat[2];
    float s = 0.f;
    for (int i = tid; i < d; i += blockDim.x) s += ln ? x[i] : x[i] * x[i];
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((tid & 31) == 0) red[tid >> 5] = s;
    __syncthreads();
    if (tid == 0) {
        float t = 0.f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
        stat[0] = ln ? t / d : 0.f;
        stat[1] = t / d;
    }
    __syncthreads();
    const float mu = stat[0];
    float rs;
    if (ln) {
        float v = 0.f;
        for (int i = tid; i < d; i += blockDim.x) {
            const float dx = x[i] - mu;
            v = fmaf(dx, dx, v);
        }
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        __syncthreads();
        if ((tid & 31) == 0) red[tid >> 5] = v;
        __syncthreads();
        if (tid == 0) {
            float t = 0.f;
            for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
            stat[1] = t / d;
        }
        __syncthreads();
    }
    rs = 1.0f / sqrtf(stat[1] + eps);
    for (int i = tid; i < d; i += blockDim.x) {
        const float xv = x[i];
        H[(size_t)m * d + i] = ln ? fmaf((xv - mu) * rs, g[i], bta[i]) : xv * rs * g[i];
    }
}

// For row m = b*np + i at position p = p0 + i: rotate q (in place, all
// heads) and k (NEOX half-split) and store k, v as fp16 at cache position p.
// One CTA per row.
__global__ void k_rope_kv(float* __restrict__ QKV, int ld, int p0, int np, int H, int Hkv, int hd, int n_ctx,
                          int row_heads, int head_off, const float* __restrict__ cs, const float* __restrict__ sn,
                          __half* __restrict__ kc, __half* __restrict__ vc) {
    const int m = blockIdx.x, b = m / np, p = p0 + (m - b * np);
    const int half = hd / 2, qd = H * hd, kd = Hkv * hd;
    float* row = QKV + (size_t)m * ld;
    for (int i = threadIdx.x; i < (H + Hkv) * half; i += blockDim.x) {
        const int h = i / half, dd = i - h * half;
        float* v = h < H ? row + h * hd : row + qd + (h - H) * hd;
        float x0 = v[dd], x1 = v[dd + half];
        if (cs) {
            const float c = cs[(size_t)p * half + dd], s = sn[(size_t)p * half + dd];
            const float y0 = x0 * c - x1 * s, y1 = x0 * s + x1 * c;
            x0 = y0;
            x1 = y1;
        }
        if (h < H) {
            v[dd] = x0;
            v[dd + half] = x1;
        } else {
            const int g = h - H;
            __half* kr = kc + (((size_t)(b * row_heads + head_off + g) * n_ctx) + p) * hd;
            kr[dd] = __float2half_rn(x0);
            kr[dd + half] = __float2half_rn(x1);
        }
    }
    for (int i = threadIdx.x; i < kd; i += blockDim.x) {
        const int g = i / hd, dd = i - g * hd;
        __half* vr = vc + (((size_t)(b * row_heads + head_off + g) * n_ctx) + p) * hd;
        vr[dd] = __float2half_rn(row[qd + kd + i]);
    }
}

// Causal attention over the prompt chunk: queries at positions p0 .. p0 + np - 1
// of row b, head h, against keys 0..p of the fp16 cache (the chunk's own keys
// were appended by k_rope_kv).  A CTA takes kQC queries of one (row, head);
// each of its four warps takes every fourth query.  The keys and values of a
// block of kKB positions are staged once in shared memory for all kQC queries
// (key rows at a pitch of hd + 8 halves, so lane j reading row j is free of
// bank conflicts); lane j scores key j of a 32-key sub-block with a full dot
// product (no shuffles per key), the sub-block updates an online softmax, and
// p.V accumulates with lanes over dimensions (DPL = head_dim / 32 per lane).
constexpr int kQC = 16, kKB = 64;

template <int DPL>
__global__ void __launch_bounds__(128) k_prefill_attn(const float* __restrict__ QKV, int ld, int p0, int np, int H,
                                                      int Hkv, int n_ctx, int row_heads, int head_off,
                                                      const __half* __restrict__ kc, const __half* __restrict__ vc,
                                                      float* __restrict__ O, int ldo) {
    constexpr int hd = 32 * DPL, KP = hd + 8, NQ = kQC / 4;
    __shared__ __align__(16) __half Ks[kKB * KP];
    __shared__ __align__(16) __half Vs[kKB * hd];
    __shared__ __align__(16) float Qs[kQC * hd];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = blockIdx.x * kQC, h = blockIdx.y, b = blockIdx.z;
    const int g = h / (H / Hkv);
    const int nq = min(kQC, np - c0);            // queries of this CTA
    const int p_last = p0 + c0 + nq - 1;         // the chunk's last position
    const __half* K = kc + ((size_t)(b * row_heads + head_off + g) * n_ctx) * hd;
    const __half* Vv = vc + ((size_t)(b * row_heads + head_off + g) * n_ctx) * hd;
    const float scale = 1.0f / sqrtf((float)hd);
    for (int i = threadIdx.x; i < nq * hd; i += blockDim.x) {
        const int qi = i / hd, e = i - qi * hd;
        Qs[qi * hd + e] = QKV[(size_t)(b * np + c0 + qi) * ld + h * hd + e] * scale;
    }
    float m[NQ], l[NQ], acc[NQ][DPL];
#pragma unroll
    for (int t = 0; t < NQ; ++t) {
        m[t] = -INFINITY;
        l[t] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[t][e] = 0.f;
    }
    for (int kb0 = 0; kb0 <= p_last; kb0 += kKB) {
        const int nk = min(kKB, p_last + 1 - kb0);
        __syncthreads();  // every warp is done with the previous block (and Qs is written)
        for (int i = threadIdx.x; i < nk * (hd / 8); i += blockDim.x) {
            const int j = i / (hd / 8), c = i - j * (hd / 8);
            *reinterpret_cast<uint4*>(Ks + j * KP + 8 * c) = *reinterpret_cast<const uint4*>(K + (size_t)(kb0 + j) * hd + 8 * c);
            *reinterpret_cast<uint4*>(Vs + j * hd + 8 * c) = *reinterpret_cast<const uint4*>(Vv + (size_t)(kb0 + j) * hd + 8 * c);
        }
        __syncthreads();
#pragma unroll
        for (int t = 0; t < NQ; ++t) {
            const int qi = warp + 4 * t;
            if (qi >= nq) continue;
            const int p = p0 + c0 + qi;
            const float* q = Qs + qi * hd;
            for (int sb = 0; sb < nk && kb0 + sb <= p; sb += 32) {
                const int j = sb + lane;                 // key kb0 + j of the block
                const bool valid = j < nk && kb0 + j <= p;
                float s = -INFINITY;
                if (valid) {
                    float d = 0.f;
                    const __half* kr = Ks + j * KP;
#pragma unroll
                    for (int c = 0; c < hd / 8; ++c) {
                        const uint4 kw = *reinterpret_cast<const uint4*>(kr + 8 * c);
                        const __half2* k2 = reinterpret_cast<const __half2*>(&kw);
                        const float4 qa = *reinterpret_cast<const float4*>(q + 8 * c);
                        const float4 qb = *reinterpret_cast<const float4*>(q + 8 * c + 4);
                        const float2 f0 = __half22float2(k2[0]), f1 = __half22float2(k2[1]);
                        const float2 f2 = __half22float2(k2[2]), f3 = __half22float2(k2[3]);
                        d = fmaf(qa.x, f0.x, d); d = fmaf(qa.y, f0.y, d);
                        d = fmaf(qa.z, f1.x, d); d = fmaf(qa.w, f1.y, d);
                        d = fmaf(qb.x, f2.x, d); d = fmaf(qb.y, f2.y, d);
                        d = fmaf(qb.z, f3.x, d); d = fmaf(qb.w, f3.y, d);
                    }
                    s = d;
                }
                float cm = s;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
                const float mnew = fmaxf(m[t], cm);
                const float corr = expf(m[t] - mnew);
                const float pj = valid ? expf(s - mnew) : 0.f;
                float ps = pj;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
                l[t] = l[t] * corr + ps;
#pragma unroll
                for (int e = 0; e < DPL; ++e) acc[t][e] *= corr;
                const int nv = min(32, min(nk - sb, p + 1 - (kb0 + sb)));  // valid keys of the sub-block
                for (int jj = 0; jj < nv; ++jj) {
                    const float pb = __shfl_sync(0xffffffffu, pj, jj);
                    const __half* vr = Vs + (sb + jj) * hd + lane * DPL;
                    if constexpr (DPL == 2) {
                        const float2 v2 = __half22float2(*reinterpret_cast<const __half2*>(vr));
                        acc[t][0] = fmaf(pb, v2.x, acc[t][0]);
                        acc[t][1] = fmaf(pb, v2.y, acc[t][1]);
                    } else {
#pragma unroll
                        for (int e = 0; e < DPL; ++e) acc[t][e] = fmaf(pb, __half2float(vr[e]), acc[t][e]);
                    }
                }
                m[t] = mnew;
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NQ; ++t) {
        const int qi = warp + 4 * t;
        if (qi >= nq) continue;
#pragma unroll
        for (int e = 0; e < DPL; ++e) O[(size_t)(b * np + c0 + qi) * ldo + h * hd + lane * DPL + e] = acc[t][e] / l[t];
    }
}

}  // namespace

cudaError_t launch_embed_rows(const float* table, const float* pos_table, const int32_t* tok, int ld, int B, int p0,
                              int np, int d, int V, float* X, int* err, cudaStream_t st) {
    if (d % 4 || B < 1 || np < 1) return cudaErrorInvalidValue;
    k_embed_rows<<<B * np, 256, 0, st>>>(table, pos_table, tok, ld, p0, np, d, V, X, err);
    return cudaGetLastError();
}

cudaError_t launch_rownorm(const float* X, int ldx, int M, int d, int ln, const float* g, const float* b, float eps,
                           float* H, cudaStream_t st) {
    if (M < 1 || ldx < d) return cudaErrorInvalidValue;
    k_rownorm<<<M, 256, 0, st>>>(X, ldx, d, ln, g, b, eps, H);
    return cudaGetLastError();
}

cudaError_t launch_rope_kv(float* QKV, int ld, int B, int p0, int np, int H, int Hkv, int hd, int n_ctx, int row_heads,
                           int head_off, const float* cs, const float* sn, __half* kc, __half* vc, cudaStream_t st) {
    if (hd % 2 || p0 < 0 || p0 + np > n_ctx) return cudaErrorInvalidValue;
    k_rope_kv<<<B * np, 128, 0, st>>>(QKV, ld, p0, np, H, Hkv, hd, n_ctx, row_heads, head_off, cs, sn, kc, vc);
    return cudaGetLastError();
}

cudaError_t launch_prefill_attn(const float* QKV, int ld, int B, int p0, int np, int H, int Hkv, int hd, int n_ctx,
                                int row_heads, int head_off, const __half* kc, const __half* vc, float* O, int ldo,
                                cudaStream_t st) {
    if (H % Hkv || p0 < 0 || p0 + np > n_ctx || np < 1) return cudaErrorInvalidValue;
    const dim3 grid((np + kQC - 1) / kQC, H, B);
    switch (hd) {
        case 64:
            k_prefill_attn<2><<<grid, 128, 0, st>>>(QKV, ld, p0, np, H, Hkv, n_ctx, row_heads, head_off, kc, vc, O, ldo);
            break;
        case 128:
            k_prefill_attn<4><<<grid, 128, 0, st>>>(QKV, ld, p0, np, H, Hkv, n_ctx, row_heads, head_off, kc, vc, O, ldo);
            break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace sd
