// Block-level sampler (temperature -> top-k -> top-p -> index-order draw),
// shared by the sampler kernel and the persistent step kernel.
// "Chatterbox -> ggml Port: Development Journal", section 3.2 (order) and the
// defaults table of section 3.9; "Every Frame Is a Memory Read", section 5.6
// (top-p over the top-k survivors, drawn in full-vocabulary index order).
//
//   greedy   argmax, ties to the lowest index;
//   top-k    4-pass 8-bit radix select of the k-th largest order-preserving
//            key (one warp finds each digit) -- every logit >= it survives;
//   softmax  p_i = exp((z_i - max) / T) over the survivors, fp32, fixed order;
//   top-p    survivors sorted by (p desc, index asc) with a bitonic sort of
//            64-bit keys (logit key << 32 | ~index); the shortest prefix whose
//            mass reaches top_p * Z is kept;
//   draw     the smallest vocabulary index whose cumulative kept mass (index
//            order, block prefix scan) exceeds u times the kept total.
#pragma once
#include "sd_internal.cuh"

namespace sd {
namespace sample_detail {

constexpr int kMaxV = 16384;

struct SampleScratch {
    float f[72];
    int i[40];
    int hist[256];
    uint32_t sel[3];  // prefix, mask, remaining
    int cnt;
};

static __device__ __forceinline__ uint32_t ord_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

static __device__ __forceinline__ int pow2_ceil(int n) {
    int c = 1;
    while (c < n) c <<= 1;
    return c;
}

// exclusive scan of one float per thread (fixed order); returns the block total in *total
static __device__ float block_exclusive_scan(float v, float* s_warp, float* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        float w = lane < (int)(blockDim.x >> 5) ? s_warp[lane] : 0.f;
        float wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += t;
        }
        s_warp[32 + lane] = wi - w;  // exclusive prefix of warp totals
        if (lane == 31) s_warp[64] = wi;
    }
    __syncthreads();
    const float r = s_warp[32 + warp] + inc - v;
    *total = s_warp[64];
    __syncthreads();
    return r;
}

static __device__ float block_sum_f(float v, float* s_warp) {
    float t;
    block_exclusive_scan(v, s_warp, &t);
    return t;
}

static __device__ int block_min_i(int v, int* s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        int w = threadIdx.x < (blockDim.x >> 5) ? s[threadIdx.x] : 0x7fffffff;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w = min(w, __shfl_xor_sync(0xffffffffu, w, o));
        if (threadIdx.x == 0) s[32] = w;
    }
    __syncthreads();
    const int r = s[32];
    __syncthreads();
    return r;
}

static __device__ int block_max_i(int v, int* s) { return -block_min_i(-v, s); }

// Samples one token from logits lg[0..V) with draw u (used by every thread of
// the calling block; every thread gets the token).  Shared memory: `smraw`
// holds sample_smem_bytes(V); `ss` the small scratch.  The block size is any
// multiple of 32 up to 1024.
static __device__ int sample_block(const float* lg, int V, const SampParams sp, const float* u_ptr,
                            unsigned char* smraw, SampleScratch& ss, int* err) {
    const int tid = threadIdx.x, kST = blockDim.x;
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(smraw);   // [pow2_ceil(V)]
    float* z = reinterpret_cast<float*>(smraw + sizeof(unsigned long long) * pow2_ceil(V));  // [V] logits, then [V] p
    float* s_f = ss.f;
    int* s_i = ss.i;
    int* s_hist = ss.hist;
    uint32_t* s_sel = ss.sel;
    int& s_cnt = ss.cnt;

    // written by other CTAs in a persistent kernel: read through L2, all loads in flight at once
    for (int i0 = 0; i0 < V; i0 += 16 * kST) {
        float r[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int i = i0 + j * kST + tid;
            r[j] = i < V ? __ldcg(lg + i) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int i = i0 + j * kST + tid;
            if (i < V) z[i] = r[j];
        }
    }
    __syncthreads();

    int tok;
    if (sp.greedy || sp.top_k == 1 || sp.temperature <= 0.f) {
        float best = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = tid; i < V; i += kST)
            if (z[i] > best) { best = z[i]; bi = i; }   // strided scan: first hit is the lowest index
        // reduce (value desc, index asc)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
        }
        if ((tid & 31) == 0) { s_f[tid >> 5] = best; s_i[tid >> 5] = bi; }
        __syncthreads();
        if (tid < 32) {
            const bool have = tid < (kST >> 5);
            best = have ? s_f[tid] : -INFINITY;
            bi = have ? s_i[tid] : 0x7fffffff;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, best, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
            }
            if (tid == 0) s_i[32] = bi;
        }
        __syncthreads();
        tok = s_i[32];
    } else {
        // ---- top-k threshold by radix select on order-preserving keys
        const int k = (sp.top_k < 1 || sp.top_k > V) ? V : sp.top_k;
        if (tid == 0) { s_sel[0] = 0u; s_sel[1] = 0u; s_sel[2] = (uint32_t)k; }
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += kST) s_hist[i] = 0;
            __syncthreads();
            const uint32_t prefix = s_sel[0], mask = s_sel[1];
            // lanes with equal digits add once (logits crowd into few high-order bins)
            for (int i0 = 0; i0 < V; i0 += kST) {
                const int i = i0 + tid;
                const uint32_t key = i < V ? ord_key(z[i]) : 0u;
                const bool in = i < V && (key & mask) == prefix;
                const unsigned act = __ballot_sync(0xffffffffu, in);
                if (in) {
                    const uint32_t digit = (key >> shift) & 255u;
                    const unsigned peers = __match_any_sync(act, digit);
                    if ((tid & 31) == __ffs(peers) - 1) atomicAdd(&s_hist[digit], __popc(peers));
                }
            }
            __syncthreads();
            if (tid < 32) {
                // lane l owns bins 255-8l .. 248-8l (descending); find the digit whose
                // cumulative count from the top reaches the remaining rank
                const uint32_t rem = s_sel[2];
                uint32_t c[8], own = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) { c[j] = (uint32_t)s_hist[255 - 8 * tid - j]; own += c[j]; }
                uint32_t incl = own;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (tid >= o) incl += t;
                }
                const uint32_t excl = incl - own;
                const unsigned hit = __ballot_sync(0xffffffffu, excl < rem && incl >= rem);
                if (tid == __ffs(hit) - 1) {
                    uint32_t cum = excl;
                    int digit = 255 - 8 * tid;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (cum + c[j] >= rem) { digit = 255 - 8 * tid - j; break; }
                        cum += c[j];
                    }
                    s_sel[0] = prefix | ((uint32_t)digit << shift);
                    s_sel[1] = mask | (255u << shift);
                    s_sel[2] = rem - cum;
                }
            }
            __syncthreads();
        }
        const uint32_t thr = s_sel[0];

        // ---- max and softmax mass of the survivors
        float mx = -INFINITY;
        for (int i = tid; i < V; i += kST) mx = fmaxf(mx, z[i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if ((tid & 31) == 0) s_f[tid >> 5] = mx;
        __syncthreads();
        mx = s_f[0];
        for (int w = 1; w < (kST >> 5); ++w) mx = fmaxf(mx, s_f[w]);
        __syncthreads();
        const float invT = 1.0f / sp.temperature;
        float* pv = z + V;  // [V] probabilities of the survivors (0 elsewhere)
        for (int i = tid; i < V; i += kST) pv[i] = ord_key(z[i]) >= thr ? expf((z[i] - mx) * invT) : 0.f;
        __syncthreads();
        auto pval = [&](int i) { return pv[i]; };

        // ---- top-p: cut key over the (p desc, index asc) order
        bool use_cut = false;
        unsigned long long cut = 0ull;
        if (sp.top_p < 1.0f) {
            float zp = 0.f;
            for (int i = tid; i < V; i += kST) zp += pv[i];
            const float Z = block_sum_f(zp, s_f);
            if (tid == 0) s_cnt = 0;
            __syncthreads();
            for (int i0 = 0; i0 < V; i0 += kST) {
                const int i = i0 + tid;
                const uint32_t key = i < V ? ord_key(z[i]) : 0u;
                const bool keep = i < V && key >= thr;
                const unsigned bal = __ballot_sync(0xffffffffu, keep);
                int base = 0;
                if ((tid & 31) == 0 && bal) base = atomicAdd(&s_cnt, __popc(bal));
                base = __shfl_sync(0xffffffffu, base, 0);
                if (keep) {
                    const int slot = base + __popc(bal & ((1u << (tid & 31)) - 1u));
                    keys[slot] = ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)i);
                }
            }
            __syncthreads();
            const int nk = s_cnt;
            const int cap = pow2_ceil(nk < 2 ? 2 : nk);
            for (int i = nk + tid; i < cap; i += kST) keys[i] = 0ull;
            __syncthreads();
            for (int size = 2; size <= cap; size <<= 1) {
                for (int stride = size >> 1; stride > 0; stride >>= 1) {
                    for (int i = tid; i < (cap >> 1); i += kST) {
                        const int lo = 2 * stride * (i / stride) + (i % stride);
                        const int hi = lo + stride;
                        const bool desc = (lo & size) == 0;
                        const unsigned long long x = keys[lo], y = keys[hi];
                        if (desc ? (x < y) : (x > y)) { keys[lo] = y; keys[hi] = x; }
                    }
                    __syncthreads();
                }
            }
            // cumulative mass in sorted order: contiguous segment per thread
            const int seg = (nk + kST - 1) / kST;
            const int a0 = tid * seg, a1 = min(nk, a0 + seg);
            float loc = 0.f;
            for (int t = a0; t < a1; ++t) loc += pval((int)(0xFFFFFFFFu - (uint32_t)(keys[t] & 0xFFFFFFFFull)));
            float tot;
            float run = block_exclusive_scan(loc, s_f, &tot);
            const float target = sp.top_p * Z;
            int c = 0x7fffffff;
            for (int t = a0; t < a1; ++t) {
                run += pval((int)(0xFFFFFFFFu - (uint32_t)(keys[t] & 0xFFFFFFFFull)));
                if (run >= target) { c = t; break; }
            }
            c = block_min_i(c, s_i);
            if (c == 0x7fffffff) c = nk - 1;
            cut = keys[c];
            use_cut = true;
            __syncthreads();
        }

        // ---- draw in vocabulary order over the kept set
        auto kept = [&](int i) {
            const uint32_t key = ord_key(z[i]);
            if (key < thr) return false;
            if (!use_cut) return true;
            const unsigned long long ck = ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)i);
            return ck >= cut;
        };
        const int seg = (V + kST - 1) / kST;
        const int v0 = tid * seg, v1 = min(V, v0 + seg);
        float loc = 0.f;
        for (int i = v0; i < v1; ++i)
            if (kept(i)) loc += pval(i);
        float ZS;
        float run = block_exclusive_scan(loc, s_f, &ZS);
        const float target = (*u_ptr) * ZS;
        int cand = 0x7fffffff;
        for (int i = v0; i < v1; ++i) {
            if (!kept(i)) continue;
            run += pval(i);
            if (run > target) { cand = i; break; }
        }
        cand = block_min_i(cand, s_i);
        if (cand == 0x7fffffff) {
            // u * ZS at or beyond the rounded total: the last kept index
            int lk = -1;
            for (int i = v0; i < v1; ++i)
                if (kept(i)) lk = i;
            cand = block_max_i(lk, s_i);
        }
        tok = cand;
    }
    if (tok < 0 || tok >= V) {
        if (tid == 0 && err) atomicExch(err, 2);
        tok = 0;
    }
    __syncthreads();
    return tok;
}

}  // namespace sample_detail

inline size_t sample_smem_bytes_dev(int V) {
    int c = 1;
    while (c < V) c <<= 1;
    return sizeof(unsigned long long) * (size_t)c + 2 * sizeof(float) * (size_t)V;
}

}  // namespace sd
