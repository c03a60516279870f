// On-device sampler: temperature -> top-k -> top-p -> draw
// ("Chatterbox -> ggml Port: Development Journal", section 3.2 and the
// defaults table of section 3.9; "Every Frame Is a Memory Read", section 5.6:
// top-p over the top-k survivors, scattered back into a full-vocabulary draw).
//
// One 1024-thread CTA per row, logits staged in shared memory:
//   greedy   argmax, ties to the lowest index;
//   top-k    4-pass 8-bit radix select of the k-th largest order-preserving
//            key -- every logit >= it survives (ties at the threshold kept);
//   softmax  p_i = exp((z_i - max) / T) over the survivors, fp32, fixed
//            summation order;
//   top-p    survivors sorted by (p desc, index asc) with a bitonic sort of
//            64-bit keys (logit key << 32 | ~index); the shortest prefix whose
//            mass reaches top_p * Z is kept;
//   draw     the smallest vocabulary index whose cumulative kept mass (index
//            order, block-wide prefix scan) exceeds u times the kept total.
#include "sd_internal.cuh"

namespace sd {
namespace {

constexpr int kST = 1024;
constexpr int kMaxV = 16384;

__device__ __forceinline__ uint32_t ord_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int pow2_ceil(int n) {
    int c = 1;
    while (c < n) c <<= 1;
    return c;
}

// exclusive scan of one float per thread (fixed order); returns the block total in *total
__device__ float block_exclusive_scan(float v, float* s_warp, float* total) {
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
        float w = s_warp[lane];
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

__device__ float block_sum_f(float v, float* s_warp) {
    float t;
    block_exclusive_scan(v, s_warp, &t);
    return t;
}

__device__ int block_min_i(int v, int* s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        int w = s[threadIdx.x];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w = min(w, __shfl_xor_sync(0xffffffffu, w, o));
        if (threadIdx.x == 0) s[32] = w;
    }
    __syncthreads();
    const int r = s[32];
    __syncthreads();
    return r;
}

__device__ int block_max_i(int v, int* s) { return -block_min_i(-v, s); }

__global__ void __launch_bounds__(kST) k_sample(const SampleArgs a) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x, tid = threadIdx.x;
    const int V = a.V;
    extern __shared__ __align__(16) unsigned char smraw[];
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(smraw);   // [pow2_ceil(V)]
    float* z = reinterpret_cast<float*>(smraw + sizeof(unsigned long long) * pow2_ceil(V));  // [V]
    __shared__ float s_f[72];
    __shared__ int s_i[40];
    __shared__ int s_hist[256];
    __shared__ uint32_t s_sel[3];  // prefix, mask, remaining
    __shared__ int s_cnt;

    const SampParams sp = *a.sp;
    const float* lg = a.logits + (size_t)b * a.ld;
    for (int i = tid; i < V; i += kST) z[i] = lg[i];
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
            best = s_f[tid];
            bi = s_i[tid];
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
            for (int i = tid; i < V; i += kST) {
                const uint32_t key = ord_key(z[i]);
                if ((key & mask) == prefix) atomicAdd(&s_hist[(key >> shift) & 255u], 1);
            }
            __syncthreads();
            if (tid == 0) {
                uint32_t rem = s_sel[2], cum = 0;
                int digit = 0;
                for (int d = 255; d >= 0; --d) {
                    if (cum + (uint32_t)s_hist[d] >= rem) { digit = d; rem -= cum; break; }
                    cum += (uint32_t)s_hist[d];
                }
                s_sel[0] = prefix | ((uint32_t)digit << shift);
                s_sel[1] = mask | (255u << shift);
                s_sel[2] = rem;
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
        for (int w = 1; w < 32; ++w) mx = fmaxf(mx, s_f[w]);
        __syncthreads();
        const float invT = 1.0f / sp.temperature;
        auto pval = [&](int i) { return expf((z[i] - mx) * invT); };

        // ---- top-p: cut key over the (p desc, index asc) order
        bool use_cut = false;
        unsigned long long cut = 0ull;
        if (sp.top_p < 1.0f) {
            float zp = 0.f;
            for (int i = tid; i < V; i += kST)
                if (ord_key(z[i]) >= thr) zp += pval(i);
            const float Z = block_sum_f(zp, s_f);
            if (tid == 0) s_cnt = 0;
            __syncthreads();
            for (int i = tid; i < V; i += kST) {
                const uint32_t key = ord_key(z[i]);
                if (key >= thr) {
                    const int slot = atomicAdd(&s_cnt, 1);
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
        float u;
        if (a.u_seq && *a.u_seq)
            u = (*a.u_seq)[(size_t)(*a.step_idx) * gridDim.x + b];
        else
            u = a.u[(size_t)b * a.u_stride + a.u_off];
        const float target = u * ZS;
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
    if (tid == 0) {
        if (tok < 0 || tok >= V) {
            if (a.err) atomicExch(a.err, 2);
            tok = 0;
        }
        a.out[(size_t)b * a.out_stride + a.out_off] = tok;
        if (a.out_seq && *a.out_seq)
            (*a.out_seq)[(size_t)(*a.step_idx) * gridDim.x + b] = tok;
    }
}

}  // namespace

size_t sample_smem_bytes(int V) {
    int c = 1;
    while (c < V) c <<= 1;
    return sizeof(unsigned long long) * (size_t)c + sizeof(float) * (size_t)V;
}

cudaError_t launch_sample(const SampleArgs& a, int rows, cudaStream_t st) {
    if (a.V < 1 || a.V > kMaxV) return cudaErrorInvalidValue;
    const size_t smem = sample_smem_bytes(a.V);
    cudaError_t e = cudaFuncSetAttribute(k_sample, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_k(k_sample, dim3(rows), dim3(kST), smem, st, a);
}

}  // namespace sd
