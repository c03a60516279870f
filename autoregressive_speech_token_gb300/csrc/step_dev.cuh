// Device helpers shared by the persistent decode-step kernels (k_step.cu,
// k_cstep.cu): bounded waits on flag-carrying exchange words and on
// mbarriers, bulk asynchronous copies into shared memory, the per-CTA
// LayerNorm / RMSNorm of a staged activation row, and the dot products of one
// 16-byte unit of Q4_0 / Q8_0 codes with a lane's activations.  Both kernels
// run 512 compute threads that synchronise on named barrier 1, plus one
// producer warp that never joins it.
#pragma once
#include "k_gemv.cuh"

namespace sd {
namespace stepdev {

using namespace gemv_detail;

constexpr int kThreads = 512;             // compute threads
constexpr int kWarps = kThreads / 32;
constexpr int kBlock = kThreads + 32;     // + the producer warp
constexpr int kErrTimeout = 6;            // error-word code of an expired wait

__device__ __forceinline__ int ld_volatile(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

// barrier of the compute threads (named barrier 1)
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }
__device__ __forceinline__ int csync_and(int pred) {
    int r;
    asm volatile(
        "{ .reg .pred p, q; setp.ne.s32 p, %1, 0; bar.red.and.pred q, 1, 512, p; selp.s32 %0, 1, 0, q; }"
        : "=r"(r)
        : "r"(pred)
        : "memory");
    return r;
}

__device__ __forceinline__ unsigned long long gtime() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ flag-carrying words

__device__ __forceinline__ void ll_store(unsigned long long* p, float v, unsigned e) {
    const unsigned long long w = ((unsigned long long)e << 32) | (unsigned long long)__float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

__device__ __forceinline__ unsigned long long ll_load(const unsigned long long* p) {
    unsigned long long w;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}

// Polls one word until it carries epoch e; false on timeout or a recorded
// error.  After a few polls it backs off (a short sleep between loads), which
// frees L2 bandwidth for the producers' stores.
static __device__ __noinline__ bool ll_spin(const unsigned long long* p, unsigned e, unsigned long long* w, int* err,
                                     long long budget) {
    const long long t0 = clock64();
    for (unsigned it = 1;; ++it) {
        *w = ll_load(p);
        if ((unsigned)(*w >> 32) == e) return true;
        if (it > 4u) __nanosleep(64);
        if ((it & 63u) == 0u) {
            if (ld_volatile(err)) return false;
            if (clock64() - t0 > budget) {
                atomicCAS(err, 0, kErrTimeout);
                return false;
            }
        }
    }
}

// dst[o * n_in + i] = value of word src[o * stride + i] (epoch e), o < n_out, i < n_in;

// ------------------------------------------------------------------ weight records

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mb_init(uint32_t mb) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mb) : "memory");
}

__device__ __forceinline__ void mb_expect(uint32_t mb, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t mb) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(mb) : "memory");
}

// L2 policies for bulk copies: evict-first for data read once per step (the weight stream,
// more bytes per step than L2 holds), so that the step's code, KV cache and exchange words stay
// resident while the weights stream through; evict-normal otherwise.
__device__ __forceinline__ uint64_t l2_policy(bool evict_first) {
    uint64_t p;
    if (evict_first)
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    else
        asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void bulk_g2s_pol(uint32_t dst, const void* src, uint32_t bytes, uint32_t mb, uint64_t pol) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(mb), "l"(pol) : "memory");
}

__device__ __forceinline__ bool mb_try(uint32_t mb, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(mb), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for an mbarrier phase; honours the error flag unless `drain`.
static __device__ bool mb_wait(uint32_t mb, uint32_t parity, int* err, long long budget, bool drain) {
    if (mb_try(mb, parity)) return true;
    const long long t0 = clock64();
    for (unsigned it = 1;; ++it) {
        if (mb_try(mb, parity)) return true;
        if ((it & 15u) == 0u) {
            if (!drain && ld_volatile(err)) return false;
            if (clock64() - t0 > budget) {
                if (!drain) atomicCAS(err, 0, kErrTimeout);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void row_range(int R, int i, int G, int& r0, int& r1) {
    r0 = (int)((long long)R * i / G);
    r1 = (int)((long long)R * (i + 1) / G);
}

// ------------------------------------------------------------------ compute helpers

// LayerNorm (biased variance) or RMSNorm of the padded rows x[b][pidx(0..K)),
// b < NB, written to xn (same layout).  Each thread holds at most two float4
// of a row in registers (K <= 4096), so the row is read from shared memory
// once; the sums go through warp shuffles and a 16-entry table per row in
// `red` (>= 2 * NB * 16 floats, 16-byte aligned) in a fixed order.  LayerNorm
// is two-pass: the mean first, then the squared deviations of the held values.
template <int NB>
__device__ void norm_to(const float* x, float* xn, int K, bool ln, const float* g, const float* gb, float eps,
                        float* red) {
    constexpr int V = 2;
    const int KP = padded(K), K4 = K >> 2, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float4 v[NB][V];
    auto table_sum = [&](const float* t) {
        const float4* r4 = reinterpret_cast<const float4*>(t);
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps / 4; ++w) {
            const float4 q = r4[w];
            tot += (q.x + q.y) + (q.z + q.w);
        }
        return tot;
    };
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k4 = tid + j * kThreads;
            v[b][j] = k4 < K4 ? reinterpret_cast<const float4*>(x + b * KP)[k4 + (k4 >> 3)]
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 q = v[b][j];
            if (ln) s += (q.x + q.y) + (q.z + q.w);
            else s += fmaf(q.x, q.x, q.y * q.y) + fmaf(q.z, q.z, q.w * q.w);
        }
        s = warp_sum(s);
        if (lane == 0) red[b * kWarps + warp] = s;
    }
    csync();
    float mu[NB], ms[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const float tot = table_sum(red + b * kWarps);
        mu[b] = ln ? tot / (float)K : 0.f;
        ms[b] = tot / (float)K;
    }
    if (ln) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            float q = 0.f;
#pragma unroll
            for (int j = 0; j < V; ++j) {
                if (tid + j * kThreads >= K4) continue;
                const float a0 = v[b][j].x - mu[b], a1 = v[b][j].y - mu[b];
                const float a2 = v[b][j].z - mu[b], a3 = v[b][j].w - mu[b];
                q += fmaf(a0, a0, a1 * a1) + fmaf(a2, a2, a3 * a3);
            }
            q = warp_sum(q);
            if (lane == 0) red[(NB + b) * kWarps + warp] = q;
        }
        csync();
#pragma unroll
        for (int b = 0; b < NB; ++b) ms[b] = table_sum(red + (NB + b) * kWarps) / (float)K;
    }
    const float4* g4 = reinterpret_cast<const float4*>(g);
    const float4* b4 = reinterpret_cast<const float4*>(gb);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const float rs = 1.0f / sqrtf(ms[b] + eps);
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int k4 = tid + j * kThreads;
            if (k4 >= K4) continue;
            const float4 gg = g4[k4];
            float4 o = v[b][j];
            if (ln) {
                const float4 oo = b4[k4];
                o.x = fmaf((o.x - mu[b]) * rs, gg.x, oo.x);
                o.y = fmaf((o.y - mu[b]) * rs, gg.y, oo.y);
                o.z = fmaf((o.z - mu[b]) * rs, gg.z, oo.z);
                o.w = fmaf((o.w - mu[b]) * rs, gg.w, oo.w);
            } else {
                o.x = o.x * rs * gg.x;
                o.y = o.y * rs * gg.y;
                o.z = o.z * rs * gg.z;
                o.w = o.w * rs * gg.w;
            }
            reinterpret_cast<float4*>(xn + b * KP)[k4 + (k4 >> 3)] = o;
        }
    }
    csync();
}

// Partial dot products of one 16-byte weight unit with the lane's activations,
// in four independent accumulators (a short dependency chain).
__device__ __forceinline__ float dot4_q4(const uint4 w, const float* x) {
    const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t lo = (wd[i] >> (8 * k)) & 0xFu;
            const uint32_t hi = (wd[i] >> (8 * k + 4)) & 0xFu;
            const float flo = __int_as_float(0x4B000000u | lo) - (kMagic + 8.0f);
            const float fhi = __int_as_float(0x4B000000u | hi) - (kMagic + 8.0f);
            s[k] = fmaf(flo, x[4 * i + k], s[k]);
            s[k] = fmaf(fhi, x[16 + 4 * i + k], s[k]);
        }
    }
    return (s[0] + s[1]) + (s[2] + s[3]);
}

__device__ __forceinline__ float dot4_s8(const uint4 w, const float* x) {
    const uint32_t wd[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t u = (wd[i] >> (8 * k)) & 0xFFu;
            s[k] = fmaf(__int_as_float(0x4B000000u | u) - (kMagic + 128.0f), x[4 * i + k], s[k]);
        }
    }
    return (s[0] + s[1]) + (s[2] + s[3]);
}


}  // namespace stepdev
}  // namespace sd
