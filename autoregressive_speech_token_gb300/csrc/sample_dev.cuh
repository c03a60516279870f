// Block-level sampler (temperature -> top-k -> top-p -> index-order draw),
// shared by the sampler kernel and the persistent step kernels.
// "Chatterbox -> ggml Port: Development Journal", section 3.2 (order) and the
// defaults table of section 3.9; "Every Frame Is a Memory Read", section 5.6
// (top-p over the top-k survivors, drawn in full-vocabulary index order).
//
//   greedy   argmax, ties to the lowest index;
//   top-k    4-pass 8-bit radix select of the k-th largest order-preserving
//            logit key (counts; equal digits of a warp combine by match_any
//            into the warp's own histogram row, rows merged in fixed order) --
//            every logit whose key is >= it survives;
//   softmax  the survivors are compacted in index order with p_i =
//            exp((z_i - max) / T) (fp32), each mass also as a 2^-31
//            fixed-point integer so that every sum below is exact and
//            independent of summation order;
//   top-p    the survivors in (p desc, index asc) order are cut at the
//            shortest prefix whose mass reaches top_p * Z: a second 4-pass
//            radix select over the compacted survivors, on mass instead of
//            counts, finds the key of the element where the cumulative mass
//            crosses, and a prefix scan over its ties (index order) finds the
//            element itself;
//   draw     the smallest vocabulary index whose cumulative kept mass
//            (index order) exceeds u times the kept total.
// Shared memory: z[V], the compacted survivor indices and probabilities,
// one 256-bin count histogram per warp, and a small fixed scratch.  No sort.
#pragma once
#include "sd_internal.cuh"

// The block barrier and thread count the sampler uses: the whole block by
// default; a kernel whose block has threads outside the sampler (a producer
// warp) defines both before including this header.
#ifndef SAMPLE_SYNC
#define SAMPLE_SYNC() __syncthreads()
#define SAMPLE_NT ((int)blockDim.x)
#endif

namespace sd {
namespace sample_detail {

constexpr int kMaxV = 16384;
struct SampleScratch {
    float f[72];
    int i[40];
    unsigned long long q[72];
    unsigned hist[256];
    unsigned long long mass[256];
    uint32_t sel[4];  // key prefix, mask, remaining count; (top-p) tie index
    unsigned long long rem;
};

static __device__ __forceinline__ uint32_t ord_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// p * 2^31 truncated to an integer, for p in [0, 1], by integer operations on
// the float's fields (a float-to-64-bit-integer conversion is slow here).
static __device__ __forceinline__ unsigned long long fixq(float p) {
    const uint32_t u = __float_as_uint(p);
    const int e = (int)(u >> 23) - 127;  // p = 1.m * 2^e
    if (e < -31) return 0ull;            // below 2^-31 (and zero)
    const uint32_t m = (u & 0x7FFFFFu) | 0x800000u;
    const int sh = e + 8;                // p * 2^31 = m * 2^(e + 31 - 23)
    return sh >= 0 ? (unsigned long long)m << sh : (unsigned long long)(m >> (-sh));
}

// bytes of one [V] array of the sampler (z, survivor indices, survivor probabilities)
static __host__ __device__ __forceinline__ size_t sample_array_bytes(int V) { return ((size_t)4 * V + 15) & ~(size_t)15; }

// exclusive scan of one u64 per thread in thread order; *total = block total
static __device__ unsigned long long block_exclusive_scan_u64(unsigned long long v, unsigned long long* s,
                                                              unsigned long long* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = SAMPLE_NT >> 5;
    unsigned long long inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) s[warp] = inc;
    SAMPLE_SYNC();
    if (warp == 0) {
        const unsigned long long w = lane < nw ? s[lane] : 0ull;
        unsigned long long wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long t = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += t;
        }
        s[32 + lane] = wi - w;
        if (lane == 31) s[64] = wi;
    }
    SAMPLE_SYNC();
    const unsigned long long r = s[32 + warp] + inc - v;
    *total = s[64];
    SAMPLE_SYNC();
    return r;
}

static __device__ int block_min_i(int v, int* s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = v;
    SAMPLE_SYNC();
    if (threadIdx.x < 32) {
        int w = threadIdx.x < (SAMPLE_NT >> 5) ? s[threadIdx.x] : 0x7fffffff;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w = min(w, __shfl_xor_sync(0xffffffffu, w, o));
        if (threadIdx.x == 0) s[32] = w;
    }
    SAMPLE_SYNC();
    const int r = s[32];
    SAMPLE_SYNC();
    return r;
}

static __device__ float block_max_f(float v, float* s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = v;
    SAMPLE_SYNC();
    if (threadIdx.x < 32) {
        float w = threadIdx.x < (SAMPLE_NT >> 5) ? s[threadIdx.x] : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w = fmaxf(w, __shfl_xor_sync(0xffffffffu, w, o));
        if (threadIdx.x == 0) s[32] = w;
    }
    SAMPLE_SYNC();
    const float r = s[32];
    SAMPLE_SYNC();
    return r;
}

// One digit of a radix select over the active elements, from the top:
// finds the digit d (bits shift..shift+7 under the current prefix) at which
// the cumulative weight of higher digits stays below the remaining rank and
// reaches it within d.  Weights are per-digit totals in `w` (counts or fixed
// masses).  Run by warp 0.
template <typename T>
static __device__ __forceinline__ void select_digit(const T* w, T rem, int shift, uint32_t* sel, T* rem_out) {
    const int lane = threadIdx.x & 31;
    T c[8], own = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        c[j] = w[255 - 8 * lane - j];
        own += c[j];
    }
    T incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const T t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    const T excl = incl - own;
    const unsigned hit = __ballot_sync(0xffffffffu, excl < rem && incl >= rem);
    if (hit && lane == __ffs(hit) - 1) {
        T cum = excl;
        int digit = 255 - 8 * lane;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (cum + c[j] >= rem) {
                digit = 255 - 8 * lane - j;
                break;
            }
            cum += c[j];
        }
        sel[0] |= (uint32_t)digit << shift;
        sel[1] |= 255u << shift;
        *rem_out = rem - cum;
    }
}

// Samples one token from the logits already in shared memory (the first V
// floats of `smraw`, which holds sample_smem_bytes_dev(V, threads) bytes) with draw
// *u_ptr; every thread gets the token.  `ss` is the small scratch.  Block
// size: any multiple of 32 up to 1024.
static __device__ __noinline__ int sample_smem(int V, const SampParams sp, const float* u_ptr, unsigned char* smraw,
                                  SampleScratch& ss, int* err) {
    const int tid = threadIdx.x, nt = SAMPLE_NT, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
    const size_t arr = sample_array_bytes(V);
    float* z = reinterpret_cast<float*>(smraw);               // [V] logits
    int* ci = reinterpret_cast<int*>(smraw + arr);            // [V] survivor indices, ascending
    float* cp = reinterpret_cast<float*>(smraw + 2 * arr);    // [V] survivor probabilities
    unsigned* pc = reinterpret_cast<unsigned*>(smraw + 3 * arr);  // [nw][256] per-warp digit counts

    int tok;
    if (sp.greedy || sp.top_k == 1 || sp.temperature <= 0.f) {
        float best = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = tid; i < V; i += nt)
            if (z[i] > best) { best = z[i]; bi = i; }   // strided scan: first hit is the lowest index
        const float mx = block_max_f(best, ss.f);
        tok = block_min_i(best == mx ? bi : 0x7fffffff, ss.i);
    } else {
        float mloc = -INFINITY;
        for (int i = tid; i < V; i += nt) mloc = fmaxf(mloc, z[i]);
        const float mx = block_max_f(mloc, ss.f);

        // ---- top-k: key of the k-th largest logit (counts, 4 x 8-bit digits); each warp
        // counts into its own histogram row, so equal digits collide only within a warp.
        const int k = (sp.top_k < 1 || sp.top_k > V) ? V : sp.top_k;
        uint32_t thr = 0u;
        if (k < V) {
            if (tid == 0) { ss.sel[0] = 0u; ss.sel[1] = 0u; ss.sel[2] = (uint32_t)k; }
            for (int shift = 24; shift >= 0; shift -= 8) {
                // the first digit (sign and high exponent bits) is shared by most logits: each
                // warp counts into its own row, rows merged in fixed order; later digits are
                // spread, and one shared histogram takes few colliding atomics
                const bool first = shift == 24;
                if (first)
                    for (int i = tid; i < nw * 256; i += nt) pc[i] = 0u;
                else
                    for (int i = tid; i < 256; i += nt) ss.hist[i] = 0u;
                SAMPLE_SYNC();
                const uint32_t prefix = ss.sel[0], mask = ss.sel[1];
                unsigned* row = first ? pc + warp * 256 : ss.hist;
                for (int i = tid; i < V; i += nt) {
                    const uint32_t key = ord_key(z[i]);
                    if ((key & mask) == prefix) atomicAdd(&row[(key >> shift) & 255u], 1u);
                }
                SAMPLE_SYNC();
                if (first) {
                    for (int bn = tid; bn < 256; bn += nt) {
                        unsigned t = 0u;
                        for (int w = 0; w < nw; ++w) t += pc[w * 256 + bn];
                        ss.hist[bn] = t;
                    }
                    SAMPLE_SYNC();
                }
                if (tid < 32) {
                    uint32_t rem_out = 0;
                    select_digit<uint32_t>(ss.hist, ss.sel[2], shift, ss.sel, &rem_out);
                    const unsigned any = __ballot_sync(0xffffffffu, rem_out != 0u);
                    if (any && lane == __ffs(any) - 1) ss.sel[2] = rem_out;
                }
                SAMPLE_SYNC();
            }
            thr = ss.sel[0];
        }

        // ---- survivors compacted in index order (contiguous segment per thread), with their
        // probabilities and the exact fixed-point total
        const float invT = 1.0f / sp.temperature;
        int ns;
        unsigned long long Zq;
        {
            const int seg = (V + nt - 1) / nt;
            const int a0 = min(V, tid * seg), a1 = min(V, a0 + seg);
            int cnt = 0;
            for (int i = a0; i < a1; ++i) cnt += ord_key(z[i]) >= thr;
            unsigned long long tot;
            int off = (int)block_exclusive_scan_u64((unsigned long long)cnt, ss.q, &tot);
            ns = (int)tot;
            unsigned long long zl = 0ull;
            for (int i = a0; i < a1; ++i) {
                if (ord_key(z[i]) < thr) continue;
                const float p = expf((z[i] - mx) * invT);
                ci[off] = i;
                cp[off] = p;
                zl += fixq(p);
                ++off;
            }
            block_exclusive_scan_u64(zl, ss.q, &Zq);  // barrier: the compacted arrays are complete
        }

        // ---- top-p over the survivors: crossing key by a mass radix select, then its ties
        bool cut = false;
        uint32_t tkey = 0u;
        int tidx = 0x7fffffff;
        if (sp.top_p < 1.0f) {
            if (tid == 0) {
                const unsigned long long T = (unsigned long long)ceil((double)sp.top_p * (double)Zq);
                ss.sel[0] = 0u; ss.sel[1] = 0u; ss.rem = T > 0ull ? T : 1ull;
            }
            unsigned* mh = pc;        // per-digit sums of the masses' high and low 16-bit halves
            unsigned* ml = pc + 256;  // (32-bit shared atomics; exact: at most 2^14 * 2^16 each)
            for (int shift = 24; shift >= 0; shift -= 8) {
                for (int i = tid; i < 512; i += nt) pc[i] = 0u;
                SAMPLE_SYNC();
                const uint32_t prefix = ss.sel[0], mask = ss.sel[1];
                for (int j0 = 0; j0 < ns; j0 += nt) {
                    const int j = j0 + tid;
                    const uint32_t key = j < ns ? ord_key(z[ci[j]]) : 0u;
                    bool in = j < ns && (key & mask) == prefix;
                    const uint32_t digit = (key >> shift) & 255u;
                    const unsigned long long q = in ? fixq(cp[j]) : 0ull;
                    if (shift != 24) {
                        // later digits are spread: direct atomics collide little
                        if (in) {
                            atomicAdd(&mh[digit], (unsigned)(q >> 16));
                            atomicAdd(&ml[digit], (unsigned)(q & 0xFFFFu));
                        }
                        continue;
                    }
                    // first digit: one full-warp reduction per distinct digit among the active lanes
                    unsigned pend = __ballot_sync(0xffffffffu, in);
                    while (pend) {
                        const uint32_t dg = __shfl_sync(0xffffffffu, digit, __ffs(pend) - 1);
                        const bool mine = in && digit == dg;
                        const unsigned hi = __reduce_add_sync(0xffffffffu, mine ? (unsigned)(q >> 16) : 0u);
                        const unsigned lo = __reduce_add_sync(0xffffffffu, mine ? (unsigned)(q & 0xFFFFu) : 0u);
                        if (lane == __ffs(pend) - 1) {
                            atomicAdd(&mh[dg], hi);
                            atomicAdd(&ml[dg], lo);
                        }
                        pend &= ~__ballot_sync(0xffffffffu, mine);
                        if (mine) in = false;
                    }
                }
                SAMPLE_SYNC();
                for (int bn = tid; bn < 256; bn += nt)
                    ss.mass[bn] = ((unsigned long long)mh[bn] << 16) + (unsigned long long)ml[bn];
                SAMPLE_SYNC();
                if (tid < 32) {
                    unsigned long long rem_out = 0ull;
                    select_digit<unsigned long long>(ss.mass, ss.rem, shift, ss.sel, &rem_out);
                    const unsigned any = __ballot_sync(0xffffffffu, rem_out != 0ull);
                    if (any && lane == __ffs(any) - 1) ss.rem = rem_out;
                }
                SAMPLE_SYNC();
            }
            tkey = ss.sel[0];
            const unsigned long long rem = ss.rem;  // mass still needed from the elements with key == tkey
            const int seg = (ns + nt - 1) / nt;
            const int b0 = min(ns, tid * seg), b1 = min(ns, b0 + seg);
            unsigned long long loc = 0ull;
            for (int j = b0; j < b1; ++j)
                if (ord_key(z[ci[j]]) == tkey) loc += fixq(cp[j]);
            unsigned long long tot;
            unsigned long long run = block_exclusive_scan_u64(loc, ss.q, &tot);
            int c = 0x7fffffff;
            for (int j = b0; j < b1; ++j) {
                if (ord_key(z[ci[j]]) != tkey) continue;
                run += fixq(cp[j]);
                if (run >= rem) { c = ci[j]; break; }
            }
            tidx = block_min_i(c, ss.i);
            cut = true;
        }

        // ---- draw in vocabulary order over the kept survivors (exact fixed-point prefix sums)
        auto kept = [&](int j) {
            if (!cut) return true;
            const uint32_t key = ord_key(z[ci[j]]);
            return key > tkey || (key == tkey && ci[j] <= tidx);
        };
        const int seg = (ns + nt - 1) / nt;
        const int b0 = min(ns, tid * seg), b1 = min(ns, b0 + seg);
        unsigned long long loc = 0ull;
        for (int j = b0; j < b1; ++j)
            if (kept(j)) loc += fixq(cp[j]);
        unsigned long long ZS;
        unsigned long long run = block_exclusive_scan_u64(loc, ss.q, &ZS);
        if (tid == 0) ss.rem = (unsigned long long)floor((double)(*u_ptr) * (double)ZS);
        SAMPLE_SYNC();
        const unsigned long long target = ss.rem;
        int cand = 0x7fffffff;
        for (int j = b0; j < b1; ++j) {
            if (!kept(j)) continue;
            run += fixq(cp[j]);
            if (run > target) { cand = ci[j]; break; }
        }
        tok = block_min_i(cand, ss.i);
    }
    if (tok < 0 || tok >= V) {
        if (tid == 0 && err) atomicExch(err, 2);
        tok = 0;
    }
    SAMPLE_SYNC();
    return tok;
}

// ---------------------------------------------------------------- fast path
//
// The same sampler (the same survivors, fixed-point masses, cut and draw as
// sample_smem) located through value histograms instead of radix passes.  The
// logits are binned linearly between their minimum and maximum (kFB bins, bin
// 0 holding the largest): the bin of a value is a monotone function of it, so
// equal values share a bin and every value of a bin is at least every value of
// a later bin.  One count histogram and one prefix over the bins find the bin
// holding the k-th largest logit; the exact k-th largest key is then selected
// among that bin's members.  The top-p cut is found the same way on a histogram
// of fixed-point masses: the bin where the cumulative mass (from the top)
// reaches T = ceil(top_p * Z), then, among its members in (key desc, index asc)
// order, the element where it does.  The draw target is floor(u * ZS).  Both
// products are formed exactly in integers (a float times a 64-bit integer, a
// 128-bit product), the same on every thread.  Every block-wide reduction or
// scan takes one barrier: the warps leave their partials in shared memory and
// each warp then folds all of them itself.  A bin with more than kFC members (a
// degenerate distribution) falls back to sample_smem.  The caller must pass a
// barrier before it reuses the sampler's shared memory.
constexpr int kFB = 2048, kFC = 1024;

// shared memory after z[V]: the survivors' masses q[V] (u32), the count and mass histograms, the candidates
static __host__ __device__ __forceinline__ size_t sample_fast_extra_bytes(int V) {
    return sample_array_bytes(V) + (size_t)kFB * 4 + (size_t)kFB * 8 + (size_t)kFC * (4 + 4 + 4) + 64;
}

static __device__ __forceinline__ int vbin(float z, float mx, float sc) {
    const float f = (mx - z) * sc;  // >= 0, non-decreasing as z decreases
    return f >= (float)(kFB - 1) ? kFB - 1 : (int)f;
}

static __device__ float block_min_f(float v, float* s) {
    return -block_max_f(-v, s);
}

static __device__ __forceinline__ unsigned warp_incl_scan_u32(unsigned v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

static __device__ __forceinline__ unsigned long long warp_incl_scan_u64(unsigned long long v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// ceil(p * n) (up) or floor(p * n) for a float p in [0, 1] and an integer n, exactly:
// p = m * 2^-sh with a 24-bit m, and m * n is formed in 128 bits
static __device__ __forceinline__ unsigned long long mul_frac(float p, unsigned long long n, bool up) {
    if (!(p > 0.f) || n == 0ull) return 0ull;
    if (p >= 1.0f) return n;
    const uint32_t u = __float_as_uint(p);
    const int ex = (int)(u >> 23);  // p > 0: the sign bit is clear
    const unsigned long long m = ex ? ((u & 0x7FFFFFu) | 0x800000u) : (u & 0x7FFFFFu);
    const int sh = ex ? 150 - ex : 149;  // p = m * 2^-sh, sh >= 24 for p < 1
    const unsigned long long lo = m * n, hi = __umul64hi(m, n);
    unsigned long long q;
    bool rem;
    if (sh >= 128) {
        q = 0ull;
        rem = true;
    } else if (sh >= 64) {
        q = hi >> (sh - 64);
        rem = lo != 0ull || (sh > 64 && (hi & ((1ull << (sh - 64)) - 1ull)) != 0ull);
    } else {
        q = (hi << (64 - sh)) | (lo >> sh);
        rem = (lo & ((1ull << sh) - 1ull)) != 0ull;
    }
    return q + ((up && rem) ? 1ull : 0ull);
}

// f(i, z[i]) for this thread's elements i = tid, tid + nt, ... < V, the loads issued four at a time
template <typename F>
static __device__ __forceinline__ void for_strided(const float* z, int V, F&& f) {
    const int tid = threadIdx.x, nt = SAMPLE_NT;
    for (int i0 = tid; i0 < V; i0 += 4 * nt) {
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * nt;
            v[j] = i < V ? z[i] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * nt;
            if (i < V) f(i, v[j]);
        }
    }
}

// as for_strided, with qv[i] loaded beside z[i]
template <typename F>
static __device__ __forceinline__ void for_strided_q(const float* z, const unsigned* qv, int V, F&& f) {
    const int tid = threadIdx.x, nt = SAMPLE_NT;
    for (int i0 = tid; i0 < V; i0 += 4 * nt) {
        float v[4];
        unsigned q[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * nt;
            v[j] = i < V ? z[i] : 0.f;
            q[j] = i < V ? qv[i] : 0u;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * nt;
            if (i < V) f(i, v[j], q[j]);
        }
    }
}

// f(i, z[i], qv[i]) for i in [a0, a1) in order, the loads issued eight at a time; f returns false to stop
template <typename F>
static __device__ __forceinline__ void for_segment(const float* z, const unsigned* qv, int a0, int a1, F&& f) {
    for (int b = a0; b < a1; b += 8) {
        float v[8];
        unsigned q[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int i = b + j;
            v[j] = i < a1 ? z[i] : 0.f;
            q[j] = i < a1 ? qv[i] : 0u;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (b + j < a1 && !f(b + j, v[j], q[j])) return;
    }
}

static __device__ __noinline__ int sample_fast(int V, const SampParams sp, const float* u_ptr, unsigned char* smraw,
                                               SampleScratch& ss, int* err) {
    const int tid = threadIdx.x, nt = SAMPLE_NT, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
    if (sp.greedy || sp.top_k == 1 || sp.temperature <= 0.f || nt * 4 != kFB)
        return sample_smem(V, sp, u_ptr, smraw, ss, err);
    const size_t arr = sample_array_bytes(V);
    const float* z = reinterpret_cast<const float*>(smraw);
    // each survivor's mass p * 2^31 (truncated, <= 2^31: fits 32 bits); 0 for the others
    unsigned* qv = reinterpret_cast<unsigned*>(smraw + arr);               // [V]
    unsigned* cnt = reinterpret_cast<unsigned*>(smraw + 2 * arr);          // [kFB]
    // per-bin masses as sums of their high and low 16-bit halves (32-bit shared atomics; exact:
    // at most 2^14 terms of at most 2^16 each)
    unsigned* mh = cnt + kFB;                                              // [kFB]
    unsigned* ml = mh + kFB;                                               // [kFB]
    uint32_t* ckey = ml + kFB;                                             // [kFC]
    int* cidx = reinterpret_cast<int*>(ckey + kFC);                        // [kFC]
    unsigned* cq = reinterpret_cast<unsigned*>(cidx + kFC);                // [kFC]

    // ---- the range of the logits; the histograms cleared on the way
    float mloc = -INFINITY, nloc = INFINITY;
    for_strided(z, V, [&](int, float v) {
        mloc = fmaxf(mloc, v);
        nloc = fminf(nloc, v);
    });
    for (int b = tid; b < kFB; b += nt) {
        cnt[b] = 0u;
        mh[b] = 0u;
        ml[b] = 0u;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
        nloc = fminf(nloc, __shfl_xor_sync(0xffffffffu, nloc, o));
    }
    if (lane == 0) {
        ss.f[warp] = mloc;
        ss.f[32 + warp] = nloc;
    }
    if (tid == 0) {
        ss.i[0] = 0;
        ss.i[1] = 0;
    }
    SAMPLE_SYNC();
    float mx = ss.f[0], mn = ss.f[32];
    for (int w = 1; w < nw; ++w) {
        mx = fmaxf(mx, ss.f[w]);
        mn = fminf(mn, ss.f[32 + w]);
    }
    // (capped: a range near the smallest normal would make the scale infinite, and 0 * inf is not 0)
    const float sc = mx > mn ? fminf((float)(kFB - 1) / (mx - mn), 1e30f) : 0.f;
    const int k = (sp.top_k < 1 || sp.top_k > V) ? V : sp.top_k;
    const float invT = 1.0f / sp.temperature;

    // ---- top-k threshold key
    uint32_t thr = 0u;
    if (k < V) {
        for_strided(z, V, [&](int, float v) { atomicAdd(&cnt[vbin(v, mx, sc)], 1u); });
        SAMPLE_SYNC();
        const uint4 c4 = reinterpret_cast<const uint4*>(cnt)[tid];  // bins 4 tid .. 4 tid + 3
        const unsigned own = c4.x + c4.y + c4.z + c4.w;
        const unsigned inc = warp_incl_scan_u32(own);
        if (lane == 31) ss.i[8 + warp] = (int)inc;
        SAMPLE_SYNC();
        unsigned cum = inc - own;
        for (int w = 0; w < warp; ++w) cum += (unsigned)ss.i[8 + w];
        const unsigned cb[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (cum < (unsigned)k && cum + cb[j] >= (unsigned)k) {
                ss.i[2] = 4 * tid + j;   // the bin of the k-th largest
                ss.i[3] = k - (int)cum;  // its rank inside the bin (1 = the bin's largest)
                ss.i[4] = (int)cb[j];
            }
            cum += cb[j];
        }
        SAMPLE_SYNC();
        const int bk = ss.i[2], rk = ss.i[3], nbk = ss.i[4];
        if (nbk > kFC) return sample_smem(V, sp, u_ptr, smraw, ss, err);
        for_strided(z, V, [&](int, float v) {
            if (vbin(v, mx, sc) == bk) ckey[atomicAdd(&ss.i[0], 1)] = ord_key(v);
        });
        SAMPLE_SYNC();
        for (int c = tid; c < nbk; c += nt) {
            const uint32_t key = ckey[c];
            int gt = 0, ge = 0;
            for (int j = 0; j < nbk; ++j) {
                gt += ckey[j] > key;
                ge += ckey[j] >= key;
            }
            if (gt < rk && rk <= ge) ss.sel[0] = key;  // every writer writes the same key
        }
        SAMPLE_SYNC();
        thr = ss.sel[0];
    }

    // ---- survivors' fixed-point masses: the total, and (for top-p) per bin
    const bool topp = sp.top_p < 1.0f;
    unsigned long long zl = 0ull;
    for_strided(z, V, [&](int i, float v) {
        unsigned q = 0u;
        if (ord_key(v) >= thr) {
            q = (unsigned)fixq(expf((v - mx) * invT));
            if (topp && q) {
                const int bn = vbin(v, mx, sc);
                atomicAdd(&mh[bn], q >> 16);
                atomicAdd(&ml[bn], q & 0xFFFFu);
            }
        }
        qv[i] = q;
        zl += q;
    });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zl += __shfl_xor_sync(0xffffffffu, zl, o);
    if (lane == 0) ss.q[warp] = zl;
    SAMPLE_SYNC();  // also: the mass histograms and qv are complete
    unsigned long long Zq = 0ull;
    for (int w = 0; w < nw; ++w) Zq += ss.q[w];

    // ---- top-p cut: (tkey, tidx) of the element where the (key desc, index asc) cumulative mass
    // reaches T = ceil(top_p * Z)
    bool cut = false;
    uint32_t tkey = 0u;
    int tidx = 0x7fffffff;
    if (topp) {
        unsigned long long T = mul_frac(sp.top_p, Zq, true);
        if (T == 0ull) T = 1ull;
        const uint4 h4 = reinterpret_cast<const uint4*>(mh)[tid], l4 = reinterpret_cast<const uint4*>(ml)[tid];
        const unsigned long long mb[4] = {((unsigned long long)h4.x << 16) + l4.x, ((unsigned long long)h4.y << 16) + l4.y,
                                          ((unsigned long long)h4.z << 16) + l4.z, ((unsigned long long)h4.w << 16) + l4.w};
        const unsigned long long own = mb[0] + mb[1] + mb[2] + mb[3];
        const unsigned long long inc = warp_incl_scan_u64(own);
        if (lane == 31) ss.q[16 + warp] = inc;
        SAMPLE_SYNC();
        unsigned long long cum = inc - own;
        for (int w = 0; w < warp; ++w) cum += ss.q[16 + w];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (cum < T && cum + mb[j] >= T) {
                ss.i[5] = 4 * tid + j;  // the bin where the cumulative mass reaches T
                ss.rem = T - cum;       // mass still needed inside it
            }
            cum += mb[j];
        }
        SAMPLE_SYNC();
        const int bp = ss.i[5];
        const unsigned long long remT = ss.rem;
        // its members that carry mass (a survivor without mass cannot be where the mass crosses,
        // nor change anything before it)
        for_strided_q(z, qv, V, [&](int i, float v, unsigned q) {
            if (q == 0u || vbin(v, mx, sc) != bp) return;
            const int c = atomicAdd(&ss.i[1], 1);
            if (c < kFC) {
                ckey[c] = ord_key(v);
                cidx[c] = i;
                cq[c] = q;
            }
        });
        SAMPLE_SYNC();
        const int np = ss.i[1];
        if (np > kFC) return sample_smem(V, sp, u_ptr, smraw, ss, err);
        for (int c = tid; c < np; c += nt) {
            const uint32_t key = ckey[c];
            const int idx = cidx[c];
            unsigned long long pre = 0ull;  // mass before this element in (key desc, index asc) order
            for (int j = 0; j < np; ++j)
                if (ckey[j] > key || (ckey[j] == key && cidx[j] < idx)) pre += cq[j];
            if (pre < remT && pre + (unsigned long long)cq[c] >= remT) {
                ss.sel[1] = key;
                ss.sel[2] = (uint32_t)idx;
            }
        }
        SAMPLE_SYNC();
        tkey = ss.sel[1];
        tidx = (int)ss.sel[2];
        cut = true;
    }

    // ---- draw in vocabulary order over the kept elements (exact fixed-point prefix sums; each
    // thread takes one contiguous segment)
    auto kept = [&](int i, float v) {
        if (!cut) return true;  // qv is 0 for the elements under the top-k threshold
        const uint32_t key = ord_key(v);
        return key > tkey || (key == tkey && i <= tidx);
    };
    const int seg = (V + nt - 1) / nt;
    const int a0 = min(V, tid * seg), a1 = min(V, a0 + seg);
    unsigned long long loc = 0ull;
    for_segment(z, qv, a0, a1, [&](int i, float v, unsigned q) {
        if (q && kept(i, v)) loc += q;
        return true;
    });
    const unsigned long long inc = warp_incl_scan_u64(loc);
    if (lane == 31) ss.q[32 + warp] = inc;
    SAMPLE_SYNC();
    unsigned long long run = inc - loc, ZS = 0ull;
    for (int w = 0; w < nw; ++w) {
        const unsigned long long t = ss.q[32 + w];
        ZS += t;
        if (w < warp) run += t;
    }
    const unsigned long long target = mul_frac(*u_ptr, ZS, false);
    int cand = 0x7fffffff;
    for_segment(z, qv, a0, a1, [&](int i, float v, unsigned q) {
        if (q == 0u || !kept(i, v)) return true;
        run += q;
        if (run > target) {
            cand = i;
            return false;
        }
        return true;
    });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
    if (lane == 0) ss.hist[warp] = (unsigned)cand;
    SAMPLE_SYNC();
    int tok = 0x7fffffff;
    for (int w = 0; w < nw; ++w) tok = min(tok, (int)ss.hist[w]);
    if (tok < 0 || tok >= V) {
        if (tid == 0 && err) atomicExch(err, 2);
        tok = 0;
    }
    return tok;
}

constexpr int kRS = 17;   // elements per thread held in registers (V <= 17 * SAMPLE_NT)

static __device__ __forceinline__ int lower_bound_u64(const unsigned long long* a, int n, unsigned long long t) {
    int lo = 0, hi = n;  // first index in [0, n) with a[i] >= t, or n
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] >= t) hi = mid; else lo = mid + 1;
    }
    return lo;
}

// The same search over the kFB non-decreasing bin prefixes `pre` by one warp, in two rounds of
// loads: cend[c] = pre[64c + 63] picks the 64-bin chunk, then each lane tests one pair of bins.
// Every lane returns min(first bin with pre >= t, n).
static __device__ __forceinline__ int lower_bound_warp(const unsigned long long* pre, const unsigned long long* cend,
                                                       int n, unsigned long long t) {
    const int lane = threadIdx.x & 31;
    const unsigned mc = __ballot_sync(0xffffffffu, cend[lane] >= t);
    if (!mc) return n;
    const int c = __ffs(mc) - 1;
    const ulonglong2 e = reinterpret_cast<const ulonglong2*>(pre)[32 * c + lane];  // bins 64c + 2 lane, + 1
    const unsigned m1 = __ballot_sync(0xffffffffu, e.y >= t), m0 = __ballot_sync(0xffffffffu, e.x >= t);
    const int l = __ffs(m1) - 1;  // m1 != 0: the chunk's last bin reaches t
    const int b = 64 * c + 2 * l + (((m0 >> l) & 1u) ? 0 : 1);
    return b < n ? b : n;
}

// The path every kernel takes first for a sampled row (512 threads, V <= 17 * 512): the same
// survivors, cut and draw as sample_fast, with each thread's logits and fixed-point masses held
// in registers over a contiguous segment of the vocabulary (odd segment length: the loads hit
// 32 distinct banks).  One pass builds the count and mass histograms over the value bins
// together (masses of every element; the bins above the k-th largest hold survivors only), one
// scan gives each bin's inclusive mass prefix, and one pass collects the members of the k-th
// bin and of the bins where the top-p cut can fall (the cut's T = ceil(top_p * Z) is bracketed
// by Z's bounds before the k-th bin is resolved).  Warp 0 then resolves the threshold key, Z,
// T and the cut element; the draw scans the kept masses in vocabulary order.  Eight barriers.
static __device__ __noinline__ int sample_reg(int V, const SampParams sp, const float* u_ptr, unsigned char* smraw,
                                              SampleScratch& ss, int* err) {
    const int tid = threadIdx.x, nt = SAMPLE_NT, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
    int S = (V + nt - 1) / nt;
    S |= 1;  // odd: lane stride S hits 32 distinct banks
    if (sp.greedy || sp.top_k == 1 || sp.temperature <= 0.f || nt * 4 != kFB || S > kRS)
        return sample_fast(V, sp, u_ptr, smraw, ss, err);
    const size_t arr = sample_array_bytes(V);
    const float* z = reinterpret_cast<const float*>(smraw);
    unsigned* cnt = reinterpret_cast<unsigned*>(smraw + arr);             // [kFB]
    unsigned* mh = cnt + kFB;                                              // [kFB]
    unsigned* ml = mh + kFB;                                               // [kFB]
    unsigned long long* pre = reinterpret_cast<unsigned long long*>(mh);   // [kFB] after the scan
    uint32_t* ckey = ml + kFB;                                             // [kFC]
    unsigned* cbi = ckey + kFC;                                            // [kFC] bin << 14 | index
    unsigned* cq = cbi + kFC;                                              // [kFC]
    const int a0 = tid * S;

    // ---- P1: this thread's logits into registers; range; histograms cleared
    float v[kRS];
    float mloc = -INFINITY, nloc = INFINITY;
#pragma unroll
    for (int j = 0; j < kRS; ++j) {
        const int i = a0 + j;
        v[j] = (j < S && i < V) ? z[i] : 0.f;
        if (j < S && i < V) {
            mloc = fmaxf(mloc, v[j]);
            nloc = fminf(nloc, v[j]);
        }
    }
    for (int b = tid; b < kFB; b += nt) {
        cnt[b] = 0u;
        mh[b] = 0u;
        ml[b] = 0u;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
        nloc = fminf(nloc, __shfl_xor_sync(0xffffffffu, nloc, o));
    }
    if (lane == 0) {
        ss.f[warp] = mloc;
        ss.f[32 + warp] = nloc;
    }
    if (tid == 0) {
        ss.i[0] = 0;
        ss.i[2] = 0;
        ss.i[3] = 1;
        ss.i[6] = -1;
        ss.q[40] = 0ull;
    }
    SAMPLE_SYNC();
    float mx = ss.f[0], mn = ss.f[32];
    for (int w = 1; w < nw; ++w) {
        mx = fmaxf(mx, ss.f[w]);
        mn = fminf(mn, ss.f[32 + w]);
    }
    const float sc = mx > mn ? fminf((float)(kFB - 1) / (mx - mn), 1e30f) : 0.f;
    const int k = (sp.top_k < 1 || sp.top_k > V) ? V : sp.top_k;
    const bool topk = k < V, topp = sp.top_p < 1.0f;
    const float invT = 1.0f / sp.temperature;

    // ---- P2: masses of every element; count and mass histograms over the bins
    unsigned q[kRS];
#pragma unroll
    for (int j = 0; j < kRS; ++j) {
        q[j] = 0u;
        if (j < S && a0 + j < V) {
            q[j] = (unsigned)fixq(expf((v[j] - mx) * invT));
            const int bn = vbin(v[j], mx, sc);
            atomicAdd(&cnt[bn], 1u);
            if (q[j]) {
                atomicAdd(&mh[bn], q[j] >> 16);
                atomicAdd(&ml[bn], q[j] & 0xFFFFu);
            }
        }
    }
    SAMPLE_SYNC();

    // ---- P3: scans of counts and masses over the bins (4 bins per thread)
    const uint4 c4 = reinterpret_cast<const uint4*>(cnt)[tid];
    const uint4 h4 = reinterpret_cast<const uint4*>(mh)[tid], l4 = reinterpret_cast<const uint4*>(ml)[tid];
    const unsigned cb[4] = {c4.x, c4.y, c4.z, c4.w};
    const unsigned long long mb[4] = {((unsigned long long)h4.x << 16) + l4.x, ((unsigned long long)h4.y << 16) + l4.y,
                                      ((unsigned long long)h4.z << 16) + l4.z, ((unsigned long long)h4.w << 16) + l4.w};
    const unsigned ownc = cb[0] + cb[1] + cb[2] + cb[3];
    const unsigned long long ownm = mb[0] + mb[1] + mb[2] + mb[3];
    const unsigned incc = warp_incl_scan_u32(ownc);
    const unsigned long long incm = warp_incl_scan_u64(ownm);
    if (lane == 31) {
        ss.i[8 + warp] = (int)incc;
        ss.q[16 + warp] = incm;
    }
    SAMPLE_SYNC();

    // ---- P4: inclusive mass prefix per bin; the bin of the k-th largest
    {
        unsigned cc = incc - ownc;
        unsigned long long cm = incm - ownm;
        for (int w = 0; w < warp; ++w) {
            cc += (unsigned)ss.i[8 + w];
            cm += ss.q[16 + w];
        }
        unsigned long long pr[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (topk && cc < (unsigned)k && cc + cb[j] >= (unsigned)k) {
                ss.i[2] = 4 * tid + j;   // the bin of the k-th largest
                ss.i[3] = k - (int)cc;   // its rank inside the bin (1 = the bin's largest)
                ss.i[4] = (int)cb[j];
                ss.q[40] = cm;           // the mass of the bins before it
            }
            cc += cb[j];
            cm += mb[j];
            pr[j] = cm;
        }
        reinterpret_cast<ulonglong2*>(pre)[2 * tid] = make_ulonglong2(pr[0], pr[1]);
        reinterpret_cast<ulonglong2*>(pre)[2 * tid + 1] = make_ulonglong2(pr[2], pr[3]);
        if ((tid & 15) == 15) ss.mass[tid >> 4] = pr[3];  // prefix at the end of 64-bin chunk tid / 16
    }
    SAMPLE_SYNC();

    // ---- P5: the members of the k-th bin and of the bins where the top-p cut can fall
    unsigned long long Ztot = 0ull;
    for (int w = 0; w < nw; ++w) Ztot += ss.q[16 + w];
    const int bk = topk ? ss.i[2] : kFB;               // kFB: no top-k bin
    const unsigned long long mAbove = topk ? ss.q[40] : Ztot;
    int blo = kFB, bhi = -1;
    if (topp) {
        const unsigned long long zhi = topk ? pre[bk] : Ztot;  // Z lies in [mAbove, zhi]
        unsigned long long tlo = mul_frac(sp.top_p, mAbove, true), thi = mul_frac(sp.top_p, zhi, true);
        if (tlo == 0ull) tlo = 1ull;
        if (thi == 0ull) thi = 1ull;
        const int lim = topk ? bk : kFB;
        blo = lower_bound_warp(pre, ss.mass, lim, tlo);
        bhi = lower_bound_warp(pre, ss.mass, lim, thi);
        if (bhi >= lim) bhi = lim - 1;
    }
#pragma unroll
    for (int j = 0; j < kRS; ++j) {
        const int i = a0 + j;
        if (j < S && i < V) {
            const int bn = vbin(v[j], mx, sc);
            if (bn == bk || (bn >= blo && bn <= bhi)) {
                const int c = atomicAdd(&ss.i[0], 1);
                if (c < kFC) {
                    ckey[c] = ord_key(v[j]);
                    cbi[c] = ((unsigned)bn << 14) | (unsigned)i;
                    cq[c] = q[j];
                }
            }
        }
    }
    SAMPLE_SYNC();
    const int nm = ss.i[0];
    if (nm > kFC) return sample_smem(V, sp, u_ptr, smraw, ss, err);

    // ---- P6 (warp 0): the top-k threshold key and the top-p cut element
    if (warp == 0 && nm <= 32) {
        // members in the lanes' registers; pairwise comparisons by shuffles
        const bool has = lane < nm;
        const uint32_t mk = has ? ckey[lane] : 0u;
        const unsigned mbi = has ? cbi[lane] : 0u, mq = has ? cq[lane] : 0u;
        const int mbin = has ? (int)(mbi >> 14) : -1, midx = (int)(mbi & 0x3FFFu);
        const int rk = topk ? ss.i[3] : 0;
        uint32_t thr = 0u;
        unsigned long long sk = 0ull;
        if (topk) {
            int gt = 0, ge = 0;
            for (int j = 0; j < nm; ++j) {
                const uint32_t kj = __shfl_sync(0xffffffffu, mk, j);
                const int bj = __shfl_sync(0xffffffffu, mbin, j);
                if (bj == bk) {
                    gt += kj > mk;
                    ge += kj >= mk;
                }
            }
            const bool mine = has && mbin == bk;
            if (mine && gt < rk) sk = mq;  // a survivor of the k-th bin: fewer than rk members above it
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sk += __shfl_xor_sync(0xffffffffu, sk, o);
            const unsigned bt = __ballot_sync(0xffffffffu, mine && gt < rk && rk <= ge);
            thr = bt ? __shfl_sync(0xffffffffu, mk, __ffs(bt) - 1) : 0u;
        }
        const unsigned long long Zq = topk ? mAbove + sk : Ztot;
        unsigned cutl = 0u;
        if (topp) {
            unsigned long long T = mul_frac(sp.top_p, Zq, true);
            if (T == 0ull) T = 1ull;
            int bp;
            unsigned long long before;
            if (topk && T > mAbove) {
                bp = bk;
                before = mAbove;
            } else {
                bp = lower_bound_warp(pre, ss.mass, topk ? bk : kFB, T);
                before = bp > 0 ? pre[bp - 1] : 0ull;
            }
            const unsigned long long rem = T - before;
            unsigned long long p0 = 0ull;  // mass before this member in (key desc, index asc) order
            for (int j = 0; j < nm; ++j) {
                const uint32_t kj = __shfl_sync(0xffffffffu, mk, j);
                const int bj = __shfl_sync(0xffffffffu, mbin, j), ij = __shfl_sync(0xffffffffu, midx, j);
                const unsigned qj = __shfl_sync(0xffffffffu, mq, j);
                if (bj == bp && kj >= thr && (kj > mk || (kj == mk && ij < midx))) p0 += qj;
            }
            cutl = __ballot_sync(0xffffffffu, has && mbin == bp && mk >= thr && p0 < rem && p0 + mq >= rem);
        }
        if (lane == 0) {
            ss.sel[0] = thr;
            ss.i[5] = cutl ? 1 : 0;
        }
        if (cutl && lane == __ffs(cutl) - 1) {
            ss.sel[1] = mk;
            ss.sel[2] = (uint32_t)midx;
        }
    } else if (warp == 0) {
        const int rk = topk ? ss.i[3] : 0;
        // survivors of the k-th bin: fewer than rk of its members above them
        uint32_t thr = 0u;
        unsigned long long sk = 0ull;
        if (topk) {
            for (int c = lane; c < nm; c += 32) {
                if ((int)(cbi[c] >> 14) != bk) continue;
                const uint32_t key = ckey[c];
                int gt = 0, ge = 0;
                for (int j = 0; j < nm; ++j) {
                    if ((int)(cbi[j] >> 14) != bk) continue;
                    gt += ckey[j] > key;
                    ge += ckey[j] >= key;
                }
                if (gt < rk) sk += cq[c];
                if (gt < rk && rk <= ge) ss.sel[0] = key;  // every writer writes the same key
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sk += __shfl_xor_sync(0xffffffffu, sk, o);
            __syncwarp();
            thr = ss.sel[0];
        }
        const unsigned long long Zq = topk ? mAbove + sk : Ztot;
        if (lane == 0) {
            ss.sel[0] = thr;
            ss.i[5] = 0;  // no cut
        }
        __syncwarp();
        if (topp) {
            unsigned long long T = mul_frac(sp.top_p, Zq, true);
            if (T == 0ull) T = 1ull;
            // the bin where the cumulative (bins in order) mass reaches T, and the mass needed inside it
            int bp;
            unsigned long long before;
            if (topk && T > mAbove) {
                bp = bk;
                before = mAbove;
            } else {
                bp = lower_bound_u64(pre, topk ? bk : kFB, T);
                before = bp > 0 ? pre[bp - 1] : 0ull;
            }
            const unsigned long long rem = T - before;
            for (int c = lane; c < nm; c += 32) {
                if ((int)(cbi[c] >> 14) != bp) continue;
                const uint32_t key = ckey[c];
                if (key < thr) continue;
                const int idx = (int)(cbi[c] & 0x3FFFu);
                unsigned long long p0 = 0ull;  // mass before this element in (key desc, index asc) order
                for (int j = 0; j < nm; ++j) {
                    if ((int)(cbi[j] >> 14) != bp || ckey[j] < thr) continue;
                    const int jx = (int)(cbi[j] & 0x3FFFu);
                    if (ckey[j] > key || (ckey[j] == key && jx < idx)) p0 += cq[j];
                }
                if (p0 < rem && p0 + (unsigned long long)cq[c] >= rem) {
                    ss.sel[1] = key;
                    ss.sel[2] = (uint32_t)idx;
                    ss.i[5] = 1;
                }
            }
        }
    }
    SAMPLE_SYNC();
    const uint32_t thr = ss.sel[0];
    const bool cut = ss.i[5] != 0;
    const uint32_t tkey = ss.sel[1];
    const int tidx = (int)ss.sel[2];

    // ---- P7: kept mass of this thread's segment, scanned in thread (= vocabulary) order
    unsigned long long loc = 0ull;
#pragma unroll
    for (int j = 0; j < kRS; ++j) {
        const int i = a0 + j;
        if (j < S && i < V && q[j]) {
            const uint32_t key = ord_key(v[j]);
            if (!(key >= thr && (!cut || key > tkey || (key == tkey && i <= tidx)))) q[j] = 0u;  // not kept
        }
        loc += q[j];
    }
    const unsigned long long inc = warp_incl_scan_u64(loc);
    if (lane == 31) ss.q[32 + warp] = inc;
    SAMPLE_SYNC();
    unsigned long long run = inc - loc, ZS = 0ull;
    for (int w = 0; w < nw; ++w) {
        const unsigned long long t = ss.q[32 + w];
        ZS += t;
        if (w < warp) run += t;
    }
    const unsigned long long target = mul_frac(*u_ptr, ZS, false);
    if (run <= target && target < run + loc) {
#pragma unroll
        for (int j = 0; j < kRS; ++j) {
            run += q[j];
            if (run > target) {
                ss.i[6] = a0 + j;
                break;
            }
        }
    }
    SAMPLE_SYNC();
    int tok = ss.i[6];
    if (tok < 0 || tok >= V) {
        if (tid == 0 && err) atomicExch(err, 2);
        tok = 0;
    }
    return tok;
}

// As sample_reg, loading the logits lg[0..V) first (through L2: they may
// have been written by other CTAs of the same kernel).  With a history mask
// `seen` and sp.rep_penalty != 1 the logit of every seen token is divided by the
// penalty when positive and multiplied by it otherwise, as it is loaded ("Every
// Frame Is a Memory Read", section 2: the Talker's repetition penalty; the HF
// rule of the journal's table of fixes).
static __device__ int sample_block(const float* lg, int V, const SampParams sp, const float* u_ptr,
                                   unsigned char* smraw, SampleScratch& ss, int* err,
                                   const uint8_t* seen = nullptr) {
    const int tid = threadIdx.x, nt = SAMPLE_NT;
    float* z = reinterpret_cast<float*>(smraw);
    const bool pen = seen && sp.rep_penalty != 1.0f;
    for (int i0 = 0; i0 < V; i0 += 8 * nt) {
        float r[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int i = i0 + j * nt + tid;
            r[j] = i < V ? __ldcg(lg + i) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int i = i0 + j * nt + tid;
            if (i < V) {
                float v = r[j];
                if (pen && seen[i]) v = v > 0.f ? v / sp.rep_penalty : v * sp.rep_penalty;
                z[i] = v;
            }
        }
    }
    SAMPLE_SYNC();
    return sample_reg(V, sp, u_ptr, smraw, ss, err);
}

}  // namespace sample_detail

// shared memory of sample_fast / sample_smem / sample_block for V logits and `threads` threads
inline size_t sample_smem_bytes_dev(int V, int threads) {
    const size_t radix = 3 * sample_detail::sample_array_bytes(V) + (size_t)(threads / 32) * 256 * sizeof(unsigned);
    const size_t fast = sample_detail::sample_array_bytes(V) + sample_detail::sample_fast_extra_bytes(V);
    return radix > fast ? radix : fast;
}

}  // namespace sd
