// Persistent decode step for the GPT-2- and Llama-style T3 (rows B <= 2,
// Q8_0/Q4_0 weights): one cooperative launch runs n decode steps, each phase
// of each layer spread over every SM, phases separated by a grid barrier.
//
// "Every Frame Is a Memory Read", section 3: a decode step is a memory read --
// its time is bytes / bandwidth only if the weight stream never stalls.  With
// one kernel per operation the stream stops at every dependency (a launch, a
// tail, a cold start).  Here the weight stream is decoupled from the
// dependency chain: at the start of each layer every CTA issues bulk L2
// prefetches (cp.async.bulk.prefetch.L2) for all of its weight rows of the
// *next* layer, so HBM keeps streaming while the current layer's phases wait
// on each other; compute then reads its rows from L2.
//
// Per step: embed -> for each layer [QKV rows (LayerNorm/RMSNorm prologue,
// bias) | attention work items (split-KV, RoPE, fp16 KV append, last-item
// log-sum-exp combine) | O rows (+bias +residual) | FC or gate/up rows
// (+GELU / SwiGLU) | proj/down rows (+bias +residual)] -> head rows -> one
// CTA per row samples the next token.  Row ranges are static per CTA.
//
// Every grid barrier is a counter incremented once per CTA and waited on with
// a clock64() budget: on expiry the CTA records an error, and every later
// barrier of every CTA falls through, so the kernel always exits.  Buffers
// written by other CTAs are read through L2 (ld.global.cg).
#include "attn_dev.cuh"
#include "k_gemv.cuh"
#include "sample_dev.cuh"

namespace sd {
namespace step_detail {

using namespace gemv_detail;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kErrTimeout = 6;

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ int ld_volatile(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

__device__ __forceinline__ void prefetch_l2(const void* p, size_t bytes) {
    const char* c = reinterpret_cast<const char*>(p);
    while (bytes) {
        const unsigned n = bytes > 65536 ? 65536u : (unsigned)bytes;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c), "r"(n) : "memory");
        c += n;
        bytes -= n;
    }
}

__device__ __forceinline__ void row_range(int R, int i, int G, int& r0, int& r1) {
    r0 = (int)((long long)R * i / G);
    r1 = (int)((long long)R * (i + 1) / G);
}

__device__ __forceinline__ size_t qrow_bytes(const QMat& W) {
    return W.kind == SD_Q4_0 ? (size_t)W.cols / 2 : (size_t)W.cols;
}
__device__ __forceinline__ size_t srow_bytes(const QMat& W) {
    return W.kind == SD_A8G64 ? (size_t)(W.cols / 64) * 4 : (size_t)(W.cols / 32) * 2;
}

__device__ void prefetch_rows(const QMat& W, int r0, int r1) {
    if (r1 <= r0) return;
    const size_t qb = qrow_bytes(W), sb = srow_bytes(W);
    prefetch_l2(W.q + (size_t)r0 * qb, (size_t)(r1 - r0) * qb);
    prefetch_l2(reinterpret_cast<const char*>(W.s) + (size_t)r0 * sb, (size_t)(r1 - r0) * sb);
}

// Grid barrier: returns false once any CTA has recorded an error (then it
// no longer waits).  `target` = (barriers passed so far + 1) * gridDim.x.
__device__ __forceinline__ bool grid_sync(unsigned* bar, unsigned target, int* err, long long budget) {
    __syncthreads();
    __shared__ int s_ok;
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(bar, 1u);
        int ok = ld_volatile(err) == 0;
        if (ok) {
            const long long t0 = clock64();
            unsigned it = 0;
            while (ld_acquire(bar) < target) {
                if ((++it & 255u) == 0) {
                    if (ld_volatile(err) != 0) { ok = 0; break; }
                    if (clock64() - t0 > budget) {
                        atomicCAS(err, 0, kErrTimeout);
                        ok = 0;
                        break;
                    }
                }
            }
        }
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// Copy a norm's gain (and offset) into shared memory ahead of the barrier
// that precedes its use: they are constants.
__device__ __forceinline__ void preload_vec(const float* src, int n, float* dst) {
    if (!src) return;
    for (int i = threadIdx.x; i < (n >> 2); i += blockDim.x)
        reinterpret_cast<float4*>(dst)[i] = __ldg(reinterpret_cast<const float4*>(src) + i);
}

// Stage activation rows [NB][K] (global, written by other CTAs) into shared
// memory, optionally normalised (LayerNorm with gain/offset, or RMSNorm) with
// the gain/offset already in shared memory (s_g, s_b).
template <int NB>
__device__ void stage_x(const float* x, int x_stride, int K, int pro, const float* s_g, const float* s_b, float eps,
                        float* s_x, float* scr) {
    const int K4 = K >> 2;
    float4* xs4 = reinterpret_cast<float4*>(s_x);
    for (int i = threadIdx.x; i < NB * K4; i += blockDim.x) {
        const int b = i / K4, k4 = i - b * K4;
        xs4[i] = __ldcg(reinterpret_cast<const float4*>(x + (size_t)b * x_stride) + k4);
    }
    __syncthreads();
    if (pro == PRO_NONE) return;
    float v[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        float sum = 0.f;
        for (int k = threadIdx.x; k < K; k += blockDim.x) {
            const float xv = s_x[b * K + k];
            sum += (pro == PRO_LN) ? xv : xv * xv;
        }
        v[b] = sum;
    }
    block_sum<NB>(v, scr);
    float mu[NB], rs[NB];
    if (pro == PRO_LN) {
#pragma unroll
        for (int b = 0; b < NB; ++b) mu[b] = v[b] / (float)K;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            float sum = 0.f;
            for (int k = threadIdx.x; k < K; k += blockDim.x) {
                const float dx = s_x[b * K + k] - mu[b];
                sum = fmaf(dx, dx, sum);
            }
            v[b] = sum;
        }
        block_sum<NB>(v, scr);
#pragma unroll
        for (int b = 0; b < NB; ++b) rs[b] = 1.0f / sqrtf(v[b] / (float)K + eps);
    } else {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            mu[b] = 0.f;
            rs[b] = 1.0f / sqrtf(v[b] / (float)K + eps);
        }
    }
    const float4* g4 = reinterpret_cast<const float4*>(s_g);
    const float4* b4 = reinterpret_cast<const float4*>(s_b);
    for (int i = threadIdx.x; i < NB * K4; i += blockDim.x) {
        const int b = i / K4, k4 = i - b * K4;
        const float4 gg = g4[k4];
        float4 xx = xs4[i];
        if (pro == PRO_LN) {
            const float4 o = b4[k4];
            xx.x = fmaf((xx.x - mu[b]) * rs[b], gg.x, o.x);
            xx.y = fmaf((xx.y - mu[b]) * rs[b], gg.y, o.y);
            xx.z = fmaf((xx.z - mu[b]) * rs[b], gg.z, o.z);
            xx.w = fmaf((xx.w - mu[b]) * rs[b], gg.w, o.w);
        } else {
            xx.x = xx.x * rs[b] * gg.x;
            xx.y = xx.y * rs[b] * gg.y;
            xx.z = xx.z * rs[b] * gg.z;
            xx.w = xx.w * rs[b] * gg.w;
        }
        xs4[i] = xx;
    }
    __syncthreads();
}

template <int QK, int R>
struct GemvPre {
    uint4 w[R][Unit<QK>::kU];
    float d[R][Unit<QK>::kU];
};

// Warp layout of a row tile: WK warps along K (1024 elements each), WR row
// groups of R rows.
struct GemvGeom {
    int K, WK, WR, kw, rg, lane;
    bool active;
};
__device__ __forceinline__ GemvGeom gemv_geom(int K) {
    GemvGeom g;
    g.K = K;
    g.WK = (K + 1023) >> 10;
    g.WR = kWarps / g.WK;
    const int warp = threadIdx.x >> 5;
    g.lane = threadIdx.x & 31;
    g.kw = warp % g.WK;
    g.rg = warp / g.WK;
    g.active = g.rg < g.WR;
    return g;
}

template <int QK, int R>
__device__ __forceinline__ void gemv_load(GemvPre<QK, R>& p, const QMat& W, int base, int r1, const GemvGeom& g) {
    constexpr int U = Unit<QK>::kU;
    const int K = W.cols;
    const int row_bytes = (QK == SD_Q4_0) ? (K >> 1) : K;
    const int spr = K >> 5;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int r = base + g.rg * R + i;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = (QK == SD_Q4_0) ? (g.kw * 1024 + g.lane * 32) : (g.kw * 1024 + u * 512 + g.lane * 16);
            const bool ok = g.active && r < r1 && e < K;
            const int boff = (QK == SD_Q4_0) ? (e >> 1) : e;
            p.w[i][u] = ok ? __ldcs(reinterpret_cast<const uint4*>(W.q + (size_t)r * row_bytes + boff))
                           : make_uint4(0u, 0u, 0u, 0u);
            p.d[i][u] = ok ? __half2float(__ldg(reinterpret_cast<const __half*>(W.s) + (size_t)r * spr + (e >> 5)))
                           : 0.f;
        }
    }
}

// Constants of a phase, issued before the barrier that precedes it: the first
// pass of weight rows into registers, this CTA's bias slice into s_bias.
template <int QK, int R>
__device__ __forceinline__ void gemv_preload(GemvPre<QK, R>& p, const QMat& W, int r0, int r1, const float* bias,
                                             float* s_bias) {
    gemv_load<QK, R>(p, W, r0, r1, gemv_geom(W.cols));
    if (bias)
        for (int i = threadIdx.x; i < r1 - r0; i += blockDim.x) s_bias[i] = __ldg(bias + r0 + i);
}

// Rows [r0, r1) of y = W x (+bias, activation, +resid), activations in shared
// memory, first pass of weights already in registers (p), bias slice in
// s_bias.  resid/out_own: this CTA's own rows of the residual stream (shared
// memory), read and updated when non-null.  Partial sums of the WK warps meet
// in shared memory in a fixed order.
__device__ __forceinline__ void inner_stamp(unsigned long long* t, int k) {
    if (t && blockIdx.x == 0 && threadIdx.x == 0) {
        unsigned long long v;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(v));
        t[k] = v;
    }
}

template <int QK, int NB, int R>
__device__ void gemv_finish(GemvPre<QK, R>& p, const QMat& W, int r0, int r1, const float* s_x, int epi,
                            const float* s_bias, float* own, int own_stride, float* y, int y_stride, float* s_tot,
                            unsigned long long* tin = nullptr) {
    constexpr int U = Unit<QK>::kU;
    constexpr int EPU = (QK == SD_Q4_0) ? 32 : 16;
    const GemvGeom g = gemv_geom(W.cols);
    const int K = W.cols;
    float xr[NB][32];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = (QK == SD_Q4_0) ? (g.kw * 1024 + g.lane * 32) : (g.kw * 1024 + u * 512 + g.lane * 16);
            const bool in = g.active && e < K;
#pragma unroll
            for (int j = 0; j < EPU; j += 4) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (in) v = *reinterpret_cast<const float4*>(&s_x[b * K + e + j]);
                xr[b][u * EPU + j] = v.x; xr[b][u * EPU + j + 1] = v.y;
                xr[b][u * EPU + j + 2] = v.z; xr[b][u * EPU + j + 3] = v.w;
            }
        }
    inner_stamp(tin, 0);
    for (int base = r0; base < r1; base += g.WR * R) {
        if (base != r0) gemv_load<QK, R>(p, W, base, r1, g);
        if (g.active) {
            float acc[R][NB];
#pragma unroll
            for (int i = 0; i < R; ++i)
#pragma unroll
                for (int b = 0; b < NB; ++b) acc[i][b] = 0.f;
#pragma unroll
            for (int i = 0; i < R; ++i)
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        const float dq = (QK == SD_Q4_0) ? dot_q4(p.w[i][u], &xr[b][0]) : dot_s8(p.w[i][u], &xr[b][u * EPU]);
                        acc[i][b] = fmaf(p.d[i][u], dq, acc[i][b]);
                    }
            inner_stamp(tin, 1);
#pragma unroll
            for (int i = 0; i < R; ++i)
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const float sv = warp_sum(acc[i][b]);
                    if (g.lane == 0) s_tot[((g.rg * R + i) * NB + b) * g.WK + g.kw] = sv;
                }
            inner_stamp(tin, 2);
        }
        __syncthreads();
        inner_stamp(tin, 3);
        const int n_out = g.WR * R * NB;
        for (int t = threadIdx.x; t < n_out; t += blockDim.x) {
            const int b = t % NB;
            const int i = (t / NB) % R;
            const int gg = t / (NB * R);
            const int r = base + gg * R + i;
            if (r >= r1) continue;
            float v = 0.f;
            for (int k = 0; k < g.WK; ++k) v += s_tot[((gg * R + i) * NB + b) * g.WK + k];
            if (epi == EPI_SWIGLU) {
                if ((i & 1) == 0) {
                    float up = 0.f;
                    for (int k = 0; k < g.WK; ++k) up += s_tot[((gg * R + i + 1) * NB + b) * g.WK + k];
                    y[(size_t)b * y_stride + (r >> 1)] = silu(v) * up;
                }
            } else {
                if (s_bias) v += s_bias[r - r0];
                if (epi == EPI_GELU) v = gelu_tanh(v);
                if (own) {
                    v += own[b * own_stride + (r - r0)];
                    own[b * own_stride + (r - r0)] = v;
                }
                y[(size_t)b * y_stride + r] = v;
            }
        }
        inner_stamp(tin, 4);
        __syncthreads();
        inner_stamp(tin, 5);
    }
}

constexpr int kMaxBiasRows = 256;  // bias slice of one phase for one CTA
constexpr int kMaxOwn = 128;       // residual-stream rows owned by one CTA

template <int QK, int NB>
__global__ void __launch_bounds__(kThreads, 1) k_step(const StepArgs a) {
    constexpr int R = (NB == 1) ? 4 : 2;
    extern __shared__ __align__(16) unsigned char smraw[];
    __shared__ float s_scr[33 * NB];
    __shared__ float s_tot[kWarps * R * NB];
    __shared__ __align__(16) float s_bias[kMaxBiasRows];
    __shared__ float s_own[NB * kMaxOwn];
    __shared__ attn_detail::AttnScratch s_attn;
    __shared__ sample_detail::SampleScratch s_samp;

    const int G = gridDim.x, cta = blockIdx.x;
    const int d = a.d, qd = a.H * a.hd, kd = a.Hkv * a.hd, qkv_rows = qd + 2 * kd;
    const int kmax = max(max(d, a.ff), qd);
    // dynamic shared memory: [NB][kmax] staged activations, then [kmax] norm gain, [kmax] norm offset;
    // the attention staging and the sampler reuse the same bytes in their own phases
    float* s_x = reinterpret_cast<float*>(smraw);
    float* s_g = s_x + NB * kmax;
    float* s_b = s_g + kmax;
    const bool swiglu = !a.gpt2;
    const int pro = a.gpt2 ? PRO_LN : PRO_RMS;
    unsigned nbar = 0;
    // trace: 4 stamps per barrier interval -- staged, computed, preloaded, barrier passed
    auto stamp = [&](int k) {
        if (a.trace && cta == 0 && threadIdx.x == 0 && (int)nbar < a.trace_cap) {
            unsigned long long t;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
            a.trace[4 * nbar + k] = t;
        }
    };
    auto sync = [&]() {
        stamp(2);
        const bool ok = grid_sync(a.bar, (nbar + 1) * (unsigned)G, a.err, a.spin_budget);
        stamp(3);
        ++nbar;
        return ok;
    };

    // this CTA's static row ranges; o0..o1 (rows of the residual stream) serve embed, O and proj
    int q0, q1, o0, o1, f0, f1, h0, h1;
    row_range(qkv_rows, cta, G, q0, q1);
    row_range(d, cta, G, o0, o1);
    row_range(a.ff, cta, G, f0, f1);
    if (swiglu) { f0 *= 2; f1 *= 2; }          // gate/up rows are interleaved in pairs
    row_range(a.V, cta, G, h0, h1);

    auto prefetch_layer = [&](int l) {
        if (threadIdx.x != 0 || l >= a.n_layer || a.prefetch <= 0) return;
        const StepLayer& L = a.layers[l];
        prefetch_rows(L.wqkv, q0, q1);
        prefetch_rows(L.wo, o0, o1);
        prefetch_rows(L.wfc, f0, f1);
        prefetch_rows(L.wproj, o0, o1);
    };
    GemvPre<QK, R> pre;
    // constants of a layer's QKV phase (or of the head when l == n_layer)
    auto preload_qkv = [&](int l) {
        if (l < a.n_layer) {
            const StepLayer& L = a.layers[l];
            preload_vec(L.n1g, d, s_g);
            preload_vec(L.n1b, d, s_b);
            gemv_preload<QK, R>(pre, L.wqkv, q0, q1, L.bqkv, s_bias);
        } else {
            preload_vec(a.nfg, d, s_g);
            preload_vec(a.nfb, d, s_b);
            gemv_preload<QK, R>(pre, a.head, h0, h1, nullptr, s_bias);
        }
    };
    if (threadIdx.x == 0 && a.trace) {
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        a.trace[4 * a.trace_cap] = t;  // launch start, in the slot after the barrier stamps
    }
    prefetch_layer(0);
    prefetch_layer(1);
    preload_qkv(0);

    for (int s = 0; s < a.n_steps; ++s) {
        const int pos = __ldcg(a.pos);
        if (pos < 0 || pos >= a.n_ctx) {
            if (threadIdx.x == 0) atomicCAS(a.err, 0, 1);
            break;
        }
        // ---- embedding of this CTA's residual rows: x[b][r] = wte[tok][r] (+ wpe[pos][r])
        for (int i = threadIdx.x; i < NB * (o1 - o0); i += blockDim.x) {
            const int b = i / (o1 - o0), r = o0 + i % (o1 - o0);
            int tok = __ldcg(a.tok + b);
            if (tok < 0 || tok >= a.V) {
                atomicCAS(a.err, 0, 3);
                tok = 0;
            }
            float v = __ldg(a.wte + (size_t)tok * d + r);
            if (a.wpe) v += __ldg(a.wpe + (size_t)pos * d + r);
            s_own[b * kMaxOwn + (r - o0)] = v;
            a.x[(size_t)b * d + r] = v;
        }
        if (!sync()) break;

        bool ok = true;
        for (int l = 0; l < a.n_layer && ok; ++l) {
            const StepLayer& L = a.layers[l];
            // ---- QKV (norm prologue, bias)
            stage_x<NB>(a.x, d, d, pro, s_g, s_b, a.eps, s_x, s_scr);
            stamp(0);
            gemv_finish<QK, NB, R>(pre, L.wqkv, q0, q1, s_x, EPI_LINEAR, L.bqkv ? s_bias : nullptr, nullptr, 0,
                                   a.qkv, qkv_rows, s_tot);
            stamp(1);
            const int items = NB * a.Hkv * a.nsplit;
            if (threadIdx.x == 0 && a.prefetch > 0) {
                // the cached K/V rows this CTA's attention items will read, and the next layer's weights
                const int n = pos + 1, chunk = (n + a.nsplit - 1) / a.nsplit;
                for (int it = cta; it < items; it += G) {
                    const int split = it % a.nsplit, g = (it / a.nsplit) % a.Hkv, b = it / (a.nsplit * a.Hkv);
                    const int c0 = split * chunk, c1 = min(n - 1, c0 + chunk);  // rows < pos are cached
                    if (c1 > c0) {
                        const size_t hb = ((size_t)(b * a.n_layer * a.Hkv + l * a.Hkv + g) * a.n_ctx) * a.hd;
                        prefetch_l2(a.kc + hb + (size_t)c0 * a.hd, (size_t)(c1 - c0) * a.hd * 2);
                        prefetch_l2(a.vc + hb + (size_t)c0 * a.hd, (size_t)(c1 - c0) * a.hd * 2);
                    }
                }
            }
            if (l + 1 < a.n_layer) prefetch_layer(l + 1);
            else if (threadIdx.x == 0 && a.prefetch > 0) prefetch_rows(a.head, h0, h1);
            if (!(ok = sync())) break;
            // ---- attention items
            {
                AttnArgs at;
                at.q = a.qkv; at.q_stride = qkv_rows; at.knew = a.qkv + qd; at.vnew = a.qkv + qd + kd;
                at.kc = a.kc; at.vc = a.vc; at.row_heads = a.n_layer * a.Hkv; at.head_off = l * a.Hkv;
                at.n_head = a.H; at.n_kv = a.Hkv; at.hd = a.hd; at.n_ctx = a.n_ctx; at.nsplit = a.nsplit;
                at.pos_ptr = a.pos; at.rope_cos = a.rope_cos; at.rope_sin = a.rope_sin; at.part = a.part;
                at.counters = a.counters; at.out = a.o; at.out_stride = qd; at.err = a.err;
                stamp(0);
                for (int it = cta; it < items; it += G) {
                    const int split = it % a.nsplit, g = (it / a.nsplit) % a.Hkv, b = it / (a.nsplit * a.Hkv);
                    attn_detail::attn_item(at, split, g, b, reinterpret_cast<float*>(smraw), s_attn);
                }
                stamp(1);
            }
            gemv_preload<QK, R>(pre, L.wo, o0, o1, L.bo, s_bias);
            if (!(ok = sync())) break;
            // ---- O projection (+bias +residual)
            stage_x<NB>(a.o, qd, qd, PRO_NONE, nullptr, nullptr, 0.f, s_x, s_scr);
            stamp(0);
            gemv_finish<QK, NB, R>(pre, L.wo, o0, o1, s_x, EPI_LINEAR, L.bo ? s_bias : nullptr, s_own, kMaxOwn,
                                   a.x, d, s_tot);
            stamp(1);
            preload_vec(L.n2g, d, s_g);
            preload_vec(L.n2b, d, s_b);
            gemv_preload<QK, R>(pre, L.wfc, f0, f1, L.bfc, s_bias);
            if (!(ok = sync())) break;
            // ---- FC / gate-up (norm prologue, GELU / SwiGLU)
            stage_x<NB>(a.x, d, d, pro, s_g, s_b, a.eps, s_x, s_scr);
            stamp(0);
            gemv_finish<QK, NB, R>(pre, L.wfc, f0, f1, s_x, swiglu ? EPI_SWIGLU : EPI_GELU,
                                   L.bfc ? s_bias : nullptr, nullptr, 0, a.u, a.ff, s_tot,
                                   (a.trace && s == 0 && l == 1) ? a.trace + 4 * (size_t)a.trace_cap + 1 : nullptr);
            stamp(1);
            gemv_preload<QK, R>(pre, L.wproj, o0, o1, L.bproj, s_bias);
            if (!(ok = sync())) break;
            // ---- proj / down (+bias +residual)
            stage_x<NB>(a.u, a.ff, a.ff, PRO_NONE, nullptr, nullptr, 0.f, s_x, s_scr);
            stamp(0);
            gemv_finish<QK, NB, R>(pre, L.wproj, o0, o1, s_x, EPI_LINEAR, L.bproj ? s_bias : nullptr, s_own,
                                   kMaxOwn, a.x, d, s_tot);
            stamp(1);
            preload_qkv(l + 1);
            if (!(ok = sync())) break;
        }
        if (!ok) break;
        // ---- head (final norm prologue)
        stage_x<NB>(a.x, d, d, pro, s_g, s_b, a.eps, s_x, s_scr);
        gemv_finish<QK, NB, R>(pre, a.head, h0, h1, s_x, EPI_LINEAR, nullptr, nullptr, 0, a.logits, a.V, s_tot);
        // the next step's first layers stream in while the sampler runs
        if (s + 1 < a.n_steps) {
            prefetch_layer(0);
            prefetch_layer(1);
        }
        if (!sync()) break;
        // ---- sampler: CTA b samples row b
        if (cta < NB) {
            const float* up = a.u_seq ? a.u_seq + (size_t)s * NB + cta : a.u1 + cta;
            const int tok = sample_detail::sample_block(a.logits + (size_t)cta * a.V, a.V, *a.sp, up, smraw, s_samp,
                                                        a.err);
            if (threadIdx.x == 0) {
                a.tok[cta] = tok;
                if (a.out_seq) a.out_seq[(size_t)s * NB + cta] = tok;
                if (cta == 0) *a.pos = pos + 1;
            }
        }
        if (s + 1 < a.n_steps) preload_qkv(0);
        if (!sync()) break;
    }
}

}  // namespace step_detail

size_t step_smem_bytes(const StepArgs& a) {
    const int B = a.B;
    int kmax = a.d > a.ff ? a.d : a.ff;
    if (a.H * a.hd > kmax) kmax = a.H * a.hd;
    size_t need = sizeof(float) * (size_t)(B + 2) * kmax;
    AttnArgs at;
    at.n_head = a.H; at.n_kv = a.Hkv; at.hd = a.hd; at.n_ctx = a.n_ctx; at.nsplit = a.nsplit;
    const size_t att = attention_smem_bytes_dev(at);
    const size_t smp = sample_smem_bytes_dev(a.V);
    if (att > need) need = att;
    if (smp > need) need = smp;
    return need;
}

cudaError_t launch_step(const StepArgs& a, int grid, cudaStream_t st) {
    using namespace step_detail;
    const size_t smem = step_smem_bytes(a);
    void (*kern)(const StepArgs) = nullptr;
    if (a.quant == SD_Q8_0) kern = a.B == 1 ? k_step<SD_Q8_0, 1> : k_step<SD_Q8_0, 2>;
    else if (a.quant == SD_Q4_0) kern = a.B == 1 ? k_step<SD_Q4_0, 1> : k_step<SD_Q4_0, 2>;
    else return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

int step_max_grid(const StepArgs& a, int sm_count) {
    using namespace step_detail;
    const size_t smem = step_smem_bytes(a);
    void (*kern)(const StepArgs) = nullptr;
    if (a.quant == SD_Q8_0) kern = a.B == 1 ? k_step<SD_Q8_0, 1> : k_step<SD_Q8_0, 2>;
    else if (a.quant == SD_Q4_0) kern = a.B == 1 ? k_step<SD_Q4_0, 1> : k_step<SD_Q4_0, 2>;
    else return 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess) return 0;
    return per_sm >= 1 ? sm_count : 0;
}

}  // namespace sd
