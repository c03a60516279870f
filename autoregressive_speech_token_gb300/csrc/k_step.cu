// Persistent decode step for the GPT-2- and Llama-style T3 (rows B <= 2,
// Q8_0/Q4_0 weights): one cooperative launch runs n decode steps.
//
// "Every Frame Is a Memory Read", section 3: a decode step is a memory read,
// and its time is bytes / bandwidth only if the weight stream never waits on
// the dependency chain.  Two mechanisms keep the two apart here.
//
// Weight stream.  Every CTA owns fixed row ranges of every matrix.  A ring
// buffer in shared memory receives, by bulk asynchronous copies
// (cp.async.bulk with mbarrier completion), the CTA's rows of the matrices in
// the order the step consumes them -- codes, scales, bias and norm gains of one
// phase per record -- as far ahead as the ring holds (two to three layers).
// A producer warp (one lane) issues records whenever space frees and never
// joins the compute barriers; compute never waits on HBM.
//
// Activation exchange.  A phase's outputs are published as 64-bit words
// (epoch << 32 | float bits) written with one relaxed store each; a consumer
// polls the words it needs until each carries the current epoch.  One L2
// round trip both synchronises and delivers the data -- there is no grid
// barrier.  Epochs are unique per (step, layer) over the life of the context,
// so no buffer needs clearing.  Every poll is bounded: on expiry the CTA
// records an error and the kernel returns.
//
// Per step (pos = position of the consumed token): embedding -> per layer
// [QKV rows with the LayerNorm/RMSNorm prologue and bias | attention items:
// (row, kv head, key split) with RoPE, the fp16 KV append and a partial
// softmax | O rows: combine the partials, +bias +residual | FC or gate/up rows:
// norm prologue, GELU or SwiGLU | proj/down rows: +bias +residual] -> head
// rows with the final norm -> CTA b samples row b.  ("Chatterbox -> ggml
// Port: Development Journal", section 3.2 for the layer order; sections
// 3.12-3.13 for the cache layout [head][pos][dim] and the causal extent.)
#include "step_dev.cuh"

// The 512 compute threads synchronise on named barrier 1; warp 16 (the
// weight-stream producer) runs its own loop and never joins them.
#define SAMPLE_SYNC() asm volatile("bar.sync 1, 512;" ::: "memory")
#define SAMPLE_NT 512
#include "sample_dev.cuh"

namespace sd {
namespace step_detail {

using namespace gemv_detail;
using namespace stepdev;

constexpr int kNMB = 16;         // records in flight at most (a power of two)
constexpr int kMaxOwn = 64;      // residual-stream rows owned by one CTA
constexpr int kMaxPart = 1024;   // per-slice GEMV partial sums (rows x batch rows x K slices)
constexpr int kMaxHPG = 8;       // query heads per KV head
constexpr int kKC = 128;         // cached keys staged per attention sub-chunk

enum PhaseKind { PK_EMBED = 0, PK_QKV, PK_ATTN, PK_O, PK_FC, PK_PROJ, PK_HEAD, PK_SAMPLE };


// Every exchange word is written to kRep replicas (kRep x the buffer, the
// buffer's size apart); CTA c polls replica c % kRep, so that one line is
// polled by a quarter of the grid instead of all of it.
constexpr int kRep = 4;

__device__ __forceinline__ void ll_store_rep(unsigned long long* p, size_t stride, float v, unsigned e) {
#pragma unroll
    for (int r = 0; r < kRep; ++r) ll_store(p + r * stride, v, e);
}

// with `pad`, dst[o * padded(n_in) + pidx(i)] (the GEMV's bank-conflict-free layout).
// Per-thread result; the caller combines it with __syncthreads_and.
__device__ bool ll_read(const unsigned long long* src, int n_out, int stride, int n_in, unsigned e, float* dst,
                        int* err, long long budget, bool pad = false) {
    const int n = n_out * n_in;
    const int np = padded(n_in);
    bool ok = true;
    for (int i0 = threadIdx.x; i0 < n && ok; i0 += 4 * kThreads) {
        unsigned long long w[4];
        const unsigned long long* p[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * kThreads;
            p[j] = i < n ? src + (size_t)(i / n_in) * stride + (i % n_in) : nullptr;
            w[j] = p[j] ? ll_load(p[j]) : 0ull;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (!p[j] || !ok) continue;
            if ((unsigned)(w[j] >> 32) != e) ok = ll_spin(p[j], e, &w[j], err, budget);
            const int i = i0 + j * kThreads;
            dst[pad ? (i / n_in) * np + pidx(i % n_in) : i] = __uint_as_float((unsigned)w[j]);
        }
    }
    return ok;
}


// One phase's record for this CTA: rows [r0, r1) of a matrix, with the scale
// and bias windows widened to 16-byte boundaries, and the norm gains.
struct Slice {
    const uint8_t* q;
    const uint8_t* s;
    const float *bias, *g1, *g2;
    int r0, r1, row_bytes, srow, s_lo, b_lo, K;
    int o_sc, o_bias, o_g1, o_g2;  // offsets in the record (codes at 0)
    int n_codes, n_sc, n_bias, n_g;
    int bytes;                     // record size in the ring (128-byte multiple)
};

// j: index of the slice within a step (4 per layer: QKV, O, FC, proj; then the head)
__device__ Slice make_slice(const StepArgs& a, const StepLayer* tab, int j, int cta, int G) {
    const int L = a.n_layer;
    const int kind = j < 4 * L ? (j & 3) : 4;
    const int l = j >> 2;
    Slice s;
    QMat W;
    s.bias = nullptr; s.g1 = nullptr; s.g2 = nullptr;
    if (kind == 0) {
        W = tab[l].wqkv; s.bias = tab[l].bqkv; s.g1 = tab[l].n1g; s.g2 = tab[l].n1b;
        row_range(W.rows, cta, G, s.r0, s.r1);
    } else if (kind == 1) {
        W = tab[l].wo; s.bias = tab[l].bo;
        row_range(W.rows, cta, G, s.r0, s.r1);
    } else if (kind == 2) {
        W = tab[l].wfc; s.bias = tab[l].bfc; s.g1 = tab[l].n2g; s.g2 = tab[l].n2b;
        if (a.gpt2) {
            row_range(W.rows, cta, G, s.r0, s.r1);
        } else {  // gate/up rows interleaved in pairs
            row_range(W.rows / 2, cta, G, s.r0, s.r1);
            s.r0 *= 2; s.r1 *= 2;
        }
    } else if (kind == 3) {
        W = tab[l].wproj; s.bias = tab[l].bproj;
        row_range(W.rows, cta, G, s.r0, s.r1);
    } else {
        W = a.head; s.g1 = a.nfg; s.g2 = a.nfb;
        row_range(W.rows, cta, G, s.r0, s.r1);
    }
    if (!a.gpt2) s.g2 = nullptr;  // RMSNorm: gain only
    s.K = W.cols;
    s.row_bytes = W.kind == SD_Q4_0 ? W.cols / 2 : W.cols;
    s.srow = (W.cols / 32) * 2;
    const int nr = s.r1 - s.r0;
    s.n_codes = nr * s.row_bytes;
    s.s_lo = (s.r0 * s.srow) & ~15;
    s.n_sc = (((s.r1 * s.srow) + 15) & ~15) - s.s_lo;
    s.o_sc = s.n_codes;
    int off = s.o_sc + s.n_sc;
    s.b_lo = s.r0 & ~3;
    s.n_bias = s.bias ? ((((s.r1 + 3) & ~3) - s.b_lo) * 4) : 0;
    s.o_bias = off;
    off += s.n_bias;
    s.n_g = s.g1 ? W.cols * 4 : 0;
    s.o_g1 = off;
    off += s.n_g;
    s.o_g2 = off;
    off += s.g2 ? s.n_g : 0;
    s.bytes = (off + 127) & ~127;
    s.q = W.q + (size_t)s.r0 * s.row_bytes;
    s.s = reinterpret_cast<const uint8_t*>(W.s) + s.s_lo;
    if (s.bias) s.bias += s.b_lo;
    return s;
}

// Slice j of a step from the per-kind geometry computed once per launch
// (rows, windows and record layout are the same in every layer; only the
// pointers change).
__device__ __forceinline__ Slice slice_at(const StepArgs& a, const StepLayer* tab, const Slice* geo, int j) {
    const int L = a.n_layer;
    const int kind = j < 4 * L ? (j & 3) : 4;
    const int l = j >> 2;
    Slice s = geo[kind];
    const QMat* W;
    const float *bias = nullptr, *g1 = nullptr, *g2 = nullptr;
    if (kind == 0) { W = &tab[l].wqkv; bias = tab[l].bqkv; g1 = tab[l].n1g; g2 = tab[l].n1b; }
    else if (kind == 1) { W = &tab[l].wo; bias = tab[l].bo; }
    else if (kind == 2) { W = &tab[l].wfc; bias = tab[l].bfc; g1 = tab[l].n2g; g2 = tab[l].n2b; }
    else if (kind == 3) { W = &tab[l].wproj; bias = tab[l].bproj; }
    else { W = &a.head; g1 = a.nfg; g2 = a.nfb; }
    s.q = W->q + (size_t)s.r0 * s.row_bytes;
    s.s = reinterpret_cast<const uint8_t*>(W->s) + s.s_lo;
    s.bias = (s.bias && bias) ? bias + s.b_lo : nullptr;
    s.g1 = s.g1 ? g1 : nullptr;
    s.g2 = s.g2 ? g2 : nullptr;
    return s;
}

// y[i * NB + b] = sum_k W[r0 + i][k] x[b][k] for i < nr, with the codes and
// scales of rows r0.. in shared memory.  Warp layout as the streaming GEMV: a
// warp owns a 1024-element K slice (lane activations in registers) and visits
// rows rg, rg + WR, ... two at a time (independent chains); only warps that
// own a row load the activations.  With one K slice (K <= 1024) lane 0 writes
// the row sums directly; otherwise the WK slices of a row meet in s_part in
// fixed order.
template <int QK, int NB>
__device__ void gemv_rec(const uint8_t* codes, const uint8_t* sc, int K, int nr, const float* x, float* s_part,
                         float* s_y) {
    constexpr int U = Unit<QK>::kU;
    constexpr int EPU = (QK == SD_Q4_0) ? 32 : 16;
    const int WK = (K + 1023) >> 10, WR = kWarps / WK;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kw = warp % WK, rg = warp / WK;
    const int row_bytes = (QK == SD_Q4_0) ? (K >> 1) : K;
    const int spr = K >> 5;
    const int KP = padded(K);  // x rows are in the padded layout
    if (rg < WR && rg < nr) {
        float xr[NB][32];
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e = (QK == SD_Q4_0) ? (kw * 1024 + lane * 32) : (kw * 1024 + u * 512 + lane * 16);
                const bool in = e < K;
#pragma unroll
                for (int j = 0; j < EPU; j += 4) {
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (in) v = *reinterpret_cast<const float4*>(&x[b * KP + pidx(e + j)]);
                    xr[b][u * EPU + j] = v.x; xr[b][u * EPU + j + 1] = v.y;
                    xr[b][u * EPU + j + 2] = v.z; xr[b][u * EPU + j + 3] = v.w;
                }
            }
        for (int i = rg; i < nr; i += 2 * WR) {
            const int i2 = i + WR;
            const bool two = i2 < nr;  // warp-uniform
            float acc0[NB], acc1[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                acc0[b] = 0.f;
                acc1[b] = 0.f;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e = (QK == SD_Q4_0) ? (kw * 1024 + lane * 32) : (kw * 1024 + u * 512 + lane * 16);
                if (e < K) {
                    const int off = (QK == SD_Q4_0) ? (e >> 1) : e;
                    const uint4 w0 = *reinterpret_cast<const uint4*>(codes + (size_t)i * row_bytes + off);
                    const float d0 = __half2float(reinterpret_cast<const __half*>(sc)[(size_t)i * spr + (e >> 5)]);
                    uint4 w1 = make_uint4(0u, 0u, 0u, 0u);
                    float d1 = 0.f;
                    if (two) {
                        w1 = *reinterpret_cast<const uint4*>(codes + (size_t)i2 * row_bytes + off);
                        d1 = __half2float(reinterpret_cast<const __half*>(sc)[(size_t)i2 * spr + (e >> 5)]);
                    }
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        const float t0 = (QK == SD_Q4_0) ? dot4_q4(w0, &xr[b][0]) : dot4_s8(w0, &xr[b][u * EPU]);
                        acc0[b] = fmaf(d0, t0, acc0[b]);
                        if (two) {
                            const float t1 =
                                (QK == SD_Q4_0) ? dot4_q4(w1, &xr[b][0]) : dot4_s8(w1, &xr[b][u * EPU]);
                            acc1[b] = fmaf(d1, t1, acc1[b]);
                        }
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    acc0[b] += __shfl_xor_sync(0xffffffffu, acc0[b], o);
                    acc1[b] += __shfl_xor_sync(0xffffffffu, acc1[b], o);
                }
            if (lane == 0) {
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    if (WK == 1) {
                        s_y[i * NB + b] = acc0[b];
                        if (two) s_y[i2 * NB + b] = acc1[b];
                    } else {
                        s_part[(i * NB + b) * WK + kw] = acc0[b];
                        if (two) s_part[(i2 * NB + b) * WK + kw] = acc1[b];
                    }
                }
            }
        }
    }
    csync();
    if (WK > 1) {
        for (int t = threadIdx.x; t < nr * NB; t += kThreads) {
            float v = 0.f;
            for (int k = 0; k < WK; ++k) v += s_part[t * WK + k];
            s_y[t] = v;
        }
        csync();
    }
}

// Attention splits for n = pos + 1 keys: at most max_split chunks of about
// split_len keys, none empty.
__device__ __forceinline__ void attn_split(const StepArgs& a, int n, int& S, int& chunk) {
    S = (n + a.split_len - 1) / a.split_len;
    if (S > a.max_split) S = a.max_split;
    if (S < 1) S = 1;
    chunk = (n + S - 1) / S;
    S = (n + chunk - 1) / chunk;
}

// One warp's share of an attention sub-chunk: keys 0..cnt-1 of the staged
// rows Kw (pitch HD + 8 halves) and Vw (pitch HD), lane = key for the scores,
// lanes over dimensions for p V; the running (o, m, l) of query head h is
// updated in place in st + h * (HD + 2).  Loops have fixed trip counts so
// loads and shuffles pipeline; staged rows past cnt are never multiplied (they
// may hold any bits, and 0 * inf is not 0).
template <int HD>
__device__ __forceinline__ void attn_warp(const float* q, const __half* Kw, const __half* Vw, float* st, int HPG,
                                          int cnt) {
    constexpr int DPL = HD / 32, W = HD + 2;
    const int lane = threadIdx.x & 31;
    const bool valid = lane < cnt;
    const __half* kr = Kw + lane * (HD + 8);  // rows >= cnt are staging space: read, then masked
    for (int h = 0; h < HPG; ++h) {
        float* r = st + h * W;
        const float4* q4 = reinterpret_cast<const float4*>(q + h * HD);
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
        for (int d8 = 0; d8 < HD; d8 += 8) {
            const uint4 kv = *reinterpret_cast<const uint4*>(kr + d8);
            const float4 qa = q4[d8 >> 2], qb = q4[(d8 >> 2) + 1];
            const float2 k0 = __half22float2(*reinterpret_cast<const __half2*>(&kv.x));
            const float2 k1 = __half22float2(*reinterpret_cast<const __half2*>(&kv.y));
            const float2 k2 = __half22float2(*reinterpret_cast<const __half2*>(&kv.z));
            const float2 k3 = __half22float2(*reinterpret_cast<const __half2*>(&kv.w));
            s0 = fmaf(qa.x, k0.x, s0);
            s1 = fmaf(qa.y, k0.y, s1);
            s2 = fmaf(qa.z, k1.x, s2);
            s3 = fmaf(qa.w, k1.y, s3);
            s0 = fmaf(qb.x, k2.x, s0);
            s1 = fmaf(qb.y, k2.y, s1);
            s2 = fmaf(qb.z, k3.x, s2);
            s3 = fmaf(qb.w, k3.y, s3);
        }
        const float sc = valid ? (s0 + s1) + (s2 + s3) : -INFINITY;
        float mx = sc;
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
        const float mold = r[HD];
        const float mnew = fmaxf(mold, mx);
        const float p = valid ? expf(sc - mnew) : 0.f;
        const float corr = expf(mold - mnew);
        const float ps = warp_sum(p);
        float ov[DPL];
#pragma unroll
        for (int dd = 0; dd < DPL; ++dd) ov[dd] = 0.f;
        const __half* vr = Vw + lane * DPL;
#pragma unroll 8
        for (int jj = 0; jj < 32; ++jj) {
            const float pj = __shfl_sync(0xffffffffu, p, jj);
            if (jj >= cnt) continue;  // rows past the warp's keys hold stale staging data (warp-uniform)
            if (DPL == 2) {
                const float2 v = __half22float2(*reinterpret_cast<const __half2*>(vr + jj * HD));
                ov[0] = fmaf(pj, v.x, ov[0]);
                ov[1] = fmaf(pj, v.y, ov[1]);
            } else {
                const uint2 vv = *reinterpret_cast<const uint2*>(vr + jj * HD);
                const float2 v0 = __half22float2(*reinterpret_cast<const __half2*>(&vv.x));
                const float2 v1 = __half22float2(*reinterpret_cast<const __half2*>(&vv.y));
                ov[0] = fmaf(pj, v0.x, ov[0]);
                ov[1] = fmaf(pj, v0.y, ov[1]);
                ov[DPL - 2] = fmaf(pj, v1.x, ov[DPL - 2]);
                ov[DPL - 1] = fmaf(pj, v1.y, ov[DPL - 1]);
            }
        }
        float* ro = r + lane * DPL;
#pragma unroll
        for (int dd = 0; dd < DPL; ++dd) ro[dd] = fmaf(ro[dd], corr, ov[dd]);
        __syncwarp();
        if (lane == 0) {
            r[HD] = mnew;
            r[HD + 1] = fmaf(r[HD + 1], corr, ps);
        }
        __syncwarp();
    }
}

// One attention item: row b, kv head g, keys [c0, c1) of n = pos + 1.  Writes
// the unnormalised partial o (per query head of the group) with its running
// max m and sum l.  sm: the activation region (>= the attention floats of
// act_region_bytes).
//
// Keys are staged kKC at a time (cp.async, issued before the wait for q).
// Four warps own 32 keys each, lane = key: a lane forms its key's score with
// the whole head dimension (no shuffles; staged key rows are (hd + 8) halves
// apart so that the lanes' rows fall in distinct banks), the warp keeps an
// online softmax (m, l) and accumulates p V with lanes over dimensions.  The
// four warp partials are combined in shared memory and published.
__device__ bool attn_item(const StepArgs& a, int l, int b, int g, int c, int S, int chunk, int pos, unsigned e,
                          float* sm, int* err, size_t rs_qkv, size_t rs_part, unsigned long long* tr) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // cycle stamps of the sub-steps (traced CTA, thread 0): tr[k] += cycles since the previous stamp
    long long tc = (tr && tid == 0) ? clock64() : 0;
    auto stamp = [&](int k) {
        if (tr && tid == 0) {
            const long long t = clock64();
            tr[k] += (unsigned long long)(t - tc);
            tc = t;
        }
    };
    constexpr int kAW = kKC / 32;        // warps that own keys
    const int hd = a.hd, half = hd >> 1, HPG = a.H / a.Hkv, n = pos + 1;
    const int qd = a.H * a.hd, kd = a.Hkv * a.hd, qkv_rows = qd + 2 * kd;
    const int c0 = c * chunk, c1 = min(n, c0 + chunk);
    const bool last = c1 == n;
    const int KP = hd + 8;               // staged key row pitch (halves)
    const int W = hd + 2;                // partial record: o[hd], m, l
    float* q = sm;                       // [HPG][hd]
    float* kn = q + HPG * hd;            // [hd]
    float* vn = kn + hd;                 // [hd]
    float* wp = vn + hd;                 // [kAW][HPG][W] warp partials
    __half* Ks = reinterpret_cast<__half*>(wp + kAW * HPG * W);  // [kKC][KP] (16-byte aligned: see act_region_bytes)
    __half* Vs = Ks + kKC * KP;                                   // [kKC][hd]
    const size_t hb = ((size_t)(b * a.n_layer * a.Hkv + l * a.Hkv + g) * a.n_ctx) * hd;
    const __half* Kg = a.kc + hb;
    const __half* Vg = a.vc + hb;
    const int u16 = hd / 8;              // 16-byte units per cached row

    // cached rows [j0, j1) (the position being decoded comes from kn / vn), as
    // asynchronous 16-byte copies (cp.async, through L2): all in flight at once,
    // completed by stage_wait()
    auto stage = [&](int j0, int j1) {
        const int nu = (j1 - j0) * u16;
        for (int t = tid; t < 2 * nu; t += kThreads) {
            const bool isv = t >= nu;
            const int uu = isv ? t - nu : t, r = uu / u16, un = uu - r * u16;
            if (j0 + r == pos) continue;
            const __half* src = (isv ? Vg : Kg) + (size_t)(j0 + r) * hd + un * 8;
            __half* dst = isv ? Vs + r * hd + un * 8 : Ks + r * KP + un * 8;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    auto stage_wait = [&]() { asm volatile("cp.async.wait_all;" ::: "memory"); };
    stage(c0, min(c1, c0 + kKC));  // issued before the wait for this step's q

    const unsigned long long* src = a.ll_qkv + (size_t)(blockIdx.x & (kRep - 1)) * rs_qkv;
    bool ok = ll_read(src + (size_t)b * qkv_rows + (size_t)g * HPG * hd, 1, 0, HPG * hd, e, q, err, a.spin_budget);
    if (last && ok) {
        ok = ll_read(src + (size_t)b * qkv_rows + qd + (size_t)g * hd, 1, 0, hd, e, kn, err, a.spin_budget);
        if (ok) ok = ll_read(src + (size_t)b * qkv_rows + qd + kd + (size_t)g * hd, 1, 0, hd, e, vn, err,
                             a.spin_budget);
    }
    if (!csync_and(ok)) return false;
    stamp(0);
    // RoPE (NEOX half split) at pos on q and the new k; q scaled by 1/sqrt(hd)
    const float scale = 1.0f / sqrtf((float)hd);
    for (int i = tid; i < (HPG + 1) * half; i += kThreads) {
        const int h = i / half, dd = i - h * half;
        if (h == HPG && !last) continue;
        float* v = h < HPG ? q + h * hd : kn;
        float x0 = v[dd], x1 = v[dd + half];
        if (a.rope_cos) {
            const float cs = a.rope_cos[(size_t)pos * half + dd], sn = a.rope_sin[(size_t)pos * half + dd];
            const float y0 = x0 * cs - x1 * sn, y1 = x0 * sn + x1 * cs;
            x0 = y0;
            x1 = y1;
        }
        if (h < HPG) {
            x0 *= scale;
            x1 *= scale;
        }
        v[dd] = x0;
        v[dd + half] = x1;
    }
    csync();
    if (last) {
        // append the new position to the cache (fp16, round to nearest); the fence after
        // the partial is published orders it before every later word this CTA
        // publishes, which the next step's readers observe before they read the cache
        for (int dd = tid; dd < hd; dd += kThreads) {
            a.kc[hb + (size_t)pos * hd + dd] = __float2half_rn(kn[dd]);
            a.vc[hb + (size_t)pos * hd + dd] = __float2half_rn(vn[dd]);
        }
    }
    // the warps' running state (o, m, l) per query head lives in their partial slots
    if (warp < kAW)
        for (int h = 0; h < HPG; ++h) {
            float* r = wp + (warp * HPG + h) * W;
            for (int dd = lane; dd < hd; dd += 32) r[dd] = 0.f;
            if (lane == 0) {
                r[hd] = -INFINITY;
                r[hd + 1] = 0.f;
            }
        }
    for (int j0 = c0; j0 < c1; j0 += kKC) {
        const int j1 = min(c1, j0 + kKC), nk = j1 - j0;
        if (j0 != c0) {
            csync();
            stage(j0, j1);
        }
        stamp(1);
        stage_wait();
        if (pos >= j0 && pos < j1)
            for (int dd = tid; dd < hd; dd += kThreads) {
                Ks[(pos - j0) * KP + dd] = __float2half_rn(kn[dd]);
                Vs[(pos - j0) * hd + dd] = __float2half_rn(vn[dd]);
            }
        csync();
        stamp(2);
        if (warp < kAW && warp * 32 < nk) {
            if (hd == 64) attn_warp<64>(q, Ks + warp * 32 * KP, Vs + warp * 32 * hd, wp + warp * HPG * W, HPG,
                                        min(32, nk - warp * 32));
            else attn_warp<128>(q, Ks + warp * 32 * KP, Vs + warp * 32 * hd, wp + warp * HPG * W, HPG,
                                min(32, nk - warp * 32));
        }
        stamp(3);
    }
    csync();
    stamp(4);
    for (int t = tid; t < HPG * (hd + 2); t += kThreads) {
        const int h = t / (hd + 2), k = t - h * (hd + 2);
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAW; ++w) M = fmaxf(M, wp[(w * HPG + h) * W + hd]);
        float v = M;
        if (k != hd) {
            v = 0.f;
#pragma unroll
            for (int w = 0; w < kAW; ++w) {
                const float mw = wp[(w * HPG + h) * W + hd];
                if (mw != -INFINITY) v = fmaf(expf(mw - M), wp[(w * HPG + h) * W + k], v);
            }
        }
        ll_store_rep(a.ll_part + (((size_t)(b * a.H + g * HPG + h) * a.max_split + c) * W + k), rs_part, v, e);
    }
    stamp(5);
    if (last) __threadfence();
    csync();
    stamp(6);
    return true;
}

// ------------------------------------------------------------------ the kernel

template <int QK, int NB>
__global__ void __launch_bounds__(kBlock, 1) k_step(const StepArgs a) {
    extern __shared__ __align__(128) unsigned char sm[];
    unsigned char* ring = sm;
    float* act = reinterpret_cast<float*>(sm + a.ring_bytes);
    // normalised input rows [NB][padded(d)], after the largest staged input
    float* xn = act + a.B * padded(a.d > a.ff ? (a.d > a.H * a.hd ? a.d : a.H * a.hd) : (a.ff > a.H * a.hd ? a.ff : a.H * a.hd));
    StepLayer* tab = reinterpret_cast<StepLayer*>(sm + a.ring_bytes + a.act_bytes);
    __shared__ __align__(8) unsigned long long s_mb[kNMB];
    __shared__ long long s_rec[kNMB];  // ring position (monotonic bytes) of record i % kNMB
    __shared__ int s_off[kNMB];        // the same position within the ring
    __shared__ int s_nc;               // records consumed (compute thread 0 -> producer)
    __shared__ int s_done;             // compute threads finished (normally or on an error)
    __shared__ float s_own[NB * kMaxOwn];
    __shared__ unsigned long long s_trc[16];  // traced CTA: sub-step cycle sums (thread 0), flushed at the end
    __shared__ float s_part[kMaxPart];
    __shared__ float s_y[kMaxPart];
    __shared__ __align__(16) float s_red[33 * NB + 8];
    __shared__ sample_detail::SampleScratch s_samp;
    __shared__ Slice s_geo[5];

    const int G = gridDim.x, cta = blockIdx.x, tid = threadIdx.x;
    const int L = a.n_layer, d = a.d, qd = a.H * a.hd, kd = a.Hkv * a.hd, qkv_rows = qd + 2 * kd;
    const int per_step = 4 * L + 1;
    const int total = a.n_steps * per_step;
    const int RB = a.ring_bytes;
    const long long budget = a.spin_budget;
    const uint64_t wpol = l2_policy(a.w_evict_first != 0);
    const bool ln = a.gpt2 != 0;
    int o0, o1;
    row_range(d, cta, G, o0, o1);

    {
        const int words = L * (int)(sizeof(StepLayer) / 4);
        for (int i = tid; i < words; i += kBlock)
            reinterpret_cast<int*>(tab)[i] = reinterpret_cast<const int*>(a.layers)[i];
    }
    __syncthreads();
    if (tid < 5) s_geo[tid] = make_slice(a, tab, tid < 4 ? tid : 4 * L, cta, G);
    if (tid == 0) {
        for (int k = 0; k < kNMB; ++k) mb_init(smem_u32(&s_mb[k]));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_nc = 0;
        s_done = 0;
    }
    if (tid < 16) s_trc[tid] = 0ull;
    __syncthreads();

    // ---- producer warp: streams this CTA's weight records into the ring, as
    // far ahead as the ring and the barriers allow (positions tracked
    // incrementally: no divisions), until every record of the launch is issued
    if (tid >= kThreads) {
        if (tid != kThreads) return;
        int ni = 0, pj = 0, hoff = 0;
        long long head = 0, idle0 = clock64();
        bool ok = true;
        while (ni < total) {
            const int nc = ld_volatile(&s_nc);
            if (ld_volatile(&s_done)) break;
            bool issued = false;
            if (ni - nc < kNMB) {
                const Slice sl = slice_at(a, tab, s_geo, pj);
                long long start = head;
                int off = hoff;
                if (off + sl.bytes > RB) {
                    start += RB - off;
                    off = 0;
                }
                if (!(ni > nc && start + sl.bytes - s_rec[nc & (kNMB - 1)] > RB)) {
                    const uint32_t dst = smem_u32(ring + off);
                    const uint32_t mb = smem_u32(&s_mb[ni & (kNMB - 1)]);
                    s_rec[ni & (kNMB - 1)] = start;
                    s_off[ni & (kNMB - 1)] = off;
                    mb_expect(mb, (uint32_t)(sl.n_codes + sl.n_sc + sl.n_bias + (sl.g1 ? sl.n_g : 0) +
                                             (sl.g2 ? sl.n_g : 0)));
                    bulk_g2s_pol(dst, sl.q, (uint32_t)sl.n_codes, mb, wpol);
                    bulk_g2s_pol(dst + sl.o_sc, sl.s, (uint32_t)sl.n_sc, mb, wpol);
                    if (sl.bias) bulk_g2s_pol(dst + sl.o_bias, sl.bias, (uint32_t)sl.n_bias, mb, wpol);
                    if (sl.g1) bulk_g2s_pol(dst + sl.o_g1, sl.g1, (uint32_t)sl.n_g, mb, wpol);
                    if (sl.g2) bulk_g2s_pol(dst + sl.o_g2, sl.g2, (uint32_t)sl.n_g, mb, wpol);
                    head = start + sl.bytes;
                    hoff = off + sl.bytes;
                    ++ni;
                    if (++pj == per_step) pj = 0;
                    issued = true;
                    idle0 = clock64();
                }
            }
            if (!issued) {
                if (clock64() - idle0 > budget) {  // the consumers stopped advancing
                    atomicCAS(a.err, 0, kErrTimeout);
                    ok = false;
                    break;
                }
                __nanosleep(128);
            }
        }
        // copies still in flight into this CTA's ring finish before the CTA exits
        const long long t0 = clock64();
        while (!ld_volatile(&s_done) && ok && clock64() - t0 < budget) __nanosleep(256);
        for (int i = ld_volatile(&s_nc); i < ni; ++i)
            mb_wait(smem_u32(&s_mb[i & (kNMB - 1)]), (uint32_t)((i / kNMB) & 1), a.err, budget, true);
        return;
    }

    // ---- compute threads
    // replica strides (words) of the exchange buffers; this CTA reads replica `rep`
    const size_t rs_x = (size_t)NB * d, rs_qkv = (size_t)NB * qkv_rows, rs_u = (size_t)NB * a.ff;
    const size_t rs_part = (size_t)NB * a.H * a.max_split * (a.hd + 2), rs_lg = (size_t)NB * a.V, rs_tok = 32;
    const int rep = cta & (kRep - 1);
    const unsigned gen0 = *reinterpret_cast<const volatile unsigned*>(a.gen);
    const int pos0 = ld_volatile(a.pos);
    int nc = 0;  // records consumed (uniform over the compute threads)

    // trace: CTA 0 sums, per phase kind, the wait for its inputs, the wait for
    // its weight record and the rest (ns)
    unsigned long long t_a = 0, t_b = 0, t_w = 0;
    // per-thread wait for record nc (normally complete long before); the caller
    // joins it with the input wait in one barrier
    auto rec_ready = [&]() -> bool {
        const unsigned long long tw0 = (a.trace && cta == 0 && tid == 0) ? gtime() : 0ull;
        const bool r = mb_wait(smem_u32(&s_mb[nc & (kNMB - 1)]), (uint32_t)((nc / kNMB) & 1), a.err, budget, false);
        if (a.trace && cta == 0 && tid == 0) t_w += gtime() - tw0;
        return r;
    };
    auto rec_base = [&]() -> const unsigned char* { return ring + s_off[nc & (kNMB - 1)]; };
    // a record is consumed: its ring space is free for the producer
    auto done_rec = [&]() {
        csync();
        ++nc;
        if (tid == 0) *reinterpret_cast<volatile int*>(&s_nc) = nc;
    };
    // publish stamps (trace_pub): latest and earliest CTA per (step, layer, phase)
    auto tr_pub = [&](int s_, int l_, int ph) {
        if (a.trace_pub && tid == 0 && s_ < kTraceSteps) {
            const unsigned long long t = gtime();
            const size_t i = ((size_t)s_ * L + l_) * kTracePhases + ph;
            atomicMax(a.trace_pub + i, t);
            atomicMin(a.trace_pub + (size_t)kTraceSteps * L * kTracePhases + i, t);
        }
    };
    auto tr_begin = [&]() { if (a.trace && cta == 0 && tid == 0) { t_a = gtime(); t_w = 0; } };
    auto tr_waited = [&]() { if (a.trace && cta == 0 && tid == 0) t_b = gtime(); };
    auto tr_end = [&](int kind) {
        if (a.trace && cta == 0 && tid == 0) {
            const unsigned long long t = gtime();
            a.trace[3 * kind] += t_b - t_a;
            a.trace[3 * kind + 1] += t_w;
            a.trace[3 * kind + 2] += t - t_b - t_w;
        }
    };

    bool ok = true;
    for (int s = 0; s < a.n_steps && ok; ++s) {
        const int pos = pos0 + s;
        const unsigned eb = 1u + (gen0 + (unsigned)s) * (unsigned)(L + 1);  // epoch of layer 0 in this step
        // ---- embedding (every CTA builds the whole input row; it owns rows o0..o1)
        tr_begin();
        {
            int tk[NB];
            bool okr = true;
            if (s == 0) {
#pragma unroll
                for (int b = 0; b < NB; ++b) tk[b] = ld_volatile(a.tok + b);
            } else {
                if (tid < NB) {
                    const unsigned long long* tp = a.ll_tok + rep * rs_tok + tid;
                    unsigned long long w = ll_load(tp);
                    const unsigned et = eb - 1u;  // layer L of the previous step
                    if ((unsigned)(w >> 32) != et) okr = ll_spin(tp, et, &w, a.err, budget);
                    reinterpret_cast<int*>(s_red)[tid] = (int)(unsigned)w;
                }
                okr = csync_and(okr) != 0;
#pragma unroll
                for (int b = 0; b < NB; ++b) tk[b] = reinterpret_cast<int*>(s_red)[b];
                csync();
            }
            if (!okr) { ok = false; break; }
            __threadfence();  // order this step's cache reads after the previous steps' appends
            tr_waited();
            for (int i = tid; i < NB * d; i += kThreads) {
                const int b = i / d, k = i - b * d;
                int t = tk[b];
                if (t < 0 || t >= a.V_in) {
                    atomicCAS(a.err, 0, 3);
                    t = 0;
                }
                float v = __ldg(a.wte + (size_t)t * d + k);
                if (a.wpe) v += __ldg(a.wpe + (size_t)pos * d + k);
                act[b * padded(d) + pidx(k)] = v;
                if (k >= o0 && k < o1) s_own[b * kMaxOwn + (k - o0)] = v;
            }
            csync();
            tr_end(PK_EMBED);
        }

        for (int l = 0; l < L && ok; ++l) {
            const unsigned e = eb + (unsigned)l;
            // ---- QKV rows (norm prologue, bias)
            tr_begin();
            {
                bool okr = l > 0 ? ll_read(a.ll_xb + rep * rs_x, NB, d, d, e - 1u, act, a.err, budget, true) : true;
                okr = okr && rec_ready();
                if (!(ok = csync_and(okr) != 0)) break;
            }
            tr_waited();
            tr_pub(s, l, 0);
            {
                // sub-phase stamps of the QKV phase (CTA 0): slice, record wait, norm, matvec, publish
                unsigned long long ts = (a.trace && cta == 0 && tid == 0) ? gtime() : 0ull;
                auto sub = [&](int k) {
                    if (a.trace && cta == 0 && tid == 0) {
                        const unsigned long long t = gtime();
                        a.trace[24 + k] += t - ts;
                        ts = t;
                    }
                };
                const Slice sl = slice_at(a, tab, s_geo, 4 * l);
                sub(0);
                const unsigned char* rec = rec_base();
                sub(1);
                norm_to<NB>(act, xn, d, ln, reinterpret_cast<const float*>(rec + sl.o_g1),
                            reinterpret_cast<const float*>(rec + sl.o_g2), a.eps, s_red);
                sub(2);
                const int nr = sl.r1 - sl.r0;
                gemv_rec<QK, NB>(rec, rec + sl.o_sc + (sl.r0 * sl.srow - sl.s_lo), d, nr, xn, s_part, s_y);
                sub(3);
                const float* bias = reinterpret_cast<const float*>(rec + sl.o_bias) + (sl.r0 - sl.b_lo);
                for (int t = tid; t < nr * NB; t += kThreads) {
                    const int i = t / NB, b = t - i * NB;
                    float v = s_y[t];
                    if (sl.bias) v += bias[i];
                    ll_store_rep(a.ll_qkv + (size_t)b * qkv_rows + sl.r0 + i, rs_qkv, v, e);
                }
                tr_pub(s, l, 1);
                done_rec();
                sub(4);
            }
            tr_end(PK_QKV);
            // ---- attention items
            tr_begin();
            int S, chunk;
            attn_split(a, pos + 1, S, chunk);
            {
                const int items = NB * a.Hkv * S;
                tr_waited();
                for (int it = cta; it < items && ok; it += G) {
                    const int c = it % S, g = (it / S) % a.Hkv, b = it / (S * a.Hkv);
                    ok = attn_item(a, l, b, g, c, S, chunk, pos, e, act, a.err, rs_qkv, rs_part,
                                   (a.trace && cta == 0) ? s_trc + 8 : nullptr);
                    tr_pub(s, l, 2);
                }
                if (!ok) break;
            }
            tr_end(PK_ATTN);
            // ---- O rows: combine the partials, +bias +residual
            tr_begin();
            {
                const int W = a.hd + 2;
                float* pp = act + NB * padded(qd);  // [NB*H][S][W]
                bool okr = ll_read(a.ll_part + rep * rs_part, NB * a.H, a.max_split * W, S * W, e, pp, a.err, budget);
                okr = okr && rec_ready();
                if (!(ok = csync_and(okr) != 0)) break;
                tr_waited();
                for (int t = tid; t < NB * qd; t += kThreads) {
                    const int bh = t / a.hd, dd = t - bh * a.hd;
                    const float* P = pp + (size_t)bh * S * W;
                    float M = -INFINITY;
                    for (int c = 0; c < S; ++c) M = fmaxf(M, P[c * W + a.hd]);
                    float num = 0.f, den = 0.f;
                    for (int c = 0; c < S; ++c) {
                        const float w = expf(P[c * W + a.hd] - M);
                        num = fmaf(w, P[c * W + dd], num);
                        den = fmaf(w, P[c * W + a.hd + 1], den);
                    }
                    act[(t / qd) * padded(qd) + pidx(t % qd)] = num / den;  // o[b][h * hd + dd], padded
                }
                csync();
                const Slice sl = slice_at(a, tab, s_geo, 4 * l + 1);
                const unsigned char* rec = rec_base();
                const int nr = sl.r1 - sl.r0;
                gemv_rec<QK, NB>(rec, rec + sl.o_sc + (sl.r0 * sl.srow - sl.s_lo), qd, nr, act, s_part, s_y);
                const float* bias = reinterpret_cast<const float*>(rec + sl.o_bias) + (sl.r0 - sl.b_lo);
                for (int t = tid; t < nr * NB; t += kThreads) {
                    const int i = t / NB, b = t - i * NB;
                    float v = s_y[t];
                    if (sl.bias) v += bias[i];
                    v += s_own[b * kMaxOwn + i];
                    s_own[b * kMaxOwn + i] = v;
                    ll_store_rep(a.ll_xa + (size_t)b * d + sl.r0 + i, rs_x, v, e);
                }
                tr_pub(s, l, 3);
                done_rec();
            }
            tr_end(PK_O);
            // ---- FC / gate-up rows (norm prologue, GELU / SwiGLU)
            tr_begin();
            {
                long long tc = (a.trace && cta == 0 && tid == 0) ? clock64() : 0;
                auto stamp = [&](int k) {
                    if (a.trace && cta == 0 && tid == 0) {
                        const long long t = clock64();
                        s_trc[k] += (unsigned long long)(t - tc);
                        tc = t;
                    }
                };
                const bool stall = a.test_budget > 0 && s == 0 && l == 0 && cta == 0;  // test hook
                bool okr = ll_read(a.ll_xa + rep * rs_x, NB, d, d, stall ? e + 0x40000000u : e, act, a.err,
                                   stall ? a.test_budget : budget, true);
                okr = okr && rec_ready();
                if (!(ok = csync_and(okr) != 0)) break;
                tr_waited();
                stamp(0);
                const Slice sl = slice_at(a, tab, s_geo, 4 * l + 2);
                const unsigned char* rec = rec_base();
                norm_to<NB>(act, xn, d, ln, reinterpret_cast<const float*>(rec + sl.o_g1),
                            reinterpret_cast<const float*>(rec + sl.o_g2), a.eps, s_red);
                stamp(1);
                const int nr = sl.r1 - sl.r0;
                gemv_rec<QK, NB>(rec, rec + sl.o_sc + (sl.r0 * sl.srow - sl.s_lo), d, nr, xn, s_part, s_y);
                stamp(2);
                const float* bias = reinterpret_cast<const float*>(rec + sl.o_bias) + (sl.r0 - sl.b_lo);
                if (ln) {
                    for (int t = tid; t < nr * NB; t += kThreads) {
                        const int i = t / NB, b = t - i * NB;
                        float v = s_y[t];
                        if (sl.bias) v += bias[i];
                        ll_store_rep(a.ll_u + (size_t)b * a.ff + sl.r0 + i, rs_u, gelu_tanh(v), e);
                    }
                } else {
                    for (int t = tid; t < (nr / 2) * NB; t += kThreads) {
                        const int i = t / NB, b = t - i * NB;
                        const float gt = s_y[(2 * i) * NB + b], up = s_y[(2 * i + 1) * NB + b];
                        ll_store_rep(a.ll_u + (size_t)b * a.ff + sl.r0 / 2 + i, rs_u, silu(gt) * up, e);
                    }
                }
                tr_pub(s, l, 4);
                stamp(3);
                done_rec();
                stamp(4);
            }
            tr_end(PK_FC);
            // ---- proj / down rows (+bias +residual)
            tr_begin();
            {
                bool okr = ll_read(a.ll_u + rep * rs_u, NB, a.ff, a.ff, e, act, a.err, budget, true);
                okr = okr && rec_ready();
                if (!(ok = csync_and(okr) != 0)) break;
                tr_waited();
                const Slice sl = slice_at(a, tab, s_geo, 4 * l + 3);
                const unsigned char* rec = rec_base();
                const int nr = sl.r1 - sl.r0;
                gemv_rec<QK, NB>(rec, rec + sl.o_sc + (sl.r0 * sl.srow - sl.s_lo), a.ff, nr, act, s_part, s_y);
                const float* bias = reinterpret_cast<const float*>(rec + sl.o_bias) + (sl.r0 - sl.b_lo);
                for (int t = tid; t < nr * NB; t += kThreads) {
                    const int i = t / NB, b = t - i * NB;
                    float v = s_y[t];
                    if (sl.bias) v += bias[i];
                    v += s_own[b * kMaxOwn + i];
                    s_own[b * kMaxOwn + i] = v;
                    ll_store_rep(a.ll_xb + (size_t)b * d + sl.r0 + i, rs_x, v, e);
                }
                tr_pub(s, l, 5);
                done_rec();
            }
            tr_end(PK_PROJ);
        }
        if (!ok) break;
        // ---- head rows (final norm prologue)
        const unsigned eh = eb + (unsigned)L;
        tr_begin();
        {
            bool okr = ll_read(a.ll_xb + rep * rs_x, NB, d, d, eh - 1u, act, a.err, budget, true);
            okr = okr && rec_ready();
            if (!(ok = csync_and(okr) != 0)) break;
            tr_waited();
            const Slice sl = slice_at(a, tab, s_geo, 4 * L);
            const unsigned char* rec = rec_base();
            norm_to<NB>(act, xn, d, ln, reinterpret_cast<const float*>(rec + sl.o_g1),
                        reinterpret_cast<const float*>(rec + sl.o_g2), a.eps, s_red);
            const int nr = sl.r1 - sl.r0;
            gemv_rec<QK, NB>(rec, rec + sl.o_sc + (sl.r0 * sl.srow - sl.s_lo), d, nr, xn, s_part, s_y);
            for (int t = tid; t < nr * NB; t += kThreads) {
                const int i = t / NB, b = t - i * NB;
                const float v = s_y[t];
                a.logits[(size_t)b * a.V + sl.r0 + i] = v;
                ll_store_rep(a.ll_logits + (size_t)b * a.V + sl.r0 + i, rs_lg, v, eh);
            }
            done_rec();
        }
        tr_end(PK_HEAD);
        // ---- sampler: CTA b samples row b
        if (cta < NB) {
            tr_begin();
            float* z = act;
            ok = csync_and(
                     ll_read(a.ll_logits + rep * rs_lg + (size_t)cta * a.V, 1, 0, a.V, eh, z, a.err, budget)) != 0;
            if (!ok) break;
            tr_waited();
            const float* up = a.u_seq ? a.u_seq + (size_t)s * NB + cta : a.u1 + cta;
            const int tok = sample_detail::sample_reg(a.V, *a.sp, up, reinterpret_cast<unsigned char*>(z), s_samp,
                                                       a.err);
            if (tid == 0) {
                a.tok[cta] = tok;
                if (a.out_seq) a.out_seq[(size_t)s * NB + cta] = tok;
                ll_store_rep(a.ll_tok + cta, rs_tok, __int_as_float(tok), eh);
            }
            tr_end(PK_SAMPLE);
        }
    }
    // final counters (CTA 0; every other CTA read gen and pos at its start).  The
    // generation advances even after an error, so that no later epoch can match
    // a word this launch wrote.
    if (cta == 0 && tid == 0) {
        if (ok) *a.pos = pos0 + a.n_steps;
        *a.gen = gen0 + (unsigned)a.n_steps;
    }
    // the producer drains its copies in flight and exits once it sees this
    csync();
    if (a.trace && cta == 0 && tid < 16) a.trace[32 + tid] += s_trc[tid];
    if (tid == 0) {
        *reinterpret_cast<volatile int*>(&s_nc) = nc;
        __threadfence_block();
        *reinterpret_cast<volatile int*>(&s_done) = 1;
    }
}

// Bytes of the activation region: staged input rows, the attention item
// workspace, the O-phase partials and the sampler's arrays.
size_t act_region_bytes(const StepArgs& a) {
    const int qd = a.H * a.hd, HPG = a.H / a.Hkv;
    int kmax = a.d > a.ff ? a.d : a.ff;
    if (qd > kmax) kmax = qd;
    size_t need = sizeof(float) * ((size_t)a.B * padded(kmax) + (size_t)a.B * padded(a.d));
    const size_t o_phase = sizeof(float) * ((size_t)a.B * padded(qd) + (size_t)a.B * a.H * a.max_split * (a.hd + 2));
    // attention: q, the new k and v, the warp partials (a multiple of 4 floats, so the fp16
    // staging after them is 16-byte aligned), then keys at a pitch of hd + 8 halves and values
    const size_t attn_floats = (size_t)HPG * a.hd + 2 * a.hd + (size_t)(kKC / 32) * HPG * (a.hd + 2);
    const size_t attn = sizeof(float) * attn_floats + sizeof(__half) * (size_t)kKC * (2 * a.hd + 8);
    const size_t smp = sample_smem_bytes_dev(a.V, kThreads);
    if (o_phase > need) need = o_phase;
    if (attn > need) need = attn;
    if (smp > need) need = smp;
    return (need + 127) & ~(size_t)127;
}

template <int QK, int NB>
void* kernel_ptr() {
    return reinterpret_cast<void*>(k_step<QK, NB>);
}

void* pick(const StepArgs& a) {
    if (a.quant == SD_Q8_0) return a.B == 1 ? kernel_ptr<SD_Q8_0, 1>() : kernel_ptr<SD_Q8_0, 2>();
    if (a.quant == SD_Q4_0) return a.B == 1 ? kernel_ptr<SD_Q4_0, 1>() : kernel_ptr<SD_Q4_0, 2>();
    return nullptr;
}

}  // namespace step_detail

size_t step_smem_bytes(const StepArgs& a) {
    return (size_t)a.ring_bytes + (size_t)a.act_bytes + sizeof(StepLayer) * (size_t)a.n_layer;
}

// Fills ring_bytes / act_bytes / max_split of `a` (taken as the plan) and
// returns the grid, or 0 when the configuration does not fit the kernel.
int step_plan_grid(StepArgs& a, int sm_count) {
    using namespace step_detail;
    void* kern = pick(a);
    if (!kern || a.B < 1 || a.B > 2 || a.n_layer < 1) return 0;
    const int qd = a.H * a.hd, kd = a.Hkv * a.hd, qkv_rows = qd + 2 * kd;
    const int HPG = a.Hkv > 0 ? a.H / a.Hkv : 0;
    if (a.Hkv < 1 || a.H % a.Hkv || HPG > kMaxHPG || (a.hd != 64 && a.hd != 128) || HPG * a.hd > kThreads) return 0;
    if (a.d > 8 * kThreads) return 0;  // norm_to holds at most two float4 of a row per thread
    if (a.V > sample_detail::kMaxV || a.d % 32 || a.ff % 32 || qd % 32) return 0;
    int G = sm_count < a.d ? sm_count : a.d;
    if (G > qkv_rows || G > a.ff || G > a.V) return 0;
    if ((a.d + G - 1) / G > kMaxOwn) return 0;
    // partial-sum staging of every slice: rows per CTA x batch rows x K slices
    auto fits = [&](int rows, int K) { return ((rows + G - 1) / G + 2) * a.B * ((K + 1023) / 1024) <= kMaxPart; };
    if (!fits(qkv_rows, a.d) || !fits(a.d, qd) || !fits(a.gpt2 ? a.ff : 2 * a.ff, a.d) || !fits(a.d, a.ff) ||
        !fits(a.V, a.d))
        return 0;
    a.max_split = G / (a.B * a.Hkv);
    if (a.max_split > 8) a.max_split = 8;
    if (a.max_split < 1) a.max_split = 1;
    a.act_bytes = (int)act_region_bytes(a);
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return 0;
    const int limit = 227 * 1024 - (int)fa.sharedSizeBytes - 1024;
    const int ring = (limit - a.act_bytes - (int)(sizeof(StepLayer) * a.n_layer)) & ~127;
    // the largest record: per slice, the rows one CTA owns (+2 for pair rounding)
    // times the row's codes and scales, plus the bias and gain windows
    auto rec = [&](int rows, int K, bool gains) {
        const int nr = (rows + G - 1) / G + 2;
        const int rowb = a.quant == SD_Q4_0 ? K / 2 : K;
        return nr * (rowb + K / 16) + 32 + (nr + 8) * 4 + (gains ? 8 * a.d : 0) + 128;
    };
    int max_rec = rec(qkv_rows, a.d, true);
    const int cand[4] = {rec(a.d, qd, false), rec(a.gpt2 ? a.ff : 2 * a.ff, a.d, true), rec(a.d, a.ff, false),
                         rec(a.V, a.d, true)};
    for (int i = 0; i < 4; ++i) max_rec = cand[i] > max_rec ? cand[i] : max_rec;
    if (ring < 2 * max_rec) return 0;
    a.ring_bytes = ring;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)step_smem_bytes(a)) !=
        cudaSuccess)
        return 0;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kBlock, step_smem_bytes(a)) != cudaSuccess ||
        per_sm < 1)
        return 0;
    return G;
}

cudaError_t launch_step(const StepArgs& a, int grid, cudaStream_t st) {
    using namespace step_detail;
    void* kern = pick(a);
    if (!kern || grid < 1) return cudaErrorInvalidValue;
    const size_t smem = step_smem_bytes(a);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kBlock);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {const_cast<StepArgs*>(&a)};
    return cudaLaunchKernelExC(&cfg, kern, args);
}

}  // namespace sd
