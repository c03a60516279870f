// Cluster persistent decode step for the GPT-2- and Llama-style T3 (rows
// B <= 2, Q8_0/Q4_0 weights): one launch runs n decode steps on `ncl`
// thread-block clusters of `cs` CTAs each.
//
// "Every Frame Is a Memory Read", section 3: a decode step is a memory read,
// and it runs at bandwidth only if the chain of dependent operations between
// the weight reads is short.  The layer order is that of "Chatterbox -> ggml
// Port: Development Journal", section 3.2 (norm -> QKV -> attention over the
// cache -> O + residual -> norm -> FC/gate-up -> proj/down + residual); the
// cache layout [head][pos][dim] and the causal extent are those of sections
// 3.12-3.13.  This kernel arranges the layer so that only two exchanges per
// layer cross the whole GPU:
//
//   cluster c owns KV heads [c*kpc, (c+1)*kpc) and their query heads.  Every
//   CTA normalises the full residual row; rank r computes its share of the
//   cluster's q, k, v rows and sends them to every rank of the cluster
//   (distributed shared memory, st.async completing on an mbarrier); rank r
//   attends over its share of the cached keys and sends its partial softmax
//   state (o, m, l) to every rank; every rank combines the partials and
//   multiplies the head outputs by the cluster's column slab of Wo, for its
//   own residual rows -- a split-K partial of the O projection.
//
//   Exchange 1 (global): rank r of every cluster publishes its rows of the
//   cluster's partial as epoch-tagged words; rank r of every cluster reads
//   the same rows of all clusters' partials, sums them in cluster order, adds
//   bias and residual and sends the rows to the ranks of its own cluster.
//   Every cluster so holds the same residual row, bit for bit.
//
//   Cluster c also owns FFN activations [c*upc, (c+1)*upc): rank r computes
//   its FC / gate-up rows with the GELU / SwiGLU epilogue, sends the
//   activations to every rank, and every rank multiplies them by the
//   cluster's column slab of the down projection for its rows -- exchange 2
//   as exchange 1.
//
// Weights reach each CTA through the producer warp's bulk-copy ring, as in
// the flat persistent step; every wait (exchange word, mbarrier, ring) is
// bounded, and on expiry the kernel records an error and returns.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <utility>
#include <vector>

#include "step_dev.cuh"

#define SAMPLE_SYNC() asm volatile("bar.sync 1, 512;" ::: "memory")
#define SAMPLE_NT 512
#include "sample_dev.cuh"

namespace sd {
namespace cstep_detail {

using namespace gemv_detail;
using namespace stepdev;

constexpr int kNMB = 16;      // weight records in flight at most (a power of two)
constexpr int kTokRep = 8;    // replicas of the sampled-token word

enum XB { XB_QKV = 0, XB_PART = 1, XB_X = 2, XB_U = 3 };

// ------------------------------------------------------------------ cluster primitives

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
// every thread of every CTA of the cluster (the producer warp included)
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t mapa(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
// 4-byte store into a cluster CTA's shared memory; completes `bytes` on its mbarrier
__device__ __forceinline__ void st_async(uint32_t raddr, float v, uint32_t rmb) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(raddr),
                 "r"(__float_as_uint(v)), "r"(rmb)
                 : "memory");
}
// one arrival on a cluster CTA's mbarrier, releasing (at cluster scope) every
// write that happens before it -- the KV-cache append among them
__device__ __forceinline__ void mb_arrive_remote(uint32_t rmb) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(rmb) : "memory");
}
__device__ __forceinline__ void mb_init_n(uint32_t mb, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mb), "r"(n) : "memory");
}
// the receiving CTA's own arrival for the next phase, with the bytes it expects
__device__ __forceinline__ void mb_arm(uint32_t mb, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mb_try_cl(uint32_t mb, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(mb), "r"(parity)
        : "memory");
    return ok != 0;
}
// bounded wait for an exchange phase (cluster-scope acquire of the data)
__device__ bool xb_wait(uint32_t mb, uint32_t parity, int* err, long long budget) {
    if (mb_try_cl(mb, parity)) return true;
    const long long t0 = clock64();
    for (unsigned it = 1;; ++it) {
        if (mb_try_cl(mb, parity)) return true;
        if ((it & 15u) == 0u) {
            if (ld_volatile(err)) return false;
            if (clock64() - t0 > budget) {
                atomicCAS(err, 0, kErrTimeout);
                return false;
            }
        }
    }
}

// ------------------------------------------------------------------ weight records

// One phase's record for this CTA: code rows [r0, r1) of a matrix (scale
// window widened to 16 bytes), bias rows [br0, br0 + r1 - r0) (window widened
// likewise), and the norm gains.
struct CSlice {
    const uint8_t* q;
    const uint8_t* s;
    const float *bias, *g1, *g2;
    int r0, r1, br0, row_bytes, srow, s_lo, b_lo, K;
    int o_sc, o_bias, o_g1, o_g2;
    int n_codes, n_sc, n_bias, n_g;
    int bytes;
};

// matrix, bias and gains of slice kind k (0 QKV, 1 O, 2 FC, 3 proj, 4 head) of layer l
__device__ __forceinline__ void kind_ptrs(const CStepArgs& a, const StepLayer* tab, int kind, int l, const QMat*& W,
                                          const float*& bias, const float*& g1, const float*& g2) {
    bias = nullptr; g1 = nullptr; g2 = nullptr;
    if (kind == 0) { W = &tab[l].wqkv; bias = tab[l].bqkv; g1 = tab[l].n1g; g2 = tab[l].n1b; }
    else if (kind == 1) { W = &tab[l].wo; bias = tab[l].bo; }
    else if (kind == 2) { W = &tab[l].wfc; bias = tab[l].bfc; g1 = tab[l].n2g; g2 = tab[l].n2b; }
    else if (kind == 3) { W = &tab[l].wproj; bias = tab[l].bproj; }
    else { W = &a.head; g1 = a.nfg; g2 = a.nfb; }
    if (!a.gpt2) g2 = nullptr;  // RMSNorm: gain only
}

__device__ CSlice make_cslice(const CStepArgs& a, const StepLayer* tab, int kind, int cl, int rank) {
    const int G = a.ncl * a.cs, gi = cl * a.cs + rank;
    const QMat* W;
    const float *bias, *g1, *g2;
    kind_ptrs(a, tab, kind, 0, W, bias, g1, g2);
    CSlice s;
    int r0, r1, br0;
    if (kind == 0) {
        row_range(a.rpc, rank, a.cs, r0, r1);
        r0 += cl * a.rpc; r1 += cl * a.rpc; br0 = r0;
    } else if (kind == 1 || kind == 3) {
        row_range(a.d, rank, a.cs, r0, r1);
        br0 = r0;
        r0 += cl * a.d; r1 += cl * a.d;
    } else if (kind == 2) {
        row_range(a.upc, rank, a.cs, r0, r1);
        r0 += cl * a.upc; r1 += cl * a.upc;
        if (!a.gpt2) { r0 *= 2; r1 *= 2; }  // gate/up rows interleaved in pairs
        br0 = r0;
    } else {
        row_range(a.V, gi, G, r0, r1);
        br0 = r0;
    }
    s.r0 = r0; s.r1 = r1; s.br0 = br0;
    s.K = W->cols;
    s.row_bytes = W->kind == SD_Q4_0 ? W->cols / 2 : W->cols;
    s.srow = (W->cols / 32) * 2;
    const int nr = r1 - r0;
    s.n_codes = nr * s.row_bytes;
    s.s_lo = (r0 * s.srow) & ~15;
    s.n_sc = (((r1 * s.srow) + 15) & ~15) - s.s_lo;
    s.o_sc = (s.n_codes + 15) & ~15;
    int off = s.o_sc + s.n_sc;
    s.b_lo = br0 & ~3;
    s.n_bias = bias ? ((((br0 + nr + 3) & ~3) - s.b_lo) * 4) : 0;
    s.o_bias = off;
    off += s.n_bias;
    s.n_g = g1 ? a.d * 4 : 0;
    s.o_g1 = off;
    off += s.n_g;
    s.o_g2 = off;
    off += g2 ? s.n_g : 0;
    s.bytes = (off + 127) & ~127;
    s.q = nullptr; s.s = nullptr;
    s.bias = bias; s.g1 = g1; s.g2 = g2;  // presence only; pointers per layer in cslice_at
    return s;
}

// slice j of a step (4 per layer, then the head): the per-kind geometry with
// this layer's pointers
__device__ __forceinline__ CSlice cslice_at(const CStepArgs& a, const StepLayer* tab, const CSlice* geo, int j) {
    const int L = a.n_layer;
    const int kind = j < 4 * L ? (j & 3) : 4;
    const int l = j >> 2;
    CSlice s = geo[kind];
    const QMat* W;
    const float *bias, *g1, *g2;
    kind_ptrs(a, tab, kind, l < L ? l : 0, W, bias, g1, g2);
    s.q = W->q + (size_t)s.r0 * s.row_bytes;
    s.s = reinterpret_cast<const uint8_t*>(W->s) + s.s_lo;
    s.bias = (s.bias && bias) ? bias + s.b_lo : nullptr;
    s.g1 = s.g1 ? g1 : nullptr;
    s.g2 = s.g2 ? g2 : nullptr;
    return s;
}

// ------------------------------------------------------------------ matvec over a record

// y[i * NB + b] = sum_k W[i][k] x[b][k] for the record's rows i < nr (codes
// row-major, fp16 block scales [nr][K/32] at sc); x rows are in the padded
// layout with row stride xs.  A row is split over LPR lanes (LPR = the row's
// 16-byte units, rounded up to a power of two, at most 32), each lane keeping
// the activations of its units in registers; a warp visits RPW = 32 / LPR rows
// at once, two row groups per iteration.  The LPR lane sums meet by xor
// shuffles (a fixed order).
template <int QK, int NB>
__device__ void cgemv(const uint8_t* codes, const uint8_t* sc, int K, int nr, const float* x, int xs, float* y) {
    constexpr int EPU = (QK == SD_Q4_0) ? 32 : 16;
    constexpr int MAXU = (QK == SD_Q4_0) ? 1 : 2;
    const int UPR = K / EPU;
    const int LPR = UPR >= 32 ? 32 : ((UPR & (UPR - 1)) ? 32 : UPR);
    const int RPW = 32 / LPR;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane % LPR, rl = lane / LPR;
    const int row_bytes = (QK == SD_Q4_0) ? (K >> 1) : K, spr = K >> 5;
    const int step = kWarps * RPW;
    const __half* sh = reinterpret_cast<const __half*>(sc);
    if (warp * RPW < nr) {
        float xr[NB][MAXU * EPU];
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int j = 0; j < MAXU; ++j) {
                const int u = sub + j * LPR;
#pragma unroll
                for (int t = 0; t < EPU; t += 4) {
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (u < UPR) v = *reinterpret_cast<const float4*>(&x[b * xs + pidx(u * EPU + t)]);
                    xr[b][j * EPU + t] = v.x; xr[b][j * EPU + t + 1] = v.y;
                    xr[b][j * EPU + t + 2] = v.z; xr[b][j * EPU + t + 3] = v.w;
                }
            }
        for (int i0 = warp * RPW; i0 < nr; i0 += 2 * step) {
            const int i1 = i0 + rl, i2 = i0 + step + rl;
            const bool v1 = i1 < nr, v2 = i2 < nr;
            float a1[NB], a2[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b) { a1[b] = 0.f; a2[b] = 0.f; }
#pragma unroll
            for (int j = 0; j < MAXU; ++j) {
                const int u = sub + j * LPR;
                if (u < UPR) {
                    const int e = u * EPU, off = (QK == SD_Q4_0) ? (e >> 1) : e;
                    uint4 w1 = make_uint4(0u, 0u, 0u, 0u), w2 = w1;
                    float d1 = 0.f, d2 = 0.f;
                    if (v1) {
                        w1 = *reinterpret_cast<const uint4*>(codes + (size_t)i1 * row_bytes + off);
                        d1 = __half2float(sh[(size_t)i1 * spr + (e >> 5)]);
                    }
                    if (v2) {
                        w2 = *reinterpret_cast<const uint4*>(codes + (size_t)i2 * row_bytes + off);
                        d2 = __half2float(sh[(size_t)i2 * spr + (e >> 5)]);
                    }
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        const float t1 = (QK == SD_Q4_0) ? dot4_q4(w1, &xr[b][0]) : dot4_s8(w1, &xr[b][j * EPU]);
                        a1[b] = fmaf(d1, t1, a1[b]);
                        if (v2) {
                            const float t2 =
                                (QK == SD_Q4_0) ? dot4_q4(w2, &xr[b][0]) : dot4_s8(w2, &xr[b][j * EPU]);
                            a2[b] = fmaf(d2, t2, a2[b]);
                        }
                    }
                }
            }
            for (int o = 1; o < LPR; o <<= 1)
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    a1[b] += __shfl_xor_sync(0xffffffffu, a1[b], o);
                    a2[b] += __shfl_xor_sync(0xffffffffu, a2[b], o);
                }
            if (sub == 0) {
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    if (v1) y[i1 * NB + b] = a1[b];
                    if (v2) y[i2 * NB + b] = a2[b];
                }
            }
        }
    }
    csync();
}

// ------------------------------------------------------------------ attention over the rank's keys

// One warp's online-softmax pass over keys [0, nk) of a staged sub-chunk
// (K and V rows of HD halves): LPK = HD / 8 lanes per key, each holding 8
// dimensions; KPP = 32 / LPK keys per warp pass.  (m: running max, uniform
// over the warp; l and o: per key slot, summed over the slots at the end.)
template <int HD>
__device__ __forceinline__ void attn_keys(const float (&q)[8], const __half* Ks, const __half* Vs, int nk, float& m,
                                          float& l, float (&o)[8]) {
    constexpr int LPK = HD / 8, KPP = 32 / LPK;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ks = lane / LPK, dg = lane % LPK;
    for (int j0 = warp * KPP; j0 < nk; j0 += kWarps * KPP) {
        const int j = j0 + ks;
        const bool valid = j < nk;
        uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
        if (valid) {
            kv = *reinterpret_cast<const uint4*>(Ks + (size_t)j * HD + dg * 8);
            vv = *reinterpret_cast<const uint4*>(Vs + (size_t)j * HD + dg * 8);
        }
        const float2 k0 = __half22float2(*reinterpret_cast<const __half2*>(&kv.x));
        const float2 k1 = __half22float2(*reinterpret_cast<const __half2*>(&kv.y));
        const float2 k2 = __half22float2(*reinterpret_cast<const __half2*>(&kv.z));
        const float2 k3 = __half22float2(*reinterpret_cast<const __half2*>(&kv.w));
        float s = fmaf(q[0], k0.x, q[1] * k0.y) + fmaf(q[2], k1.x, q[3] * k1.y);
        s += fmaf(q[4], k2.x, q[5] * k2.y) + fmaf(q[6], k3.x, q[7] * k3.y);
#pragma unroll
        for (int w = 1; w < LPK; w <<= 1) s += __shfl_xor_sync(0xffffffffu, s, w);
        s = valid ? s : -INFINITY;
        float pm = s;
#pragma unroll
        for (int w = LPK; w < 32; w <<= 1) pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, w));
        const float mn = fmaxf(m, pm);  // finite: key j0 (slot 0) is valid
        const float corr = expf(m - mn);
        const float p = valid ? expf(s - mn) : 0.f;
        l = fmaf(l, corr, p);
        const float2 v0 = __half22float2(*reinterpret_cast<const __half2*>(&vv.x));
        const float2 v1 = __half22float2(*reinterpret_cast<const __half2*>(&vv.y));
        const float2 v2 = __half22float2(*reinterpret_cast<const __half2*>(&vv.z));
        const float2 v3 = __half22float2(*reinterpret_cast<const __half2*>(&vv.w));
        o[0] = fmaf(o[0], corr, p * v0.x); o[1] = fmaf(o[1], corr, p * v0.y);
        o[2] = fmaf(o[2], corr, p * v1.x); o[3] = fmaf(o[3], corr, p * v1.y);
        o[4] = fmaf(o[4], corr, p * v2.x); o[5] = fmaf(o[5], corr, p * v2.y);
        o[6] = fmaf(o[6], corr, p * v3.x); o[7] = fmaf(o[7], corr, p * v3.y);
        m = mn;
    }
}

// ------------------------------------------------------------------ cross-cluster reduction

// Rows [xr0, xr0 + nr) of the residual stream after a split-K exchange: for
// each (row i, batch row b), the partials P[c][b][xr0 + i] of clusters c < ncl
// (epoch-tagged words) are summed in a fixed order -- TPR lanes of a group
// take clusters j, j + TPR, ... in increasing order and meet by xor shuffles
// -- then bias and the residual are added and the row is sent to every rank of
// the cluster (st.async into x, completing on its mbarrier mb_x).  All loads of
// a lane are issued before the first is waited for.  False on a timeout.
template <int NB>
__device__ bool reduce_bcast(const unsigned long long* P, int ncl, int d, int xr0, int nr, unsigned e,
                             const float* bias, const float* xs, int PD, uint32_t a_x, uint32_t mb_x, int cs, int* err,
                             long long budget) {
    int TPR = 1;
    while (TPR < 8 && 2 * TPR <= ncl && 2 * TPR * nr * NB <= kThreads) TPR <<= 1;
    const int total = nr * NB * TPR;
    bool ok = true;
    for (int base = 0; base < total; base += kThreads) {
        const int t = base + (int)threadIdx.x;
        const bool valid = t < total;
        const int ib = t / TPR, j = t - ib * TPR;
        const int i = ib / NB, b = ib - i * NB;
        float acc = 0.f;
        if (valid && ok) {
            for (int c0 = j; c0 < ncl && ok; c0 += 4 * TPR) {
                unsigned long long w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int c = c0 + q * TPR;
                    w[q] = c < ncl ? ll_load(P + ((size_t)c * NB + b) * d + xr0 + i) : 0ull;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int c = c0 + q * TPR;
                    if (c >= ncl || !ok) continue;
                    if ((unsigned)(w[q] >> 32) != e)
                        ok = ll_spin(P + ((size_t)c * NB + b) * d + xr0 + i, e, &w[q], err, budget);
                    acc += __uint_as_float((unsigned)w[q]);
                }
            }
        }
        for (int o = 1; o < TPR; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        float v = 0.f;
        if (valid && ok) {
            if (bias) acc += bias[i];
            v = xs[b * PD + pidx(xr0 + i)] + acc;
        }
        __syncwarp();  // every lane of the group has read the old row before one of them overwrites it
        if (valid && ok) {
            const uint32_t addr = a_x + 4u * (uint32_t)(b * PD + pidx(xr0 + i));
            for (int dst = j; dst < cs; dst += TPR) st_async(mapa(addr, dst), v, mapa(mb_x, dst));
        }
    }
    return ok;
}

// ------------------------------------------------------------------ the kernel

struct Geo {
    int cl, rank, gi, G;
    int xr0, xr1, qr0, qr1, fr0, fr1, hr0, hr1;
};

template <int QK, int NB>
__global__ void __launch_bounds__(kBlock, 1) k_cstep(const CStepArgs a) {
    extern __shared__ __align__(128) unsigned char sm[];
    unsigned char* ring = sm;
    unsigned char* actb = sm + a.ring_bytes;
    float* xs = reinterpret_cast<float*>(actb + a.o_x);     // [NB][padded(d)] residual rows
    float* xn = reinterpret_cast<float*>(actb + a.o_xn);    // [NB][padded(kin)] matvec input
    float* ub = reinterpret_cast<float*>(actb + a.o_u);     // [NB][padded(upc)] cluster FFN activations
    float* qkv = reinterpret_cast<float*>(actb + a.o_qkv);  // [NB][rpc] cluster q, k, v rows
    float* part = reinterpret_cast<float*>(actb + a.o_part);  // [cs][NB * hpc][hd + 4] rank partials
    float* ys = reinterpret_cast<float*>(actb + a.o_y);     // [rows][NB] matvec output
    float* wp = reinterpret_cast<float*>(actb + a.o_wp);    // [16][hd + 4] warp partials
    __half* stg = reinterpret_cast<__half*>(actb + a.o_stage);  // K then V [NB * kpc][kkc][hd]
    StepLayer* tab = reinterpret_cast<StepLayer*>(sm + a.ring_bytes + a.act_bytes);
    __shared__ __align__(8) unsigned long long s_mb[kNMB];
    __shared__ __align__(8) unsigned long long s_xb[4];
    __shared__ long long s_rec[kNMB];
    __shared__ int s_off[kNMB];
    __shared__ int s_nc, s_done;
    __shared__ __align__(16) float s_red[64];
    __shared__ int s_tok[2];
    __shared__ sample_detail::SampleScratch s_samp;
    __shared__ CSlice s_geo[5];
    __shared__ unsigned long long s_trc[kCTraceSub];

    const int tid = threadIdx.x;
    Geo g;
    g.cl = (int)cluster_index();
    g.rank = (int)cluster_rank();
    g.G = a.ncl * a.cs;
    g.gi = g.cl * a.cs + g.rank;
    row_range(a.d, g.rank, a.cs, g.xr0, g.xr1);
    row_range(a.rpc, g.rank, a.cs, g.qr0, g.qr1);
    row_range(a.upc, g.rank, a.cs, g.fr0, g.fr1);
    row_range(a.V, g.gi, g.G, g.hr0, g.hr1);
    const int L = a.n_layer, d = a.d, hd = a.hd, cs = a.cs;
    const int per_step = 4 * L + 1, total = a.n_steps * per_step;
    const int RB = a.ring_bytes;
    const long long budget = a.spin_budget;
    const bool ln = a.gpt2 != 0;
    const int PD = padded(d), PU = padded(a.upc), PO = padded(a.ko);
    const int W2 = hd + 4;  // partial record stride
    // bytes each exchange phase delivers to this CTA
    auto xb_bytes_of = [&](int k) -> uint32_t {
        return k == XB_QKV ? (uint32_t)(4 * NB * a.rpc)
             : k == XB_PART ? (uint32_t)(4 * cs * NB * a.hpc * (hd + 2))
             : k == XB_X ? (uint32_t)(4 * NB * d) : (uint32_t)(4 * NB * a.upc);
    };

    {
        const int words = L * (int)(sizeof(StepLayer) / 4);
        for (int i = tid; i < words; i += kBlock)
            reinterpret_cast<int*>(tab)[i] = reinterpret_cast<const int*>(a.layers)[i];
    }
    __syncthreads();
    if (tid < 5) s_geo[tid] = make_cslice(a, tab, tid, g.cl, g.rank);
    if (tid < kCTraceSub) s_trc[tid] = 0ull;
    if (tid == 0) {
        for (int k = 0; k < kNMB; ++k) mb_init(smem_u32(&s_mb[k]));
        // the partial exchange also counts one release arrival per rank (see the attention phase)
        for (int k = 0; k < 4; ++k) mb_init_n(smem_u32(&s_xb[k]), k == XB_PART ? 1 + a.cs : 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_nc = 0;
        s_done = 0;
    }
    __syncthreads();
    if (tid == 0)
        for (int k = 0; k < 4; ++k) mb_arm(smem_u32(&s_xb[k]), xb_bytes_of(k));
    // every CTA's exchange barriers are initialised and armed before any rank sends
    cluster_sync_all();

    // ---- producer warp: streams this CTA's weight records into the ring
    if (tid >= kThreads) {
        if (tid == kThreads) {
            int ni = 0, pj = 0, hoff = 0;
            long long head = 0, idle0 = clock64();
            bool ok = true;
            while (ni < total) {
                const int nc = ld_volatile(&s_nc);
                if (ld_volatile(&s_done)) break;
                bool issued = false;
                if (ni - nc < kNMB) {
                    const CSlice sl = cslice_at(a, tab, s_geo, pj);
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
                        bulk_g2s(dst, sl.q, (uint32_t)sl.n_codes, mb);
                        bulk_g2s(dst + sl.o_sc, sl.s, (uint32_t)sl.n_sc, mb);
                        if (sl.bias) bulk_g2s(dst + sl.o_bias, sl.bias, (uint32_t)sl.n_bias, mb);
                        if (sl.g1) bulk_g2s(dst + sl.o_g1, sl.g1, (uint32_t)sl.n_g, mb);
                        if (sl.g2) bulk_g2s(dst + sl.o_g2, sl.g2, (uint32_t)sl.n_g, mb);
                        head = start + sl.bytes;
                        hoff = off + sl.bytes;
                        ++ni;
                        if (++pj == per_step) pj = 0;
                        issued = true;
                        idle0 = clock64();
                    }
                }
                if (!issued) {
                    if (clock64() - idle0 > budget) {
                        atomicCAS(a.err, 0, kErrTimeout);
                        ok = false;
                        break;
                    }
                    __nanosleep(128);
                }
            }
            const long long t0 = clock64();
            while (!ld_volatile(&s_done) && ok && clock64() - t0 < budget) __nanosleep(256);
            for (int i = ld_volatile(&s_nc); i < ni; ++i)
                mb_wait(smem_u32(&s_mb[i & (kNMB - 1)]), (uint32_t)((i / kNMB) & 1), a.err, budget, true);
        }
        __syncwarp();
        cluster_sync_all();
        if (ld_volatile(a.err)) __nanosleep(20000);  // stores in flight from other ranks land first
        return;
    }

    // ---- compute threads
    const unsigned gen0 = *reinterpret_cast<const volatile unsigned*>(a.gen);
    const int pos0 = ld_volatile(a.pos);
    int nc = 0;
    unsigned ph_qkv = 0u, ph_part = 0u, ph_x = 0u, ph_u = 0u;  // completed phases of each exchange barrier
    // this CTA's exchange barriers and receive buffers (shared-window addresses; mapa() gives rank r's)
    const uint32_t mb_qkv = smem_u32(&s_xb[XB_QKV]), mb_part = smem_u32(&s_xb[XB_PART]);
    const uint32_t mb_x = smem_u32(&s_xb[XB_X]), mb_u = smem_u32(&s_xb[XB_U]);
    const uint32_t a_x = smem_u32(xs), a_qkv = smem_u32(qkv), a_part = smem_u32(part), a_u = smem_u32(ub);

    auto rec_ready = [&]() -> bool {
        return mb_wait(smem_u32(&s_mb[nc & (kNMB - 1)]), (uint32_t)((nc / kNMB) & 1), a.err, budget, false);
    };
    auto rec_base = [&]() -> const unsigned char* { return ring + s_off[nc & (kNMB - 1)]; };
    auto done_rec = [&]() {
        csync();
        ++nc;
        if (tid == 0) *reinterpret_cast<volatile int*>(&s_nc) = nc;
    };
    // waits for the next phase of an exchange barrier (every compute thread), re-arms it
    auto xwait = [&](uint32_t mb, unsigned& ph, uint32_t bytes) -> bool {
        bool ok = xb_wait(mb, ph & 1u, a.err, budget);
        if (ok && tid == 0) mb_arm(mb, bytes);
        ++ph;
        return csync_and(ok) != 0;
    };
    // CTA 0, thread 0: cycles since the previous stamp, added to sub-step k
    const bool trc = a.trace && g.gi == 0 && tid == 0;
    long long tc0 = trc ? clock64() : 0;
    auto stamp = [&](int k) {
        if (trc) {
            const long long t = clock64();
            s_trc[k] += (unsigned long long)(t - tc0);
            tc0 = t;
        }
    };
    auto tr_pub = [&](int s_, int l_, int phs) {
        if (a.trace_pub && tid == 0 && s_ < kTraceSteps) {
            const unsigned long long t = gtime();
            const size_t i = ((size_t)s_ * L + l_) * kCTracePhases + phs;
            atomicMax(a.trace_pub + i, t);
            atomicMin(a.trace_pub + (size_t)kTraceSteps * L * kCTracePhases + i, t);
        }
    };

    // KV staging of layer l (cp.async, through L2): item it = b * kpc + gg, keys [c0, min(c1, c0 + kkc))
    // except the position being decoded (it comes from this step's k, v)
    auto stage = [&](int l, int pos, int c0, int c1) {
        const int u16 = hd / 8, j1 = min(c1, c0 + a.kkc), nk = j1 - c0;
        const int items = NB * a.kpc, per = nk * u16;
        __half* Ks = stg;
        __half* Vs = stg + (size_t)items * a.kkc * hd;
        for (int t = tid; t < 2 * items * per; t += kThreads) {
            const bool isv = t >= items * per;
            const int tt = isv ? t - items * per : t;
            const int it = tt / per, rem = tt - it * per, r = rem / u16, un = rem - r * u16;
            if (c0 + r == pos) continue;
            const int b = it / a.kpc, gg = g.cl * a.kpc + (it - b * a.kpc);
            const size_t hb = ((size_t)(b * L + l) * a.Hkv + gg) * a.n_ctx * hd;
            const __half* src = (isv ? a.vc : a.kc) + hb + (size_t)(c0 + r) * hd + un * 8;
            __half* dst = (isv ? Vs : Ks) + ((size_t)it * a.kkc + r) * hd + un * 8;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    bool ok = true;
    for (int s = 0; s < a.n_steps && ok; ++s) {
        const int pos = pos0 + s, n = pos + 1;
        const unsigned eb = 1u + (gen0 + (unsigned)s) * (unsigned)(L + 1);
        int c0, c1;
        row_range(n, g.rank, cs, c0, c1);
        stamp(26);
        stage(0, pos, c0, c1);
        // ---- embedding: every CTA builds the whole input row
        {
            bool okr = true;
            if (tid < NB) {
                int t;
                if (s == 0) {
                    t = ld_volatile(a.tok + tid);
                } else {
                    const unsigned long long* tp = a.ll_tok + (g.gi % kTokRep) * 32 + tid;
                    unsigned long long w = ll_load(tp);
                    if ((unsigned)(w >> 32) != eb - 1u) okr = ll_spin(tp, eb - 1u, &w, a.err, budget);
                    t = (int)(unsigned)w;
                }
                if (t < 0 || t >= a.V) {
                    atomicCAS(a.err, 0, 3);
                    t = 0;
                }
                s_tok[tid] = t;
            }
            if (!csync_and(okr)) { ok = false; break; }
            for (int i = tid; i < NB * d; i += kThreads) {
                const int b = i / d, k = i - b * d;
                float v = __ldg(a.wte + (size_t)s_tok[b] * d + k);
                if (a.wpe) v += __ldg(a.wpe + (size_t)pos * d + k);
                xs[b * PD + pidx(k)] = v;
            }
            csync();
            stamp(27);
        }
        for (int l = 0; l < L && ok; ++l) {
            const unsigned e = eb + (unsigned)l;
            // ---- norm and this rank's q, k, v rows -> every rank of the cluster
            {
                bool okr = l > 0 ? xwait(mb_x, ph_x, xb_bytes_of(XB_X)) : true;
                stamp(0);
                if (okr) okr = csync_and(rec_ready()) != 0;
                if (!okr) { ok = false; break; }
                stamp(1);
                tr_pub(s, l, 0);
                const CSlice sl = cslice_at(a, tab, s_geo, 4 * l);
                const unsigned char* rec = rec_base();
                norm_to<NB>(xs, xn, d, ln, reinterpret_cast<const float*>(rec + sl.o_g1),
                            reinterpret_cast<const float*>(rec + sl.o_g2), a.eps, s_red);
                stamp(2);
                const int nr = sl.r1 - sl.r0;
                cgemv<QK, NB>(rec, rec + sl.o_sc + (sl.r0 * sl.srow - sl.s_lo), d, nr, xn, PD, ys);
                stamp(3);
                const float* bias = sl.bias ? reinterpret_cast<const float*>(rec + sl.o_bias) + (sl.br0 - sl.b_lo)
                                            : nullptr;
                for (int t = tid; t < nr * NB * cs; t += kThreads) {
                    const int dst = t % cs, ib = t / cs, i = ib / NB, b = ib - i * NB;
                    float v = ys[i * NB + b];
                    if (bias) v += bias[i];
                    st_async(mapa(a_qkv + 4u * (uint32_t)(b * a.rpc + g.qr0 + i), dst), v,
                             mapa(mb_qkv, dst));
                }
                tr_pub(s, l, 1);
                done_rec();
                stamp(4);
            }
            // ---- attention over this rank's keys [c0, c1)
            {
                if (!xwait(mb_qkv, ph_qkv, xb_bytes_of(XB_QKV))) { ok = false; break; }
                stamp(5);
                const int qd = a.hpc * hd, kd = a.kpc * hd, half = hd >> 1, hpg = a.hpc / a.kpc;
                const float scale = 1.0f / sqrtf((float)hd);
                const bool last = c1 == n;  // this rank holds the position being decoded
                // RoPE (NEOX half split) at pos on q and k; q scaled by 1/sqrt(hd)
                for (int i = tid; i < NB * (a.hpc + a.kpc) * half; i += kThreads) {
                    const int b = i / ((a.hpc + a.kpc) * half), r = i - b * (a.hpc + a.kpc) * half;
                    const int h = r / half, dd = r - h * half;
                    float* v = qkv + b * a.rpc + h * hd;  // q heads, then k heads (contiguous)
                    float x0 = v[dd], x1 = v[dd + half];
                    if (a.rope_cos) {
                        const float c = a.rope_cos[(size_t)pos * half + dd], sn = a.rope_sin[(size_t)pos * half + dd];
                        const float y0 = x0 * c - x1 * sn, y1 = x0 * sn + x1 * c;
                        x0 = y0;
                        x1 = y1;
                    }
                    if (h < a.hpc) {
                        x0 *= scale;
                        x1 *= scale;
                    }
                    v[dd] = x0;
                    v[dd + half] = x1;
                }
                csync();
                const int items = NB * a.kpc;
                __half* Ks = stg;
                __half* Vs = stg + (size_t)items * a.kkc * hd;
                if (last) {
                    // append the new position to the cache (fp16, round to nearest) and to the staging
                    for (int i = tid; i < items * hd; i += kThreads) {
                        const int it = i / hd, dd = i - it * hd, b = it / a.kpc, gl = it - b * a.kpc;
                        const int gg = g.cl * a.kpc + gl;
                        const __half kh = __float2half_rn(qkv[b * a.rpc + qd + gl * hd + dd]);
                        const __half vh = __float2half_rn(qkv[b * a.rpc + qd + kd + gl * hd + dd]);
                        const size_t hb = ((size_t)(b * L + l) * a.Hkv + gg) * a.n_ctx * hd + (size_t)pos * hd + dd;
                        a.kc[hb] = kh;
                        a.vc[hb] = vh;
                        if (pos - c0 < a.kkc) {
                            Ks[((size_t)it * a.kkc + (pos - c0)) * hd + dd] = kh;
                            Vs[((size_t)it * a.kkc + (pos - c0)) * hd + dd] = vh;
                        }
                    }
                }
                asm volatile("cp.async.wait_all;" ::: "memory");
                csync();
                stamp(6);
                const int warp = tid >> 5, lane = tid & 31;
                bool first_staged = true;  // the staging holds each item's first sub-chunk
                for (int it = 0; it < items; ++it) {
                    const int b = it / a.kpc, gl = it - b * a.kpc;
                    for (int h = 0; h < hpg; ++h) {
                        const int qh = gl * hpg + h;  // query head within the cluster
                        const int LPK = hd / 8, dg = lane % LPK;
                        float q[8];
#pragma unroll
                        for (int t = 0; t < 8; ++t) q[t] = qkv[b * a.rpc + qh * hd + dg * 8 + t];
                        float m = -INFINITY, lsum = 0.f, o[8];
#pragma unroll
                        for (int t = 0; t < 8; ++t) o[t] = 0.f;
                        for (int j0 = c0; j0 < c1; j0 += a.kkc) {
                            const int j1 = min(c1, j0 + a.kkc);
                            if (!(j0 == c0 && first_staged)) {
                                // a later sub-chunk (or the first one again after it was replaced)
                                csync();
                                const int u16 = hd / 8, per = (j1 - j0) * u16;
                                for (int t = tid; t < 2 * per; t += kThreads) {
                                    const bool isv = t >= per;
                                    const int tt = isv ? t - per : t, r = tt / u16, un = tt - r * u16;
                                    __half* dst = (isv ? Vs : Ks) + ((size_t)it * a.kkc + r) * hd + un * 8;
                                    if (j0 + r == pos) {
                                        const float* srcf = qkv + b * a.rpc + qd + (isv ? kd : 0) + gl * hd + un * 8;
#pragma unroll
                                        for (int w = 0; w < 8; ++w) dst[w] = __float2half_rn(srcf[w]);
                                        continue;
                                    }
                                    const int gg = g.cl * a.kpc + gl;
                                    const size_t hb = ((size_t)(b * L + l) * a.Hkv + gg) * a.n_ctx * hd;
                                    const __half* src = (isv ? a.vc : a.kc) + hb + (size_t)(j0 + r) * hd + un * 8;
                                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)),
                                                 "l"(src)
                                                 : "memory");
                                }
                                asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
                                csync();
                                first_staged = false;
                            }
                            if (hd == 64)
                                attn_keys<64>(q, Ks + (size_t)it * a.kkc * hd, Vs + (size_t)it * a.kkc * hd, j1 - j0,
                                              m, lsum, o);
                            else
                                attn_keys<128>(q, Ks + (size_t)it * a.kkc * hd, Vs + (size_t)it * a.kkc * hd, j1 - j0,
                                               m, lsum, o);
                        }
                        stamp(7);
                        // sum the key slots of the warp, then the warps (in warp order)
                        for (int w = LPK; w < 32; w <<= 1) {
                            lsum += __shfl_xor_sync(0xffffffffu, lsum, w);
#pragma unroll
                            for (int t = 0; t < 8; ++t) o[t] += __shfl_xor_sync(0xffffffffu, o[t], w);
                        }
                        if (lane < LPK) {
#pragma unroll
                            for (int t = 0; t < 8; ++t) wp[warp * W2 + dg * 8 + t] = o[t];
                            if (lane == 0) {
                                wp[warp * W2 + hd] = m;
                                wp[warp * W2 + hd + 1] = lsum;
                            }
                        }
                        csync();
                        const int bh = b * a.hpc + qh;
                        for (int t = tid; t < (hd + 2) * cs; t += kThreads) {
                            const int dst = t / (hd + 2), k = t - dst * (hd + 2);
                            float M = -INFINITY;
#pragma unroll 4
                            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wp[w * W2 + hd]);
                            float v = M;
                            if (k != hd) {
                                v = 0.f;
                                for (int w = 0; w < kWarps; ++w) {
                                    const float mw = wp[w * W2 + hd];
                                    if (mw != -INFINITY) v = fmaf(expf(mw - M), wp[w * W2 + k], v);
                                }
                            }
                            st_async(mapa(a_part + 4u * (uint32_t)((g.rank * NB * a.hpc + bh) * W2 + k), dst), v,
                                     mapa(mb_part, dst));
                        }
                        csync();
                    }
                }
                // one release arrival per rank: a reader of this KV head's cache in a later step
                // (another rank of this cluster) acquires the append through this barrier
                if (tid < cs) mb_arrive_remote(mapa(mb_part, tid));
                tr_pub(s, l, 2);
                stamp(8);
                // the staging is free: the next layer's keys
                if (l + 1 < L) stage(l + 1, pos, c0, c1);
            }
            // ---- combine the ranks' partials; O slab for this rank's rows -> global partial words
            {
                if (!xwait(mb_part, ph_part, xb_bytes_of(XB_PART))) { ok = false; break; }
                stamp(9);
                for (int t = tid; t < NB * a.hpc * hd; t += kThreads) {
                    const int bh = t / hd, dd = t - bh * hd;
                    float M = -INFINITY;
                    for (int r = 0; r < cs; ++r) M = fmaxf(M, part[(r * NB * a.hpc + bh) * W2 + hd]);
                    float num = 0.f, den = 0.f;
                    for (int r = 0; r < cs; ++r) {
                        const float* P = part + (r * NB * a.hpc + bh) * W2;
                        if (P[hd] == -INFINITY) continue;
                        const float w = expf(P[hd] - M);
                        num = fmaf(w, P[dd], num);
                        den = fmaf(w, P[hd + 1], den);
                    }
                    const int b = bh / a.hpc, qh = bh - b * a.hpc;
                    xn[b * PO + pidx(qh * hd + dd)] = num / den;
                }
                csync();
                stamp(10);
                if (!csync_and(rec_ready())) { ok = false; break; }
                stamp(11);
                const CSlice sl = cslice_at(a, tab, s_geo, 4 * l + 1);
                const unsigned char* rec = rec_base();
                const int nr = sl.r1 - sl.r0;
                cgemv<QK, NB>(rec, rec + sl.o_sc + (sl.r0 * sl.srow - sl.s_lo), a.ko, nr, xn, PO, ys);
                stamp(12);
                for (int t = tid; t < nr * NB; t += kThreads) {
                    const int i = t / NB, b = t - i * NB;
                    ll_store(a.ll_po + ((size_t)g.cl * NB + b) * d + g.xr0 + i, ys[t], e);
                }
                tr_pub(s, l, 3);
                stamp(13);
                // ---- exchange 1: rows [xr0, xr1) of every cluster's partial, summed in cluster order
                const float* bias = sl.bias ? reinterpret_cast<const float*>(rec + sl.o_bias) + (sl.br0 - sl.b_lo)
                                            : nullptr;
                const bool okr = reduce_bcast<NB>(a.ll_po, a.ncl, d, g.xr0, nr, e, bias, xs, PD, a_x, mb_x, cs, a.err,
                                                  budget);
                if (!csync_and(okr)) { ok = false; break; }
                tr_pub(s, l, 4);
                done_rec();
                stamp(14);
            }
            // ---- norm and this rank's FC / gate-up rows -> cluster FFN activations
            {
                bool okr = xwait(mb_x, ph_x, xb_bytes_of(XB_X));
                stamp(15);
                if (okr) okr = csync_and(rec_ready()) != 0;
                if (!okr) { ok = false; break; }
                stamp(16);
                const CSlice sl = cslice_at(a, tab, s_geo, 4 * l + 2);
                const unsigned char* rec = rec_base();
                norm_to<NB>(xs, xn, d, ln, reinterpret_cast<const float*>(rec + sl.o_g1),
                            reinterpret_cast<const float*>(rec + sl.o_g2), a.eps, s_red);
                stamp(17);
                const int nr = sl.r1 - sl.r0;
                cgemv<QK, NB>(rec, rec + sl.o_sc + (sl.r0 * sl.srow - sl.s_lo), d, nr, xn, PD, ys);
                stamp(18);
                const float* bias = sl.bias ? reinterpret_cast<const float*>(rec + sl.o_bias) + (sl.br0 - sl.b_lo)
                                            : nullptr;
                const int nu = ln ? nr : nr / 2;
                for (int t = tid; t < nu * NB * cs; t += kThreads) {
                    const int dst = t % cs, ib = t / cs, i = ib / NB, b = ib - i * NB;
                    float v;
                    if (ln) {
                        v = ys[i * NB + b];
                        if (bias) v += bias[i];
                        v = gelu_tanh(v);
                    } else {
                        v = silu(ys[(2 * i) * NB + b]) * ys[(2 * i + 1) * NB + b];
                    }
                    st_async(mapa(a_u + 4u * (uint32_t)(b * PU + pidx(g.fr0 + i)), dst), v, mapa(mb_u, dst));
                }
                tr_pub(s, l, 5);
                done_rec();
                stamp(19);
            }
            // ---- down-projection slab for this rank's rows -> exchange 2
            {
                bool okr = xwait(mb_u, ph_u, xb_bytes_of(XB_U));
                stamp(20);
                if (okr) okr = csync_and(rec_ready()) != 0;
                if (!okr) { ok = false; break; }
                stamp(21);
                const CSlice sl = cslice_at(a, tab, s_geo, 4 * l + 3);
                const unsigned char* rec = rec_base();
                const int nr = sl.r1 - sl.r0;
                cgemv<QK, NB>(rec, rec + sl.o_sc + (sl.r0 * sl.srow - sl.s_lo), a.upc, nr, ub, PU, ys);
                stamp(22);
                for (int t = tid; t < nr * NB; t += kThreads) {
                    const int i = t / NB, b = t - i * NB;
                    ll_store(a.ll_pp + ((size_t)g.cl * NB + b) * d + g.xr0 + i, ys[t], e);
                }
                tr_pub(s, l, 6);
                stamp(23);
                const float* bias = sl.bias ? reinterpret_cast<const float*>(rec + sl.o_bias) + (sl.br0 - sl.b_lo)
                                            : nullptr;
                okr = reduce_bcast<NB>(a.ll_pp, a.ncl, d, g.xr0, nr, e, bias, xs, PD, a_x, mb_x, cs, a.err, budget);
                if (!csync_and(okr)) { ok = false; break; }
                tr_pub(s, l, 7);
                done_rec();
                stamp(24);
            }
        }
        if (!ok) break;
        // ---- head rows (final norm)
        const unsigned eh = eb + (unsigned)L;
        {
            bool okr = xwait(mb_x, ph_x, xb_bytes_of(XB_X));
            if (okr) okr = csync_and(rec_ready()) != 0;
            if (!okr) { ok = false; break; }
            const CSlice sl = cslice_at(a, tab, s_geo, 4 * L);
            const unsigned char* rec = rec_base();
            norm_to<NB>(xs, xn, d, ln, reinterpret_cast<const float*>(rec + sl.o_g1),
                        reinterpret_cast<const float*>(rec + sl.o_g2), a.eps, s_red);
            const int nr = sl.r1 - sl.r0;
            cgemv<QK, NB>(rec, rec + sl.o_sc + (sl.r0 * sl.srow - sl.s_lo), d, nr, xn, PD, ys);
            for (int t = tid; t < nr * NB; t += kThreads) {
                const int i = t / NB, b = t - i * NB;
                a.logits[(size_t)b * a.V + sl.r0 + i] = ys[t];
                ll_store(a.ll_logits + (size_t)b * a.V + sl.r0 + i, ys[t], eh);
            }
            done_rec();
            stamp(25);
        }
        // ---- sampler: CTA b samples row b
        if (g.gi < NB) {
            float* z = reinterpret_cast<float*>(stg);
            const int b = g.gi;
            bool okr = true;
            for (int i0 = tid; i0 < a.V && okr; i0 += 4 * kThreads) {
                unsigned long long w[4];
                const unsigned long long* p[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int i = i0 + j * kThreads;
                    p[j] = i < a.V ? a.ll_logits + (size_t)b * a.V + i : nullptr;
                    w[j] = p[j] ? ll_load(p[j]) : 0ull;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (!p[j] || !okr) continue;
                    if ((unsigned)(w[j] >> 32) != eh) okr = ll_spin(p[j], eh, &w[j], a.err, budget);
                    z[i0 + j * kThreads] = __uint_as_float((unsigned)w[j]);
                }
            }
            if (!csync_and(okr)) { ok = false; break; }
            const float* up = a.u_seq ? a.u_seq + (size_t)s * NB + b : a.u1 + b;
            const int tk = sample_detail::sample_smem(a.V, *a.sp, up, reinterpret_cast<unsigned char*>(z), s_samp,
                                                      a.err);
            if (tid == 0) {
                a.tok[b] = tk;
                if (a.out_seq) a.out_seq[(size_t)s * NB + b] = tk;
#pragma unroll
                for (int r = 0; r < kTokRep; ++r) ll_store(a.ll_tok + r * 32 + b, __int_as_float(tk), eh);
            }
            csync();
        }
    }
    if (g.gi == 0 && tid == 0) {
        if (ok) *a.pos = pos0 + a.n_steps;
        *a.gen = gen0 + (unsigned)a.n_steps;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    csync();
    if (a.trace && g.gi == 0 && tid < kCTraceSub) a.trace[tid] += s_trc[tid];
    if (tid == 0) {
        *reinterpret_cast<volatile int*>(&s_nc) = nc;
        __threadfence_block();
        *reinterpret_cast<volatile int*>(&s_done) = 1;
    }
    // no CTA of the cluster leaves while another may still send into its shared memory
    cluster_sync_all();
    if (ld_volatile(a.err)) __nanosleep(20000);
}

template <int QK, int NB>
void* kernel_ptr() {
    return reinterpret_cast<void*>(k_cstep<QK, NB>);
}

void* pick(const CStepArgs& a) {
    if (a.quant == SD_Q8_0) return a.B == 1 ? kernel_ptr<SD_Q8_0, 1>() : kernel_ptr<SD_Q8_0, 2>();
    if (a.quant == SD_Q4_0) return a.B == 1 ? kernel_ptr<SD_Q4_0, 1>() : kernel_ptr<SD_Q4_0, 2>();
    return nullptr;
}

// ------------------------------------------------------------------ slab gather (set-up)

__global__ void k_slab_gather(const uint8_t* q, const __half* s, int R, int K, int W, int q4, const int* perm,
                              uint8_t* qo, __half* so) {
    const int rb = q4 ? K / 2 : K, wb = q4 ? W / 2 : W;  // code bytes per source row / per slab row
    const int ns = K / W;
    const long long chunks = (long long)R * rb / 16;
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < chunks;
         t += (long long)gridDim.x * blockDim.x) {
        const int i = (int)(t / (rb / 16)), cb = (int)(t % (rb / 16)) * 16;  // out row i, byte cb of the full row
        const int sl = cb / wb, ib = cb - sl * wb;
        const int src = perm ? perm[i] : i;
        *reinterpret_cast<uint4*>(qo + ((size_t)sl * R + i) * wb + ib) =
            *reinterpret_cast<const uint4*>(q + (size_t)src * rb + cb);
    }
    const int spr = K / 32, sps = W / 32;
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < (long long)R * spr;
         t += (long long)gridDim.x * blockDim.x) {
        const int i = (int)(t / spr), j = (int)(t % spr);
        const int sl = j / sps, jj = j - sl * sps;
        const int src = perm ? perm[i] : i;
        so[((size_t)sl * R + i) * sps + jj] = s[(size_t)src * spr + j];
    }
    (void)ns;
}

}  // namespace cstep_detail

size_t cstep_smem_bytes(const CStepArgs& a) {
    return (size_t)a.ring_bytes + (size_t)a.act_bytes + sizeof(StepLayer) * (size_t)a.n_layer;
}

// Activation-region layout for the plan in `a` (B, d, upc, ko, rpc, hpc, kpc, cs, hd, kkc); returns its bytes.
static size_t cstep_layout(CStepArgs& a, int yrows) {
    using gemv_detail::padded;
    const int B = a.B;
    auto al = [](size_t v) { return (v + 127) & ~(size_t)127; };
    size_t off = 0;
    const int kin = a.d > a.ko ? a.d : a.ko;
    a.o_x = (int)off; off = al(off + 4 * (size_t)B * padded(a.d));
    a.o_xn = (int)off; off = al(off + 4 * (size_t)B * padded(kin));
    a.o_u = (int)off; off = al(off + 4 * (size_t)B * padded(a.upc));
    a.o_qkv = (int)off; off = al(off + 4 * (size_t)B * a.rpc);
    a.o_part = (int)off; off = al(off + 4 * (size_t)a.cs * B * a.hpc * (a.hd + 4));
    a.o_y = (int)off; off = al(off + 4 * (size_t)yrows * B);
    a.o_wp = (int)off; off = al(off + 4 * (size_t)stepdev::kWarps * (a.hd + 4));
    a.o_stage = (int)off;
    const size_t stage = 2 * sizeof(__half) * (size_t)B * a.kpc * a.kkc * a.hd;
    const size_t smp = sample_smem_bytes_dev(a.V, stepdev::kThreads);
    off = al(off + (stage > smp ? stage : smp));
    return off;
}

int cstep_plan(CStepArgs& a, int sm_count) {
    using namespace cstep_detail;
    void* kern = pick(a);
    if (!kern || a.B < 1 || a.B > 2 || a.n_layer < 1 || a.Hkv < 1 || a.H % a.Hkv) return 0;
    if ((a.hd != 64 && a.hd != 128) || a.d % 32 || a.ff % 32 || a.V > sample_detail::kMaxV) return 0;
    if (a.d > 8 * stepdev::kThreads) return 0;  // norm_to holds at most two float4 of a row per thread
    const int maxk = a.quant == SD_Q4_0 ? 1024 : 1024;  // one (Q4_0) or two (Q8_0) 16-byte units per lane
    if (a.d > maxk) return 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) return 0;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return 0;
    const int limit = 227 * 1024 - (int)fa.sharedSizeBytes - 1024;
    int best = 0;
    CStepArgs pick_a = a;
    const bool dbg = getenv("SD_PLAN_DEBUG") != nullptr;
    // candidates: ncl divides Hkv, cs any size from 16 down to 2 (the part's GPCs do not all
    // hold the same number of clusters of a size); the most CTAs that can be resident wins,
    // then the most clusters (fewer heads per cluster)
    std::vector<std::pair<int, int>> cand;  // (ncl, cs), best first: the most CTAs, then the most clusters
    for (int ncl = a.Hkv; ncl >= 1; --ncl)
        if (a.Hkv % ncl == 0)
            for (int cs = 16; cs >= 2; --cs)
                if (ncl * cs <= sm_count) cand.push_back({ncl, cs});
    std::stable_sort(cand.begin(), cand.end(), [](const std::pair<int, int>& x, const std::pair<int, int>& y) {
        const int gx = x.first * x.second, gy = y.first * y.second;
        return gx != gy ? gx > gy : x.first > y.first;
    });
    for (const auto& nc : cand) {
        if (best) break;
        {
            const int ncl = nc.first, cs = nc.second;
            CStepArgs t = a;
            t.ncl = ncl; t.cs = cs;
            t.kpc = a.Hkv / ncl; t.hpc = a.H / ncl;
            t.rpc = (t.hpc + 2 * t.kpc) * a.hd;
            t.ko = t.hpc * a.hd;
            t.upc = a.ff / ncl;
            if (a.ff % ncl || t.upc % 32 || t.ko > maxk || t.upc > maxk) continue;
            if (ncl * cs > a.V || cs > a.d || t.upc < cs || t.rpc < cs) continue;
            // keys per rank staged at once: the whole share of a full context where it fits
            const int G = ncl * cs;
            auto cdiv = [](int x, int y) { return (x + y - 1) / y; };
            const int urows = a.gpt2 ? cdiv(t.upc, cs) : 2 * cdiv(t.upc, cs);
            int yrows = cdiv(t.rpc, cs) + 1;
            yrows = std::max(yrows, cdiv(a.d, cs) + 1);
            yrows = std::max(yrows, urows + 2);
            yrows = std::max(yrows, cdiv(a.V, G) + 1);
            t.kkc = std::min(256, std::max(32, ((cdiv(a.n_ctx, cs) + 31) / 32) * 32));
            int act = (int)cstep_layout(t, yrows);
            while (t.kkc > 32 && act > limit / 2) {
                t.kkc -= 32;
                act = (int)cstep_layout(t, yrows);
            }
            t.act_bytes = act;
            const int ring = (limit - act - (int)(sizeof(StepLayer) * a.n_layer)) & ~127;
            // the largest record: rows x (codes + scales) + bias and gain windows
            auto rec = [&](int rows, int K, bool gains) {
                const int rowb = a.quant == SD_Q4_0 ? K / 2 : K;
                return rows * (rowb + K / 16) + 64 + (rows + 8) * 4 + (gains ? 8 * a.d : 0) + 256;
            };
            // records in step order: QKV, O, FC, proj per layer, then the head; the ring holds
            // any two consecutive ones of a layer, so the next record streams in while one is in
            // use (the head record, once per step, may have to wait for the ring to drain)
            const int rq = rec(cdiv(t.rpc, cs), a.d, true), ro = rec(cdiv(a.d, cs), t.ko, false);
            const int rf = rec(urows, a.d, true), rp = rec(cdiv(a.d, cs), t.upc, false);
            const int rh = rec(cdiv(a.V, G), a.d, true);
            const int need = std::max({rq + ro, ro + rf, rf + rp, rp + rq, rh});
            if (dbg)
                fprintf(stderr, "cstep plan: ncl %d cs %d act %d ring %d records %d %d %d %d %d kkc %d\n", ncl, cs,
                        act, ring, rq, ro, rf, rp, rh, t.kkc);
            if (ring < need) continue;
            t.ring_bytes = ring;
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cstep_smem_bytes(t)) !=
                cudaSuccess)
                continue;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(G);
            cfg.blockDim = dim3(stepdev::kBlock);
            cfg.dynamicSmemBytes = cstep_smem_bytes(t);
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = cs;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int nclu = 0;
            const cudaError_t oe = cudaOccupancyMaxActiveClusters(&nclu, kern, &cfg);
            if (dbg) fprintf(stderr, "cstep plan: ncl %d cs %d: %d clusters fit (%s)\n", ncl, cs, nclu, cudaGetErrorString(oe));
            if (oe != cudaSuccess || nclu < ncl) {
                cudaGetLastError();
                continue;
            }
            if (G > best || (G == best && ncl > pick_a.ncl)) {
                best = G;
                pick_a = t;
            }
        }
    }
    if (!best) return 0;
    a = pick_a;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cstep_smem_bytes(a)) !=
        cudaSuccess)
        return 0;
    return best;
}

cudaError_t launch_cstep(const CStepArgs& a, cudaStream_t st) {
    using namespace cstep_detail;
    void* kern = pick(a);
    if (!kern || a.ncl < 1 || a.cs < 1) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.ncl * a.cs);
    cfg.blockDim = dim3(stepdev::kBlock);
    cfg.dynamicSmemBytes = cstep_smem_bytes(a);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {const_cast<CStepArgs*>(&a)};
    return cudaLaunchKernelExC(&cfg, kern, args);
}

cudaError_t launch_slab_gather(const QMat& src, int W, const int* perm, uint8_t* q_out, __half* s_out,
                               cudaStream_t st) {
    if ((src.kind != SD_Q4_0 && src.kind != SD_Q8_0) || W < 32 || W % 32 || src.cols % W) return cudaErrorInvalidValue;
    const int q4 = src.kind == SD_Q4_0;
    if ((q4 ? W / 2 : W) % 16) return cudaErrorInvalidValue;
    cstep_detail::k_slab_gather<<<1024, 256, 0, st>>>(src.q, reinterpret_cast<const __half*>(src.s), src.rows,
                                                      src.cols, W, q4, perm, q_out, s_out);
    return cudaGetLastError();
}

}  // namespace sd
