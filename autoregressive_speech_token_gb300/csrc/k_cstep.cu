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
//   attends over its blocks of 32 cached positions (block j belongs to rank
//   j % cs, so a position is appended and later read by the same CTA and the
//   cache needs no cross-CTA ordering) and sends its partial softmax
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
// Every matvec is a run of mma.sync m16n8k16 over 16-row tiles of exact fp16
// codes against the activations split into fp16 hi and lo parts (see the
// tensor-core matvec below): the decode step's arithmetic is issue-bound on
// CUDA cores at this grid size, and the tensor cores take a 16 x 16 block of
// weights per instruction.  Weights reach each CTA through a ring of bulk
// asynchronous copies in shared memory, issued by thread 0 whenever it is
// about to wait anyway, as far ahead as the ring holds; every wait (exchange
// word, mbarrier, ring) is bounded, and on expiry the kernel records an error,
// finishes the step on whatever data it has and returns.
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
constexpr int kRB = 8;        // exchange words one thread of a reduction loads at once
constexpr int kTokRep = 8;    // replicas of the sampled-token word

// exchange barriers: q/k/v rows, attention partials, residual rows after the O projection (x')
// and after the down projection (x''), FFN activations -- one phase per layer each
enum XB { XB_QKV = 0, XB_PART = 1, XB_X0 = 2, XB_X1 = 3, XB_U = 4 };

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
// every thread of every CTA of the cluster
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
// non-blocking test of an mbarrier phase (this CTA's view)
__device__ __forceinline__ bool mb_test(uint32_t mb, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(mb), "r"(parity)
        : "memory");
    return ok != 0;
}
// one arrival on this CTA's mbarrier (release at CTA scope)
__device__ __forceinline__ void mb_arrive_local(uint32_t mb) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mb) : "memory");
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
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(mb), "r"(parity)
        : "memory");
    return ok != 0;
}
// bounded wait for a phase of this CTA's mbarrier: bytes written by st.async or bulk copies that
// completed the phase are visible to the waiting thread once it returns true
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

// ------------------------------------------------------------------ fragment-major weights

// The cluster step's matrices are stored 16 rows (a tile) by 32 columns (a
// block) at a time, in the order the tensor-core matvec consumes them: per
// (tile, block), the 32 lanes' code words for rows g and g + 8 of the tile
// (lane 4g + t) -- Q4_0: the word of code bytes 4t..4t+3 of each row, Q8_0:
// the two words of code bytes 8t..8t+7 -- then, after all (tile, block)
// pairs of the matrix, the tiles' fp16 block scales [tile][block][16 rows].
// A warp's loads of one (tile, block) are then 256 (Q4_0) or 512 (Q8_0)
// contiguous bytes, free of bank conflicts, and a range of whole tiles is one
// contiguous copy.  Rows past the matrix end are zero codes with zero scales.
template <int QK>
struct Frag {
    static constexpr int W = (QK == SD_Q4_0) ? 1 : 2;  // code words per lane per row and block
    static constexpr int TB = 256 * W;                 // code bytes of one (tile, block)
};
__host__ __device__ __forceinline__ int frag_tb(int quant) { return quant == SD_Q4_0 ? 256 : 512; }

// ------------------------------------------------------------------ weight records

// One phase's record for this CTA: tiles [t0, t0 + nt) of a fragment-major
// matrix (codes, then scales), the bias of rows [br0, br0 + nr) (window widened
// to 16 bytes), and the norm gains (padded layout).  Pointers are per layer.
struct CSlice {
    int t0, nt, nr, br0, KB;
    int o_sc, o_bias, o_g1, o_g2;
    int n_codes, n_sc, n_bias, n_g, b_lo;
    int bytes;
    int has_bias, has_g1, has_g2;
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

// tiles [t0, t1) of N tiles for part i of G (in whole tiles)
__host__ __device__ __forceinline__ void tile_range(int N, int i, int G, int& t0, int& t1) {
    t0 = N * i / G;
    t1 = N * (i + 1) / G;
}

__device__ CSlice make_cslice(const CStepArgs& a, const StepLayer* tab, int kind, int cl, int rank) {
    const int G = a.ncl * a.cs, gi = cl * a.cs + rank;
    const QMat* W;
    const float *bias, *g1, *g2;
    kind_ptrs(a, tab, kind, 0, W, bias, g1, g2);
    CSlice s;
    int t0, t1;
    if (kind == 0) {
        const int N = a.rpc / 16;
        tile_range(N, rank, a.cs, t0, t1);
        t0 += cl * N; t1 += cl * N;
        s.br0 = 16 * t0;
        s.nr = 16 * (t1 - t0);
    } else if (kind == 1 || kind == 3) {
        const int N = a.d / 16;
        tile_range(N, rank, a.cs, t0, t1);
        s.br0 = 16 * t0;  // residual rows of this rank
        s.nr = 16 * (t1 - t0);
        t0 += cl * N; t1 += cl * N;
    } else if (kind == 2) {
        const int N = (a.gpt2 ? a.upc : 2 * a.upc) / 16;  // gate/up rows interleaved in pairs
        tile_range(N, rank, a.cs, t0, t1);
        t0 += cl * N; t1 += cl * N;
        s.br0 = 16 * t0;
        s.nr = 16 * (t1 - t0);
    } else {
        tile_range((a.V + 15) / 16, gi, G, t0, t1);
        s.br0 = 16 * t0;
        s.nr = min(16 * t1, a.V) - 16 * t0;
    }
    s.t0 = t0;
    s.nt = t1 - t0;
    s.KB = W->cols / 32;
    s.n_codes = s.nt * s.KB * frag_tb(W->kind);
    s.n_sc = s.nt * s.KB * 32;
    s.o_sc = s.n_codes;
    int off = s.o_sc + s.n_sc;
    s.b_lo = s.br0 & ~3;
    s.n_bias = bias ? ((((s.br0 + s.nr + 3) & ~3) - s.b_lo) * 4) : 0;
    s.o_bias = off;
    off += s.n_bias;
    s.n_g = g1 ? padded(a.d) * 4 : 0;  // gains are stored in the padded activation layout
    s.o_g1 = off;
    off += s.n_g;
    s.o_g2 = off;
    off += g2 ? s.n_g : 0;
    s.bytes = (off + 127) & ~127;
    s.has_bias = bias != nullptr;
    s.has_g1 = g1 != nullptr;
    s.has_g2 = g2 != nullptr;
    return s;
}

// ------------------------------------------------------------------ tensor-core matvec over a record

// The record's rows are the M = 16 side of mma.sync m16n8k16: the codes are
// small integers, exact in fp16 (byte v placed under the exponent of 1024 is
// the half 1024 + v; one half2 subtraction removes the offset), and the fp32
// activations enter as B columns 2b (hi = fp16(x)) and 2b + 1 (lo = fp16(x -
// hi)), so x = hi + lo to 22 bits and every product is exact in fp32.  A
// block's two 16-wide k-steps accumulate in fp32 and are scaled by the rows'
// block scales.  Inside a block the MMA k index is permuted -- the same
// permutation for codes and activations, so the dot product is unchanged --
// so that a lane's codes of a row are one word per step: step s of a block
// takes elements 16s + 4t + j (Q4_0: low nibbles of code bytes 4t..4t+3 for
// s = 0, high nibbles for s = 1) or 8t + 4s + j (Q8_0: code bytes 8t..8t+7),
// j = 0..3, which sit at k = 2t, 2t+1 (j = 0, 1) and 2t+8, 2t+9 (j = 2, 3).

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
    const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
}

// the four codes of word w (elements j = 0..3) of step s -> halves for
// k = 2t, 2t+1 (lo) and 2t+8, 2t+9 (hi)
template <int QK>
__device__ __forceinline__ void code_pair(uint32_t w, int s, uint32_t& lo, uint32_t& hi) {
    uint32_t off;
    if constexpr (QK == SD_Q4_0) {
        w = (s ? (w >> 4) : w) & 0x0F0F0F0Fu;
        off = 0x64086408u;  // 1024 + 8
    } else {
        w ^= 0x80808080u;   // signed byte v -> v + 128
        off = 0x64806480u;  // 1024 + 128
    }
    lo = hsub2_u(__byte_perm(w, 0x64646464u, 0x4140), off);
    hi = hsub2_u(__byte_perm(w, 0x64646464u, 0x4342), off);
}

// Half index of element e (of a K-long activation row) in the B-fragment
// buffer [block][step][column][lane t][4 halves j]; batch row b's hi part is
// column 2b, its lo part column 2b + 1.
template <int QK, int NB>
__device__ __forceinline__ int bf_index(int e, int col) {
    const int kb = e >> 5, r = e & 31, j = r & 3;
    int s, t;
    if (QK == SD_Q4_0) { s = r >> 4; t = (r >> 2) & 3; }
    else { t = r >> 3; s = (r >> 2) & 1; }
    return ((((kb * 2 + s) * 2 * NB + col) * 4 + t) << 2) + j;
}

template <int QK, int NB>
__device__ __forceinline__ void bf_put(__half* bf, int e, int b, float x) {
    const __half h = __float2half_rn(x);
    bf[bf_index<QK, NB>(e, 2 * b)] = h;
    bf[bf_index<QK, NB>(e, 2 * b + 1)] = __float2half_rn(x - __half2float(h));
}

// B fragments of activation rows src[b][pidx(k)] (row stride ss), k < K, as
// they are.  Ends with a CTA barrier.
template <int QK, int NB>
__device__ void bf_plain(const float* src, int ss, int K, __half* bf) {
#pragma unroll
    for (int b = 0; b < NB; ++b)
        for (int e = threadIdx.x; e < K; e += kThreads) bf_put<QK, NB>(bf, e, b, src[b * ss + pidx(e)]);
    csync();
}

// B fragments of the LayerNorm (biased variance) or RMSNorm of x[b][pidx(k)],
// k < K <= 2 * kThreads, with gains g1 and offsets g2 in the padded layout.
// One pass: the sums of (x - c) and (x - c)^2 with the shift c = x[0] (the
// shifted-data variance, exact in real arithmetic and free of the cancellation
// of the plain one-pass form when |mean| >> deviation), per warp by shuffles,
// then across the warps through `red` (>= 4 * NB * kWarps floats, each warp
// reducing the table again by shuffles in a fixed order).  Ends with a CTA
// barrier.
template <int QK, int NB>
__device__ void bf_norm(const float* x, int xs, int K, bool ln, const float* g1, const float* g2, float eps,
                        float* red, __half* bf) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float v[NB][2], c[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        c[b] = ln ? x[b * xs] : 0.f;
        float s1 = 0.f, s2 = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int e = tid + j * kThreads;
            v[b][j] = e < K ? x[b * xs + pidx(e)] : 0.f;
            const float dv = e < K ? v[b][j] - c[b] : 0.f;
            s1 += dv;
            s2 = fmaf(dv, dv, s2);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            s1 += __shfl_xor_sync(0xffffffffu, s1, o);
            s2 += __shfl_xor_sync(0xffffffffu, s2, o);
        }
        if (lane == 0) {
            red[(2 * b) * kWarps + warp] = s1;
            red[(2 * b + 1) * kWarps + warp] = s2;
        }
    }
    csync();
    const float inv = 1.0f / (float)K;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        float s1 = lane < kWarps ? red[(2 * b) * kWarps + lane] : 0.f;
        float s2 = lane < kWarps ? red[(2 * b + 1) * kWarps + lane] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {  // lanes past the table hold zeros; every lane gets the totals
            s1 += __shfl_xor_sync(0xffffffffu, s1, o);
            s2 += __shfl_xor_sync(0xffffffffu, s2, o);
        }
        const float m1 = s1 * inv;  // mean of x - c
        const float var = ln ? fmaxf(s2 * inv - m1 * m1, 0.f) : s2 * inv;
        const float mu = ln ? c[b] + m1 : 0.f;
        const float r = 1.0f / sqrtf(var + eps);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int e = tid + j * kThreads;
            if (e >= K) continue;
            const float gg = g1[pidx(e)];
            const float y = ln ? fmaf((v[b][j] - mu) * r, gg, g2[pidx(e)]) : v[b][j] * r * gg;
            bf_put<QK, NB>(bf, e, b, y);
        }
    }
    csync();
}

// sum_k W[i][k] x[b][k] for the record's rows i < nr (tiles of fragment-major
// codes and scales), x given as B fragments.  Units of (tile, k-slice) go to
// the warps -- KS slices per tile, as many as leave no warp idle, at most four -- and each
// unit's partial sums go to red[unit][16][NB]; after a CTA barrier the slices
// are added in order and emit(i, b, y) (PAIRS: emit(i, b, y_2i, y_2i+1) for
// row pairs) runs once per output.  The codes are read straight from the
// record in shared memory.
template <int QK, int NB, bool PAIRS, typename Emit>
__device__ __forceinline__ void mma_rows(const uint8_t* codes, const uint8_t* sc, int K, int nt, int nr,
                                         const __half* bf, float* red, Emit&& emit) {
    constexpr int W = Frag<QK>::W;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int KB = K >> 5;
    int KS = kWarps / nt;
    if (KS < 1) KS = 1;
    if (KS > 4) KS = 4;  // measured: past four slices the extra reduction costs more than the shorter runs save
    if (KS > KB) KS = KB;
    const int units = nt * KS;
    const __half* sh = reinterpret_cast<const __half*>(sc);
    const uint2* bfv = reinterpret_cast<const uint2*>(bf);
    for (int u = warp; u < units; u += kWarps) {
        const int rt = u / KS, s = u - rt * KS;
        const int kb0 = KB * s / KS, kb1 = KB * (s + 1) / KS;
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 2
        for (int kb = kb0; kb < kb1; ++kb) {
            const int tb = rt * KB + kb;
            uint32_t w0[W], w1[W];
            if constexpr (W == 1) {
                const uint2 aw = reinterpret_cast<const uint2*>(codes)[tb * 32 + lane];
                w0[0] = aw.x;
                w1[0] = aw.y;
            } else {
                const uint4 aw = reinterpret_cast<const uint4*>(codes)[tb * 32 + lane];
                w0[0] = aw.x; w0[W - 1] = aw.y;
                w1[0] = aw.z; w1[W - 1] = aw.w;
            }
            float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int st = 0; st < 2; ++st) {
                uint32_t a0, a1, a2, a3;
                code_pair<QK>(w0[W == 1 ? 0 : st], st, a0, a2);
                code_pair<QK>(w1[W == 1 ? 0 : st], st, a1, a3);
                uint2 bb = make_uint2(0u, 0u);
                if (g < 2 * NB) bb = bfv[((kb * 2 + st) * 2 * NB + g) * 4 + t];
                mma16816(c, a0, a1, a2, a3, bb.x, bb.y);
            }
            const float d0 = __half2float(sh[tb * 16 + g]), d1 = __half2float(sh[tb * 16 + g + 8]);
            acc0 = fmaf(d0, c[0] + c[1], acc0);
            acc1 = fmaf(d1, c[2] + c[3], acc1);
        }
        if (t < NB) {
            red[(u * 16 + g) * NB + t] = acc0;
            red[(u * 16 + g + 8) * NB + t] = acc1;
        }
    }
    csync();
    // the KS slices of an output meet by xor shuffles: lane s of a group of KSP (a power of two
    // >= KS) lanes loads slice s (a fixed order); the group then holds the sum
    int lk = 0;
    while ((1 << lk) < KS) ++lk;
    const int KSP = 1 << lk;
    const int outs = PAIRS ? (nr >> 1) * NB : nr * NB;
    for (int base = 0; base < outs * KSP; base += kThreads) {
        const int x = base + tid, o = x >> lk, s = x & (KSP - 1);
        const bool live = o < outs;
        int row, b;
        if (PAIRS) {
            const int k = NB == 1 ? o : o / NB;
            b = o - k * NB;
            row = 2 * k;
        } else {
            row = NB == 1 ? o : o / NB;
            b = o - row * NB;
        }
        const int rt = row >> 4, rr = row & 15;
        float v0 = 0.f, v1 = 0.f;
        if (live && s < KS) {
            v0 = red[((rt * KS + s) * 16 + rr) * NB + b];
            if (PAIRS) v1 = red[((rt * KS + s) * 16 + rr + 1) * NB + b];
        }
        for (int m = 1; m < KSP; m <<= 1) {
            v0 += __shfl_xor_sync(0xffffffffu, v0, m);
            if (PAIRS) v1 += __shfl_xor_sync(0xffffffffu, v1, m);
        }
        if (live && s == 0) emit(PAIRS ? row >> 1 : row, b, v0, v1);
    }
}

// ------------------------------------------------------------------ attention over the rank's keys

// One warp's pass over keys [j0, j0 + 32) of a staged sub-chunk of nk keys
// (rows of HD halves): lane = key.  A lane forms its key's score over the
// whole head dimension, reading the row's 16-byte chunks in an order rotated
// by the lane so that a quarter warp touches distinct bank groups; the warp
// keeps an online softmax (m, l: uniform over the warp; o: DPL dimensions per
// lane) and accumulates p V with lanes over dimensions.
template <int HD>
__device__ __forceinline__ void attn_lk(const float* q, const __half* Ks, const __half* Vs, int j0, int nk, float& m,
                                        float& l, float (&o)[HD / 32]) {
    constexpr int CH = HD / 8, DPL = HD / 32;
    const int lane = threadIdx.x & 31;
    const int j = j0 + lane;
    const bool valid = j < nk;
    float s = -INFINITY;
    if (valid) {
        const __half* kr = Ks + (size_t)j * HD;
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int cc = (c + lane) & (CH - 1);
            const uint4 kv = *reinterpret_cast<const uint4*>(kr + cc * 8);
            const float4 qa = *reinterpret_cast<const float4*>(q + cc * 8);
            const float4 qb = *reinterpret_cast<const float4*>(q + cc * 8 + 4);
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
        s = (s0 + s1) + (s2 + s3);
    }
    float mx = s;
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
    const float mn = fmaxf(m, mx);  // finite: key j0 (lane 0) is valid
    const float corr = expf(m - mn);
    const float p = valid ? expf(s - mn) : 0.f;
    l = fmaf(l, corr, warp_sum(p));
    float ov[DPL];
#pragma unroll
    for (int dd = 0; dd < DPL; ++dd) ov[dd] = 0.f;
    const int cnt = min(32, nk - j0);
    const __half* vr = Vs + (size_t)j0 * HD + lane * DPL;
#pragma unroll 8
    for (int jj = 0; jj < 32; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
        if (jj >= cnt) continue;  // warp-uniform
        if (DPL == 2) {
            const float2 v = __half22float2(*reinterpret_cast<const __half2*>(vr + (size_t)jj * HD));
            ov[0] = fmaf(pj, v.x, ov[0]);
            ov[1] = fmaf(pj, v.y, ov[1]);
        } else {
            const uint2 vv = *reinterpret_cast<const uint2*>(vr + (size_t)jj * HD);
            const float2 v0 = __half22float2(*reinterpret_cast<const __half2*>(&vv.x));
            const float2 v1 = __half22float2(*reinterpret_cast<const __half2*>(&vv.y));
            ov[0] = fmaf(pj, v0.x, ov[0]);
            ov[1] = fmaf(pj, v0.y, ov[1]);
            ov[DPL - 2] = fmaf(pj, v1.x, ov[DPL - 2]);
            ov[DPL - 1] = fmaf(pj, v1.y, ov[DPL - 1]);
        }
    }
#pragma unroll
    for (int dd = 0; dd < DPL; ++dd) o[dd] = fmaf(o[dd], corr, ov[dd]);
    m = mn;
}

// ------------------------------------------------------------------ cross-cluster reduction

// Rows [xr0, xr0 + nr) of the residual stream after a split-K exchange: for
// each (row i, batch row b), the partials P[c][b][xr0 + i] of clusters c < ncl
// (epoch-tagged words) are summed in a fixed order -- TPR lanes of a group
// take clusters j, j + TPR, ... in increasing order and meet by xor shuffles
// -- then bias and the residual are added and the row is sent to every rank of
// the cluster (st.async into x, completing on its mbarrier mb_x).  A lane
// issues up to kRB loads before it waits for the first (all of them when
// ncl <= kRB * TPR: one L2 round trip per reduction).  A wait that expires
// leaves the error word set and the sum undefined (the step is then abandoned).
template <int NB>
__device__ void reduce_bcast(const unsigned long long* P, int ncl, int d, int xr0, int nr, unsigned e,
                             const float* bias, const float* xs, int PD, uint32_t a_x, uint32_t mb_x, int cs, int* err,
                             long long budget) {
    int lt = 0;  // TPR = 1 << lt
    while (lt < 3 && (2 << lt) <= ncl && (2 << lt) * nr * NB <= kThreads) ++lt;
    const int TPR = 1 << lt;
    const int total = nr * NB * TPR;
    bool ok = true;
    for (int base = 0; base < total; base += kThreads) {
        const int t = base + (int)threadIdx.x;
        const bool valid = t < total;
        const int ib = t >> lt, j = t & (TPR - 1);
        const int i = ib / NB, b = ib - i * NB;
        float acc = 0.f;
        if (valid) {
            for (int c0 = j; c0 < ncl; c0 += kRB * TPR) {
                // the (up to) kRB words are loaded together and polled until all carry epoch e,
                // so the wait ends one load after the last of them lands; they are added in
                // cluster order
                const unsigned long long* pw[kRB];
                unsigned long long w[kRB];
                unsigned pend = 0u;
#pragma unroll
                for (int q = 0; q < kRB; ++q) {
                    const int c = c0 + q * TPR;
                    pw[q] = P + ((size_t)(c < ncl ? c : 0) * NB + b) * d + xr0 + i;
                    w[q] = 0ull;
                    if (c < ncl) pend |= 1u << q;
                }
                const long long t0 = clock64();
                for (unsigned it = 0; pend && ok; ++it) {
#pragma unroll
                    for (int q = 0; q < kRB; ++q)
                        if (pend & (1u << q)) w[q] = ll_load(pw[q]);
#pragma unroll
                    for (int q = 0; q < kRB; ++q)
                        if ((pend & (1u << q)) && (unsigned)(w[q] >> 32) == e) pend &= ~(1u << q);
                    if (!pend) break;
                    if (it > 2u) __nanosleep(32);
                    if ((it & 31u) == 31u) {
                        if (ld_volatile(err)) ok = false;
                        else if (clock64() - t0 > budget) {
                            atomicCAS(err, 0, kErrTimeout);
                            ok = false;
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < kRB; ++q)
                    if (c0 + q * TPR < ncl) acc += __uint_as_float((unsigned)w[q]);
            }
        }
        for (int o = 1; o < TPR; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        float v = 0.f;
        if (valid) {
            if (bias) acc += bias[i];
            v = xs[b * PD + pidx(xr0 + i)] + acc;
        }
        __syncwarp();  // every lane of the group has read the old row before one of them overwrites it
        if (valid) {
            const uint32_t addr = a_x + 4u * (uint32_t)(b * PD + pidx(xr0 + i));
            for (int dst = j; dst < cs; dst += TPR) st_async(mapa(addr, dst), v, mapa(mb_x, dst));
        }
    }
}

// ------------------------------------------------------------------ the kernel

constexpr int kCBlock = kThreads;  // 16 warps, no producer warp: a thread may hold 128 registers

template <int QK, int NB>
__global__ void __launch_bounds__(kCBlock, 1) k_cstep(const CStepArgs a) {
    extern __shared__ __align__(128) unsigned char sm[];
    unsigned char* ring = sm;
    unsigned char* actb = sm + a.ring_bytes;
    float* xs = reinterpret_cast<float*>(actb + a.o_x);       // [NB][padded(d)] residual rows
    float* ub = reinterpret_cast<float*>(actb + a.o_u);       // [NB][padded(upc)] cluster FFN activations
    float* qkv = reinterpret_cast<float*>(actb + a.o_qkv);    // [NB][rpc] cluster q, k, v rows
    float* part = reinterpret_cast<float*>(actb + a.o_part);  // [cs][NB * hpc][hd + 4] rank partials
    float* wq = reinterpret_cast<float*>(actb + a.o_wq);      // [16][hd] each warp's rotated query
    float* wp = reinterpret_cast<float*>(actb + a.o_wp);      // [16][hd + 4] warp partials
    __half* bf = reinterpret_cast<__half*>(actb + a.o_bf);    // B fragments of the current matvec input
    float* red = reinterpret_cast<float*>(actb + a.o_red);    // matvec partial sums
    __half* stg = reinterpret_cast<__half*>(actb + a.o_stage);  // K then V [NB * kpc][kkc][hd]
    StepLayer* tab = reinterpret_cast<StepLayer*>(sm + a.ring_bytes + a.act_bytes);
    __shared__ __align__(8) unsigned long long s_mb[kNMB];     // record landed
    __shared__ __align__(8) unsigned long long s_empty[kNMB];  // record consumed by every warp
    __shared__ __align__(8) unsigned long long s_xb[5];        // exchange phases received
    __shared__ __align__(8) unsigned long long s_kv;           // KV staging landed
    __shared__ long long s_rec[kNMB];
    __shared__ int s_off[kNMB];
    __shared__ int s_tok[2];
    __shared__ __align__(16) float s_red[4 * 2 * kWarps];
    __shared__ sample_detail::SampleScratch s_samp;
    __shared__ CSlice s_geo[5];
    __shared__ unsigned long long s_trc[kCTraceSub];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cl = (int)cluster_index(), rank = (int)cluster_rank();
    const int gi = cl * a.cs + rank;
    const int L = a.n_layer, d = a.d, hd = a.hd, cs = a.cs;
    const int per_step = 4 * L + 1, total = a.n_steps * per_step;
    const int RB = a.ring_bytes;
    const long long budget = a.spin_budget;
    const uint64_t wpol = l2_policy(a.w_evict_first != 0);
    const bool ln = a.gpt2 != 0;
    const int PD = padded(d), PU = padded(a.upc);
    const int W2 = hd + 4;  // partial record stride
    const int lhd = 31 - __clz(hd);
    // attention roles, fixed for the launch: (row, query head) pair pr of this warp and its index
    // wi among the WG warps of the pair; b_, qh_, gl_: its batch row, query head and KV head
    const int hpg = a.hpc / a.kpc, nph = NB * a.hpc;
    const int WG = nph >= kWarps ? 1 : kWarps / nph;
    const int pr = warp / WG, wi = warp - pr * WG;
    const int b_ = pr < nph ? pr / a.hpc : 0;
    const int qh_ = pr < nph ? pr - b_ * a.hpc : 0;
    const int gl_ = qh_ / hpg;
    // combine-and-send entries of this thread: (pair, component) = (cp_p, cp_k) for u = tid
    const int cp_p = tid / (hd + 2), cp_k = tid - cp_p * (hd + 2);
    // bytes each exchange phase delivers to this CTA
    auto xb_bytes_of = [&](int k) -> uint32_t {
        return k == XB_QKV ? (uint32_t)(4 * NB * a.rpc)
             : k == XB_PART ? (uint32_t)(4 * cs * NB * a.hpc * (hd + 2))
             : k == XB_U ? (uint32_t)(4 * NB * a.upc) : (uint32_t)(4 * NB * d);
    };

    {
        const int words = L * (int)(sizeof(StepLayer) / 4);
        for (int i = tid; i < words; i += kCBlock)
            reinterpret_cast<int*>(tab)[i] = reinterpret_cast<const int*>(a.layers)[i];
    }
    __syncthreads();
    if (tid < 5) s_geo[tid] = make_cslice(a, tab, tid, cl, rank);
    if (tid < kCTraceSub) s_trc[tid] = 0ull;
    if (tid == 0) {
        for (int k = 0; k < kNMB; ++k) {
            mb_init(smem_u32(&s_mb[k]));
            mb_init_n(smem_u32(&s_empty[k]), kWarps);
        }
        for (int k = 0; k < 5; ++k) mb_init_n(smem_u32(&s_xb[k]), 1);
        mb_init(smem_u32(&s_kv));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (tid == 0)
        for (int k = 0; k < 5; ++k) mb_arm(smem_u32(&s_xb[k]), xb_bytes_of(k));
    // every CTA's exchange barriers are initialised and armed before any rank sends
    cluster_sync_all();
    // this rank's rows: residual rows (O / proj), cluster q/k/v rows, FFN activations
    const int xr0 = s_geo[1].br0, nx = s_geo[1].nr;
    const int qr0 = s_geo[0].br0 - cl * a.rpc;
    const int fr0 = (s_geo[2].br0 - cl * (ln ? a.upc : 2 * a.upc)) >> (ln ? 0 : 1);

    const unsigned gen0 = *reinterpret_cast<const volatile unsigned*>(a.gen);
    const int pos0 = ld_volatile(a.pos);
    int nc = 0;  // records this warp has consumed (the same sequence in every warp)
    // completed phases of the exchange barriers and of the KV staging barrier
    unsigned ph_qkv = 0u, ph_part = 0u, ph_x0 = 0u, ph_x1 = 0u, ph_u = 0u, ph_kv = 0u;
    const uint32_t mb_qkv = smem_u32(&s_xb[XB_QKV]), mb_part = smem_u32(&s_xb[XB_PART]);
    const uint32_t mb_x0 = smem_u32(&s_xb[XB_X0]), mb_x1 = smem_u32(&s_xb[XB_X1]), mb_u = smem_u32(&s_xb[XB_U]);
    const uint32_t mb_kv = smem_u32(&s_kv);
    const uint32_t a_x = smem_u32(xs), a_qkv = smem_u32(qkv), a_part = smem_u32(part), a_u = smem_u32(ub);

    // ---- weight ring, run by thread 0: records issued (p_ni), records every warp has consumed
    // (p_nc), the next record's slice index within a step (p_pj), the ring head (p_head, p_hoff)
    int p_ni = 0, p_nc = 0, p_pj = 0, p_hoff = 0;
    long long p_head = 0;
    // issues records while they fit: at most kNMB in flight, and a record never overwrites the
    // oldest record a warp still reads; with nothing in flight any record fits
    auto pump = [&]() {
        while (p_nc < p_ni && mb_test(smem_u32(&s_empty[p_nc & (kNMB - 1)]), (uint32_t)((p_nc / kNMB) & 1)))
            ++p_nc;
        while (p_ni < total && p_ni - p_nc < kNMB) {
            const int kind = p_pj < 4 * L ? (p_pj & 3) : 4;
            const CSlice& G0 = s_geo[kind];
            const int bytes = G0.bytes;
            long long start = p_head;
            int off = p_hoff;
            if (off + bytes > RB) {
                start += RB - off;
                off = 0;
            }
            if (p_ni > p_nc && start + bytes - s_rec[p_nc & (kNMB - 1)] > RB) break;
            const int l = p_pj >> 2;
            const QMat* Wm;
            const float *bias, *g1, *g2;
            kind_ptrs(a, tab, kind, l < L ? l : 0, Wm, bias, g1, g2);
            const uint32_t dst = smem_u32(ring + off);
            const uint32_t mb = smem_u32(&s_mb[p_ni & (kNMB - 1)]);
            s_rec[p_ni & (kNMB - 1)] = start;
            s_off[p_ni & (kNMB - 1)] = off;
            const int nb_ = G0.has_bias ? G0.n_bias : 0, ng = G0.has_g1 ? G0.n_g : 0, ng2 = G0.has_g2 ? G0.n_g : 0;
            const size_t tbase = (size_t)G0.t0 * G0.KB;
            const size_t sc_off = (size_t)((Wm->rows + 15) / 16) * G0.KB * frag_tb(Wm->kind);
            mb_expect(mb, (uint32_t)(G0.n_codes + G0.n_sc + nb_ + ng + ng2));
            bulk_g2s_pol(dst, Wm->q + tbase * frag_tb(Wm->kind), (uint32_t)G0.n_codes, mb, wpol);
            bulk_g2s_pol(dst + G0.o_sc, Wm->q + sc_off + tbase * 32, (uint32_t)G0.n_sc, mb, wpol);
            if (nb_) bulk_g2s_pol(dst + G0.o_bias, bias + G0.b_lo, (uint32_t)nb_, mb, wpol);
            if (ng) bulk_g2s_pol(dst + G0.o_g1, g1, (uint32_t)ng, mb, wpol);
            if (ng2) bulk_g2s_pol(dst + G0.o_g2, g2, (uint32_t)ng2, mb, wpol);
            p_head = start + bytes;
            p_hoff = off + bytes;
            ++p_ni;
            if (++p_pj == per_step) p_pj = 0;
        }
    };
    // waits for record nc to land (thread 0 keeps the ring topped up meanwhile, so the record is
    // issued as soon as it fits); false on an expired wait or a recorded error
    auto rec_wait = [&]() -> bool {
        const uint32_t mb = smem_u32(&s_mb[nc & (kNMB - 1)]), par = (uint32_t)((nc / kNMB) & 1);
        if (mb_test(mb, par)) return true;  // landed (thread 0 refills the ring when it has to wait)
        const long long t0 = clock64();
        for (unsigned it = 1;; ++it) {
            if (tid == 0) pump();
            if (mb_try(mb, par)) return true;
            if ((it & 15u) == 0u) {
                if (ld_volatile(a.err)) return false;
                if (clock64() - t0 > budget) {
                    atomicCAS(a.err, 0, kErrTimeout);
                    return false;
                }
            }
        }
    };
    auto rec_base = [&]() -> const unsigned char* { return ring + s_off[nc & (kNMB - 1)]; };
    // this warp is done with record nc
    auto rec_done = [&]() {
        __syncwarp();
        if (lane == 0) mb_arrive_local(smem_u32(&s_empty[nc & (kNMB - 1)]));
        ++nc;
    };
    // waits for the next phase of an exchange barrier; thread 0 re-arms it at once.  (Every barrier
    // is re-armed before this CTA's next CTA-wide barrier, and no rank sends the next phase's data
    // before this CTA has passed that barrier.)
    auto xwait = [&](uint32_t mb, unsigned& ph, uint32_t bytes) -> bool {
        if (tid == 0 && !mb_test(mb, ph & 1u)) pump();  // idle time: refill the weight ring
        const bool ok = xb_wait(mb, ph & 1u, a.err, budget);
        if (ok && tid == 0) mb_arm(mb, bytes);
        ++ph;
        return ok;
    };
    // CTA 0, thread 0: cycles since the previous stamp, added to sub-step k
    const bool trc = a.trace && gi == a.trace_gi && tid == 0;
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
            if (a.trace_cta && s_ < kCtaSteps) a.trace_cta[i * (a.ncl * a.cs) + gi] = t;
        }
    };
    // KV staging: the cached keys are owned in blocks of 32 positions, block j by rank j % cs, so the
    // rank that appends a position is the only one that ever reads it back (no cross-CTA ordering of
    // the cache is needed).  Staging fill: this rank's blocks q0..q1-1 (block j = rank + q * cs) of
    // layer l for every (row, KV head) item, without the position being decoded (its key comes
    // from this step): two bulk copies per item and block (thread 0)
    int kv_issued = 0;
    const int SB = a.kkc / 32;  // blocks per staging fill
    auto kv_fetch = [&](int l, int pos, int q0, int q1) {
        ++kv_issued;
        // the staging was last read by generic loads; the cache was appended by generic stores
        asm volatile("fence.proxy.async.shared::cta;\n\tfence.proxy.async.global;" ::: "memory");
        const int items = NB * a.kpc;
        uint32_t total = 0u;
        for (int q = q0; q < q1; ++q) {
            const int j = rank + q * cs, nrow = min(32, pos - 32 * j);
            if (nrow > 0) total += (uint32_t)(nrow * hd * 2);
        }
        mb_expect(mb_kv, 2u * (uint32_t)items * total);
        for (int q = q0; q < q1; ++q) {
            const int j = rank + q * cs, nrow = min(32, pos - 32 * j);
            if (nrow <= 0) continue;
            for (int it = 0; it < items; ++it) {
                const int b = it / a.kpc, gg = cl * a.kpc + (it - b * a.kpc);
                const size_t hb = ((size_t)(b * L + l) * a.Hkv + gg) * a.n_ctx * hd + (size_t)(32 * j) * hd;
                const size_t so = ((size_t)it * a.kkc + (q - q0) * 32) * hd;
                bulk_g2s(smem_u32(stg + so), a.kc + hb, (uint32_t)(nrow * hd * 2), mb_kv);
                bulk_g2s(smem_u32(stg + (size_t)items * a.kkc * hd + so), a.vc + hb, (uint32_t)(nrow * hd * 2), mb_kv);
            }
        }
    };
    // matvec operands of the current record
    auto rec_codes = [&](const unsigned char* rec) { return reinterpret_cast<const uint8_t*>(rec); };

    if (tid == 0) pump();
    bool ok = true;
    for (int s = 0; s < a.n_steps; ++s) {
        const int pos = pos0 + s, n = pos + 1;
        const unsigned eb = 1u + (gen0 + (unsigned)s) * (unsigned)(L + 1);
        const int nb = (n + 31) >> 5;                                      // key blocks
        const int nbr = nb > rank ? (nb - rank + cs - 1) / cs : 0;          // this rank's blocks
        const int jl = nb - 1;                                              // the block of pos
        stamp(26);
        if (tid == 0) kv_fetch(0, pos, 0, min(nbr, SB));
        // RoPE angles at pos for the pairs (i, i + hd/2) of this lane, i = lane, lane + 32
        float rcs[2] = {1.f, 1.f}, rsn[2] = {0.f, 0.f};
        if (a.rope_cos)
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int i = lane + 32 * t;
                if (i < hd / 2) {
                    rcs[t] = __ldg(a.rope_cos + (size_t)pos * (hd / 2) + i);
                    rsn[t] = __ldg(a.rope_sin + (size_t)pos * (hd / 2) + i);
                }
            }
        // ---- embedding: every CTA builds the whole input row
        {
            if (tid < NB) {
                int t;
                if (s == 0) {
                    t = ld_volatile(a.tok + tid);
                } else {
                    const unsigned long long* tp = a.ll_tok + (gi % kTokRep) * 32 + tid;
                    unsigned long long w = ll_load(tp);
                    if ((unsigned)(w >> 32) != eb - 1u && !ll_spin(tp, eb - 1u, &w, a.err, budget)) w = 0ull;
                    t = (int)(unsigned)w;
                }
                if (t < 0 || t >= a.V_in) {
                    atomicCAS(a.err, 0, 3);
                    t = 0;
                }
                s_tok[tid] = t;
            }
            csync();
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float* te = a.wte + (size_t)s_tok[b] * d;
                for (int k = tid; k < d; k += kThreads) {
                    float v = __ldg(te + k);
                    if (a.wpe) v += __ldg(a.wpe + (size_t)pos * d + k);
                    xs[b * PD + pidx(k)] = v;
                }
            }
            csync();
            stamp(27);
        }
        for (int l = 0; l < L; ++l) {
            const unsigned e = eb + (unsigned)l;
            const int qd = a.hpc * hd, kd = a.kpc * hd;
            // ---- norm and this rank's q, k, v rows -> every rank of the cluster
            {
                if (l > 0) xwait(mb_x1, ph_x1, xb_bytes_of(XB_X1));
                stamp(0);
                rec_wait();
                stamp(1);
                tr_pub(s, l, 0);
                const CSlice& sl = s_geo[0];
                const unsigned char* rec = rec_base();
                bf_norm<QK, NB>(xs, PD, d, ln, reinterpret_cast<const float*>(rec + sl.o_g1),
                                reinterpret_cast<const float*>(rec + sl.o_g2), a.eps, s_red, bf);
                stamp(2);
                const float* bias =
                    sl.has_bias ? reinterpret_cast<const float*>(rec + sl.o_bias) + (sl.br0 - sl.b_lo) : nullptr;
                mma_rows<QK, NB, false>(rec_codes(rec), rec + sl.o_sc, d, sl.nt, sl.nr, bf, red,
                                        [&](int i, int b, float v, float) {
                                            if (bias) v += bias[i];
                                            const uint32_t addr = a_qkv + 4u * (uint32_t)(b * a.rpc + qr0 + i);
                                            for (int dst = 0; dst < cs; ++dst)
                                                st_async(mapa(addr, dst), v, mapa(mb_qkv, dst));
                                        });
                rec_done();
                tr_pub(s, l, 1);
                stamp(3);
            }
            // ---- attention over this rank's key blocks
            {
                xwait(mb_qkv, ph_qkv, xb_bytes_of(XB_QKV));
                stamp(4);
                const int half = hd >> 1;
                const int items = NB * a.kpc;
                __half* Ks = stg;
                __half* Vs = stg + (size_t)items * a.kkc * hd;
                const float scale = 1.0f / sqrtf((float)hd);
                float m = -INFINITY, lsum = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
                const int b = b_, gl = gl_, qh = qh_;
                if (pr < nph) {
                    // this warp's query: RoPE at pos (NEOX half split), scaled by 1/sqrt(hd)
                    float* q = wq + warp * hd;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const int i = lane + 32 * t;
                        if (i >= half) continue;
                        const float x0 = qkv[b * a.rpc + qh * hd + i], x1 = qkv[b * a.rpc + qh * hd + i + half];
                        q[i] = (x0 * rcs[t] - x1 * rsn[t]) * scale;
                        q[i + half] = (x0 * rsn[t] + x1 * rcs[t]) * scale;
                    }
                }
                // the position being decoded: its rotated key and its value, fp16, into the cache
                // (one warp per item) and into the staging slot of every warp that reads it
                auto put_new = [&](int jloc, bool to_cache) {
                    const int it = b * a.kpc + gl, gg = cl * a.kpc + gl;
                    const float* kk = qkv + b * a.rpc + qd + gl * hd;
                    const float* vv = qkv + b * a.rpc + qd + kd + gl * hd;
                    const size_t hb = ((size_t)(b * L + l) * a.Hkv + gg) * a.n_ctx * hd + (size_t)pos * hd;
                    __half* ks = Ks + ((size_t)it * a.kkc + jloc) * hd;
                    __half* vs = Vs + ((size_t)it * a.kkc + jloc) * hd;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const int i = lane + 32 * t;
                        if (i >= half) continue;
                        const __half k0 = __float2half_rn(kk[i] * rcs[t] - kk[i + half] * rsn[t]);
                        const __half k1 = __float2half_rn(kk[i] * rsn[t] + kk[i + half] * rcs[t]);
                        const __half v0 = __float2half_rn(vv[i]), v1 = __float2half_rn(vv[i + half]);
                        ks[i] = k0; ks[i + half] = k1; vs[i] = v0; vs[i + half] = v1;
                        if (to_cache) {
                            a.kc[hb + i] = k0; a.kc[hb + i + half] = k1;
                            a.vc[hb + i] = v0; a.vc[hb + i + half] = v1;
                        }
                    }
                };
                __syncwarp();
                stamp(22);
                for (int q0 = 0;; q0 += SB) {
                    const int q1 = min(nbr, q0 + SB);
                    if (q0 != 0) {
                        // a later staging fill: every warp is done with the staging first
                        csync();
                        if (tid == 0) kv_fetch(l, pos, q0, q1);
                    }
                    xb_wait(mb_kv, ph_kv & 1u, a.err, budget);
                    ++ph_kv;
                    stamp(23);
                    if (pr < nph) {
                        const float* q = wq + warp * hd;
                        for (int qq = wi; q0 + qq < q1; qq += WG) {
                            const int j = rank + (q0 + qq) * cs, nk = min(32, n - 32 * j);
                            const size_t so = ((size_t)(b * a.kpc + gl) * a.kkc + qq * 32) * hd;
                            if (j == jl) {
                                // this block holds the position being decoded (row nk - 1)
                                put_new(qq * 32 + nk - 1, qh % hpg == 0);
                                asm volatile("fence.proxy.async.global;" ::: "memory");
                                __syncwarp();
                            }
                            if (hd == 64)
                                attn_lk<64>(q, Ks + so, Vs + so, 0, nk, m, lsum, *reinterpret_cast<float(*)[2]>(o));
                            else
                                attn_lk<128>(q, Ks + so, Vs + so, 0, nk, m, lsum, o);
                        }
                    }
                    if (q1 >= nbr) break;
                }
                stamp(5);
                // warp partials -> the warps of a pair combined in warp order -> every rank
                {
                    const int DPL = hd / 32;
#pragma unroll
                    for (int dd = 0; dd < 4; ++dd)
                        if (dd < DPL) wp[warp * W2 + lane * DPL + dd] = o[dd];
                    if (lane == 0) {
                        wp[warp * W2 + hd] = m;
                        wp[warp * W2 + hd + 1] = lsum;
                    }
                }
                csync();
                stamp(24);
                // only the first min(WG, blocks per fill) warps of a pair hold keys.  One warp per pair
                // folds their maxima (lane w: warp w of the pair) into M and the weights exp(m_w - M),
                // kept in wq (idle once every warp has attended); then each component is one
                // weighted sum over the warps, and the pair's M
                const int wa = min(WG, min(nbr, SB));
                float* ew = wq;  // [nph][17]: the weights, then M
                if (warp < nph) {
                    const float* P = wp + (size_t)warp * WG * W2;
                    const float mw = lane < wa ? P[lane * W2 + hd] : -INFINITY;
                    float M = mw;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
                    if (lane < wa) ew[warp * 17 + lane] = mw != -INFINITY ? expf(mw - M) : 0.f;
                    if (lane == 0) ew[warp * 17 + 16] = M;
                }
                csync();
                for (int u = tid; u < nph * (hd + 2); u += kThreads) {
                    const int p = u == tid ? cp_p : u / (hd + 2), k = u == tid ? cp_k : u - p * (hd + 2);
                    const float* P = wp + (size_t)p * WG * W2;
                    float v = ew[p * 17 + 16];
                    if (k != hd) {
                        v = 0.f;
                        for (int w = 0; w < wa; ++w) v = fmaf(ew[p * 17 + w], P[w * W2 + k], v);
                    }
                    const uint32_t addr = a_part + 4u * (uint32_t)((rank * NB * a.hpc + p) * W2 + k);
                    for (int dst = 0; dst < cs; ++dst) st_async(mapa(addr, dst), v, mapa(mb_part, dst));
                }
                stamp(25);
                // the staging is free: the next layer's keys (off the critical path, after the sends)
                if (tid == 0 && l + 1 < L) kv_fetch(l + 1, pos, 0, min(nbr, SB));
                tr_pub(s, l, 2);
                stamp(6);
            }
            // ---- combine the ranks' partials; O slab for this rank's rows -> global partial words
            {
                xwait(mb_part, ph_part, xb_bytes_of(XB_PART));
                stamp(7);
                // per (batch row, head): one warp (lane r: rank r) folds the ranks' maxima and
                // denominators into the weights exp(m_r - M) / sum_r exp(m_r - M) l_r, kept in red
                // (idle until the O matvec); then each output element is one weighted sum over ranks
                const int nbh = NB * a.hpc;
                float* cw = red;  // [nbh][16]
                if (warp < nbh) {
                    const float* P = part + (size_t)(lane * nbh + warp) * W2;
                    const float mr = lane < cs ? P[hd] : -INFINITY;
                    float M = mr;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
                    const float w = (lane < cs && mr != -INFINITY) ? expf(mr - M) : 0.f;
                    float den = lane < cs ? w * P[hd + 1] : 0.f;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
                    if (lane < cs) cw[warp * 16 + lane] = w / den;
                }
                csync();
                for (int t = tid; t < nbh * hd; t += kThreads) {
                    const int bh = t >> lhd, dd = t & (hd - 1);
                    float v = 0.f;
                    for (int r = 0; r < cs; ++r) v = fmaf(cw[bh * 16 + r], part[(r * nbh + bh) * W2 + dd], v);
                    const int bb = NB == 1 ? 0 : bh / a.hpc, qh = bh - bb * a.hpc;
                    bf_put<QK, NB>(bf, qh * hd + dd, bb, v);
                }
                csync();
                stamp(8);
                rec_wait();
                stamp(9);
                const CSlice& sl = s_geo[1];
                const unsigned char* rec = rec_base();
                unsigned long long* P = a.ll_po + (size_t)cl * NB * d;
                mma_rows<QK, NB, false>(rec_codes(rec), rec + sl.o_sc, a.ko, sl.nt, sl.nr, bf, red,
                                        [&](int i, int bb, float v, float) {
                                            ll_store(P + (size_t)bb * d + xr0 + i, v, e);
                                        });
                tr_pub(s, l, 3);
                stamp(10);
                // ---- exchange 1: rows [xr0, xr0 + nx) of every cluster's partial, summed in cluster order
                const float* bias =
                    sl.has_bias ? reinterpret_cast<const float*>(rec + sl.o_bias) + (sl.br0 - sl.b_lo) : nullptr;
                const bool stall = a.test_budget > 0 && s == 0 && l == 0 && gi == 0;  // test hook
                reduce_bcast<NB>(a.ll_po, a.ncl, d, xr0, nx, stall ? e + 0x40000000u : e, bias, xs, PD, a_x, mb_x0,
                                 cs, a.err, stall ? a.test_budget : budget);
                rec_done();
                tr_pub(s, l, 4);
                stamp(11);
            }
            // ---- norm and this rank's FC / gate-up rows -> cluster FFN activations
            {
                xwait(mb_x0, ph_x0, xb_bytes_of(XB_X0));
                stamp(12);
                rec_wait();
                stamp(13);
                const CSlice& sl = s_geo[2];
                const unsigned char* rec = rec_base();
                bf_norm<QK, NB>(xs, PD, d, ln, reinterpret_cast<const float*>(rec + sl.o_g1),
                                reinterpret_cast<const float*>(rec + sl.o_g2), a.eps, s_red, bf);
                stamp(14);
                const float* bias =
                    sl.has_bias ? reinterpret_cast<const float*>(rec + sl.o_bias) + (sl.br0 - sl.b_lo) : nullptr;
                auto send_u = [&](int i, int bb, float v) {
                    const uint32_t addr = a_u + 4u * (uint32_t)(bb * PU + pidx(fr0 + i));
                    for (int dst = 0; dst < cs; ++dst) st_async(mapa(addr, dst), v, mapa(mb_u, dst));
                };
                if (ln)
                    mma_rows<QK, NB, false>(rec_codes(rec), rec + sl.o_sc, d, sl.nt, sl.nr, bf, red,
                                            [&](int i, int bb, float v, float) {
                                                if (bias) v += bias[i];
                                                send_u(i, bb, gelu_tanh(v));
                                            });
                else
                    mma_rows<QK, NB, true>(rec_codes(rec), rec + sl.o_sc, d, sl.nt, sl.nr, bf, red,
                                           [&](int k, int bb, float gt, float up) { send_u(k, bb, silu(gt) * up); });
                rec_done();
                tr_pub(s, l, 5);
                stamp(15);
            }
            // ---- down-projection slab for this rank's rows -> exchange 2
            {
                xwait(mb_u, ph_u, xb_bytes_of(XB_U));
                stamp(16);
                rec_wait();
                stamp(17);
                bf_plain<QK, NB>(ub, PU, a.upc, bf);
                const CSlice& sl = s_geo[3];
                const unsigned char* rec = rec_base();
                unsigned long long* P = a.ll_pp + (size_t)cl * NB * d;
                mma_rows<QK, NB, false>(rec_codes(rec), rec + sl.o_sc, a.upc, sl.nt, sl.nr, bf, red,
                                        [&](int i, int bb, float v, float) {
                                            ll_store(P + (size_t)bb * d + xr0 + i, v, e);
                                        });
                tr_pub(s, l, 6);
                stamp(18);
                const float* bias =
                    sl.has_bias ? reinterpret_cast<const float*>(rec + sl.o_bias) + (sl.br0 - sl.b_lo) : nullptr;
                reduce_bcast<NB>(a.ll_pp, a.ncl, d, xr0, nx, e, bias, xs, PD, a_x, mb_x1, cs, a.err, budget);
                rec_done();
                tr_pub(s, l, 7);
                stamp(19);
            }
        }
        // ---- head rows (final norm)
        const unsigned eh = eb + (unsigned)L;
        {
            xwait(mb_x1, ph_x1, xb_bytes_of(XB_X1));
            rec_wait();
            const CSlice& sl = s_geo[4];
            const unsigned char* rec = rec_base();
            bf_norm<QK, NB>(xs, PD, d, ln, reinterpret_cast<const float*>(rec + sl.o_g1),
                            reinterpret_cast<const float*>(rec + sl.o_g2), a.eps, s_red, bf);
            const int hr0 = sl.br0;
            mma_rows<QK, NB, false>(rec_codes(rec), rec + sl.o_sc, d, sl.nt, sl.nr, bf, red,
                                    [&](int i, int bb, float v, float) {
                                        a.logits[(size_t)bb * a.V + hr0 + i] = v;
                                        ll_store(a.ll_logits + (size_t)bb * a.V + hr0 + i, v, eh);
                                    });
            rec_done();
            stamp(20);
        }
        // ---- sampler: CTA b samples row b (its shared memory overlays the activation region: every
        // buffer there is idle until the next step, and no rank sends into it before this token)
        if (gi < NB) {
            float* z = reinterpret_cast<float*>(actb);
            csync();  // the head's partial sums are read
            const int b = gi;
            // every word of the row is loaded (16 per thread at a time), then the ones not yet carrying
            // epoch eh are polled again together
            for (int i0 = tid; i0 < a.V; i0 += 16 * kThreads) {
                unsigned long long w[16];
                unsigned pend = 0u;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int i = i0 + j * kThreads;
                    w[j] = i < a.V ? ll_load(a.ll_logits + (size_t)b * a.V + i) : 0ull;
                    if (i < a.V && (unsigned)(w[j] >> 32) != eh) pend |= 1u << j;
                }
                const long long t0 = clock64();
                for (unsigned it = 0; pend; ++it) {
                    if (it > 2u) __nanosleep(32);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (pend & (1u << j)) {
                            w[j] = ll_load(a.ll_logits + (size_t)b * a.V + i0 + j * kThreads);
                            if ((unsigned)(w[j] >> 32) == eh) pend &= ~(1u << j);
                        }
                    if ((it & 31u) == 31u && (ld_volatile(a.err) || clock64() - t0 > budget)) {
                        atomicCAS(a.err, 0, kErrTimeout);
                        break;
                    }
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int i = i0 + j * kThreads;
                    if (i < a.V) z[i] = __uint_as_float((unsigned)w[j]);
                }
            }
            csync();
            stamp(28);
            const float* up = a.u_seq ? a.u_seq + (size_t)s * NB + b : a.u1 + b;
            const int tk = sample_detail::sample_reg(a.V, *a.sp, up, reinterpret_cast<unsigned char*>(z), s_samp,
                                                      a.err);
            if (tid == 0) {
                a.tok[b] = tk;
                if (a.out_seq) a.out_seq[(size_t)s * NB + b] = tk;
#pragma unroll
                for (int r = 0; r < kTokRep; ++r) ll_store(a.ll_tok + r * 32 + b, __int_as_float(tk), eh);
            }
            stamp(29);
        }
        // the step ends uniformly: on a recorded error every thread leaves here
        ok = csync_and(ld_volatile(a.err) == 0) != 0;
        stamp(21);
        if (!ok) break;
    }
    if (gi == 0 && tid == 0) {
        if (ok) *a.pos = pos0 + a.n_steps;
        *a.gen = gen0 + (unsigned)a.n_steps;
    }
    // copies still in flight into this CTA's shared memory land before the CTA exits
    if (tid == 0) {
        for (int i = p_nc; i < p_ni; ++i)
            mb_wait(smem_u32(&s_mb[i & (kNMB - 1)]), (uint32_t)((i / kNMB) & 1), a.err, budget, true);
        if (kv_issued > (int)ph_kv) mb_wait(mb_kv, ph_kv & 1u, a.err, budget, true);
    }
    csync();
    if (a.trace && gi == a.trace_gi && tid < kCTraceSub) a.trace[tid] += s_trc[tid];
    // no CTA of the cluster leaves while another may still send into its shared memory
    cluster_sync_all();
    if (!ok) __nanosleep(20000);
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

// ------------------------------------------------------------------ fragment-major repack (set-up)

// out = the fragment-major copy (see Frag) of column slab s of rows perm[i]
// (or i) of a row-major Q8_0 / Q4_0 matrix, for s < K / Wd; rows past R are
// zero.  Slabs follow each other; the scales of all slabs come after all codes.
__global__ void k_frag_pack(const uint8_t* q, const __half* sc, int R, int K, int Wd, int q4, const int* perm,
                            uint8_t* out) {
    const int rb = q4 ? K / 2 : K;           // code bytes per source row
    const int blk = q4 ? 16 : 32;            // code bytes per block
    const int W = q4 ? 1 : 2, TB = 256 * W;  // words per lane per row, bytes per (tile, block)
    const int NT = (R + 15) / 16, KB = Wd / 32, NS = K / Wd;
    const long long lanes = (long long)NS * NT * KB * 32;
    const size_t sc_base = (size_t)NS * NT * KB * TB;
    for (long long x = blockIdx.x * (long long)blockDim.x + threadIdx.x; x < lanes;
         x += (long long)gridDim.x * blockDim.x) {
        const int lane = (int)(x & 31);
        const long long tbk = x >> 5;                       // (slab, tile, block)
        const int kb = (int)(tbk % KB), tile = (int)((tbk / KB) % NT), sl = (int)(tbk / ((long long)KB * NT));
        const int g = lane >> 2, t = lane & 3;
        uint32_t* o = reinterpret_cast<uint32_t*>(out + (size_t)tbk * TB) + lane * 2 * W;
        for (int h = 0; h < 2; ++h) {
            const int row = tile * 16 + g + 8 * h;
            for (int w = 0; w < W; ++w) {
                uint32_t v = 0u;
                if (row < R) {
                    const int src = perm ? perm[row] : row;
                    const size_t off = (size_t)src * rb + (size_t)sl * (Wd / 32) * blk + (size_t)kb * blk +
                                       (size_t)(4 * W) * t + 4 * w;
                    v = *reinterpret_cast<const uint32_t*>(q + off);
                }
                o[h * W + w] = v;
            }
        }
        if (lane < 16) {
            const int row = tile * 16 + lane;
            __half hv = __float2half(0.f);
            if (row < R) {
                const int src = perm ? perm[row] : row;
                hv = sc[(size_t)src * (K / 32) + (size_t)sl * KB + kb];
            }
            reinterpret_cast<__half*>(out + sc_base)[(size_t)tbk * 16 + lane] = hv;
        }
    }
}

}  // namespace cstep_detail

size_t cstep_smem_bytes(const CStepArgs& a) {
    return (size_t)a.ring_bytes + (size_t)a.act_bytes + sizeof(StepLayer) * (size_t)a.n_layer;
}

// Activation-region layout for the plan in `a`; returns its bytes.  maxnt: the
// most tiles of one record (the matvec partial sums hold max(16, maxnt) units).
static size_t cstep_layout(CStepArgs& a, int maxnt) {
    using gemv_detail::padded;
    const int B = a.B;
    auto al = [](size_t v) { return (v + 127) & ~(size_t)127; };
    size_t off = 0;
    int kin = a.d > a.ko ? a.d : a.ko;
    if (a.upc > kin) kin = a.upc;
    a.o_x = (int)off; off = al(off + 4 * (size_t)B * padded(a.d));
    a.o_u = (int)off; off = al(off + 4 * (size_t)B * padded(a.upc));
    a.o_qkv = (int)off; off = al(off + 4 * (size_t)B * a.rpc);
    a.o_part = (int)off; off = al(off + 4 * (size_t)a.cs * B * a.hpc * (a.hd + 4));
    a.o_wq = (int)off; off = al(off + 4 * (size_t)stepdev::kWarps * a.hd);
    a.o_wp = (int)off; off = al(off + 4 * (size_t)stepdev::kWarps * (a.hd + 4));
    a.o_bf = (int)off; off = al(off + 2 * 2 * 2 * (size_t)B * kin);  // hi and lo halves per element and row
    a.o_red = (int)off; off = al(off + 4 * (size_t)(maxnt > 16 ? maxnt : 16) * 16 * B);
    a.o_stage = (int)off;
    off = al(off + 2 * sizeof(__half) * (size_t)B * a.kpc * a.kkc * a.hd);
    // the sampler overlays the whole region: while a CTA samples, every buffer above is idle and no
    // rank sends into it (the next step's exchanges need the token this sample produces)
    const size_t smp = sample_smem_bytes_dev(a.V, stepdev::kThreads);
    return off > smp ? off : al(smp);
}

int cstep_plan(CStepArgs& a, int sm_count) {
    using namespace cstep_detail;
    void* kern = pick(a);
    if (!kern || a.B < 1 || a.B > 2 || a.n_layer < 1 || a.Hkv < 1 || a.H % a.Hkv) return 0;
    if ((a.hd != 64 && a.hd != 128) || a.d % 32 || a.ff % 32 || a.V > sample_detail::kMaxV) return 0;
    if (a.d > 2 * stepdev::kThreads) return 0;  // the norm holds at most two elements of a row per thread
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
    std::vector<std::pair<int, int>> cand;
    // SD_CLUSTERS / SD_CLUSTER_SIZE restrict the candidates (measurement of other shapes)
    const int want_ncl = getenv("SD_CLUSTERS") ? atoi(getenv("SD_CLUSTERS")) : 0;
    const int want_cs = getenv("SD_CLUSTER_SIZE") ? atoi(getenv("SD_CLUSTER_SIZE")) : 0;
    for (int ncl = a.Hkv; ncl >= 1; --ncl)
        if (a.Hkv % ncl == 0 && (!want_ncl || ncl == want_ncl))
            for (int cs = 16; cs >= 2; --cs)
                if (ncl * cs <= sm_count && (!want_cs || cs == want_cs)) cand.push_back({ncl, cs});
    std::stable_sort(cand.begin(), cand.end(), [](const std::pair<int, int>& x, const std::pair<int, int>& y) {
        const int gx = x.first * x.second, gy = y.first * y.second;
        return gx != gy ? gx > gy : x.first > y.first;
    });
    const int tb = frag_tb(a.quant);
    for (const auto& nc : cand) {
        if (best) break;
        const int ncl = nc.first, cs = nc.second, G = ncl * cs;
        CStepArgs t = a;
        t.ncl = ncl; t.cs = cs;
        t.kpc = a.Hkv / ncl; t.hpc = a.H / ncl;
        t.rpc = (t.hpc + 2 * t.kpc) * a.hd;
        t.ko = t.hpc * a.hd;
        t.upc = a.ff / ncl;
        if (a.ff % ncl || t.upc % 32) continue;
        // every rank needs at least one tile of every matrix; the norm and B fragments cover a row
        const int nq = t.rpc / 16, nd = a.d / 16, nf = (a.gpt2 ? t.upc : 2 * t.upc) / 16, nh = (a.V + 15) / 16;
        if (nq < cs || nd < cs || nf < cs || nh < G || t.ko > 2 * stepdev::kThreads || t.upc > 2 * stepdev::kThreads)
            continue;
        if (a.B * t.hpc > stepdev::kWarps) continue;
        auto cdiv = [](int x, int y) { return (x + y - 1) / y; };
        const int tq = cdiv(nq, cs), td = cdiv(nd, cs), tf = cdiv(nf, cs), th = cdiv(nh, G);
        const int maxnt = std::max({tq, td, tf, th});
        // keys per rank staged at once: the whole share of a full context where it fits
        t.kkc = std::min(256, std::max(32, ((cdiv(a.n_ctx, cs) + 31) / 32) * 32));
        int act = (int)cstep_layout(t, maxnt);
        while (t.kkc > 32 && act > limit / 2) {
            t.kkc -= 32;
            act = (int)cstep_layout(t, maxnt);
        }
        t.act_bytes = act;
        const int ring = (limit - act - (int)(sizeof(StepLayer) * a.n_layer)) & ~127;
        // record bytes: tiles x blocks x (codes + scales) + bias and gain windows
        auto rec = [&](int tiles, int K, bool gains) {
            return tiles * (K / 32) * (tb + 32) + (16 * tiles + 8) * 4 + (gains ? 2 * 4 * gemv_detail::padded(a.d) : 0) +
                   128;
        };
        // records in step order: QKV, O, FC, proj per layer, then the head; the ring holds any
        // two consecutive ones of a layer, so the next record streams in while one is in use
        // (the head record, once per step, may have to wait for the ring to drain)
        const int rq = rec(tq, a.d, true), ro = rec(td, t.ko, false), rf = rec(tf, a.d, true);
        const int rp = rec(td, t.upc, false), rh = rec(th, a.d, true);
        const int need = std::max({rq + ro, ro + rf, rf + rp, rp + rq, rh});
        if (dbg)
            fprintf(stderr, "cstep plan: ncl %d cs %d act %d ring %d records %d %d %d %d %d kkc %d\n", ncl, cs, act,
                    ring, rq, ro, rf, rp, rh, t.kkc);
        if (ring < need) continue;
        t.ring_bytes = ring;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cstep_smem_bytes(t)) !=
            cudaSuccess)
            continue;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(G);
        cfg.blockDim = dim3(cstep_detail::kCBlock);
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
        best = G;
        pick_a = t;
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
    cfg.blockDim = dim3(cstep_detail::kCBlock);
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

size_t frag_bytes(int quant, int rows, int cols, int slab_cols) {
    const int nt = (rows + 15) / 16, ns = cols / slab_cols, kb = slab_cols / 32;
    return (size_t)ns * nt * kb * (cstep_detail::frag_tb(quant) + 32);
}

cudaError_t launch_frag_pack(const QMat& src, int slab_cols, const int* perm, uint8_t* out, cudaStream_t st) {
    if ((src.kind != SD_Q4_0 && src.kind != SD_Q8_0) || slab_cols < 32 || slab_cols % 32 || src.cols % slab_cols)
        return cudaErrorInvalidValue;
    cstep_detail::k_frag_pack<<<1024, 256, 0, st>>>(src.q, reinterpret_cast<const __half*>(src.s), src.rows, src.cols,
                                                    slab_cols, src.kind == SD_Q4_0, perm, out);
    return cudaGetLastError();
}

}  // namespace sd
