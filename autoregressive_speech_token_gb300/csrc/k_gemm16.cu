// Skinny tensor-core GEMM for up to 16 activation rows (the G rollouts of the
// Talker + code predictor, or a few batch rows): Y[M][N] = X[M][K] W[N][K]^T,
// M <= 16, with the GEMV epilogues.  "Every Frame Is a Memory Read", section
// 8: G rollouts share one read of the weights per step, so the kernel streams
// every quantised weight exactly once, straight from global memory into the
// MMA's B fragments, and splits K over CTAs so the whole GPU streams even when
// N is small.
//
// Arithmetic (as the 64x64 GEMM): w = d*q per quantisation block ("Chatterbox
// -> ggml Port: Development Journal", section 3.23; affine groups w = s*q + b,
// "Every Frame Is a Memory Read", section 3).  The codes are small integers,
// exact in fp16; the fp32 activations are split x = hi + lo in fp16; each
// 16-wide K step is two mma.sync m16n8k16 (hi, lo) with fp32 accumulation, and
// the block's partial sums are scaled by d (plus b * sum(x) for affine groups)
// in fp32.
//
// Element order: inside a quantisation block the MMA's k index is permuted --
// the same permutation for A and B, so each step's dot product is unchanged --
// so that a lane's B elements are consecutive code bytes: lane t (of the quad)
// loads 16 (affine), 8 (Q8_0) or 4 (Q4_0) consecutive bytes of a block with one
// load, and step s of the block takes its elements
//   affine: 16t + 4s + j,   Q8_0: 8t + 4s + j,   Q4_0: 4t + 16s + j  (j = 0..3),
// which sit at MMA k = 2t, 2t+1 (j = 0, 1) and 2t+8, 2t+9 (j = 2, 3).  The
// codes become fp16 by the exponent trick: byte v placed under the exponent of
// 1024 is the half 1024 + v, and one half2 subtraction removes the offset
// (1024, 1024 + 128 for signed bytes, 1024 + 8 for Q4_0 nibbles).
//
// CTA: 8 warps x two n8 tiles = 128 output rows; K range k_per (a multiple of
// 64 or 32, at most 1024).  The CTA stages its 16 x k_per activations (fp16
// hi/lo, rows padded so the fragment loads are bank-conflict free) and the
// block scales of its 128 rows in shared memory, while its first two batches
// of code words are already in flight; then each warp streams its rows in
// double-buffered register batches of 64 bytes per lane.  Partial sums go to a
// workspace [split][16][N]; the last CTA of each column tile (a counter per
// tile, left zero again) adds the splits in split order and applies
// bias / GELU / SwiGLU / residual, so the result does not depend on timing.
#include "sd_internal.cuh"

namespace sd {
namespace g16_detail {

constexpr int kWarps = 8, kThreads = 32 * kWarps, kTileN = 16 * kWarps, kMaxKPer = 1024, kSP = kTileN + 2;

template <int QK> struct Fmt;
template <> struct Fmt<SD_A8G64> { static constexpr int BK = 64, W = 4, NBB = 2, PAD = 4; };
template <> struct Fmt<SD_Q8_0> { static constexpr int BK = 32, W = 2, NBB = 4, PAD = 32; };
template <> struct Fmt<SD_Q4_0> { static constexpr int BK = 32, W = 1, NBB = 8, PAD = 16; };

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Streaming loads of code words: read once per step, not kept in L1.
template <int W>
__device__ __forceinline__ void ld_codes(const uint8_t* p, uint32_t (&w)[W]) {
    if constexpr (W == 4) {
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "l"(p));
    } else if constexpr (W == 2) {
        asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "l"(p));
    } else {
        asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(w[0]) : "l"(p));
    }
}

__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
    const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
}

// Four code values of word w (bytes 0..3 in element order) -> B fragment (b0: elements 0,1; b1: 2,3).
template <int QK>
__device__ __forceinline__ void code_frag(uint32_t w, int s, uint32_t& b0, uint32_t& b1) {
    uint32_t off;
    if constexpr (QK == SD_Q4_0) {
        w = (s ? (w >> 4) : w) & 0x0F0F0F0Fu;
        off = 0x64086408u;  // 1024 + 8
    } else if constexpr (QK == SD_Q8_0) {
        w ^= 0x80808080u;   // signed byte v -> unsigned v + 128
        off = 0x64806480u;  // 1024 + 128
    } else {
        off = 0x64006400u;  // 1024
    }
    b0 = hsub2_u(__byte_perm(w, 0x64646464u, 0x4140), off);
    b1 = hsub2_u(__byte_perm(w, 0x64646464u, 0x4342), off);
}

__device__ __forceinline__ float gelu_tanh(float v) {
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    return 0.5f * v * (1.0f + tanhf(c * (v + 0.044715f * v * v * v)));
}
__device__ __forceinline__ float silu(float v) { return v / (1.0f + expf(-v)); }

template <int QK>
__host__ __device__ constexpr int xs_stride(int k_per) { return k_per + Fmt<QK>::PAD; }

template <int QK>
__host__ __device__ inline size_t smem_bytes(int k_per) {
    const int nbk = k_per / Fmt<QK>::BK;
    size_t b = (size_t)2 * 16 * xs_stride<QK>(k_per) * sizeof(__half);
    b += (size_t)nbk * kSP * sizeof(float) * (QK == SD_A8G64 ? 2 : 1);
    if (QK == SD_A8G64) b += (size_t)nbk * 16 * sizeof(float);
    return b;
}

template <int QK>
__global__ void __launch_bounds__(kThreads, 2) k_gemm16(const Gemm16Args a) {
    using F = Fmt<QK>;
    constexpr int BK = F::BK, W = F::W, NBB = F::NBB, STEPS = BK / 16;
    constexpr int BLK_BYTES = (QK == SD_Q4_0) ? 16 : BK;   // code bytes of one block
    extern __shared__ __align__(16) unsigned char g16_smem[];
    __shared__ int s_last;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int N = a.W.rows, K = a.W.cols, M = a.M;
    const int n0 = blockIdx.x * kTileN;
    const int k_beg = blockIdx.y * a.k_per;
    const int kcn = min(a.k_per, K - k_beg);
    const int nbk = kcn / BK;                       // blocks of this CTA
    const int S = xs_stride<QK>(a.k_per);
    __half* xh = reinterpret_cast<__half*>(g16_smem);
    __half* xl = xh + 16 * S;
    float* ssc = reinterpret_cast<float*>(xl + 16 * S);             // [nbk][kSP] block scales
    float* sbi = ssc + (QK == SD_A8G64 ? (a.k_per / BK) * kSP : 0);  // [nbk][kSP] affine biases
    float* xsum = sbi + (QK == SD_A8G64 ? (a.k_per / BK) * kSP : 0); // [nbk][16] affine group sums

    const size_t row_bytes = (QK == SD_Q4_0) ? (size_t)(K >> 1) : (size_t)K;
    const int spb = K / BK, kb0 = k_beg / BK;
    // this lane's two weight rows (B column g of tiles 0, 1), clamped into the matrix
    const uint8_t* wr[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int n = min(n0 + warp * 16 + j * 8 + g, N - 1);
        wr[j] = a.W.q + (size_t)n * row_bytes + (size_t)kb0 * BLK_BYTES + (size_t)t * (4 * W);
    }
    auto load_batch = [&](uint32_t (&buf)[2][NBB][W], int kb) {
#pragma unroll
        for (int q = 0; q < NBB; ++q)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                if (kb + q < nbk) {
                    ld_codes<W>(wr[j] + (size_t)(kb + q) * BLK_BYTES, buf[j][q]);
                } else {
#pragma unroll
                    for (int w = 0; w < W; ++w) buf[j][q][w] = 0u;
                }
            }
    };
    uint32_t bufA[2][NBB][W], bufB[2][NBB][W];
    load_batch(bufA, 0);
    load_batch(bufB, NBB);

    // ---- stage the activations (fp16 hi/lo; rows >= M are zero) and, for affine groups, their sums
    {
        const int q4 = kcn >> 2;  // float4 per row
        for (int i = tid; i < 16 * q4; i += kThreads) {
            const int m = i / q4, k4 = i - m * q4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (m < M) v = __ldg(reinterpret_cast<const float4*>(a.x + (size_t)m * a.ldx + k_beg) + k4);
            const __half h0 = __float2half_rn(v.x), h1 = __float2half_rn(v.y);
            const __half h2 = __float2half_rn(v.z), h3 = __float2half_rn(v.w);
            __half2* ph = reinterpret_cast<__half2*>(xh + m * S + 4 * k4);
            __half2* pl = reinterpret_cast<__half2*>(xl + m * S + 4 * k4);
            ph[0] = __halves2half2(h0, h1);
            ph[1] = __halves2half2(h2, h3);
            pl[0] = __floats2half2_rn(v.x - __half2float(h0), v.y - __half2float(h1));
            pl[1] = __floats2half2_rn(v.z - __half2float(h2), v.w - __half2float(h3));
            if constexpr (QK == SD_A8G64) {
                // 16 consecutive float4 of one row form one 64-wide group; the loop keeps whole warps
                // active (16 * q4 is a multiple of 256) and groups aligned to half-warps
                float s = (v.x + v.y) + (v.z + v.w);
#pragma unroll
                for (int o = 8; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if ((k4 & 15) == 0) xsum[(k4 >> 4) * 16 + m] = s;
            }
        }
        // block scales (and affine biases) of the CTA's 128 rows, transposed to [block][row]
        for (int i = tid; i < kTileN * nbk; i += kThreads) {
            const int r = i / nbk, b = i - r * nbk, n = n0 + r;
            float sv = 0.f, bv = 0.f;
            if (n < N) {
                if constexpr (QK == SD_A8G64) {
                    const __half2 sb = __ldg(reinterpret_cast<const __half2*>(a.W.s) + (size_t)n * spb + kb0 + b);
                    sv = __low2float(sb);
                    bv = __high2float(sb);
                } else {
                    sv = __half2float(__ldg(reinterpret_cast<const __half*>(a.W.s) + (size_t)n * spb + kb0 + b));
                }
            }
            ssc[b * kSP + r] = sv;
            if constexpr (QK == SD_A8G64) sbi[b * kSP + r] = bv;
        }
    }
    __syncthreads();

    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const int cl = warp * 16 + 2 * t;  // C column (within the CTA tile) of c0/c2 in tile 0; +8 in tile 1

    auto compute_batch = [&](const uint32_t (&buf)[2][NBB][W], int kb) {
#pragma unroll
        for (int q = 0; q < NBB; ++q) {
            const int b = kb + q;
            if (b >= nbk) break;
            // A fragments of the block's steps: (row g, row g+8) x (k 2t.., k 2t+8..), hi and lo
            uint32_t ah[STEPS][4], al[STEPS][4];
            if constexpr (QK == SD_Q8_0) {
                const int h = b * BK + 8 * t;
                const uint4 h0 = *reinterpret_cast<const uint4*>(xh + g * S + h);
                const uint4 h1 = *reinterpret_cast<const uint4*>(xh + (g + 8) * S + h);
                const uint4 l0 = *reinterpret_cast<const uint4*>(xl + g * S + h);
                const uint4 l1 = *reinterpret_cast<const uint4*>(xl + (g + 8) * S + h);
                ah[0][0] = h0.x; ah[0][1] = h1.x; ah[0][2] = h0.y; ah[0][3] = h1.y;
                ah[1][0] = h0.z; ah[1][1] = h1.z; ah[1][2] = h0.w; ah[1][3] = h1.w;
                al[0][0] = l0.x; al[0][1] = l1.x; al[0][2] = l0.y; al[0][3] = l1.y;
                al[1][0] = l0.z; al[1][1] = l1.z; al[1][2] = l0.w; al[1][3] = l1.w;
            } else {
#pragma unroll
                for (int s = 0; s < STEPS; ++s) {
                    const int h = b * BK + (QK == SD_Q4_0 ? 4 * t + 16 * s : 16 * t + 4 * s);
                    const uint2 h0 = *reinterpret_cast<const uint2*>(xh + g * S + h);
                    const uint2 h1 = *reinterpret_cast<const uint2*>(xh + (g + 8) * S + h);
                    const uint2 l0 = *reinterpret_cast<const uint2*>(xl + g * S + h);
                    const uint2 l1 = *reinterpret_cast<const uint2*>(xl + (g + 8) * S + h);
                    ah[s][0] = h0.x; ah[s][1] = h1.x; ah[s][2] = h0.y; ah[s][3] = h1.y;
                    al[s][0] = l0.x; al[s][1] = l1.x; al[s][2] = l0.y; al[s][3] = l1.y;
                }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int s = 0; s < STEPS; ++s) {
                    uint32_t b0, b1;
                    code_frag<QK>(buf[j][q][QK == SD_Q4_0 ? 0 : s], s, b0, b1);
                    mma16816(c, ah[s][0], ah[s][1], ah[s][2], ah[s][3], b0, b1);
                    mma16816(c, al[s][0], al[s][1], al[s][2], al[s][3], b0, b1);
                }
                const float2 d = *reinterpret_cast<const float2*>(ssc + b * kSP + cl + 8 * j);
                acc[j][0] = fmaf(d.x, c[0], acc[j][0]);
                acc[j][1] = fmaf(d.y, c[1], acc[j][1]);
                acc[j][2] = fmaf(d.x, c[2], acc[j][2]);
                acc[j][3] = fmaf(d.y, c[3], acc[j][3]);
                if constexpr (QK == SD_A8G64) {
                    const float2 bb = *reinterpret_cast<const float2*>(sbi + b * kSP + cl + 8 * j);
                    const float s0 = xsum[b * 16 + g], s1 = xsum[b * 16 + g + 8];
                    acc[j][0] = fmaf(bb.x, s0, acc[j][0]);
                    acc[j][1] = fmaf(bb.y, s0, acc[j][1]);
                    acc[j][2] = fmaf(bb.x, s1, acc[j][2]);
                    acc[j][3] = fmaf(bb.y, s1, acc[j][3]);
                }
            }
        }
    };

    for (int kb = 0; kb < nbk; kb += 2 * NBB) {
        compute_batch(bufA, kb);
        if (kb + 2 * NBB < nbk) load_batch(bufA, kb + 2 * NBB);
        if (kb + NBB >= nbk) break;
        compute_batch(bufB, kb + NBB);
        if (kb + 3 * NBB < nbk) load_batch(bufB, kb + 3 * NBB);
    }

    // ---- partial sums of this split: ws[split][m][n]
    float* ws = a.ws + (size_t)blockIdx.y * 16 * N;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int n = n0 + cl + 8 * j;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int m = g + 8 * h;
            if (m >= M) continue;
            if (n < N) ws[(size_t)m * N + n] = acc[j][2 * h];
            if (n + 1 < N) ws[(size_t)m * N + n + 1] = acc[j][2 * h + 1];
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(a.cnt + blockIdx.x, 1) == (int)gridDim.y - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- last CTA of the column tile: sum the splits in order, epilogue
    const int ncols = min(kTileN, N - n0);
    const int outs = a.epi == EPI_SWIGLU ? ncols / 2 : ncols;
    for (int i = tid; i < M * outs; i += kThreads) {
        const int m = i / outs, jj = i - m * outs;
        // the splits' partials in split order; loads issued eight at a time (independent L2
        // round trips), the additions stay in order so the result does not depend on the grouping
        auto sum = [&](int n) {
            const int S = (int)gridDim.y;
            const float* p = a.ws + (size_t)m * N + n;
            const size_t stride = (size_t)16 * N;
            float v = 0.f;
            for (int s0 = 0; s0 < S; s0 += 8) {
                float pv[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) pv[j] = s0 + j < S ? __ldcg(p + (size_t)(s0 + j) * stride) : 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (s0 + j < S) v += pv[j];
            }
            return v;
        };
        float v;
        int oc;
        if (a.epi == EPI_SWIGLU) {
            const int n = n0 + 2 * jj;  // interleaved rows: n the gate, n + 1 the up projection
            v = silu(sum(n)) * sum(n + 1);
            oc = n >> 1;
        } else {
            oc = n0 + jj;
            v = sum(oc);
            if (a.bias) v += a.bias[oc];
            if (a.epi == EPI_GELU) v = gelu_tanh(v);
        }
        if (a.resid) v += a.resid[(size_t)m * a.ldy + oc];
        a.y[(size_t)m * a.ldy + oc] = v;
    }
    if (tid == 0) a.cnt[blockIdx.x] = 0;
}

struct Plan {
    int k_per = 0, splits = 0, tiles = 0;
};

Plan plan(int N, int K, int sm_count) {
    Plan p;
    p.tiles = (N + kTileN - 1) / kTileN;
    const int gran = (K % 64 == 0) ? 64 : 32;
    const int want = std::max(1, (2 * std::max(sm_count, 1) + p.tiles - 1) / p.tiles);
    int kp = (K + want - 1) / want;
    kp = ((kp + gran - 1) / gran) * gran;
    // at least 256 codes per CTA row range: below that the staging and the split reduction
    // cost more than the extra CTAs gain (small code-predictor matrices)
    const int kmin = std::min(K, 256) / gran * gran;
    p.k_per = std::min(std::max(kp, std::max(kmin, gran)), kMaxKPer);
    p.splits = (K + p.k_per - 1) / p.k_per;
    return p;
}

template <int QK>
cudaError_t launch_fmt(const Gemm16Args& a, const Plan& p, cudaStream_t st) {
    // the opt-in size covers the largest K range; setting it is cheap and keeps no state here
    cudaError_t e = cudaFuncSetAttribute(k_gemm16<QK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes<QK>(kMaxKPer));
    if (e != cudaSuccess) return e;
    k_gemm16<QK><<<dim3(p.tiles, p.splits), kThreads, smem_bytes<QK>(p.k_per), st>>>(a);
    return cudaGetLastError();
}

}  // namespace g16_detail

size_t gemm16_ws_floats(int N, int K, int sm_count) {
    const g16_detail::Plan p = g16_detail::plan(N, K, sm_count);
    return (size_t)p.splits * 16 * N;
}

int gemm16_tiles(int N) { return (N + g16_detail::kTileN - 1) / g16_detail::kTileN; }

cudaError_t launch_gemm16(Gemm16Args a, int sm_count, cudaStream_t st) {
    using namespace g16_detail;
    const int N = a.W.rows, K = a.W.cols;
    const int bk = a.W.kind == SD_A8G64 ? 64 : 32;
    if (a.M < 1 || a.M > 16 || N < 1 || K < bk || K % bk || !a.x || !a.y || !a.ws || !a.cnt)
        return cudaErrorInvalidValue;
    if (a.ldx % 4 || reinterpret_cast<uintptr_t>(a.x) % 16) return cudaErrorInvalidValue;
    if (a.epi == EPI_SWIGLU && (N % 2 || a.bias)) return cudaErrorInvalidValue;
    const Plan p = plan(N, K, sm_count);
    a.k_per = p.k_per;
    switch (a.W.kind) {
        case SD_Q8_0: return launch_fmt<SD_Q8_0>(a, p, st);
        case SD_Q4_0: return launch_fmt<SD_Q4_0>(a, p, st);
        case SD_A8G64: return launch_fmt<SD_A8G64>(a, p, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sd
