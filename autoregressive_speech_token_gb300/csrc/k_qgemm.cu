// Tensor-core GEMM over block-quantised weights: Y[M][N] = X[M][K] W[N][K]^T
// (+bias, GELU / SwiGLU, +residual), for prompt prefill (M = rows x prompt
// positions) and batched decode rows.
//
// The weights stay exact: the codes of a quantisation block (Q8_0 q, Q4_0 q-8,
// affine q) are small integers, exact in fp16, and the block's fp16 scale is
// applied in fp32 to the block's partial sum -- w = d*q, so
// sum_k x_k w_k = d * sum_k x_k q_k ("Chatterbox -> ggml Port: Development
// Journal", Tier A item A3 and section 3.23 for the block formats; for affine
// groups sum_k x_k (s q_k + b) = s sum_k x_k q_k + b sum_k x_k, "Every Frame Is
// a Memory Read", section 3).  The fp32 activations are split into two fp16
// terms x = x_hi + x_lo, so each k16 step is two MMAs; products accumulate in
// fp32.
//
// Tiling: a 128-thread CTA computes a 64 x 64 output tile; warp w owns rows
// 16w..16w+15 and all eight n8 tiles.  Each K block (32 weights, 64 for affine)
// is staged in shared memory: activations as fp16 hi/lo, codes as fp16, the
// block scales as fp32; rows are padded by 8 halves so the fragment loads are
// bank-conflict free.  MMA: mma.sync m16n8k16, fp16 inputs, fp32 accumulate.
#include "sd_internal.cuh"

namespace sd {
namespace {

constexpr int BM = 64, BN = 64, PAD = 8;

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ uint32_t ld_h2(const __half* p) { return *reinterpret_cast<const uint32_t*>(p); }

__device__ __forceinline__ float gelu_tanh(float t) {
    const float c = 0.7978845608028654f;
    return 0.5f * t * (1.0f + tanhf(c * (t + 0.044715f * t * t * t)));
}
__device__ __forceinline__ float silu(float t) { return t / (1.0f + expf(-t)); }

template <int QK>
__global__ void __launch_bounds__(128) k_qgemm(const QGemmArgs a) {
    constexpr int BK = (QK == SD_A8G64) ? 64 : 32;
    constexpr int LD = BK + PAD;
    __shared__ __align__(16) __half xh[BM * LD];
    __shared__ __align__(16) __half xl[BM * LD];
    __shared__ __align__(16) __half wq[BN * LD];
    __shared__ float wsc[BN], wbi[BN], xsum[BM];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int M = a.M, N = a.W.rows, K = a.W.cols;
    const int row_bytes = (QK == SD_Q4_0) ? (K >> 1) : K;

    float acc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;

    for (int k0 = 0; k0 < K; k0 += BK) {
        // ---- activations: fp32 -> fp16 hi + lo
        for (int i = tid; i < BM * BK; i += 128) {
            const int r = i / BK, c = i - r * BK;
            const float v = (m0 + r < M) ? __ldg(a.x + (size_t)(m0 + r) * a.ldx + k0 + c) : 0.f;
            const __half hi = __float2half_rn(v);
            xh[r * LD + c] = hi;
            xl[r * LD + c] = __float2half_rn(v - __half2float(hi));
        }
        if (QK == SD_A8G64) {
            // per-row sum of the group's activations (for the affine bias term)
            for (int r = tid; r < BM; r += 128) {
                float s = 0.f;
                if (m0 + r < M)
                    for (int c = 0; c < BK; ++c) s += __ldg(a.x + (size_t)(m0 + r) * a.ldx + k0 + c);
                xsum[r] = s;
            }
        }
        // ---- weight codes -> fp16 integers; block scales
        for (int i = tid; i < BN * BK; i += 128) {
            const int r = i / BK, c = i - r * BK;
            float q = 0.f;
            if (n0 + r < N) {
                const uint8_t* row = a.W.q + (size_t)(n0 + r) * row_bytes;
                if (QK == SD_Q4_0) {
                    const uint8_t byte = __ldg(row + (k0 >> 1) + (c & 15));
                    q = (float)((c < 16 ? (byte & 0xF) : (byte >> 4)) - 8);
                } else if (QK == SD_Q8_0) {
                    q = (float)(int8_t)__ldg(row + k0 + c);
                } else {
                    q = (float)__ldg(row + k0 + c);
                }
            }
            wq[r * LD + c] = __float2half_rn(q);  // exact: |q| <= 255
        }
        for (int r = tid; r < BN; r += 128) {
            float s = 0.f, b = 0.f;
            if (n0 + r < N) {
                if (QK == SD_A8G64) {
                    const __half2 sb = __ldg(reinterpret_cast<const __half2*>(a.W.s) + (size_t)(n0 + r) * (K / 64) + k0 / 64);
                    s = __low2float(sb);
                    b = __high2float(sb);
                } else {
                    s = __half2float(__ldg(reinterpret_cast<const __half*>(a.W.s) + (size_t)(n0 + r) * (K / 32) + k0 / 32));
                }
            }
            wsc[r] = s;
            wbi[r] = b;
        }
        __syncthreads();

        // ---- MMAs: the block's integer-code products, then the scale in fp32
        const int ar = warp * 16;
        uint32_t ahi[BK / 16][4], alo[BK / 16][4];
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
            const int kc = kk * 16;
            ahi[kk][0] = ld_h2(&xh[(ar + g) * LD + kc + 2 * t]);
            ahi[kk][1] = ld_h2(&xh[(ar + g + 8) * LD + kc + 2 * t]);
            ahi[kk][2] = ld_h2(&xh[(ar + g) * LD + kc + 2 * t + 8]);
            ahi[kk][3] = ld_h2(&xh[(ar + g + 8) * LD + kc + 2 * t + 8]);
            alo[kk][0] = ld_h2(&xl[(ar + g) * LD + kc + 2 * t]);
            alo[kk][1] = ld_h2(&xl[(ar + g + 8) * LD + kc + 2 * t]);
            alo[kk][2] = ld_h2(&xl[(ar + g) * LD + kc + 2 * t + 8]);
            alo[kk][3] = ld_h2(&xl[(ar + g + 8) * LD + kc + 2 * t + 8]);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
                uint32_t b[2];
                b[0] = ld_h2(&wq[(j * 8 + g) * LD + kk * 16 + 2 * t]);
                b[1] = ld_h2(&wq[(j * 8 + g) * LD + kk * 16 + 2 * t + 8]);
                mma16816(c, ahi[kk], b);
                mma16816(c, alo[kk], b);
            }
            const int nc = j * 8 + 2 * t;
            const float d0 = wsc[nc], d1 = wsc[nc + 1];
            acc[j][0] = fmaf(d0, c[0], acc[j][0]);
            acc[j][1] = fmaf(d1, c[1], acc[j][1]);
            acc[j][2] = fmaf(d0, c[2], acc[j][2]);
            acc[j][3] = fmaf(d1, c[3], acc[j][3]);
            if (QK == SD_A8G64) {
                const float s0 = xsum[ar + g], s1 = xsum[ar + g + 8];
                acc[j][0] = fmaf(wbi[nc], s0, acc[j][0]);
                acc[j][1] = fmaf(wbi[nc + 1], s0, acc[j][1]);
                acc[j][2] = fmaf(wbi[nc], s1, acc[j][2]);
                acc[j][3] = fmaf(wbi[nc + 1], s1, acc[j][3]);
            }
        }
        __syncthreads();
    }

    // ---- epilogue
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int m = m0 + warp * 16 + g + 8 * h;
            const int n = n0 + j * 8 + 2 * t;
            if (m >= M) continue;
            float v0 = acc[j][2 * h], v1 = acc[j][2 * h + 1];
            if (a.epi == EPI_SWIGLU) {
                // interleaved rows: column n (even) is the gate, n + 1 the up projection
                if (n + 1 < N) {
                    float o = silu(v0) * v1;
                    if (a.resid) o += a.resid[(size_t)m * a.ldy + (n >> 1)];
                    a.y[(size_t)m * a.ldy + (n >> 1)] = o;
                }
                continue;
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int nn = n + e;
                if (nn >= N) continue;
                float v = e ? v1 : v0;
                if (a.bias) v += a.bias[nn];
                if (a.epi == EPI_GELU) v = gelu_tanh(v);
                if (a.resid) v += a.resid[(size_t)m * a.ldy + nn];
                a.y[(size_t)m * a.ldy + nn] = v;
            }
        }
    }
}

}  // namespace

cudaError_t launch_qgemm(const QGemmArgs& a, cudaStream_t st) {
    if (a.M < 1 || a.W.rows < 1 || a.W.cols % 32 || (a.W.kind == SD_A8G64 && a.W.cols % 64)) return cudaErrorInvalidValue;
    if (a.epi == EPI_SWIGLU && a.W.rows % 2) return cudaErrorInvalidValue;
    const dim3 grid((a.W.rows + BN - 1) / BN, (a.M + BM - 1) / BM);
    switch (a.W.kind) {
        case SD_Q8_0: k_qgemm<SD_Q8_0><<<grid, 128, 0, st>>>(a); break;
        case SD_Q4_0: k_qgemm<SD_Q4_0><<<grid, 128, 0, st>>>(a); break;
        case SD_A8G64: k_qgemm<SD_A8G64><<<grid, 128, 0, st>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace sd
