// Quantised GEMV with fused norm prologue and bias/activation/residual
// epilogue: the weight-streaming matvec of the decode step.
//
// One decode step multiplies every quantised matrix once by a 1- or 2-row
// activation ("Every Frame Is a Memory Read", section 3: decode is a memory
// read; "Chatterbox -> ggml Port: Development Journal", sections 3.15-3.16:
// the matvec carries the bias and the residual add in its epilogue).
//
// Work split: a warp owns a 1024-element slice of K (lane l holds the 32
// activation values of its 16-byte weight units in registers, reused for
// every row it visits) and R rows per tile; K > 1024 is split across WK warps
// whose partial sums meet in shared memory in a fixed order (deterministic).
// Weights are read once with 128-bit streaming loads; dequantisation happens
// in registers: Q4_0 / Q5_0 / 4-bit affine nibbles (Q5_0 with its fifth bit)
// and Q8_0 / 8-bit affine bytes become exact floats through the 2^23 exponent
// trick, the block scale multiplies the block's partial sum (affine formats add
// bias times the activations' block sum).
#pragma once
#include "sd_internal.cuh"

namespace sd {
namespace gemv_detail {

constexpr float kMagic = 8388608.0f;  // 2^23: float bits 0x4B000000 | n == 2^23 + n for n < 2^23

__device__ __forceinline__ uint4 ld_stream(const uint8_t* p) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// sum over the block of NB values; every thread gets the totals (fixed order:
// warp sums, then warp 0 reduces the warp sums with shuffles).
template <int NB>
__device__ __forceinline__ void block_sum(float (&v)[NB], float* scratch) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        float s = warp_sum(v[b]);
        if (lane == 0) scratch[warp * NB + b] = s;
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const float s = warp_sum(lane < nw ? scratch[lane * NB + b] : 0.f);
            if (lane == 0) scratch[32 * NB + b] = s;
        }
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < NB; ++b) v[b] = scratch[32 * NB + b];
    __syncthreads();
}

// Activation rows staged in shared memory carry 4 floats of padding after
// every 32 elements: a lane's 32-element slice (its 16-byte weight unit) then
// starts 36 floats after its neighbour's, so the eight 16-byte loads of a
// quarter warp fall in distinct bank groups (unpadded, the 128-byte stride put
// every lane of the warp on the same four banks).
__device__ __forceinline__ int pidx(int k) { return k + ((k >> 5) << 2); }
__host__ __device__ __forceinline__ int padded(int K) { return K + (K >> 3); }

// 4-bit codes (16-byte units of 32 elements), affine formats, groups of 64
template <int QK> constexpr bool kNib = QK == SD_Q4_0 || QK == SD_Q5_0 || QK == SD_A4G32 || QK == SD_A4G64;
template <int QK> constexpr bool kAff = QK == SD_A8G64 || QK == SD_A4G32 || QK == SD_A4G64;
template <int QK> constexpr bool kG64 = QK == SD_A8G64 || QK == SD_A4G64;

template <int QK>
struct Unit {
    // 16-byte weight units per lane per 1024-element warp slice
    static constexpr int kU = kNib<QK> ? 1 : 2;
};

// Partial dot product of one 16-byte unit with the lane's activations.
__device__ __forceinline__ float dot_q4(const uint4 w, const float* x) {
    // bytes 0..15 -> elements 0..15 (low nibble) and 16..31 (high nibble)
    const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t lo = (wd[i] >> (8 * k)) & 0xFu;
            const uint32_t hi = (wd[i] >> (8 * k + 4)) & 0xFu;
            const float flo = __int_as_float(0x4B000000u | lo) - (kMagic + 8.0f);  // q - 8, exact
            const float fhi = __int_as_float(0x4B000000u | hi) - (kMagic + 8.0f);
            s = fmaf(flo, x[4 * i + k], s);
            s = fmaf(fhi, x[16 + 4 * i + k], s);
        }
    }
    return s;
}

// Q5_0: the nibbles as in dot_q4 plus the fifth bit of element j in bit j of qh; code - 16
__device__ __forceinline__ float dot_q5(const uint4 w, const uint32_t qh, const float* x) {
    const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int j = 4 * i + k;
            const uint32_t lo = ((wd[i] >> (8 * k)) & 0xFu) | (((qh >> j) & 1u) << 4);
            const uint32_t hi = ((wd[i] >> (8 * k + 4)) & 0xFu) | (((qh >> (j + 16)) & 1u) << 4);
            const float flo = __int_as_float(0x4B000000u | lo) - (kMagic + 16.0f);  // q - 16, exact
            const float fhi = __int_as_float(0x4B000000u | hi) - (kMagic + 16.0f);
            s = fmaf(flo, x[j], s);
            s = fmaf(fhi, x[16 + j], s);
        }
    }
    return s;
}

// unsigned 4-bit codes in the dot_q4 layout (affine formats)
__device__ __forceinline__ float dot_u4(const uint4 w, const float* x) {
    const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t lo = (wd[i] >> (8 * k)) & 0xFu;
            const uint32_t hi = (wd[i] >> (8 * k + 4)) & 0xFu;
            s = fmaf(__int_as_float(0x4B000000u | lo) - kMagic, x[4 * i + k], s);
            s = fmaf(__int_as_float(0x4B000000u | hi) - kMagic, x[16 + 4 * i + k], s);
        }
    }
    return s;
}

__device__ __forceinline__ float dot_s8(const uint4 w, const float* x) {
    const uint32_t wd[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t u = (wd[i] >> (8 * k)) & 0xFFu;  // q + 128 for two's-complement q
            s = fmaf(__int_as_float(0x4B000000u | u) - (kMagic + 128.0f), x[4 * i + k], s);
        }
    }
    return s;
}

__device__ __forceinline__ float dot_u8(const uint4 w, const float* x) {
    const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t u = (wd[i] >> (8 * k)) & 0xFFu;
            s = fmaf(__int_as_float(0x4B000000u | u) - kMagic, x[4 * i + k], s);
        }
    }
    return s;
}

__device__ __forceinline__ float gelu_tanh(float t) {
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    return 0.5f * t * (1.0f + tanhf(c * (t + 0.044715f * t * t * t)));
}

__device__ __forceinline__ float silu(float t) { return t / (1.0f + expf(-t)); }

// Loads tile tt's weight units and their block scales (affine: scale and
// bias as one half2) into registers; issued a tile ahead, so neither the
// codes nor the scales are waited for inside the dot products.
template <int QK, int R, int U>
__device__ __forceinline__ void load_tile(uint4 (&w)[R][U], uint32_t (&sc)[R][U], uint32_t (&hb)[R][U],
                                          const GemvArgs& a, int tt, int WR, int rg, int rows, int row_bytes, int spr,
                                          const int (&ebase)[U], int K) {
    const int r0 = tt * WR * R + rg * R;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int r = r0 + i;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            hb[i][u] = 0u;
            if (r < rows && ebase[u] < K) {
                const int boff = kNib<QK> ? (ebase[u] >> 1) : ebase[u];
                const int gi = kG64<QK> ? (ebase[u] >> 6) : (ebase[u] >> 5);
                w[i][u] = ld_stream(a.W.q + (size_t)r * row_bytes + boff);
                if (kAff<QK>) {
                    sc[i][u] = __ldg(reinterpret_cast<const unsigned int*>(a.W.s) + (size_t)r * spr + gi);
                } else if (QK == SD_Q5_0) {
                    const uint2 v = __ldg(reinterpret_cast<const uint2*>(a.W.s) + (size_t)r * spr + gi);
                    sc[i][u] = v.x;
                    hb[i][u] = v.y;
                } else {
                    sc[i][u] = __ldg(reinterpret_cast<const unsigned short*>(a.W.s) + (size_t)r * spr + gi);
                }
            } else {
                w[i][u] = make_uint4(0u, 0u, 0u, 0u);
                sc[i][u] = 0u;
            }
        }
    }
}

template <int QK, int NB, int R>
__global__ void __launch_bounds__(256) k_gemv(const GemvArgs a) {
    constexpr int U = Unit<QK>::kU;
    const int K = a.W.cols, rows = a.W.rows;
    const int WK = (K + 1023) >> 10;
    const int nw = blockDim.x >> 5;
    const int WR = nw / WK;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kw = warp % WK, rg = warp / WK;
    const int tiles = (rows + WR * R - 1) / (WR * R);
    const int row_bytes = kNib<QK> ? (K >> 1) : K;
    const int spr = kG64<QK> ? (K >> 6) : (K >> 5);

    __shared__ float s_scr[33 * NB];
    __shared__ float s_tot[8 * R * NB];
    extern __shared__ float s_x[];  // [NB][padded(K)] transformed activations (padded layout, pidx)

    // element index of the lane's unit u (units lie wholly inside or outside K)
    int ebase[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
        ebase[u] = kNib<QK> ? (kw * 1024 + lane * 32) : (kw * 1024 + u * 512 + lane * 16);
    constexpr int EPU = kNib<QK> ? 32 : 16;  // elements per unit

    // issue the first tile's weight loads before the prologue: they do not
    // depend on the activations.
    uint4 w[R][U];
    uint32_t scw[R][U], hbw[R][U];
    int t = blockIdx.x;
    pdl_trigger();
    if (t < tiles) load_tile<QK, R, U>(w, scw, hbw, a, t, WR, rg, rows, row_bytes, spr, ebase, K);
    pdl_wait();  // activations come from the previous kernel

    // ---------------------------------------------------------------- prologue
    // stage the activation rows in shared memory with 16-byte loads (one pass
    // over global memory), then normalise in place
    const int KP = padded(K);  // padded row length in shared memory
    {
        const int K4 = K >> 2;
        const float4* xg = reinterpret_cast<const float4*>(a.x);
        float4* xs4 = reinterpret_cast<float4*>(s_x);
#pragma unroll 4
        for (int i = threadIdx.x; i < NB * K4; i += blockDim.x) {
            const int b = i / K4, k4 = i - b * K4;
            xs4[(b * KP >> 2) + k4 + (k4 >> 3)] = xg[(size_t)b * (a.x_stride >> 2) + k4];
        }
    }
    __syncthreads();
    if (a.pro == PRO_LN || a.pro == PRO_RMS) {
        float v[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            float s = 0.f;
            for (int k = threadIdx.x; k < K; k += blockDim.x) {
                const float xv = s_x[b * KP + pidx(k)];
                s += (a.pro == PRO_LN) ? xv : xv * xv;
            }
            v[b] = s;
        }
        block_sum<NB>(v, s_scr);
        float mu[NB], rs[NB];
        if (a.pro == PRO_LN) {
#pragma unroll
            for (int b = 0; b < NB; ++b) mu[b] = v[b] / (float)K;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                float s = 0.f;
                for (int k = threadIdx.x; k < K; k += blockDim.x) {
                    const float dx = s_x[b * KP + pidx(k)] - mu[b];
                    s = fmaf(dx, dx, s);
                }
                v[b] = s;
            }
            block_sum<NB>(v, s_scr);
#pragma unroll
            for (int b = 0; b < NB; ++b) rs[b] = 1.0f / sqrtf(v[b] / (float)K + a.eps);
        } else {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                mu[b] = 0.f;
                rs[b] = 1.0f / sqrtf(v[b] / (float)K + a.eps);
            }
        }
        const int K4 = K >> 2;
        const float4* g4 = reinterpret_cast<const float4*>(a.ng);
        const float4* b4 = reinterpret_cast<const float4*>(a.nbias);
        float4* xs4 = reinterpret_cast<float4*>(s_x);
        for (int i = threadIdx.x; i < NB * K4; i += blockDim.x) {
            const int b = i / K4, k4 = i - b * K4;
            const int pi = (b * KP >> 2) + k4 + (k4 >> 3);
            const float4 g = g4[k4];
            float4 x = xs4[pi];
            if (a.pro == PRO_LN) {
                const float4 o = b4[k4];
                x.x = fmaf((x.x - mu[b]) * rs[b], g.x, o.x);
                x.y = fmaf((x.y - mu[b]) * rs[b], g.y, o.y);
                x.z = fmaf((x.z - mu[b]) * rs[b], g.z, o.z);
                x.w = fmaf((x.w - mu[b]) * rs[b], g.w, o.w);
            } else {
                x.x = x.x * rs[b] * g.x;
                x.y = x.y * rs[b] * g.y;
                x.z = x.z * rs[b] * g.z;
                x.w = x.w * rs[b] * g.w;
            }
            xs4[pi] = x;
        }
    }
    __syncthreads();

    // ---------------------------------------------------------------- activations -> registers
    float xr[NB][32];
    float xsum[NB][U];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float s = 0.f;
            const bool in = ebase[u] < K;
#pragma unroll
            for (int j = 0; j < EPU; j += 4) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (in) v = *reinterpret_cast<const float4*>(&s_x[b * KP + pidx(ebase[u] + j)]);
                xr[b][u * EPU + j] = v.x; xr[b][u * EPU + j + 1] = v.y;
                xr[b][u * EPU + j + 2] = v.z; xr[b][u * EPU + j + 3] = v.w;
                s += (v.x + v.y) + (v.z + v.w);
            }
            xsum[b][u] = s;
        }
    }

    // ---------------------------------------------------------------- main loop
    for (; t < tiles; t += gridDim.x) {
        const int r0 = t * WR * R + rg * R;
        float acc[R][NB];
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[i][b] = 0.f;

#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int r = r0 + i;
            if (r >= rows) continue;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (ebase[u] >= K) continue;
                if (kAff<QK>) {
                    const __half2 sb = *reinterpret_cast<const __half2*>(&scw[i][u]);
                    const float sc = __low2float(sb), bi = __high2float(sb);
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        const float dq = kNib<QK> ? dot_u4(w[i][u], &xr[b][0]) : dot_u8(w[i][u], &xr[b][u * EPU]);
                        acc[i][b] = fmaf(sc, dq, fmaf(bi, xsum[b][u], acc[i][b]));
                    }
                } else {
                    const float d = __half2float(__ushort_as_half((unsigned short)(scw[i][u] & 0xFFFFu)));
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        const float dq = (QK == SD_Q4_0)   ? dot_q4(w[i][u], &xr[b][0])
                                         : (QK == SD_Q5_0) ? dot_q5(w[i][u], hbw[i][u], &xr[b][0])
                                                           : dot_s8(w[i][u], &xr[b][u * EPU]);
                        acc[i][b] = fmaf(d, dq, acc[i][b]);
                    }
                }
            }
        }
        // prefetch the next tile while reducing this one
        const int tn = t + gridDim.x;
        if (tn < tiles) load_tile<QK, R, U>(w, scw, hbw, a, tn, WR, rg, rows, row_bytes, spr, ebase, K);

#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float s = warp_sum(acc[i][b]);
                if (lane == 0) s_tot[((rg * R + i) * NB + b) * WK + kw] = s;
            }
        __syncthreads();
        const int n_out = WR * R * NB;
        if (threadIdx.x < n_out) {
            const int b = threadIdx.x % NB;
            const int i = (threadIdx.x / NB) % R;
            const int g = threadIdx.x / (NB * R);
            const int r = t * WR * R + g * R + i;
            float v = 0.f;
            for (int k = 0; k < WK; ++k) v += s_tot[((g * R + i) * NB + b) * WK + k];
            if (r < rows) {
                if (a.epi == EPI_SWIGLU) {
                    // rows are interleaved (gate 2j, up 2j+1); the even row's thread writes
                    if ((i & 1) == 0) {
                        float up = 0.f;
                        for (int k = 0; k < WK; ++k) up += s_tot[((g * R + i + 1) * NB + b) * WK + k];
                        const int j = r >> 1;
                        float o = silu(v) * up;
                        if (a.resid) o += a.resid[(size_t)b * a.y_stride + j];
                        a.y[(size_t)b * a.y_stride + j] = o;
                    }
                } else {
                    if (a.bias) v += a.bias[r];
                    if (a.epi == EPI_GELU) v = gelu_tanh(v);
                    if (a.resid) v += a.resid[(size_t)b * a.y_stride + r];
                    a.y[(size_t)b * a.y_stride + r] = v;
                }
            }
        }
        __syncthreads();
    }
}

template <int QK, int NB>
cudaError_t launch_t(const GemvArgs& a, int sm_count, cudaStream_t st) {
    constexpr int R = (NB == 1) ? 4 : 2;
    const int K = a.W.cols;
    const int WK = (K + 1023) / 1024;
    if (WK > 8) return cudaErrorInvalidValue;
    int WR = 8 / WK;
    if (WR < 1) WR = 1;
    // fewer rows per CTA when the matrix is short, so that every SM gets work
    while (WR > 1 && (a.W.rows + WR * R - 1) / (WR * R) < sm_count) WR >>= 1;
    const int tiles = (a.W.rows + WR * R - 1) / (WR * R);
    const size_t smem = sizeof(float) * (size_t)NB * padded(K);
    if (smem > 32 * 1024) {  // with the static arrays the total passes the 48 KB default
        cudaError_t e = cudaFuncSetAttribute(k_gemv<QK, NB, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    // one wave of resident CTAs that loop over the tiles (the next tile's loads are in flight
    // while a tile is reduced, and the activation prologue is paid once per CTA); the
    // occupancy of each (K slices, row groups) shape is asked once
    const int threads = 32 * WK * WR;
    static int occ_cache[9][4] = {};  // [WK][WR index] -> resident CTAs per SM
    int& occ = occ_cache[WK][WR >= 8 ? 3 : WR >= 4 ? 2 : WR >= 2 ? 1 : 0];
    if (occ == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv<QK, NB, R>, threads, smem) != cudaSuccess || n < 1)
            n = 1;
        occ = n;
    }
    const int wave = occ * sm_count;
    const int grid = tiles < wave ? tiles : wave;
    return launch_k(k_gemv<QK, NB, R>, dim3(grid), dim3(threads), smem, st, a);
}

inline cudaError_t check_gemv(const GemvArgs& a) {
    if (!q_valid(a.W.kind) || a.W.cols % q_group(a.W.kind) || a.W.cols > 8192) return cudaErrorInvalidValue;
    if (a.epi == EPI_SWIGLU && a.W.rows % 2) return cudaErrorInvalidValue;
    if (a.x_stride % 4 || (reinterpret_cast<uintptr_t>(a.x) & 15)) return cudaErrorInvalidValue;
    if (a.nb != 1 && a.nb != 2) return cudaErrorInvalidValue;
    return cudaSuccess;
}

}  // namespace gemv_detail
}  // namespace sd
