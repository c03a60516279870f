// Prompt-prefill GEMM on the 5th-generation tensor cores (tcgen05, TMEM
// accumulator, TMA operand loads): Y[M][N] = X[M][K] W[N][K]^T with the GEMV
// epilogues (bias, GELU, interleaved SwiGLU, residual).
//
// "Chatterbox -> ggml Port: Development Journal", section 3.2: the prompt graph
// applies each layer to all prompt positions at once -- a dense contraction,
// unlike the decode step.  Precision: the weights are dequantised once at load
// (w = d*q, or fma(s, q, b) for affine groups; exact in fp32) and split, like
// the fp32 activations, into fp16 high and low parts; three fp16 MMAs per K step
// (hi*hi + hi*lo + lo*hi, fp32 accumulation) give an error near 2^-22 of the
// products, where one fp16 MMA would carry 2^-11.
//
// Tile: 128 rows x 64 outputs per CTA (more CTAs for the short prompt row
// counts), K in steps of 64 (one 128-byte swizzled row of fp16 per operand
// row), four stages of four operand tiles (X hi/lo 16 KB each, W hi/lo 8 KB
// each) = 192 KB of shared memory.  Thread 0 issues the TMA loads and the
// MMAs; the MMA completion (tcgen05.commit) frees a stage for the next load.
// The accumulator (128 x 64 fp32) lives in tensor memory; after the last K
// step each warp reads its 32 rows back (tcgen05.ld) for the epilogue.  Every
// wait is bounded: on expiry the kernel records an error, waits (bounded) for
// its own copies and MMAs, frees its tensor memory and returns.
#include <cuda.h>

#include "sd_internal.cuh"

namespace sd {
namespace tc_detail {

constexpr int kBM = 128, kBN = 64, kBK = 64, kStages = 4;
constexpr int kTileX = kBM * kBK * 2;         // 16 KB per activation tile
constexpr int kTileW = kBN * kBK * 2;         // 8 KB per weight tile
constexpr int kStageBytes = 2 * kTileX + 2 * kTileW;  // X hi, X lo, W hi, W lo
constexpr int kErrTimeout = 6;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ int ld_volatile(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

__device__ __forceinline__ void mb_init(uint32_t mb) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mb) : "memory");
}
__device__ __forceinline__ void mb_expect(uint32_t mb, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"(bytes) : "memory");
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
__device__ bool mb_wait(uint32_t mb, uint32_t parity, long long budget) {
    if (mb_try(mb, parity)) return true;
    const long long t0 = clock64();
    while (!mb_try(mb, parity))
        if (clock64() - t0 > budget) return false;
    return true;
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t mb) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mb)
        : "memory");
}

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzled
// layout TMA writes (8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);        // start address
    d |= (uint64_t)1u << 16;                        // leading byte offset (unused when swizzled)
    d |= (uint64_t)(1024u >> 4) << 32;              // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1u << 46;                        // descriptor version
    d |= (uint64_t)2u << 61;                        // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (K-major), fp32 D, M = 128, N = 64.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);

__device__ __forceinline__ void mma(uint32_t tmem, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
        ::"r"(tmem), "l"(a), "l"(b), "r"(kIdesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t mb) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mb) : "memory");
}

__device__ __forceinline__ float gelu_tanh(float t) {
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    return 0.5f * t * (1.0f + tanhf(c * (t + 0.044715f * t * t * t)));
}
__device__ __forceinline__ float silu(float t) { return t / (1.0f + expf(-t)); }

__global__ void __launch_bounds__(128, 1) k_gemm_tc(const __grid_constant__ TcGemmArgs a) {
    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
    __shared__ __align__(8) unsigned long long s_full[kStages], s_empty[kStages];
    __shared__ uint32_t s_tmem;
    __shared__ int s_ok;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * kBM;
    const int KT = a.K / kBK;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "n"(kBN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mb_init(smem_u32(&s_full[s]));
            mb_init(smem_u32(&s_empty[s]));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_ok = 1;
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s_tmem;

    if (tid == 0) {
        auto stage_ptr = [&](int s, int which) {
            const int off = which < 2 ? which * kTileX : 2 * kTileX + (which - 2) * kTileW;
            return smem_u32(sm + (size_t)s * kStageBytes + off);
        };
        auto issue = [&](int t) {
            const int s = t % kStages;
            const uint32_t mb = smem_u32(&s_full[s]);
            mb_expect(mb, kStageBytes);
            tma_2d(stage_ptr(s, 0), &a.xh, t * kBK, m0, mb);
            tma_2d(stage_ptr(s, 1), &a.xl, t * kBK, m0, mb);
            tma_2d(stage_ptr(s, 2), &a.wh, t * kBK, n0, mb);
            tma_2d(stage_ptr(s, 3), &a.wl, t * kBK, n0, mb);
        };
        bool ok = true;
        int issued = 0;
        for (; issued < KT && issued < kStages; ++issued) issue(issued);
        int mmas = 0;  // K steps whose MMAs were issued
        for (int t = 0; t < KT && ok; ++t) {
            const int s = t % kStages;
            if (!mb_wait(smem_u32(&s_full[s]), (uint32_t)((t / kStages) & 1), a.spin_budget)) { ok = false; break; }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
                const uint64_t xh = sdesc(stage_ptr(s, 0) + kk * 32), xl = sdesc(stage_ptr(s, 1) + kk * 32);
                const uint64_t wh = sdesc(stage_ptr(s, 2) + kk * 32), wl = sdesc(stage_ptr(s, 3) + kk * 32);
                mma(tmem, xh, wh, (t > 0 || kk > 0) ? 1u : 0u);
                mma(tmem, xh, wl, 1u);
                mma(tmem, xl, wh, 1u);
            }
            mma_commit(smem_u32(&s_empty[s]));
            mmas = t + 1;
            // the stage of step t-1 is free once its MMAs finished: load step t-1+kStages into it
            if (t >= 1 && issued < KT) {
                const int sp = (t - 1) % kStages;
                if (!mb_wait(smem_u32(&s_empty[sp]), (uint32_t)(((t - 1) / kStages) & 1), a.spin_budget)) {
                    ok = false;
                    break;
                }
                issue(issued++);
            }
        }
        // wait for the last MMAs (their commit is the last phase of that stage's barrier)
        if (ok && mmas > 0) {
            const int t = mmas - 1;
            ok = mb_wait(smem_u32(&s_empty[t % kStages]), (uint32_t)((t / kStages) & 1), a.spin_budget);
        }
        if (!ok) {
            s_ok = 0;
            if (a.err) atomicCAS(a.err, 0, kErrTimeout);
            // bounded drain of this CTA's outstanding loads and MMAs
            for (int t = mmas; t < issued; ++t)
                mb_wait(smem_u32(&s_full[t % kStages]), (uint32_t)((t / kStages) & 1), a.spin_budget);
            if (mmas > 0) {
                const int t = mmas - 1;
                mb_wait(smem_u32(&s_empty[t % kStages]), (uint32_t)((t / kStages) & 1), a.spin_budget);
            }
        }
    }
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    if (s_ok) {
        // epilogue: warp w holds rows 32w..32w+31 of the tile in TMEM lanes 32w..
        const int m = m0 + warp * 32 + lane;
        for (int c0 = 0; c0 < kBN; c0 += 32) {
            uint32_t r[32];
            const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0;
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
                "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                  "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                  "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                  "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                  "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                : "r"(taddr));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            if (m >= a.M) continue;
            if (a.epi == EPI_SWIGLU) {
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const int n = n0 + c0 + j;
                    if (n + 1 >= a.N) break;
                    float o = silu(__uint_as_float(r[j])) * __uint_as_float(r[j + 1]);
                    float* yp = a.y + (size_t)m * a.ldy + (n >> 1);
                    if (a.resid) o += a.resid[(size_t)m * a.ldy + (n >> 1)];
                    *yp = o;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int n = n0 + c0 + j;
                    if (n >= a.N) break;
                    float v = __uint_as_float(r[j]);
                    if (a.bias) v += a.bias[n];
                    if (a.epi == EPI_GELU) v = gelu_tanh(v);
                    if (a.resid) v += a.resid[(size_t)m * a.ldy + n];
                    a.y[(size_t)m * a.ldy + n] = v;
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kBN) : "memory");
}

// fp32 rows -> fp16 high and low parts: hi = fp16(x), lo = fp16(x - hi)
__global__ void k_split_rows(const float* __restrict__ x, int ldx, int M, int K, __half* __restrict__ hi,
                             __half* __restrict__ lo) {
    const size_t n = (size_t)M * K;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t m = i / K, k = i - m * K;
        const float v = x[m * ldx + k];
        const __half h = __float2half_rn(v);
        hi[i] = h;
        lo[i] = __float2half_rn(v - __half2float(h));
    }
}

// Repacked quantised matrix -> dequantised fp16 high and low parts [rows][cols]
__global__ void k_dequant_split(const QMat W, __half* __restrict__ hi, __half* __restrict__ lo) {
    const size_t n = (size_t)W.rows * W.cols;
    const int K = W.cols;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t r = i / K;
        const int k = (int)(i - r * K);
        const float w = q_value(W, r, k);
        const __half h = __float2half_rn(w);
        hi[i] = h;
        lo[i] = __float2half_rn(w - __half2float(h));
    }
}

}  // namespace tc_detail

namespace {
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeFn encoder() {
    static EncodeFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (EncodeFn) nullptr;
        return reinterpret_cast<EncodeFn>(p);
    }();
    return fn;
}
}  // namespace

bool tc_map_fp16(CUtensorMap* map, const void* base, int rows, int cols, bool weights) {
    EncodeFn enc = encoder();
    if (!enc || !base || rows < 1 || cols % tc_detail::kBK || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)tc_detail::kBK, (cuuint32_t)(weights ? tc_detail::kBN : tc_detail::kBM)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t tc_smem_bytes() { return (size_t)tc_detail::kStages * tc_detail::kStageBytes + 1024; }

cudaError_t launch_gemm_tc(const TcGemmArgs& a, cudaStream_t st) {
    using namespace tc_detail;
    if (a.M < 1 || a.N < 1 || a.K < kBK || a.K % kBK || !a.y) return cudaErrorInvalidValue;
    if (a.epi == EPI_SWIGLU && (a.N % 2 || a.bias)) return cudaErrorInvalidValue;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem_bytes());
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const dim3 grid((a.N + kBN - 1) / kBN, (a.M + kBM - 1) / kBM);
    k_gemm_tc<<<grid, 128, tc_smem_bytes(), st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_split_rows(const float* x, int ldx, int M, int K, __half* hi, __half* lo, cudaStream_t st) {
    if (M < 1 || K < 1) return cudaErrorInvalidValue;
    const long long n = (long long)M * K;
    const int blocks = (int)std::min<long long>((n + 255) / 256, 4096);
    tc_detail::k_split_rows<<<blocks, 256, 0, st>>>(x, ldx, M, K, hi, lo);
    return cudaGetLastError();
}

cudaError_t launch_dequant_split(const QMat& W, __half* hi, __half* lo, cudaStream_t st) {
    const long long n = (long long)W.rows * W.cols;
    if (n < 1) return cudaErrorInvalidValue;
    const int blocks = (int)std::min<long long>((n + 255) / 256, 16384);
    tc_detail::k_dequant_split<<<blocks, 256, 0, st>>>(W, hi, lo);
    return cudaGetLastError();
}

}  // namespace sd
