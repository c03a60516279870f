// Skinny GEMM for up to 16 activation rows on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators), for 8-bit affine-group weights: the G = 16
// rollouts of the Talker + code predictor ("Every Frame Is a Memory Read",
// section 8: G rollouts share one read of the weights per step).
// Y[M][N] = X[M][K] W[N][K]^T, M <= 16, with the GEMV epilogues.
//
// Roles.  The weights are the M = 128 operand (a CTA owns 128 weight rows) and
// the activations the N = 16 operand, so one tcgen05.mma (kind::f16, M 128,
// N 16, K 16) advances 128 rows by 16 codes for every rollout row at once.
//
// Exactness.  An affine group of 64 codes has w = s*q + b ("Every Frame Is a
// Memory Read", section 3).  The codes q (bytes 0..255) are exact in fp16, the
// fp32 activations are split x = hi + lo in fp16, and two MMAs per 16-wide K
// step (q*hi, q*lo) give exact products summed in fp32.  Each 64-wide group
// accumulates into its own 16 TMEM columns, so after the K loop the epilogue
// forms sum_g (s_g * D_g + b_g * sum_{k in g} x_k) in fp32 -- the scale and bias
// never pass through fp16.  (One accumulator over all groups would have needed
// the weights themselves in fp16, or a hi/lo split of them and a third MMA.)
//
// Data flow per CTA (128 threads, one CTA per SM, K range k_per <= 1024):
//   - thread 0 keeps kRaw groups of raw codes in flight: one 2-D TMA load of
//     128 rows x 64 bytes per group into a ring (zero fill past the matrix);
//   - all threads turn a landed group into fp16 codes in the 128-byte swizzled
//     K-major layout the MMA reads (16-byte chunk c of row r at chunk c ^ (r & 7)
//     of its 128-byte row, 8-row atoms 1024 bytes apart: the layout a TMA load
//     with 128-byte swizzle writes), in a ring of kAStages buffers;
//   - thread 0 issues the group's eight MMAs and commits them to an mbarrier
//     that frees the buffer kAStages groups later.
// The activations of the K range (fp16 hi/lo in the same layout), their group
// sums and the rows' scales and biases are staged once.  Partial sums go to a
// workspace [split][16][N]; the last CTA of each column tile adds the splits in
// split order and applies bias / GELU / SwiGLU / residual (as the mma.sync
// skinny GEMM), so results do not depend on timing.  Every wait is bounded: on
// expiry the kernel records an error, drains its own copies and MMAs (bounded),
// frees its tensor memory and returns.
#include <cuda.h>

#include <cstring>
#include <mutex>
#include <unordered_map>

#include "sd_internal.cuh"

namespace sd {
namespace g16tc_detail {

constexpr int kRows = 128;            // weight rows per CTA (the MMA's M)
constexpr int kG = 64;                // affine group width = one 128-byte swizzled row of fp16
constexpr int kMaxGroups = 16;        // K range per CTA <= 1024
constexpr int kRaw = 6;               // raw code groups in flight
constexpr int kAStages = 4;           // converted groups the MMAs may still be reading
constexpr int kThreads = 128;
constexpr int kTmemCols = 256;        // 16 columns per group, 16 groups
constexpr int kErrTimeout = 6;

constexpr int kRawBytes = kRows * kG;         // 8 KB: one group of codes, row-major
constexpr int kABytes = kRows * kG * 2;       // 16 KB: the group as fp16, swizzled
constexpr int kXBytes = 16 * kG * 2;          // 2 KB: 16 activation rows of a group, fp16, swizzled

// shared memory: [x hi | x lo] per group, two A buffers, the raw ring, then scales / biases / sums
constexpr size_t kOffX = 0;
constexpr size_t kOffA = kOffX + (size_t)kMaxGroups * 2 * kXBytes;
constexpr size_t kOffRaw = kOffA + (size_t)kAStages * kABytes;
constexpr size_t kOffSc = kOffRaw + (size_t)kRaw * kRawBytes;
constexpr size_t kOffBi = kOffSc + (size_t)kMaxGroups * kRows * 4;
constexpr size_t kOffXs = kOffBi + (size_t)kMaxGroups * kRows * 4;
constexpr size_t kSmemBytes = kOffXs + (size_t)kMaxGroups * 16 * 4 + 1024;  // + alignment slack

// Instruction descriptor, kind::f16: fp16 A and B (K-major), fp32 D, M = 128, N = 16.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(16 >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

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

// Shared-memory matrix descriptor of a K-major operand in the 128-byte swizzled layout
// (8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);  // start address
    d |= (uint64_t)1u << 16;                  // leading byte offset (unused when swizzled)
    d |= (uint64_t)(1024u >> 4) << 32;        // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1u << 46;                  // descriptor version
    d |= (uint64_t)2u << 61;                  // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void mma(uint32_t tmem, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
        ::"r"(tmem), "l"(a), "l"(b), "r"(kIdesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t mb) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mb) : "memory");
}

// byte offset of 16-byte chunk c (0..7) of row r in a 128-byte swizzled K-major tile
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
    const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
}
// bytes 0..3 of w -> fp16 values 0..255 as two half2 (bytes 0, 1 and 2, 3)
__device__ __forceinline__ void bytes_to_half(uint32_t w, uint32_t& h01, uint32_t& h23) {
    h01 = hsub2_u(__byte_perm(w, 0x64646464u, 0x4140), 0x64006400u);
    h23 = hsub2_u(__byte_perm(w, 0x64646464u, 0x4342), 0x64006400u);
}

__device__ __forceinline__ float gelu_tanh(float v) {
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    return 0.5f * v * (1.0f + tanhf(c * (v + 0.044715f * v * v * v)));
}
__device__ __forceinline__ float silu(float v) { return v / (1.0f + expf(-v)); }

__global__ void __launch_bounds__(kThreads, 1) k_gemm16_tc(const __grid_constant__ Gemm16TcArgs a) {
    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
    __shared__ __align__(8) unsigned long long s_full[kRaw], s_done[kAStages];
    __shared__ uint32_t s_tmem;
    __shared__ int s_ok, s_last;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Gemm16Args& g = a.g;
    const int N = g.W.rows, K = g.W.cols, M = g.M;
    const int n0 = blockIdx.x * kRows;
    const int k_beg = blockIdx.y * g.k_per;
    const int ng = min(g.k_per, K - k_beg) / kG;  // groups of this CTA (1..16)
    const int gb = k_beg / kG, spg = K / kG;
    unsigned char* xbuf = sm + kOffX;
    unsigned char* abuf = sm + kOffA;
    unsigned char* raw = sm + kOffRaw;
    float* ssc = reinterpret_cast<float*>(sm + kOffSc);  // [group][row] scales
    float* sbi = reinterpret_cast<float*>(sm + kOffBi);  // [group][row] biases
    float* xsum = reinterpret_cast<float*>(sm + kOffXs); // [group][16] activation sums

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "n"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int s = 0; s < kRaw; ++s) mb_init(smem_u32(&s_full[s]));
        for (int s = 0; s < kAStages; ++s) mb_init(smem_u32(&s_done[s]));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_ok = 1;
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s_tmem;

    // raw code groups into the ring, as far ahead as it holds
    int issued = 0;
    auto issue_raw = [&](int q) {
        const uint32_t mb = smem_u32(&s_full[q % kRaw]);
        mb_expect(mb, kRawBytes);
        tma_2d(smem_u32(raw + (size_t)(q % kRaw) * kRawBytes), &a.wq, k_beg + q * kG, n0, mb);
    };
    if (tid == 0)
        for (; issued < ng && issued < kRaw; ++issued) issue_raw(issued);

    // ---- stage the activations (fp16 hi/lo, swizzled; rows >= M zero), their group sums, and the
    // rows' scales and biases (zero past the matrix)
    for (int i = tid; i < ng * 16 * 8; i += kThreads) {
        const int q = i >> 7, m = (i >> 3) & 15, c = i & 7;  // group, row, 16-byte chunk (8 values)
        float v[8];
        if (m < M) {
            const float4* p = reinterpret_cast<const float4*>(g.x + (size_t)m * g.ldx + k_beg + q * kG + 8 * c);
            const float4 v0 = __ldg(p), v1 = __ldg(p + 1);
            v[0] = v0.x; v[1] = v0.y; v[2] = v0.z; v[3] = v0.w; v[4] = v1.x; v[5] = v1.y; v[6] = v1.z; v[7] = v1.w;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = 0.f;
        }
        uint32_t hi[4], lo[4];
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half h0 = __float2half_rn(v[2 * j]), h1 = __float2half_rn(v[2 * j + 1]);
            const __half2 hh = __halves2half2(h0, h1);
            const __half2 ll = __floats2half2_rn(v[2 * j] - __half2float(h0), v[2 * j + 1] - __half2float(h1));
            hi[j] = *reinterpret_cast<const uint32_t*>(&hh);
            lo[j] = *reinterpret_cast<const uint32_t*>(&ll);
            s += v[2 * j] + v[2 * j + 1];
        }
        unsigned char* xg = xbuf + (size_t)q * 2 * kXBytes;
        *reinterpret_cast<uint4*>(xg + swz(m, c)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(xg + kXBytes + swz(m, c)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        // the 8 chunks of (group, row) are lanes 8k..8k+7 of a warp: their sum, in a fixed order
#pragma unroll
        for (int o = 4; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (c == 0) xsum[q * 16 + m] = s;
    }
    for (int i = tid; i < ng * kRows; i += kThreads) {
        const int q = i / kRows, r = i - q * kRows, n = n0 + r;
        float sv = 0.f, bv = 0.f;
        if (n < N) {
            const __half2 sb = __ldg(reinterpret_cast<const __half2*>(g.W.s) + (size_t)n * spg + gb + q);
            sv = __low2float(sb);
            bv = __high2float(sb);
        }
        ssc[q * kRows + r] = sv;
        sbi[q * kRows + r] = bv;
    }

    // ---- K loop: convert group q, then its MMAs (issued by thread 0)
    bool ok = true;
    int qstop = ng;  // groups whose MMAs were issued
    for (int q = 0; q < ng && ok; ++q) {
        const int slot = q % kRaw, st = q % kAStages;
        // the raw group has landed, and the MMAs that read this A buffer kAStages groups ago are done
        bool w = mb_wait(smem_u32(&s_full[slot]), (uint32_t)((q / kRaw) & 1), a.budget);
        if (w && q >= kAStages)
            w = mb_wait(smem_u32(&s_done[st]), (uint32_t)(((q - kAStages) / kAStages) & 1), a.budget);
        if (!__syncthreads_and(w)) {
            ok = false;
            qstop = q;
            break;
        }
        const unsigned char* rg = raw + (size_t)slot * kRawBytes;
        unsigned char* ab = abuf + (size_t)st * kABytes;
        // 128 rows x 8 chunks of 8 codes: chunk (r, c) = raw bytes r*64 + 8c .. +7
        for (int i = tid; i < kRows * 8; i += kThreads) {
            const int r = i >> 3, c = i & 7;
            const uint2 w8 = *reinterpret_cast<const uint2*>(rg + r * kG + 8 * c);
            uint32_t h[4];
            bytes_to_half(w8.x, h[0], h[1]);
            bytes_to_half(w8.y, h[2], h[3]);
            *reinterpret_cast<uint4*>(ab + swz(r, c)) = make_uint4(h[0], h[1], h[2], h[3]);
        }
        // this thread's shared-memory writes -> the tensor cores' reads (async proxy)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (tid == 0) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t a0 = smem_u32(ab), xh = smem_u32(xbuf + (size_t)q * 2 * kXBytes), xl = xh + kXBytes;
            const uint32_t d = tmem + (uint32_t)(q * 16);
#pragma unroll
            for (int kk = 0; kk < kG / 16; ++kk) {
                const uint64_t ad = sdesc(a0 + kk * 32);
                mma(d, ad, sdesc(xh + kk * 32), kk > 0 ? 1u : 0u);
                mma(d, ad, sdesc(xl + kk * 32), 1u);
            }
            mma_commit(smem_u32(&s_done[st]));
            // the raw slot was consumed by the conversion above: refill it
            if (issued < ng) issue_raw(issued++);
        }
    }
    // the last group's commit covers every MMA before it
    if (tid == 0) {
        const bool w =
            ok && mb_wait(smem_u32(&s_done[(ng - 1) % kAStages]), (uint32_t)(((ng - 1) / kAStages) & 1), a.budget);
        if (!w) {
            s_ok = 0;
            if (a.err) atomicCAS(a.err, 0, kErrTimeout);
            // bounded drain of this CTA's copies and MMAs still in flight
            for (int q = qstop; q < issued; ++q)
                mb_wait(smem_u32(&s_full[q % kRaw]), (uint32_t)((q / kRaw) & 1), a.budget);
            if (qstop > 0)
                mb_wait(smem_u32(&s_done[(qstop - 1) % kAStages]), (uint32_t)(((qstop - 1) / kAStages) & 1), a.budget);
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    // ---- epilogue: row r = 32 * warp + lane of the tile (TMEM lane r); y[m] = sum over groups of
    // s * D_g[m] + b * xsum_g[m], groups in order
    const int r = warp * 32 + lane, n = n0 + r;
    if (s_ok) {
        float acc[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) acc[m] = 0.f;
        for (int q = 0; q < ng; ++q) {
            uint32_t v[16];
            const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(q * 16);
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
                "%13, %14, %15}, [%16];"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                  "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
                  "=r"(v[15])
                : "r"(taddr));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            const float s = ssc[q * kRows + r], b = sbi[q * kRows + r];
#pragma unroll
            for (int m = 0; m < 16; ++m) acc[m] = fmaf(s, __uint_as_float(v[m]), fmaf(b, xsum[q * 16 + m], acc[m]));
        }
        // partial sums of this split: ws[split][m][n]
        float* ws = g.ws + (size_t)blockIdx.y * 16 * N;
        if (n < N) {
#pragma unroll
            for (int m = 0; m < 16; ++m)
                if (m < M) ws[(size_t)m * N + n] = acc[m];
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
    if (!s_ok) return;  // uniform: the partial sums were not written
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(g.cnt + blockIdx.x, 1) == (int)gridDim.y - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- last CTA of the column tile: the splits in split order, then the epilogue
    const int ncols = min(kRows, N - n0);
    const int outs = g.epi == EPI_SWIGLU ? ncols / 2 : ncols;
    const int S = (int)gridDim.y;
    for (int i = tid; i < M * outs; i += kThreads) {
        const int m = i / outs, jj = i - m * outs;
        auto sum = [&](int col) {
            const float* p = g.ws + (size_t)m * N + col;
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
        if (g.epi == EPI_SWIGLU) {
            const int c = n0 + 2 * jj;  // interleaved rows: c the gate, c + 1 the up projection
            v = silu(sum(c)) * sum(c + 1);
            oc = c >> 1;
        } else {
            oc = n0 + jj;
            v = sum(oc);
            if (g.bias) v += g.bias[oc];
            if (g.epi == EPI_GELU) v = gelu_tanh(v);
        }
        if (g.resid) v += g.resid[(size_t)m * g.ldy + oc];
        g.y[(size_t)m * g.ldy + oc] = v;
    }
    if (tid == 0) g.cnt[blockIdx.x] = 0;
}

struct Plan {
    int k_per = 0, splits = 0, tiles = 0;
};

// One CTA per SM: about one wave of (tile, split) CTAs, K ranges of whole groups, at most 16
Plan plan(int N, int K, int sm_count) {
    Plan p;
    p.tiles = (N + kRows - 1) / kRows;
    const int groups = K / kG;
    const int want = std::max(1, (std::max(sm_count, 1) + p.tiles - 1) / p.tiles);
    int gp = (groups + want - 1) / want;
    gp = std::min(std::max(gp, std::min(groups, 4)), kMaxGroups);  // at least 4 groups per CTA where K allows
    p.k_per = gp * kG;
    p.splits = (groups + gp - 1) / gp;
    return p;
}

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

// The codes of W as a 2-D byte tensor [rows][cols], loaded 64 x 128 at a time (zero fill past the
// last row); encoded once per matrix.
bool code_map(const QMat& W, CUtensorMap* map) {
    static std::mutex mu;
    struct Key {
        const void* q;
        int rows, cols;
        bool operator==(const Key& o) const { return q == o.q && rows == o.rows && cols == o.cols; }
    };
    struct KeyHash {
        size_t operator()(const Key& k) const {
            return std::hash<const void*>()(k.q) ^ ((size_t)k.rows * 1000003u) ^ ((size_t)k.cols << 20);
        }
    };
    static std::unordered_map<Key, CUtensorMap, KeyHash> cache;
    std::lock_guard<std::mutex> lk(mu);
    const Key key{W.q, W.rows, W.cols};
    auto it = cache.find(key);
    if (it != cache.end()) {
        *map = it->second;
        return true;
    }
    EncodeFn enc = encoder();
    if (!enc || (reinterpret_cast<uintptr_t>(W.q) & 15) || W.cols % kG) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)W.cols, (cuuint64_t)W.rows};
    const cuuint64_t strides[1] = {(cuuint64_t)W.cols};
    const cuuint32_t box[2] = {(cuuint32_t)kG, (cuuint32_t)kRows};
    const cuuint32_t estr[2] = {1, 1};
    CUtensorMap m;
    if (enc(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(W.q), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    cache.emplace(key, m);
    *map = m;
    return true;
}

}  // namespace g16tc_detail

size_t gemm16_tc_ws_floats(int N, int K, int sm_count) {
    const g16tc_detail::Plan p = g16tc_detail::plan(N, K, sm_count);
    return (size_t)p.splits * 16 * N;
}

bool gemm16_tc_supported(const QMat& W) { return W.kind == SD_A8G64 && W.cols % g16tc_detail::kG == 0; }

cudaError_t launch_gemm16_tc(Gemm16Args g, int sm_count, int* err, cudaStream_t st) {
    using namespace g16tc_detail;
    const int N = g.W.rows, K = g.W.cols;
    if (!gemm16_tc_supported(g.W) || g.M < 1 || g.M > 16 || N < 1 || K < kG || !g.x || !g.y || !g.ws || !g.cnt)
        return cudaErrorInvalidValue;
    if (g.ldx % 4 || reinterpret_cast<uintptr_t>(g.x) % 16) return cudaErrorInvalidValue;
    if (g.epi == EPI_SWIGLU && (N % 2 || g.bias)) return cudaErrorInvalidValue;
    const Plan p = plan(N, K, sm_count);
    g.k_per = p.k_per;
    Gemm16TcArgs a;
    a.g = g;
    if (!code_map(g.W, &a.wq)) return cudaErrorInvalidValue;
    static const long long budget = [] {
        int dev = 0, khz = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev);
        return (long long)(khz > 0 ? khz : 2000000) * 200;  // 200 ms per wait
    }();
    a.budget = budget;
    a.err = err;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm16_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    k_gemm16_tc<<<dim3(p.tiles, p.splits), kThreads, kSmemBytes, st>>>(a);
    return cudaGetLastError();
}

}  // namespace sd
