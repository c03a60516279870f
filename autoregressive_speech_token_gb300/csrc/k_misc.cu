// Small kernels of the decode step: weight repack and dequantisation,
// embedding gathers (token + learned position, code-embedding sums), and the
// device-side position counter.
#include <cstdlib>

#include "sd_internal.cuh"

namespace sd {
namespace {

// Canonical blob tensor -> device layout (see QMat).  One thread per
// (row, 32- or 64-element block).  With swiglu_ff > 0 the stacked [gate; up]
// rows are interleaved: canonical row r < ff -> 2r, row ff + r -> 2r + 1.
__global__ void k_repack(int kind, const uint8_t* __restrict__ canon, int rows, int cols, int swiglu_ff,
                         uint8_t* __restrict__ q, void* __restrict__ s) {
    const int gs = q_group(kind);
    const int nblk = cols / gs;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)rows * nblk) return;
    const int r = (int)(idx / nblk), blk = (int)(idx % nblk);
    const int dr = swiglu_ff > 0 ? (r < swiglu_ff ? 2 * r : 2 * (r - swiglu_ff) + 1) : r;
    if (kind == SD_Q8_0) {
        const uint8_t* src = canon + ((size_t)r * nblk + blk) * 34;
        uint8_t* dq = q + (size_t)dr * cols + (size_t)blk * 32;
        for (int j = 0; j < 32; ++j) dq[j] = src[2 + j];
        reinterpret_cast<uint16_t*>(s)[(size_t)dr * nblk + blk] = (uint16_t)(src[0] | (src[1] << 8));
    } else if (kind == SD_Q4_0) {
        const uint8_t* src = canon + ((size_t)r * nblk + blk) * 18;
        uint8_t* dq = q + (size_t)dr * (cols / 2) + (size_t)blk * 16;
        for (int j = 0; j < 16; ++j) dq[j] = src[2 + j];
        reinterpret_cast<uint16_t*>(s)[(size_t)dr * nblk + blk] = (uint16_t)(src[0] | (src[1] << 8));
    } else if (kind == SD_Q5_0) {
        const uint8_t* src = canon + ((size_t)r * nblk + blk) * 22;
        uint8_t* dq = q + (size_t)dr * (cols / 2) + (size_t)blk * 16;
        for (int j = 0; j < 16; ++j) dq[j] = src[6 + j];
        const uint32_t qh = (uint32_t)src[2] | ((uint32_t)src[3] << 8) | ((uint32_t)src[4] << 16) | ((uint32_t)src[5] << 24);
        reinterpret_cast<uint2*>(s)[(size_t)dr * nblk + blk] = make_uint2((uint32_t)(src[0] | (src[1] << 8)), qh);
    } else if (kind == SD_A4G32 || kind == SD_A4G64) {
        // canonical: element 2i in the low nibble of byte i; device: per 32-element block, element j
        // in the low and element j+16 in the high nibble of byte j
        const uint8_t* src = canon + (size_t)r * (cols / 2) + (size_t)blk * (gs / 2);
        uint8_t* dq = q + (size_t)dr * (cols / 2) + (size_t)blk * (gs / 2);
        for (int b = 0; b < gs / 32; ++b)
            for (int j = 0; j < 16; ++j) {
                const int e0 = 32 * b + j, e1 = e0 + 16;
                const int c0 = (src[e0 >> 1] >> ((e0 & 1) * 4)) & 0xF, c1 = (src[e1 >> 1] >> ((e1 & 1) * 4)) & 0xF;
                dq[16 * b + j] = (uint8_t)(c0 | (c1 << 4));
            }
        const uint16_t* sc = reinterpret_cast<const uint16_t*>(canon + (size_t)rows * (cols / 2));
        const uint16_t* bi = sc + (size_t)rows * nblk;
        uint16_t* d = reinterpret_cast<uint16_t*>(s) + 2 * ((size_t)dr * nblk + blk);
        d[0] = sc[(size_t)r * nblk + blk];
        d[1] = bi[(size_t)r * nblk + blk];
    } else {
        const uint8_t* src = canon + (size_t)r * cols + (size_t)blk * 64;
        uint8_t* dq = q + (size_t)dr * cols + (size_t)blk * 64;
        for (int j = 0; j < 64; ++j) dq[j] = src[j];
        const uint16_t* sc = reinterpret_cast<const uint16_t*>(canon + (size_t)rows * cols);
        const uint16_t* bi = sc + (size_t)rows * nblk;
        uint16_t* d = reinterpret_cast<uint16_t*>(s) + 2 * ((size_t)dr * nblk + blk);
        d[0] = sc[(size_t)r * nblk + blk];
        d[1] = bi[(size_t)r * nblk + blk];
    }
}

// Bit-exact dequantisation of the device layout (one thread per element).
__global__ void k_dequant(QMat W, float* __restrict__ out) {
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)W.rows * W.cols) return;
    const int r = (int)(idx / W.cols), k = (int)(idx % W.cols);
    out[idx] = q_value(W, (size_t)r, k);
}

__global__ void k_embed(const EmbedArgs a) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x;
    const int pos = *a.pos_ptr;
    int tok;
    if (a.prompt && *a.prompt_on)
        tok = a.prompt[(size_t)b * a.prompt_ld + pos];
    else
        tok = a.tok[(size_t)b * a.tok_stride + a.tok_off];
    if (tok < 0 || tok >= a.V || pos < 0 || pos >= a.n_ctx) {
        if (threadIdx.x == 0 && a.err) atomicExch(a.err, 3);
        tok = 0;
    }
    const float4* e = reinterpret_cast<const float4*>(a.table + (size_t)tok * a.d);
    const float4* p = a.pos_table
                          ? reinterpret_cast<const float4*>(a.pos_table + (size_t)min(max(pos, 0), a.n_ctx - 1) * a.d)
                          : nullptr;
    float4* x = reinterpret_cast<float4*>(a.x + (size_t)b * a.d);
    for (int i = threadIdx.x; i < (a.d >> 2); i += blockDim.x) {
        float4 v = e[i];
        if (p) {
            const float4 q = p[i];
            v.x += q.x; v.y += q.y; v.z += q.z; v.w += q.w;
        }
        x[i] = v;
    }
}

__global__ void k_embed_sum(const EmbedSumArgs a) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x;
    int code[kMaxCodebooks];
    for (int j = 0; j < a.ncb; ++j) {
        int c = a.codes[b * kMaxCodebooks + j];
        if (c < 0 || c >= a.vocab[j]) {
            if (threadIdx.x == 0 && a.err) atomicExch(a.err, 4);
            c = 0;
        }
        code[j] = c;
    }
    if (a.seen0 && threadIdx.x == 0) a.seen0[(size_t)b * a.vocab[0] + code[0]] = 1;
    for (int i = threadIdx.x; i < a.d; i += blockDim.x) {
        double s = 0.0;
        for (int j = 0; j < a.ncb; ++j) s += (double)a.tables[j][(size_t)code[j] * a.d + i];
        a.e[(size_t)b * a.d + i] = (float)s;
    }
}

__global__ void k_embed_code(const EmbedCodeArgs a) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x;
    const bool forced = a.force && a.force_on && *a.force_on;
    int c = forced ? a.force[b * kMaxCodebooks + a.j] : a.codes[b * kMaxCodebooks + a.j];
    if (c < 0 || c >= a.V) {
        if (threadIdx.x == 0 && a.err) atomicExch(a.err, 5);
        c = 0;
    }
    const float4* src = reinterpret_cast<const float4*>(a.table + (size_t)c * a.d);
    float4* dst = reinterpret_cast<float4*>(a.x + (size_t)b * a.d);
    for (int i = threadIdx.x; i < (a.d >> 2); i += blockDim.x) dst[i] = src[i];
}

__global__ void k_advance(int* a, int add_a, int* b, int add_b, int* c, int set_c) {
    pdl_trigger();
    pdl_wait();
    if (a) *a += add_a;
    if (b) *b += add_b;
    if (c) *c = set_c;
}

}  // namespace

cudaError_t launch_gemv(const GemvArgs& a, int sm_count, cudaStream_t st) {
    switch (a.W.kind) {
        case SD_Q8_0: return launch_gemv_q8(a, sm_count, st);
        case SD_Q4_0: return launch_gemv_q4(a, sm_count, st);
        case SD_A8G64: return launch_gemv_a8(a, sm_count, st);
        case SD_Q5_0: return launch_gemv_q5(a, sm_count, st);
        case SD_A4G32:
        case SD_A4G64: return launch_gemv_a4(a, sm_count, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_repack(int kind, const uint8_t* canon, int rows, int cols, int swiglu_ff, uint8_t* q, void* s,
                          cudaStream_t st) {
    if (!q_valid(kind)) return cudaErrorInvalidValue;
    const int gs = q_group(kind);
    const long long n = (long long)rows * (cols / gs);
    const int threads = 256;
    k_repack<<<(unsigned)((n + threads - 1) / threads), threads, 0, st>>>(kind, canon, rows, cols, swiglu_ff, q, s);
    return cudaGetLastError();
}

cudaError_t launch_dequant(const QMat& W, float* out, cudaStream_t st) {
    const long long n = (long long)W.rows * W.cols;
    k_dequant<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(W, out);
    return cudaGetLastError();
}

cudaError_t launch_embed(const EmbedArgs& a, int B, cudaStream_t st) {
    return launch_k(k_embed, dim3(B), dim3(256), 0, st, a);
}

cudaError_t launch_embed_sum(const EmbedSumArgs& a, int B, cudaStream_t st) {
    return launch_k(k_embed_sum, dim3(B), dim3(256), 0, st, a);
}

cudaError_t launch_embed_code(const EmbedCodeArgs& a, int B, cudaStream_t st) {
    return launch_k(k_embed_code, dim3(B), dim3(256), 0, st, a);
}

cudaError_t launch_advance(int* a, int add_a, int* b, int add_b, int* c, int set_c, cudaStream_t st) {
    return launch_k(k_advance, dim3(1), dim3(1), 0, st, a, add_a, b, add_b, c, set_c);
}

// Programmatic dependent launch: SD_PDL=1 / SD_PDL=0 force it on / off;
// otherwise the graph being captured decides (set_pdl_default).  Measured on
// GB300: the Talker + code-predictor frame gains (3.98 vs 4.35 ms per frame at
// one row, 9.86 vs 10.17 ms at sixteen), the GPT-2-Medium Q4_0 step graph
// loses (0.875 vs 0.809 ms).
namespace {
thread_local bool t_pdl_default = false;
}
void set_pdl_default(bool on) { t_pdl_default = on; }
bool use_pdl() {
    static const int env = [] {
        const char* e = getenv("SD_PDL");
        return e && e[0] ? (e[0] == '1' ? 1 : 0) : -1;
    }();
    return env >= 0 ? env == 1 : t_pdl_default;
}

}  // namespace sd
