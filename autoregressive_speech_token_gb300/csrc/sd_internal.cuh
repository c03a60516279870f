// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sd.h"

namespace sd {

// Programmatic dependent launch: a kernel lets its successor launch as soon as
// all of its CTAs are running, and waits for its predecessor's results before
// its first dependent read.  Both are no-ops when launched without the
// attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch with the programmatic-serialization attribute (set when use_pdl()).
bool use_pdl();
void set_pdl_default(bool on);  // this thread's default when SD_PDL is unset
template <typename Kern, typename... Args>
cudaError_t launch_k(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = use_pdl() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

constexpr int kMaxRows = SD_MAX_ROWS;
constexpr int kMaxCodebooks = SD_MAX_CODEBOOKS;

// Device copy of a quantised matrix in the repacked layout:
//   Q8_0 : q = int8 [rows][cols],   s = __half  [rows][cols/32]
//   Q4_0 : q = bytes [rows][cols/2] (16-byte block of nibbles, element j low /
//          j+16 high nibble of byte j), s = __half [rows][cols/32]
//   Q5_0 : q = low nibbles as Q4_0, s = uint2 [rows][cols/32] = (fp16 d in the
//          low half of x, fifth bits in y: bit j = element j of the block)
//   A8G64: q = uint8 [rows][cols],  s = __half2 [rows][cols/64] = (scale, bias)
//   A4G32 / A4G64: q = nibbles as Q4_0 (unsigned codes), s = __half2
//          [rows][cols/g] = (scale, bias)
struct QMat {
    int kind = 0;
    int rows = 0, cols = 0;
    const uint8_t* q = nullptr;
    const void* s = nullptr;
};

__host__ __device__ inline bool q_valid(int k) { return k >= SD_Q8_0 && k <= SD_A4G64; }
__host__ __device__ inline bool q_affine(int k) { return k == SD_A8G64 || k == SD_A4G32 || k == SD_A4G64; }
__host__ __device__ inline bool q_nibbles(int k) { return k == SD_Q4_0 || k == SD_Q5_0 || k == SD_A4G32 || k == SD_A4G64; }
__host__ __device__ inline int q_group(int k) { return (k == SD_A8G64 || k == SD_A4G64) ? 64 : 32; }
// device layout: bytes of the code array, and side bytes (scale, scale+bias, scale+fifth bits) per group
__host__ __device__ inline size_t q_code_bytes(int k, size_t rows, size_t cols) {
    return q_nibbles(k) ? rows * cols / 2 : rows * cols;
}
__host__ __device__ inline int q_side_bytes(int k) { return q_affine(k) ? 4 : k == SD_Q5_0 ? 8 : 2; }
// bytes of one canonical blob tensor
__host__ __device__ inline size_t q_canon_bytes(int k, size_t rows, size_t cols) {
    if (k == SD_Q8_0) return rows * (cols / 32) * 34;
    if (k == SD_Q4_0) return rows * (cols / 32) * 18;
    if (k == SD_Q5_0) return rows * (cols / 32) * 22;
    return q_code_bytes(k, rows, cols) + rows * (cols / q_group(k)) * 4;
}

#ifdef __CUDACC__
// Element (r, k) of a repacked matrix: the bit-exact definition of each format.
__device__ __forceinline__ float q_value(const QMat& W, size_t r, int k) {
    const int K = W.cols, g = q_group(W.kind);
    if (W.kind == SD_Q8_0)
        return __half2float(reinterpret_cast<const __half*>(W.s)[r * (K / 32) + k / 32]) * (float)(int8_t)W.q[r * K + k];
    if (W.kind == SD_A8G64) {
        const __half2 sb = reinterpret_cast<const __half2*>(W.s)[r * (K / 64) + k / 64];
        return __fmaf_rn(__low2float(sb), (float)W.q[r * K + k], __high2float(sb));
    }
    const uint8_t byte = W.q[r * (K / 2) + (k / 32) * 16 + (k & 15)];
    const int nib = (k & 31) < 16 ? (byte & 0xF) : (byte >> 4);
    if (W.kind == SD_Q4_0)
        return __half2float(reinterpret_cast<const __half*>(W.s)[r * (K / 32) + k / 32]) * (float)(nib - 8);
    if (W.kind == SD_Q5_0) {
        const uint2 side = reinterpret_cast<const uint2*>(W.s)[r * (K / 32) + k / 32];
        const int code = nib | (int)(((side.y >> (k & 31)) & 1u) << 4);
        return __half2float(__ushort_as_half((unsigned short)(side.x & 0xFFFFu))) * (float)(code - 16);
    }
    const __half2 sb = reinterpret_cast<const __half2*>(W.s)[r * (K / g) + k / g];
    return __fmaf_rn(__low2float(sb), (float)nib, __high2float(sb));
}
#endif

enum Prologue : int { PRO_NONE = 0, PRO_LN = 1, PRO_RMS = 2 };
enum Epilogue : int { EPI_LINEAR = 0, EPI_GELU = 1, EPI_SWIGLU = 2 };

// Split-KV partial record: o[hd] (unnormalised), then m (running max) and l
// (sum of exp) -- stride hd + 4 floats.
__host__ __device__ inline int part_stride(int hd) { return hd + 4; }

struct GemvArgs {
    QMat W;
    int nb = 1;                    // activation rows (1 or 2)
    const float* x = nullptr;      // [nb][x_stride] input
    int x_stride = 0;
    int pro = PRO_NONE;
    const float* ng = nullptr;     // norm gain   (PRO_LN / PRO_RMS)
    const float* nbias = nullptr;  // norm offset (PRO_LN)
    float eps = 1e-5f;
    int epi = EPI_LINEAR;
    const float* bias = nullptr;   // [rows] (or [rows/2] after SwiGLU) -- optional
    const float* resid = nullptr;  // [nb][y_stride] added after bias -- optional, may alias y
    float* y = nullptr;            // [nb][y_stride]
    int y_stride = 0;
};

struct AttnArgs {
    const float* q = nullptr;      // query of row b, head h at q[b*q_stride + h*hd]
    int q_stride = 0;
    const float* knew = nullptr;   // new key   of row b, kv head g at knew[b*q_stride + g*hd] (nullable)
    const float* vnew = nullptr;   // new value (same layout); appended at position `pos`
    __half* kc = nullptr;          // cache [B][kv_rows][n_ctx][hd], row b, kv head g of this layer at
    __half* vc = nullptr;          //   ((b*row_heads + head_off + g) * n_ctx) * hd
    int row_heads = 0;             // kv heads per row in the cache (layers * Hkv)
    int head_off = 0;              // layer * Hkv
    int n_head = 0, n_kv = 0, hd = 0, n_ctx = 0, nsplit = 0;
    const int* pos_ptr = nullptr;  // device: attend to positions [0, *pos_ptr + pos_add]
    int pos_add = 0;
    int max_len = 0;               // upper bound of *pos_ptr + pos_add + 1 (0: n_ctx); sizes the staging
    const float* rope_cos = nullptr;  // [n_ctx][hd/2] or null (no RoPE)
    const float* rope_sin = nullptr;
    float* part = nullptr;         // [B][n_head][nsplit][hd+4] scratch
    int* counters = nullptr;       // [B][n_kv] zero between launches (the last CTA resets its entry)
    float* out = nullptr;          // o of row b, head h at out[b*out_stride + h*hd]
    int out_stride = 0;
    int* err = nullptr;
};

struct SampParams {
    float temperature;
    int32_t top_k;
    float top_p;
    int32_t greedy;
    float rep_penalty;  // applied to the logits of the tokens in the sampler's history mask (1: none)
};

struct SampleArgs {
    const float* logits = nullptr;  // row b at logits + b*ld
    int ld = 0;
    int V = 0;
    const SampParams* sp = nullptr;  // device
    // draw of row b: (*u_seq)[(*step_idx) * rows + b] when *u_seq is set, else u[b*u_stride + u_off]
    const float* u = nullptr;
    const float* const* u_seq = nullptr;  // device pointer to a device pointer (may hold null)
    const int* step_idx = nullptr;
    int u_stride = 1, u_off = 0;
    int32_t* out = nullptr;                 // out[b*out_stride + out_off]
    int out_stride = 1, out_off = 0;
    int32_t* const* out_seq = nullptr;      // if *out_seq: (*out_seq)[(*step_idx) * rows + b] = token
    int* err = nullptr;
    const uint8_t* seen = nullptr;          // history mask of row b at seen[b*seen_ld .. + V), or null
    int seen_ld = 0;
};

// ------------------------------------------------------------------ launchers
// (implemented in the kernels' translation units; all enqueue on `st`)
cudaError_t launch_gemv(const GemvArgs& a, int sm_count, cudaStream_t st);
cudaError_t launch_gemv_q8(const GemvArgs& a, int sm_count, cudaStream_t st);
cudaError_t launch_gemv_q4(const GemvArgs& a, int sm_count, cudaStream_t st);
cudaError_t launch_gemv_a8(const GemvArgs& a, int sm_count, cudaStream_t st);
cudaError_t launch_gemv_q5(const GemvArgs& a, int sm_count, cudaStream_t st);
cudaError_t launch_gemv_a4(const GemvArgs& a, int sm_count, cudaStream_t st);
cudaError_t launch_attention(const AttnArgs& a, int B, cudaStream_t st);
size_t attention_smem_bytes(const AttnArgs& a);
cudaError_t launch_sample(const SampleArgs& a, int rows, cudaStream_t st);

// Sampler ladder (op level): CFG combine -> repetition penalty -> temperature
// -> min_p -> top-p -> top-k -> draw, one CTA per row, V <= 8192.
struct LadderParams {
    float cfg_weight = 0.f, rep_penalty = 1.f, temperature = 1.f, min_p = 0.f, top_p = 1.f;
    int top_k = 0;
};
size_t sample_ladder_smem_bytes(int V);
cudaError_t launch_sample_ladder(const float* zc, const float* zu, int rows, int V, const LadderParams& p,
                                 const uint8_t* seen, const float* u, int32_t* out, cudaStream_t st);
// One decode step's token for a conditional (row 0) / unconditional (row 1) pair: the step's
// input token consumed[0] joins the history mask `seen` [V] (unless *prompt_on), then the ladder
// on logits rows 0 and 1 (row stride ld) with row 0's draw (u1[0], or (*u_seq)[*step_idx * rows]);
// the token goes to tok[0..rows) and the output sequence.
cudaError_t launch_ladder_step(const float* logits, int ld, int rows, int V, const LadderParams& p, uint8_t* seen,
                               const int* prompt_on, const int32_t* consumed, const float* u1,
                               const float* const* u_seq, const int* step_idx, float* u_slot, int32_t* t_slot,
                               int32_t* tok, int32_t* const* out_seq, int* err, cudaStream_t st);
size_t sample_smem_bytes(int V);

cudaError_t launch_repack(int kind, const uint8_t* canon, int rows, int cols, int swiglu_ff, uint8_t* q,
                          void* s, cudaStream_t st);
cudaError_t launch_dequant(const QMat& W, float* out, cudaStream_t st);

struct EmbedArgs {
    const float* table = nullptr;     // [V][d]
    const float* pos_table = nullptr; // [n_ctx][d] learned positions or null
    const int* pos_ptr = nullptr;
    const int32_t* tok = nullptr;     // token of row b at tok[b*tok_stride + tok_off]
    int tok_stride = 1, tok_off = 0;
    const int32_t* prompt = nullptr;  // if non-null and *prompt_on: token = prompt[b*prompt_ld + pos]
    const int* prompt_on = nullptr;
    int prompt_ld = 0;
    int d = 0, V = 0, n_ctx = 0;
    float* x = nullptr;               // [B][d]
    int* err = nullptr;
};
cudaError_t launch_embed(const EmbedArgs& a, int B, cudaStream_t st);

// e[b] = sum_j E_j[codes[b*16 + j]] for j < ncb (double accumulation).
struct EmbedSumArgs {
    const float* tables[kMaxCodebooks] = {};
    int vocab[kMaxCodebooks] = {};
    int ncb = 0, d = 0;
    const int32_t* codes = nullptr;   // [B][16]
    float* e = nullptr;               // [B][d]
    int* err = nullptr;
    uint8_t* seen0 = nullptr;         // if set: seen0[b*vocab[0] + code 0 of row b] = 1 (the Talker's history)
};
cudaError_t launch_embed_sum(const EmbedSumArgs& a, int B, cudaStream_t st);

// x[b] = table[code(b)] with code(b) = force_on && *force_on ? force[b*16+j] : codes[b*16+j]
struct EmbedCodeArgs {
    const float* table = nullptr;
    int V = 0, d = 0, j = 0;
    const int32_t* codes = nullptr;
    const int32_t* force = nullptr;
    const int* force_on = nullptr;
    float* x = nullptr;
    int* err = nullptr;
};
cudaError_t launch_embed_code(const EmbedCodeArgs& a, int B, cudaStream_t st);

// Persistent decode step (k_step.cu): per-layer weights and buffers.
struct StepLayer {
    const float *n1g = nullptr, *n1b = nullptr, *bqkv = nullptr, *bo = nullptr;
    const float *n2g = nullptr, *n2b = nullptr, *bfc = nullptr, *bproj = nullptr;
    QMat wqkv, wo, wfc, wproj;
};
struct StepArgs {
    int gpt2 = 1, n_layer = 0, d = 0, H = 0, Hkv = 0, hd = 0, ff = 0, V = 0, n_ctx = 0, B = 1, quant = 0;
    int V_in = 0;                        // rows of the input embedding table (vocab + prompt-vector rows)
    float eps = 1e-5f;
    const StepLayer* layers = nullptr;   // device array [n_layer]
    QMat head;
    const float *nfg = nullptr, *nfb = nullptr, *wte = nullptr, *wpe = nullptr;
    const float *rope_cos = nullptr, *rope_sin = nullptr;
    __half *kc = nullptr, *vc = nullptr;
    // flag-carrying exchange buffers: one 64-bit word per value, (epoch << 32) | float bits
    unsigned long long *ll_xa = nullptr;    // [B][d]   residual stream after the O projection
    unsigned long long *ll_xb = nullptr;    // [B][d]   residual stream after the down projection
    unsigned long long *ll_qkv = nullptr;   // [B][qkv_rows]
    unsigned long long *ll_part = nullptr;  // [B][H][max_split][hd + 2] attention partials (o, m, l)
    unsigned long long *ll_u = nullptr;     // [B][ff]  FFN activations
    unsigned long long *ll_logits = nullptr;// [B][V]
    unsigned long long *ll_tok = nullptr;   // [B]      sampled token (as float bits)
    unsigned* gen = nullptr;             // epoch generation: steps run by earlier launches
    float* logits = nullptr;             // [B][V] plain copy of the last step's logits
    int* pos = nullptr;                  // advanced by n_steps at the end
    int32_t* tok = nullptr;              // [B] input token, overwritten with the sampled one
    const float* u1 = nullptr;           // [B] draws when u_seq is null
    const float* u_seq = nullptr;        // [n_steps][B] draws, or null
    int32_t* out_seq = nullptr;          // [n_steps][B] sampled tokens, or null
    const SampParams* sp = nullptr;
    int* err = nullptr;
    int n_steps = 1;
    long long spin_budget = 0;           // clock64 cycles per wait
    int w_evict_first = 1;               // weight copies with the L2 evict-first policy
    // test hook (0: off): in the launch's first step, CTA 0's first-layer wait for the O
    // projection's output words looks for an epoch no producer writes, for this many cycles
    long long test_budget = 0;
    int ring_bytes = 0;                  // shared-memory weight ring
    int act_bytes = 0;                   // shared-memory activation / attention / sampler region
    int max_split = 1;                   // attention splits per (row, kv head) at most
    int split_len = 128;                 // cached positions per attention split (before the cap)
    unsigned long long* trace = nullptr; // optional [64]: CTA 0 per phase kind: input wait, weight wait, rest (ns); [24..29) QKV sub-phases (ns); [32..37) FC and [40..48) attention sub-steps (cycles)
    // optional publish stamps of the first kTraceSteps steps: [2][kTraceSteps][n_layer][kTracePhases]
    // (latest over CTAs, then earliest over CTAs) of the global time at which a CTA published a phase
    unsigned long long* trace_pub = nullptr;
};
size_t step_smem_bytes(const StepArgs& a);
// grid size the persistent step runs with (0: the configuration does not fit)
// fills a.ring_bytes, a.act_bytes and a.max_split as planned
int step_plan_grid(StepArgs& a, int sm_count);
constexpr int kTraceSteps = 64, kTracePhases = 6;  // phases: layer input, QKV, attention, O, FC, proj
cudaError_t launch_step(const StepArgs& a, int grid, cudaStream_t st);

// Cluster persistent decode step (k_cstep.cu).  The grid is `ncl` thread-block
// clusters of `cs` CTAs; cluster c owns KV heads [c*kpc, (c+1)*kpc) with their
// query heads, FFN activations [c*upc, (c+1)*upc) and, through split-K
// partials, a share of every residual row.  Every matrix of the layer table
// and the head are fragment-major copies (launch_frag_pack): wqkv with each
// cluster's q, k, v rows contiguous (bqkv permuted alike), wo as ncl column
// slabs of ko columns, wproj as ncl column slabs of upc columns, wfc and the
// head as they are.  Norm gains and offsets are in the padded activation
// layout (four zero floats after every 32).
struct CStepArgs {
    int gpt2 = 1, n_layer = 0, d = 0, H = 0, Hkv = 0, hd = 0, ff = 0, V = 0, n_ctx = 0, B = 1, quant = 0;
    int V_in = 0;                        // rows of the input embedding table (vocab + prompt-vector rows)
    float eps = 1e-5f;
    int ncl = 0, cs = 0;                 // clusters, CTAs per cluster
    int hpc = 0, kpc = 0;                // query heads, KV heads per cluster
    int rpc = 0, ko = 0, upc = 0;        // QKV rows, O slab width, FFN activations per cluster
    const StepLayer* layers = nullptr;   // device array [n_layer] (repacked matrices)
    QMat head;
    const float *nfg = nullptr, *nfb = nullptr, *wte = nullptr, *wpe = nullptr;
    const float *rope_cos = nullptr, *rope_sin = nullptr;
    __half *kc = nullptr, *vc = nullptr;
    // exchange words (epoch << 32 | float bits)
    unsigned long long *ll_po = nullptr;     // [ncl][B][d] O-projection partials
    unsigned long long *ll_pp = nullptr;     // [ncl][B][d] down-projection partials
    unsigned long long *ll_logits = nullptr; // [B][V]
    unsigned long long *ll_tok = nullptr;    // [8][32] sampled tokens (8 replicas, one line each)
    unsigned* gen = nullptr;
    float* logits = nullptr;
    int* pos = nullptr;
    int32_t* tok = nullptr;
    const float* u1 = nullptr;
    const float* u_seq = nullptr;
    int32_t* out_seq = nullptr;
    const SampParams* sp = nullptr;
    int* err = nullptr;
    int n_steps = 1;
    long long spin_budget = 0;
    int w_evict_first = 1;               // weight copies with the L2 evict-first policy
    // test hook (0: off): in the launch's first step, cluster 0 rank 0's first-layer wait for
    // the O-projection partials looks for an epoch no producer writes, for this many cycles
    long long test_budget = 0;
    int ring_bytes = 0, act_bytes = 0;
    int kkc = 128;                       // cached keys staged per (row, KV head) item at once
    // byte offsets in the activation region
    int o_x = 0, o_u = 0, o_qkv = 0, o_part = 0, o_wq = 0, o_wp = 0, o_bf = 0, o_red = 0, o_yv = 0, o_stage = 0;
    // optional publish stamps [2][kTraceSteps][n_layer][kCTracePhases] (latest, then earliest CTA)
    unsigned long long* trace_pub = nullptr;
    // optional [kCTraceSub]: CTA 0's clock64 cycles per sub-step, summed over the launch
    unsigned long long* trace = nullptr;
    // optional [kCtaSteps][n_layer][kCTracePhases][grid]: every CTA's publish stamps of the first steps
    unsigned long long* trace_cta = nullptr;
    int trace_gi = 0;                    // the CTA whose sub-steps `trace` accumulates
};
constexpr int kCtaSteps = 4;
constexpr int kCTraceSub = 32;  // sub-steps 28, 29: the sampler CTA's logits gather and sampling
constexpr int kCTracePhases = 8;  // x ready, QKV sent, attention sent, O published, x' sent, u sent, proj published, x'' sent
size_t cstep_smem_bytes(const CStepArgs& a);
// Chooses ncl / cs and fills the layout fields of `a`; returns the grid size,
// or 0 when the configuration does not fit the kernel.
int cstep_plan(CStepArgs& a, int sm_count);
cudaError_t launch_cstep(const CStepArgs& a, cudaStream_t st);
// Fragment-major copy of a Q8_0 or Q4_0 matrix for the cluster step (k_cstep.cu):
// column slabs of slab_cols columns, rows perm[i] (or i) of the source, padded
// to whole 16-row tiles; frag_bytes() is its size.  The cluster step's layer
// table holds such copies as QMat {kind, rows = slabs * tiles * 16, cols =
// slab_cols, q = the copy, s = unused}.
size_t frag_bytes(int quant, int rows, int cols, int slab_cols);
cudaError_t launch_frag_pack(const QMat& src, int slab_cols, const int* perm, uint8_t* out, cudaStream_t st);

// Tensor-core GEMM Y[M][N] = X[M][K] W[N][K]^T over a repacked weight, with
// the GEMV epilogues (bias, GELU, interleaved SwiGLU -> Y[M][N/2], residual).
struct QGemmArgs {
    QMat W;
    int M = 0;
    const float* x = nullptr;      // [M][ldx]
    int ldx = 0;
    int epi = EPI_LINEAR;
    const float* bias = nullptr;   // [N] (linear / GELU only) -- optional
    const float* resid = nullptr;  // [M][ldy] -- optional, may alias y
    float* y = nullptr;            // [M][ldy]
    int ldy = 0;
};
cudaError_t launch_qgemm(const QGemmArgs& a, cudaStream_t st);

// Skinny split-K tensor-core GEMM for M <= 16 rows (the same operation and
// epilogues as QGemm).  x must be 16-byte aligned with ldx a multiple of 4.
// ws holds gemm16_ws_floats(N, K) floats of partial sums; cnt holds
// gemm16_tiles(N) ints, zero before the launch and zero again after it (one
// launch at a time may use a given cnt).
struct Gemm16Args {
    QMat W;
    int M = 0;
    const float* x = nullptr;      // [M][ldx]
    int ldx = 0;
    int epi = EPI_LINEAR;
    const float* bias = nullptr;
    const float* resid = nullptr;  // may alias y
    float* y = nullptr;
    int ldy = 0;
    float* ws = nullptr;
    int* cnt = nullptr;
    int k_per = 0;                 // set by the launcher
};
size_t gemm16_ws_floats(int N, int K, int sm_count);
int gemm16_tiles(int N);
cudaError_t launch_gemm16(Gemm16Args a, int sm_count, cudaStream_t st);

// The same product on tcgen05 for 8-bit affine-group weights (k_gemm16_tc.cu): the
// codes' 2-D tensor map, the skinny-GEMM arguments, the wait budget and error word.
struct alignas(128) Gemm16TcArgs {
    CUtensorMap wq;
    Gemm16Args g;
    long long budget = 0;
    int* err = nullptr;
};
bool gemm16_tc_supported(const QMat& W);
size_t gemm16_tc_ws_floats(int N, int K, int sm_count);
cudaError_t launch_gemm16_tc(Gemm16Args g, int sm_count, int* err, cudaStream_t st);

// Tensor-core (tcgen05) GEMM for prefill: fp16 hi/lo operands loaded by TMA
// through 2-D tensor maps ([rows][K] fp16, K a multiple of 64), three MMAs per
// K step, the QGemm epilogues.
struct alignas(128) TcGemmArgs {
    CUtensorMap xh, xl;          // activations [>= M][K]
    CUtensorMap wh, wl;          // weights [N][K]
    int M = 0, N = 0, K = 0;
    int epi = EPI_LINEAR;
    const float* bias = nullptr;
    const float* resid = nullptr;
    float* y = nullptr;
    int ldy = 0;
    int* err = nullptr;
    long long spin_budget = 0;
};
// 2-D fp16 tensor map [rows][cols] with the GEMM's box (weights: 64 rows, activations: 128 rows)
bool tc_map_fp16(CUtensorMap* map, const void* base, int rows, int cols, bool weights);
size_t tc_smem_bytes();
cudaError_t launch_gemm_tc(const TcGemmArgs& a, cudaStream_t st);
cudaError_t launch_split_rows(const float* x, int ldx, int M, int K, __half* hi, __half* lo, cudaStream_t st);
cudaError_t launch_dequant_split(const QMat& W, __half* hi, __half* lo, cudaStream_t st);

// Prefill helpers: positions p0..p0+np-1 of B rows at once, activation row
// m = b*np + i for position p0 + i.
cudaError_t launch_embed_rows(const float* table, const float* pos_table, const int32_t* tok, int ld, int B, int p0,
                              int np, int d, int V, float* X, int* err, cudaStream_t st);
cudaError_t launch_rownorm(const float* X, int ldx, int M, int d, int ln, const float* g, const float* b, float eps,
                           float* H, cudaStream_t st);
cudaError_t launch_rope_kv(float* QKV, int ld, int B, int p0, int np, int H, int Hkv, int hd, int n_ctx, int row_heads,
                           int head_off, const float* cs, const float* sn, __half* kc, __half* vc, cudaStream_t st);
cudaError_t launch_prefill_attn(const float* QKV, int ld, int B, int p0, int np, int H, int Hkv, int hd, int n_ctx,
                                int row_heads, int head_off, const __half* kc, const __half* vc, float* O, int ldo,
                                cudaStream_t st);

// Message returned by sd_last_error(NULL) on this thread.
void set_last_error(const char* msg);

// *p += add for each listed counter (single thread).
cudaError_t launch_advance(int* a, int add_a, int* b, int add_b, int* c, int set_c, cudaStream_t st);

}  // namespace sd
