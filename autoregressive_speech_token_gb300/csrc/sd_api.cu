// Host runtime of libsd.so: context and memory plan, weight-blob reader and
// repack, CUDA-graph capture of the decode step / frame, and the C ABI of
// include/sd.h and include/sd_ops.h.
//
// Structure follows "Chatterbox -> ggml Port: Development Journal", section
// 3.2 (a prompt graph and a step graph sharing one persistent KV cache) and
// "Every Frame Is a Memory Read", section 5.2 (the whole code-predictor frame
// -- fifteen passes, heads, sampling, code-embedding sum -- as one captured
// graph with the random draws as inputs).  Everything that changes from step
// to step (position, tokens, draws, sampler settings) lives in device memory,
// so a captured graph is replayed unchanged; attention reads the position on
// the device and covers only [0, pos] ("Every Frame Is a Memory Read",
// section 5.3: attending over the whole fixed capacity is a loss).
#include <algorithm>
#include <array>
#include <cmath>
#include <cstdarg>
#include <cstddef>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/sd_ops.h"
#include "sd_internal.cuh"

using namespace sd;

namespace {

thread_local std::string g_err = "";

constexpr uint32_t kBlobMagic = 0x31574453u;
constexpr int kEntryBytes = 96;
constexpr int kConfigFields = 22;

struct alignas(16) DevState {
    // device-owned counters
    int32_t pos, cp_pos, step_idx, err;
    // host-written inputs (uploaded per call)
    int32_t prompt_on, force_on, pad0, pad1;
    const float* u_seq;
    int32_t* out_seq;
    SampParams samp[2];
    int32_t tok[kMaxRows];
    float u1[kMaxRows];                 // GPT-2/Llama step draws
    float u[kMaxRows * kMaxCodebooks];  // frame draws [row][codebook]
    int32_t codes_in[kMaxRows * kMaxCodebooks];
    int32_t force[kMaxRows * kMaxCodebooks];
    // device-written outputs
    int32_t codes[kMaxRows * kMaxCodebooks];
};

struct BlobTensor {
    uint32_t kind, rows, cols;
    uint64_t off, nbytes;
};

struct DLayer {
    const float *n1g = nullptr, *n1b = nullptr, *bqkv = nullptr, *bo = nullptr;
    const float *n2g = nullptr, *n2b = nullptr, *bfc = nullptr, *bproj = nullptr;
    QMat wqkv, wo, wfc, wproj;
};

struct DStack {
    bool gpt2 = false;
    int n_layer = 0, d = 0, H = 0, Hkv = 0, hd = 0, ff = 0, n_ctx = 0, nsplit = 1;
    float eps = 1e-5f, theta = 10000.f;
    std::vector<DLayer> L;
    const float *nfg = nullptr, *nfb = nullptr;
    __half *kc = nullptr, *vc = nullptr;
    float *rope_cos = nullptr, *rope_sin = nullptr;
    float *x = nullptr, *qkv = nullptr, *part = nullptr, *u = nullptr, *o = nullptr;
    int* counters = nullptr;
    int qkv_rows() const { return (H + 2 * Hkv) * hd; }
};

enum class Phase { Created, Loaded, Running };

}  // namespace

struct sd_ctx {
    sd_model_config cfg{};
    int device = 0, sm_count = 0, B = 1;
    cudaStream_t stream = nullptr;      // launches
    cudaStream_t cap = nullptr;         // private capture stream
    bool own_stream = false;
    std::string err;
    Phase phase = Phase::Created;
    int host_pos = 0;

    DStack main, cp;
    std::vector<void*> allocs;          // activations, caches, tables
    uint8_t* weights = nullptr;         // weight arena
    int64_t weight_bytes = 0, kv_bytes = 0;
    const float *wte = nullptr, *wpe = nullptr;
    QMat head, cp_proj;
    const float* emb[kMaxCodebooks] = {};
    // the input embedding table (wte, or the Talker's emb[0]) has B * max_ctx extra rows after the
    // vocabulary: sd_prefill_embeds writes row b's prompt vector p to row vocab + b * max_ctx + p
    // and feeds that row's index as the prompt token
    int v_in = 0;
    QMat cp_head[kMaxCodebooks];
    float* logits = nullptr;            // [B][V] or [B][16][Vmax]
    int logits_ld = 0, vmax = 0;
    float* ebuf = nullptr;              // [B][d] code-embedding staging (Qwen)
    float* nrm = nullptr;               // [B][max width] normalised rows (B > 2)
    float* g16_ws = nullptr;            // skinny GEMM partial sums (B > 2)
    int* g16_cnt = nullptr;             // skinny GEMM column-tile counters (zero between launches)
    bool rows_gemm_tc = false;          // SD_ROWS_GEMM=tc: 3-16 rows with affine weights on the tcgen05 skinny GEMM
    bool rows_gemm_mma = false;         // SD_ROWS_GEMM=mma: the 64x64 mma.sync GEMM for > 2 rows instead
    int32_t* prompt = nullptr;          // [B][max_ctx]

    DevState* ds = nullptr;             // device
    DevState* hs = nullptr;             // pinned host mirror
    bool force_pending = false;

    // GEMM prefill of prompt positions 0..n-2 in chunks of pf_rows activation rows (all batch rows)
    bool gemm_prefill = true;
    int pf_chunk = 0;                   // positions per chunk
    float *pf_x = nullptr, *pf_h = nullptr, *pf_qkv = nullptr, *pf_o = nullptr, *pf_u = nullptr;
    // tensor-core (tcgen05) prefill: per layer the four matrices dequantised to fp16 hi/lo with their
    // tensor maps, and the split activations ([rows][K] fp16 hi/lo, maps for K = d, q width, ffn width)
    bool tc_prefill = false;
    long long spin_budget = 0;                      // clock64 cycles a device wait may take (200 ms)
    std::vector<std::array<CUtensorMap, 8>> tc_w;   // [layer]: qkv hi/lo, o hi/lo, fc hi/lo, proj hi/lo
    __half *pf_xh = nullptr, *pf_xl = nullptr;
    CUtensorMap tc_x[3][2];                         // [d | qd | ff][hi | lo]

    cudaGraphExec_t g_step = nullptr, g_body = nullptr, g_frame = nullptr, g_prompt_last = nullptr;
    int kernels_per_step = 0;
    int count_launch = 0;

    // persistent step kernel (GPT-2/Llama): one cooperative launch per step or per decode_n
    bool persistent = false;
    StepArgs step;
    std::string trace_path;             // SD_TRACE: per-phase timings of the persistent step
    StepLayer* step_layers = nullptr;   // device [n_layer]
    int step_grid = 0;
    // cluster persistent step kernel (k_cstep.cu): preferred over the flat one where its plan fits
    bool cpersistent = false;
    bool ladder_on = false;             // sd_set_ladder: one token per step for a cond / uncond row pair
    LadderParams ladder;
    uint8_t* seen = nullptr;            // [vocab] tokens generated since sd_prefill (ladder mode)
    uint8_t* seen0 = nullptr;           // [B][vocab] codebook-0 tokens fed to the Talker since sd_prefill
    float* lad_u = nullptr;             // the ladder's draw slot
    int32_t* lad_t = nullptr;           // the ladder's token slot
    int32_t* lad_in = nullptr;          // the guided step's input token, kept across the persistent launch
    long long test_stall = 0;           // test hook (SD_TEST_STALL_US): cycles for one wait of the next persistent launch
    CStepArgs cstep;
};

namespace {

int fail(sd_ctx* c, int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (c) c->err = buf;
    g_err = buf;
    return code;
}

#define CK(call)                                                                                   \
    do {                                                                                           \
        cudaError_t e_ = (call);                                                                   \
        if (e_ != cudaSuccess) return fail(c, SD_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
    } while (0)

template <typename T>
int dalloc(sd_ctx* c, T** p, size_t bytes) {
    void* q = nullptr;
    cudaError_t e = cudaMalloc(&q, bytes ? bytes : 16);
    if (e != cudaSuccess) return fail(c, SD_ERR_OOM, "cudaMalloc(%zu): %s", bytes, cudaGetErrorString(e));
    CK(cudaMemset(q, 0, bytes ? bytes : 16));
    c->allocs.push_back(q);
    *p = reinterpret_cast<T*>(q);
    return SD_OK;
}

int validate_cfg(const sd_model_config& m) {
    if (m.arch < SD_ARCH_GPT2 || m.arch > SD_ARCH_QWEN_TTS) return 0;
    if (!q_valid(m.quant)) return 0;
    if (m.n_layer < 0 || m.d_model <= 0 || m.n_head <= 0 || m.n_kv_head <= 0 || m.head_dim <= 0) return 0;
    if (m.head_dim != 64 && m.head_dim != 128) return 0;
    if (m.n_head % m.n_kv_head || m.n_head / m.n_kv_head > 4) return 0;
    if (m.d_ff <= 0 || m.vocab <= 0 || m.vocab > 16384 || m.max_ctx <= 0 || m.batch < 1 || m.batch > kMaxRows) return 0;
    const int gs = q_group(m.quant);
    if (m.d_model % gs || m.d_ff % gs || (m.n_head * m.head_dim) % gs) return 0;
    if (m.d_model > 8192 || m.d_ff > 8192) return 0;
    if (m.arch == SD_ARCH_GPT2 && m.n_head != m.n_kv_head) return 0;
    if (m.arch == SD_ARCH_QWEN_TTS) {
        if (m.n_codebooks < 2 || m.n_codebooks > kMaxCodebooks || m.cp_layer < 0 || m.cp_d_model <= 0) return 0;
        if (m.cp_head_dim != 64 && m.cp_head_dim != 128) return 0;
        if (m.cp_n_kv_head <= 0 || m.cp_n_head % m.cp_n_kv_head || m.cp_n_head / m.cp_n_kv_head > 4) return 0;
        if (m.cp_vocab <= 0 || m.cp_vocab > 16384 || m.cp_max_ctx < m.n_codebooks) return 0;
        if (m.cp_d_model % gs || m.cp_d_ff % gs) return 0;
    }
    return 1;
}

void init_stack(DStack& s, bool gpt2, int n_layer, int d, int H, int Hkv, int hd, int ff, int n_ctx, float eps,
                float theta) {
    s.gpt2 = gpt2;
    s.n_layer = n_layer; s.d = d; s.H = H; s.Hkv = Hkv; s.hd = hd; s.ff = ff; s.n_ctx = n_ctx;
    s.eps = eps; s.theta = theta;
    // split-KV chunks: enough CTAs for the grid at typical lengths, never more than the capacity needs
    s.nsplit = n_ctx >= 256 ? 8 : (n_ctx >= 64 ? 4 : 1);

}

int alloc_stack(sd_ctx* c, DStack& s) {
    const int B = c->B;
    const size_t kv = (size_t)B * s.n_layer * s.Hkv * s.n_ctx * s.hd;
    int rc;
    if ((rc = dalloc(c, &s.kc, kv * 2)) || (rc = dalloc(c, &s.vc, kv * 2))) return rc;
    c->kv_bytes += (int64_t)kv * 4;
    const int wide = std::max(s.qkv_rows(), 2 * s.ff);
    if ((rc = dalloc(c, &s.x, sizeof(float) * B * s.d)) || (rc = dalloc(c, &s.qkv, sizeof(float) * B * wide)) ||
        (rc = dalloc(c, &s.part, sizeof(float) * B * s.H * s.nsplit * part_stride(s.hd))) ||
        (rc = dalloc(c, &s.o, sizeof(float) * B * s.H * s.hd)) || (rc = dalloc(c, &s.counters, sizeof(int) * B * s.Hkv)) ||
        (rc = dalloc(c, &s.u, sizeof(float) * B * std::max(s.ff, s.d))))
        return rc;
    if (!s.gpt2) {
        // NEOX RoPE table in double, rounded to fp32: theta_i = base^(-2i/hd), phi = pos * theta_i
        const int half = s.hd / 2;
        std::vector<float> cs((size_t)s.n_ctx * half), sn((size_t)s.n_ctx * half);
        for (int p = 0; p < s.n_ctx; ++p)
            for (int i = 0; i < half; ++i) {
                const double phi = (double)p * std::pow((double)s.theta, -2.0 * i / s.hd);
                cs[(size_t)p * half + i] = (float)std::cos(phi);
                sn[(size_t)p * half + i] = (float)std::sin(phi);
            }
        if ((rc = dalloc(c, &s.rope_cos, cs.size() * 4)) || (rc = dalloc(c, &s.rope_sin, sn.size() * 4))) return rc;
        CK(cudaMemcpy(s.rope_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice));
        CK(cudaMemcpy(s.rope_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice));
    }
    return SD_OK;
}

// ------------------------------------------------------------------ enqueue helpers

// y = W x for the context's rows: the streaming GEMV for 1-2 rows; for more
// rows (G rollouts, at most 16) the norm prologue as its own kernel and the
// skinny split-K tensor-core GEMM with the same epilogue.
int gemv(sd_ctx* c, const GemvArgs& a, cudaStream_t st) {
    cudaError_t e;
    if (a.nb <= 2) {
        e = launch_gemv(a, c->sm_count, st);
        c->count_launch++;
    } else {
        const float* x = a.x;
        int ldx = a.x_stride;
        if (a.pro != PRO_NONE) {
            e = launch_rownorm(a.x, a.x_stride, a.nb, a.W.cols, a.pro == PRO_LN, a.ng, a.nbias, a.eps, c->nrm, st);
            c->count_launch++;
            if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "row norm launch: %s", cudaGetErrorString(e));
            x = c->nrm;
            ldx = a.W.cols;
        }
        const bool skinny_ok = a.W.kind == SD_Q8_0 || a.W.kind == SD_Q4_0 || a.W.kind == SD_A8G64;
        if (!skinny_ok) {
            // formats the row GEMMs do not take: the matvec over pairs of rows (one weight read per pair)
            e = cudaSuccess;
            for (int r0 = 0; r0 < a.nb && e == cudaSuccess; r0 += 2) {
                GemvArgs p = a;
                p.pro = PRO_NONE;
                p.nb = std::min(2, a.nb - r0);
                p.x = x + (size_t)r0 * ldx;
                p.x_stride = ldx;
                p.y = a.y + (size_t)r0 * a.y_stride;
                p.resid = a.resid ? a.resid + (size_t)r0 * a.y_stride : nullptr;
                e = launch_gemv(p, c->sm_count, st);
                c->count_launch++;
            }
            c->count_launch--;
        } else if (c->rows_gemm_mma) {
            QGemmArgs g;
            g.W = a.W; g.M = a.nb; g.x = x; g.ldx = ldx; g.epi = a.epi; g.bias = a.bias; g.resid = a.resid;
            g.y = a.y; g.ldy = a.y_stride;
            e = launch_qgemm(g, st);
        } else {
            Gemm16Args g;
            g.W = a.W; g.M = a.nb; g.x = x; g.ldx = ldx; g.epi = a.epi; g.bias = a.bias; g.resid = a.resid;
            g.y = a.y; g.ldy = a.y_stride; g.ws = c->g16_ws; g.cnt = c->g16_cnt;
            e = (c->rows_gemm_tc && gemm16_tc_supported(a.W)) ? launch_gemm16_tc(g, c->sm_count, &c->ds->err, st)
                                                               : launch_gemm16(g, c->sm_count, st);
        }
        c->count_launch++;
    }
    if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "gemv launch: %s", cudaGetErrorString(e));
    return SD_OK;
}

// One transformer position through every layer of stack s (input already in s.x).
int enqueue_layers(sd_ctx* c, DStack& s, const int* pos_ptr, cudaStream_t st) {
    const int B = c->B, d = s.d, qd = s.H * s.hd, kd = s.Hkv * s.hd, qr = s.qkv_rows();
    int rc;
    for (int l = 0; l < s.n_layer; ++l) {
        DLayer& L = s.L[l];
        GemvArgs g;
        g.W = L.wqkv; g.nb = B; g.x = s.x; g.x_stride = d;
        g.pro = s.gpt2 ? PRO_LN : PRO_RMS; g.ng = L.n1g; g.nbias = L.n1b; g.eps = s.eps;
        g.epi = EPI_LINEAR; g.bias = L.bqkv; g.y = s.qkv; g.y_stride = qr;
        if ((rc = gemv(c, g, st))) return rc;

        AttnArgs a;
        a.q = s.qkv; a.q_stride = qr; a.knew = s.qkv + qd; a.vnew = s.qkv + qd + kd;
        a.kc = s.kc; a.vc = s.vc; a.row_heads = s.n_layer * s.Hkv; a.head_off = l * s.Hkv;
        a.n_head = s.H; a.n_kv = s.Hkv; a.hd = s.hd; a.n_ctx = s.n_ctx; a.nsplit = s.nsplit;
        a.pos_ptr = pos_ptr; a.rope_cos = s.rope_cos; a.rope_sin = s.rope_sin; a.part = s.part;
        a.counters = s.counters; a.out = s.o; a.out_stride = qd;
        a.err = &c->ds->err;
        cudaError_t e = launch_attention(a, B, st);
        c->count_launch++;
        if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "attention launch: %s", cudaGetErrorString(e));

        GemvArgs o;
        o.W = L.wo; o.nb = B; o.x = s.o; o.x_stride = qd; o.pro = PRO_NONE;
        o.epi = EPI_LINEAR; o.bias = L.bo; o.resid = s.x; o.y = s.x; o.y_stride = d;
        if ((rc = gemv(c, o, st))) return rc;

        GemvArgs f;
        f.W = L.wfc; f.nb = B; f.x = s.x; f.x_stride = d;
        f.pro = s.gpt2 ? PRO_LN : PRO_RMS; f.ng = L.n2g; f.nbias = L.n2b; f.eps = s.eps;
        f.epi = s.gpt2 ? EPI_GELU : EPI_SWIGLU; f.bias = L.bfc; f.y = s.u; f.y_stride = s.ff;
        if ((rc = gemv(c, f, st))) return rc;

        GemvArgs p;
        p.W = L.wproj; p.nb = B; p.x = s.u; p.x_stride = s.ff; p.pro = PRO_NONE;
        p.epi = EPI_LINEAR; p.bias = L.bproj; p.resid = s.x; p.y = s.x; p.y_stride = d;
        if ((rc = gemv(c, p, st))) return rc;
    }
    return SD_OK;
}

// logits = head(final_norm(s.x)) written to c->logits + slot * vmax
int enqueue_head(sd_ctx* c, DStack& s, const QMat& W, int slot, cudaStream_t st) {
    GemvArgs h;
    h.W = W; h.nb = c->B; h.x = s.x; h.x_stride = s.d;
    h.pro = s.gpt2 ? PRO_LN : PRO_RMS; h.ng = s.nfg; h.nbias = s.nfb; h.eps = s.eps;
    h.epi = EPI_LINEAR; h.y = c->logits + (size_t)slot * c->vmax; h.y_stride = c->logits_ld;
    return gemv(c, h, st);
}

int enqueue_sample(sd_ctx* c, int which, int slot, int V, bool t3, cudaStream_t st) {
    SampleArgs a;
    a.logits = c->logits + (size_t)slot * c->vmax; a.ld = c->logits_ld; a.V = V;
    a.sp = &c->ds->samp[which];
    a.err = &c->ds->err;
    if (t3) {
        a.u = c->ds->u1; a.u_stride = 1; a.u_off = 0;
        a.u_seq = &c->ds->u_seq; a.step_idx = &c->ds->step_idx;
        a.out = c->ds->tok; a.out_stride = 1; a.out_off = 0;
        a.out_seq = &c->ds->out_seq;
    } else {
        a.u = c->ds->u; a.u_stride = kMaxCodebooks; a.u_off = slot;
        a.out = c->ds->codes; a.out_stride = kMaxCodebooks; a.out_off = slot;
        if (which == 0) {  // the Talker's codebook-0 sampler: its history of fed codebook-0 tokens
            a.seen = c->seen0;
            a.seen_ld = c->cfg.vocab;
        }
    }
    cudaError_t e = launch_sample(a, c->B, st);
    c->count_launch++;
    if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "sampler launch: %s", cudaGetErrorString(e));
    return SD_OK;
}

int advance(sd_ctx* c, int* a, int add_a, int* b, int add_b, int* cc, int set_c, cudaStream_t st) {
    cudaError_t e = launch_advance(a, add_a, b, add_b, cc, set_c, st);
    c->count_launch++;
    if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "advance launch: %s", cudaGetErrorString(e));
    return SD_OK;
}

// Input embedding of the main stack at the current position: token table
// (+ learned positions), reading the prompt buffer while prompt_on is set.
int enqueue_embed(sd_ctx* c, cudaStream_t st) {
    EmbedArgs e;
    e.table = c->cfg.arch == SD_ARCH_QWEN_TTS ? c->emb[0] : c->wte;
    e.pos_table = c->wpe; e.pos_ptr = &c->ds->pos; e.tok = c->ds->tok;
    e.prompt = c->prompt; e.prompt_on = &c->ds->prompt_on; e.prompt_ld = c->cfg.max_ctx;
    e.d = c->main.d; e.V = c->v_in; e.n_ctx = c->cfg.max_ctx; e.x = c->main.x; e.err = &c->ds->err;
    cudaError_t err = launch_embed(e, c->B, st);
    c->count_launch++;
    if (err != cudaSuccess) return fail(c, SD_ERR_CUDA, "embed launch: %s", cudaGetErrorString(err));
    return SD_OK;
}

// The code-predictor part of a frame: 16 positions, heads 1..15, samplers.
int enqueue_cp_frame(sd_ctx* c, cudaStream_t st) {
    DStack& t = c->main;
    DStack& p = c->cp;
    const int B = c->B;
    int rc;
    if ((rc = advance(c, nullptr, 0, nullptr, 0, &c->ds->cp_pos, 0, st))) return rc;
    for (int j = 0; j < c->cfg.n_codebooks; ++j) {
        GemvArgs g;
        g.W = c->cp_proj; g.nb = B; g.epi = EPI_LINEAR; g.y = p.x; g.y_stride = p.d;
        if (j == 0) {  // Pr * final_norm(h_T)
            g.x = t.x; g.x_stride = t.d; g.pro = PRO_RMS; g.ng = t.nfg; g.eps = t.eps;
        } else {       // Pr * E_{j-1}[c_{j-1}]
            EmbedCodeArgs ec;
            ec.table = c->emb[j - 1]; ec.V = j - 1 == 0 ? c->cfg.vocab : c->cfg.cp_vocab; ec.d = t.d; ec.j = j - 1;
            ec.codes = c->ds->codes; ec.force = c->ds->force; ec.force_on = &c->ds->force_on; ec.x = c->ebuf;
            ec.err = &c->ds->err;
            cudaError_t e = launch_embed_code(ec, B, st);
            c->count_launch++;
            if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "embed_code launch: %s", cudaGetErrorString(e));
            g.x = c->ebuf; g.x_stride = t.d; g.pro = PRO_NONE;
        }
        if ((rc = gemv(c, g, st))) return rc;
        if ((rc = enqueue_layers(c, p, &c->ds->cp_pos, st))) return rc;
        if (j >= 1) {
            if ((rc = enqueue_head(c, p, c->cp_head[j], j, st))) return rc;
            if ((rc = enqueue_sample(c, 1, j, c->cfg.cp_vocab, false, st))) return rc;
        }
        if ((rc = advance(c, &c->ds->cp_pos, 1, nullptr, 0, nullptr, 0, st))) return rc;
    }
    return SD_OK;
}

// One launch of the cluster step kernel for n_steps steps.
// Test hook: the first persistent launch made outside a stream capture takes the stall budget
// (a captured graph would replay it on every step).
void take_test_stall(sd_ctx* c, cudaStream_t st, long long* budget) {
    *budget = 0;
    if (!c->test_stall) return;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return;
    *budget = c->test_stall;
    c->test_stall = 0;
}

int enqueue_cstep(sd_ctx* c, int n_steps, const float* u_seq, int32_t* out_seq, cudaStream_t st) {
    CStepArgs a = c->cstep;
    a.n_steps = n_steps;
    take_test_stall(c, st, &a.test_budget);
    a.u_seq = u_seq;
    a.out_seq = out_seq;
    if (a.trace) CK(cudaMemsetAsync(a.trace, 0, sizeof(unsigned long long) * kCTraceSub, st));
    if (a.trace_pub) {
        const size_t half = (size_t)kTraceSteps * a.n_layer * kCTracePhases;
        CK(cudaMemsetAsync(a.trace_pub, 0, sizeof(unsigned long long) * half, st));
        CK(cudaMemsetAsync(a.trace_pub + half, 0xFF, sizeof(unsigned long long) * half, st));
    }
    cudaError_t e = launch_cstep(a, st);
    c->count_launch++;
    if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "cluster step launch: %s", cudaGetErrorString(e));
    return SD_OK;
}

// One cooperative launch of the persistent step kernel for n_steps steps.
int enqueue_persistent(sd_ctx* c, int n_steps, const float* u_seq, int32_t* out_seq, cudaStream_t st) {
    if (c->cpersistent) return enqueue_cstep(c, n_steps, u_seq, out_seq, st);
    StepArgs a = c->step;
    a.n_steps = n_steps;
    take_test_stall(c, st, &a.test_budget);
    a.u_seq = u_seq;
    a.out_seq = out_seq;
    if (a.trace) CK(cudaMemsetAsync(a.trace, 0, sizeof(unsigned long long) * 64, st));
    if (a.trace_pub) {
        const size_t half = (size_t)kTraceSteps * a.n_layer * kTracePhases;
        CK(cudaMemsetAsync(a.trace_pub, 0, sizeof(unsigned long long) * half, st));
        CK(cudaMemsetAsync(a.trace_pub + half, 0xFF, sizeof(unsigned long long) * half, st));
    }
    cudaError_t e = launch_step(a, c->step_grid, st);
    c->count_launch++;
    if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "persistent step launch: %s", cudaGetErrorString(e));
    return SD_OK;
}

// Prompt positions [0, n) of the main stack's rows [0, rows) as GEMMs, in
// chunks of pf_chunk positions: embed, then per layer norm -> QKV GEMM ->
// RoPE + fp16 KV store -> causal attention over the cache -> O GEMM (+resid)
// -> norm -> FC / gate-up GEMM -> proj / down GEMM (+resid).  Leaves the KV
// cache filled for positions < n and the device position at n.
int enqueue_prefill_gemm(sd_ctx* c, int n, int rows, cudaStream_t st) {
    DStack& s = c->main;
    const int B = rows, d = s.d, qd = s.H * s.hd, kd = s.Hkv * s.hd, qr = s.qkv_rows();
    const bool qwen = c->cfg.arch == SD_ARCH_QWEN_TTS;
    auto ck = [&](cudaError_t e, const char* what) {
        return e == cudaSuccess ? SD_OK : fail(c, SD_ERR_CUDA, "prefill %s: %s", what, cudaGetErrorString(e));
    };
    // one GEMM: tcgen05 (split the activations, then the tensor-core kernel) or mma.sync
    auto gemm = [&](const QGemmArgs& g, int l, int which, int kslot) -> cudaError_t {
        if (!c->tc_prefill) return launch_qgemm(g, st);
        cudaError_t e = launch_split_rows(g.x, g.ldx, g.M, g.W.cols, c->pf_xh, c->pf_xl, st);
        if (e != cudaSuccess) return e;
        TcGemmArgs t;
        t.xh = c->tc_x[kslot][0]; t.xl = c->tc_x[kslot][1];
        t.wh = c->tc_w[l][2 * which]; t.wl = c->tc_w[l][2 * which + 1];
        t.M = g.M; t.N = g.W.rows; t.K = g.W.cols; t.epi = g.epi; t.bias = g.bias; t.resid = g.resid;
        t.y = g.y; t.ldy = g.ldy; t.err = &c->ds->err; t.spin_budget = c->spin_budget;
        c->count_launch++;
        return launch_gemm_tc(t, st);
    };
    int rc;
    for (int p0 = 0; p0 < n; p0 += c->pf_chunk) {
        const int np = std::min(c->pf_chunk, n - p0), M = B * np;
        if ((rc = ck(launch_embed_rows(qwen ? c->emb[0] : c->wte, c->wpe, c->prompt, c->cfg.max_ctx, B, p0, np, d,
                                       c->v_in, c->pf_x, &c->ds->err, st), "embed")))
            return rc;
        for (int l = 0; l < s.n_layer; ++l) {
            DLayer& L = s.L[l];
            if ((rc = ck(launch_rownorm(c->pf_x, d, M, d, s.gpt2, L.n1g, L.n1b, s.eps, c->pf_h, st), "norm"))) return rc;
            QGemmArgs g;
            g.W = L.wqkv; g.M = M; g.x = c->pf_h; g.ldx = d; g.epi = EPI_LINEAR; g.bias = L.bqkv;
            g.y = c->pf_qkv; g.ldy = qr;
            if ((rc = ck(gemm(g, l, 0, 0), "qkv gemm"))) return rc;
            if ((rc = ck(launch_rope_kv(c->pf_qkv, qr, B, p0, np, s.H, s.Hkv, s.hd, s.n_ctx, s.n_layer * s.Hkv,
                                        l * s.Hkv, s.rope_cos, s.rope_sin, s.kc, s.vc, st), "rope/kv")))
                return rc;
            if ((rc = ck(launch_prefill_attn(c->pf_qkv, qr, B, p0, np, s.H, s.Hkv, s.hd, s.n_ctx, s.n_layer * s.Hkv,
                                             l * s.Hkv, s.kc, s.vc, c->pf_o, qd, st), "attention")))
                return rc;
            QGemmArgs o;
            o.W = L.wo; o.M = M; o.x = c->pf_o; o.ldx = qd; o.epi = EPI_LINEAR; o.bias = L.bo;
            o.resid = c->pf_x; o.y = c->pf_x; o.ldy = d;
            if ((rc = ck(gemm(o, l, 1, 1), "o gemm"))) return rc;
            if ((rc = ck(launch_rownorm(c->pf_x, d, M, d, s.gpt2, L.n2g, L.n2b, s.eps, c->pf_h, st), "norm"))) return rc;
            QGemmArgs f;
            f.W = L.wfc; f.M = M; f.x = c->pf_h; f.ldx = d; f.epi = s.gpt2 ? EPI_GELU : EPI_SWIGLU; f.bias = L.bfc;
            f.y = c->pf_u; f.ldy = s.ff;
            if ((rc = ck(gemm(f, l, 2, 0), "fc gemm"))) return rc;
            QGemmArgs q;
            q.W = L.wproj; q.M = M; q.x = c->pf_u; q.ldx = s.ff; q.epi = EPI_LINEAR; q.bias = L.bproj;
            q.resid = c->pf_x; q.y = c->pf_x; q.ldy = d;
            if ((rc = ck(gemm(q, l, 3, 2), "proj gemm"))) return rc;
            c->count_launch += 8;
        }
        c->count_launch += 1;
        (void)kd;
    }
    return advance(c, &c->ds->pos, n, nullptr, 0, nullptr, 0, st);
}

enum class GraphKind { T3Step, T3Body, QwenFrame, QwenBody, QwenPromptLast };

int enqueue_graph(sd_ctx* c, GraphKind k, cudaStream_t st) {
    int rc;
    if (k == GraphKind::T3Step && c->persistent) {
        if (!c->ladder_on) return enqueue_persistent(c, 1, nullptr, nullptr, st);
        // the guided step: one persistent launch for the layers and the head (its own sampled token
        // is replaced), then the ladder on the two rows' logits; the kernel advanced the position.
        // The step's input token is kept first: the kernel overwrites tok with its own sample.
        CK(cudaMemcpyAsync(c->lad_in, c->ds->tok, sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
        if ((rc = enqueue_persistent(c, 1, nullptr, nullptr, st))) return rc;
        cudaError_t e = launch_ladder_step(c->logits, c->logits_ld, c->B, c->cfg.vocab, c->ladder, c->seen,
                                           &c->ds->prompt_on, c->lad_in, c->ds->u1, &c->ds->u_seq,
                                           &c->ds->step_idx, c->lad_u, c->lad_t, c->ds->tok, &c->ds->out_seq,
                                           &c->ds->err, st);
        c->count_launch += 3;
        if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "ladder launch: %s", cudaGetErrorString(e));
        return advance(c, nullptr, 0, &c->ds->step_idx, 1, nullptr, 0, st);
    }
    const bool qwen = c->cfg.arch == SD_ARCH_QWEN_TTS;
    if (k == GraphKind::QwenFrame) {
        EmbedSumArgs es;
        for (int j = 0; j < c->cfg.n_codebooks; ++j) {
            es.tables[j] = c->emb[j];
            es.vocab[j] = j ? c->cfg.cp_vocab : c->cfg.vocab;
        }
        es.ncb = c->cfg.n_codebooks; es.d = c->main.d; es.codes = c->ds->codes_in; es.e = c->main.x;
        es.err = &c->ds->err;
        es.seen0 = c->seen0;
        cudaError_t e = launch_embed_sum(es, c->B, st);
        c->count_launch++;
        if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "embed_sum launch: %s", cudaGetErrorString(e));
    } else {
        if ((rc = enqueue_embed(c, st))) return rc;
    }
    if ((rc = enqueue_layers(c, c->main, &c->ds->pos, st))) return rc;
    if (k == GraphKind::T3Body || k == GraphKind::QwenBody)
        return advance(c, &c->ds->pos, 1, nullptr, 0, nullptr, 0, st);
    if ((rc = enqueue_head(c, c->main, c->head, 0, st))) return rc;
    if (c->ladder_on && !qwen) {
        cudaError_t e = launch_ladder_step(c->logits, c->logits_ld, c->B, c->cfg.vocab, c->ladder, c->seen,
                                           &c->ds->prompt_on, c->ds->tok, c->ds->u1, &c->ds->u_seq,
                                           &c->ds->step_idx, c->lad_u, c->lad_t, c->ds->tok, &c->ds->out_seq,
                                           &c->ds->err, st);
        c->count_launch += 3;
        if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "ladder launch: %s", cudaGetErrorString(e));
    } else if ((rc = enqueue_sample(c, 0, 0, c->cfg.vocab, !qwen, st))) {
        return rc;
    }
    if (qwen && (rc = enqueue_cp_frame(c, st))) return rc;
    return advance(c, &c->ds->pos, 1, &c->ds->step_idx, 1, nullptr, 0, st);
}

int capture(sd_ctx* c, GraphKind k, cudaGraphExec_t* out, int* n_kernels) {
    cudaGraph_t g = nullptr;
    c->count_launch = 0;
    CK(cudaStreamBeginCapture(c->cap, cudaStreamCaptureModeThreadLocal));
    // programmatic dependent launch inside the Talker + code-predictor graphs (many short
    // kernels whose weight loads can start before their predecessor ends)
    set_pdl_default(c->cfg.arch == SD_ARCH_QWEN_TTS);
    int rc = enqueue_graph(c, k, c->cap);
    set_pdl_default(false);
    cudaError_t e = cudaStreamEndCapture(c->cap, &g);
    if (rc) {
        if (g) cudaGraphDestroy(g);
        return rc;
    }
    if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "end capture: %s", cudaGetErrorString(e));
    e = cudaGraphInstantiate(out, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(e));
    if (n_kernels) *n_kernels = c->count_launch;
    return SD_OK;
}

// ------------------------------------------------------------------ weights

struct Blob {
    std::unordered_map<std::string, BlobTensor> t;
    const uint8_t* base = nullptr;  // device pointer to the blob bytes
};

int find_f32(sd_ctx* c, Blob& b, const std::string& name, int64_t n, uint8_t*& arena, const float** out) {
    auto it = b.t.find(name);
    if (it == b.t.end() || it->second.kind != 0 || (int64_t)it->second.rows * it->second.cols != n)
        return fail(c, SD_ERR_BLOB, "blob: missing or mis-shaped fp32 tensor '%s'", name.c_str());
    CK(cudaMemcpyAsync(arena, b.base + it->second.off, n * 4, cudaMemcpyDeviceToDevice, c->stream));
    *out = reinterpret_cast<const float*>(arena);
    arena += (n * 4 + 255) / 256 * 256;
    return SD_OK;
}

size_t qbytes(int kind, int rows, int cols) {
    const size_t q = q_code_bytes(kind, rows, cols);
    const size_t s = (size_t)rows * (cols / q_group(kind)) * q_side_bytes(kind);
    return (q + 255) / 256 * 256 + (s + 255) / 256 * 256;
}

// A Talker + code-predictor blob may store the code predictor's matrices (c<l>.*, cp.*) in a
// format of their own; every other matrix is in the config's format.
bool own_format_allowed(const sd_ctx* c, const std::string& name) {
    return c->cfg.arch == SD_ARCH_QWEN_TTS &&
           (name.rfind("cp.", 0) == 0 || (name.size() > 1 && name[0] == 'c' && name[1] >= '0' && name[1] <= '9'));
}

int find_q(sd_ctx* c, Blob& b, const std::string& name, int rows, int cols, int swiglu_ff, uint8_t*& arena,
           QMat* out) {
    auto it = b.t.find(name);
    if (it == b.t.end() || (int)it->second.rows != rows || (int)it->second.cols != cols)
        return fail(c, SD_ERR_BLOB, "blob: missing or mis-shaped matrix '%s'", name.c_str());
    const int kind = (int)it->second.kind;
    if (!q_valid(kind) || cols % q_group(kind) || (kind != c->cfg.quant && !own_format_allowed(c, name)))
        return fail(c, SD_ERR_BLOB, "blob: matrix '%s' has format %d (config: %d)", name.c_str(), kind, c->cfg.quant);
    if (it->second.nbytes < q_canon_bytes(kind, rows, cols))
        return fail(c, SD_ERR_BLOB, "blob: matrix '%s' is truncated", name.c_str());
    const size_t qsz = q_code_bytes(kind, rows, cols);
    uint8_t* q = arena;
    uint8_t* s = arena + (qsz + 255) / 256 * 256;
    cudaError_t e = launch_repack(kind, b.base + it->second.off, rows, cols, swiglu_ff, q, s, c->stream);
    if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "repack: %s", cudaGetErrorString(e));
    arena += qbytes(kind, rows, cols);
    out->kind = kind; out->rows = rows; out->cols = cols; out->q = q; out->s = s;
    return SD_OK;
}

// Walks every tensor of the model either to size the arena (dry) or to fill it.
int load_all(sd_ctx* c, Blob& b, uint8_t* arena, size_t* total) {
    const sd_model_config& m = c->cfg;
    const bool dry = arena == nullptr;
    size_t sum = 0;
    int rc = SD_OK;
    auto F = [&](const std::string& n, int64_t cnt, const float** out) {
        if (rc) return;
        if (dry) { sum += (cnt * 4 + 255) / 256 * 256; return; }
        rc = find_f32(c, b, n, cnt, arena, out);
    };
    // the input embedding table, followed by B * max_ctx zeroed rows for prompt vectors
    const int64_t in_extra = (int64_t)c->B * m.max_ctx * m.d_model;
    auto FI = [&](const std::string& n, int64_t cnt, const float** out) {
        if (rc) return;
        const size_t bytes = (size_t)((cnt + in_extra) * 4 + 255) / 256 * 256;
        if (dry) { sum += bytes; return; }
        uint8_t* slot = arena;
        if ((rc = find_f32(c, b, n, cnt, arena, out))) return;
        arena = slot + bytes;
        if (cudaMemsetAsync(slot + cnt * 4, 0, (size_t)in_extra * 4, c->stream) != cudaSuccess)
            rc = fail(c, SD_ERR_CUDA, "clearing the prompt-vector rows failed");
    };
    auto Q = [&](const std::string& n, int rows, int cols, int swiglu_ff, QMat* out) {
        if (rc) return;
        if (dry) {
            auto it = b.t.find(n);
            const int k = it != b.t.end() && q_valid((int)it->second.kind) ? (int)it->second.kind : m.quant;
            sum += qbytes(k, rows, cols);
            return;
        }
        rc = find_q(c, b, n, rows, cols, swiglu_ff, arena, out);
    };
    auto stack = [&](DStack& s, const char* pfx) {
        s.L.resize(s.n_layer);
        const int d = s.d, qd = s.H * s.hd;
        for (int l = 0; l < s.n_layer; ++l) {
            DLayer& L = s.L[l];
            const std::string p = pfx + std::to_string(l) + ".";
            if (s.gpt2) {
                F(p + "ln1.g", d, &L.n1g); F(p + "ln1.b", d, &L.n1b);
                Q(p + "wqkv", s.qkv_rows(), d, 0, &L.wqkv); F(p + "bqkv", s.qkv_rows(), &L.bqkv);
                Q(p + "wo", d, qd, 0, &L.wo); F(p + "bo", d, &L.bo);
                F(p + "ln2.g", d, &L.n2g); F(p + "ln2.b", d, &L.n2b);
                Q(p + "wfc", s.ff, d, 0, &L.wfc); F(p + "bfc", s.ff, &L.bfc);
                Q(p + "wproj", d, s.ff, 0, &L.wproj); F(p + "bproj", d, &L.bproj);
            } else {
                F(p + "rms1.g", d, &L.n1g);
                Q(p + "wqkv", s.qkv_rows(), d, 0, &L.wqkv);
                Q(p + "wo", d, qd, 0, &L.wo);
                F(p + "rms2.g", d, &L.n2g);
                Q(p + "wgu", 2 * s.ff, d, s.ff, &L.wfc);
                Q(p + "wdown", d, s.ff, 0, &L.wproj);
            }
        }
    };
    if (m.arch == SD_ARCH_GPT2) {
        FI("wte", (int64_t)m.vocab * m.d_model, &c->wte);
        F("wpe", (int64_t)m.max_ctx * m.d_model, &c->wpe);
        stack(c->main, "l");
        F("lnf.g", m.d_model, &c->main.nfg); F("lnf.b", m.d_model, &c->main.nfb);
        Q("whead", m.vocab, m.d_model, 0, &c->head);
    } else if (m.arch == SD_ARCH_LLAMA) {
        FI("wte", (int64_t)m.vocab * m.d_model, &c->wte);
        stack(c->main, "l");
        F("normf.g", m.d_model, &c->main.nfg);
        Q("whead", m.vocab, m.d_model, 0, &c->head);
    } else {
        for (int j = 0; j < m.n_codebooks; ++j) {
            if (j == 0) FI("emb.0", (int64_t)m.vocab * m.d_model, &c->emb[0]);
            else F("emb." + std::to_string(j), (int64_t)m.cp_vocab * m.d_model, &c->emb[j]);
        }
        stack(c->main, "t");
        F("t.normf.g", m.d_model, &c->main.nfg);
        Q("t.head", m.vocab, m.d_model, 0, &c->head);
        Q("cp.proj", m.cp_d_model, m.d_model, 0, &c->cp_proj);
        stack(c->cp, "c");
        F("cp.normf.g", m.cp_d_model, &c->cp.nfg);
        for (int j = 1; j < m.n_codebooks; ++j)
            Q("cp.head." + std::to_string(j), m.cp_vocab, m.cp_d_model, 0, &c->cp_head[j]);
    }
    if (total) *total = sum;
    return rc;
}

// Per-call inputs: a GPT-2/Llama step uploads [prompt_on, u) (flags, sequence
// pointers, samplers, tokens, step draws); a frame also uploads the frame draws,
// previous codes and forced codes.
constexpr size_t kStepH2D = offsetof(DevState, u) - offsetof(DevState, prompt_on);
constexpr size_t kStepD2H = offsetof(DevState, u1);
// sd_frame uploads the inputs through the forced codes and reads the codes back as well
constexpr size_t kFrameH2D = offsetof(DevState, codes) - offsetof(DevState, prompt_on);
constexpr size_t kFrameD2H = kStepD2H + sizeof(DevState::codes);
// Tensor-core prefill: every main-stack matrix dequantised once into fp16 high
// and low parts with its TMA tensor maps, and the split-activation buffers.
// SD_PREFILL=mma keeps the mma.sync GEMM; a shape the kernel does not take
// (a width not a multiple of 64) keeps it too.
int setup_tc_prefill(sd_ctx* c) {
    c->tc_prefill = false;
    const char* env = getenv("SD_PREFILL");
    // the mma.sync prefill GEMM takes Q8_0, Q4_0 and 8-bit affine; other formats prefill through
    // the tensor-core GEMM or, where that does not apply, the per-position step graphs
    const bool mma_ok = c->cfg.quant == SD_Q8_0 || c->cfg.quant == SD_Q4_0 || c->cfg.quant == SD_A8G64;
    if (!c->gemm_prefill) return SD_OK;
    if (env && strcmp(env, "mma") == 0) {
        if (!mma_ok) c->gemm_prefill = false;
        return SD_OK;
    }
    DStack& s = c->main;
    const int qd = s.H * s.hd;
    if (s.d % 64 || qd % 64 || s.ff % 64) {
        if (!mma_ok) c->gemm_prefill = false;
        return SD_OK;
    }
    c->tc_w.assign(s.n_layer, std::array<CUtensorMap, 8>{});
    int rc;
    for (int l = 0; l < s.n_layer; ++l) {
        const QMat* mats[4] = {&s.L[l].wqkv, &s.L[l].wo, &s.L[l].wfc, &s.L[l].wproj};
        for (int w = 0; w < 4; ++w) {
            const QMat& W = *mats[w];
            const size_t n = (size_t)W.rows * W.cols;
            __half* buf = nullptr;
            if ((rc = dalloc(c, &buf, 2 * n * sizeof(__half)))) return rc;
            CK(launch_dequant_split(W, buf, buf + n, c->stream));
            if (!tc_map_fp16(&c->tc_w[l][2 * w], buf, W.rows, W.cols, true) ||
                !tc_map_fp16(&c->tc_w[l][2 * w + 1], buf + n, W.rows, W.cols, true))
                return fail(c, SD_ERR_CUDA, "tensor map for a prefill weight could not be encoded");
        }
    }
    const int R = c->B * c->pf_chunk, kmax = std::max(std::max(s.d, qd), s.ff);
    if ((rc = dalloc(c, &c->pf_xh, sizeof(__half) * (size_t)R * kmax)) ||
        (rc = dalloc(c, &c->pf_xl, sizeof(__half) * (size_t)R * kmax)))
        return rc;
    const int ks[3] = {s.d, qd, s.ff};
    for (int k = 0; k < 3; ++k)
        if (!tc_map_fp16(&c->tc_x[k][0], c->pf_xh, R, ks[k], false) ||
            !tc_map_fp16(&c->tc_x[k][1], c->pf_xl, R, ks[k], false))
            return fail(c, SD_ERR_CUDA, "tensor map for the prefill activations could not be encoded");
    CK(cudaStreamSynchronize(c->stream));
    c->tc_prefill = true;
    return SD_OK;
}

// Which persistent step kernel runs the decode steps of a GPT-2/Llama T3 with
// Q8_0/Q4_0 weights: 0 none (the per-operation graph), 1 the cluster kernel
// where its plan fits and the flat one otherwise, 2 the flat kernel only, 3
// the cluster kernel only.  Default: 1 for one row; 3 for two rows (where the
// flat kernel is slower than the graph, so the graph is the fallback).
// SD_PERSISTENT = 0 | 1 | flat | cluster overrides.
int persistent_mode(int rows) {
    const char* e = getenv("SD_PERSISTENT");
    if (e && !strcmp(e, "flat")) return 2;
    if (e && !strcmp(e, "cluster")) return 3;
    if (e && e[0] == '0') return 0;
    if (e && e[0] == '1') return 1;
    return rows == 1 ? 1 : 3;
}

// Cluster step plan, repacked matrices (cluster-major QKV rows, Wo and the
// down projection as column slabs) and exchange buffers.  Leaves
// c->cpersistent false when the plan does not fit.
int setup_cstep(sd_ctx* c) {
    const sd_model_config& m = c->cfg;
    DStack& s = c->main;
    CStepArgs& a = c->cstep;
    a = CStepArgs();
    a.gpt2 = s.gpt2 ? 1 : 0; a.n_layer = s.n_layer; a.d = s.d; a.H = s.H; a.Hkv = s.Hkv; a.hd = s.hd; a.ff = s.ff;
    a.V = m.vocab; a.n_ctx = s.n_ctx; a.B = c->B; a.quant = m.quant; a.eps = s.eps;
    a.head = c->head; a.nfg = s.nfg; a.nfb = s.nfb; a.wte = c->wte; a.wpe = c->wpe; a.V_in = c->v_in;
    a.rope_cos = s.rope_cos; a.rope_sin = s.rope_sin; a.kc = s.kc; a.vc = s.vc;
    a.logits = c->logits;
    a.pos = &c->ds->pos; a.tok = c->ds->tok; a.u1 = c->ds->u1; a.sp = &c->ds->samp[0]; a.err = &c->ds->err;
    const int grid = cstep_plan(a, c->sm_count);
    cudaGetLastError();
    if (grid <= 0) return SD_OK;
    int rc;
    // q, k, v rows of each cluster's heads, contiguous
    const int qd = s.H * s.hd, kd = s.Hkv * s.hd, R = s.qkv_rows();
    std::vector<int> perm(R);
    for (int cl = 0; cl < a.ncl; ++cl)
        for (int i = 0; i < a.rpc; ++i) {
            const int qn = a.hpc * s.hd, kn = a.kpc * s.hd;
            int src;
            if (i < qn) src = cl * qn + i;
            else if (i < qn + kn) src = qd + cl * kn + (i - qn);
            else src = qd + kd + cl * kn + (i - qn - kn);
            perm[cl * a.rpc + i] = src;
        }
    int* dperm = nullptr;
    if ((rc = dalloc(c, &dperm, sizeof(int) * R))) return rc;
    CK(cudaMemcpy(dperm, perm.data(), sizeof(int) * R, cudaMemcpyHostToDevice));
    // fragment-major copy of a matrix: column slabs of `width` columns, rows permuted by pm
    auto frag = [&](const QMat& W, int width, const int* pm, QMat* out) -> int {
        uint8_t* q = nullptr;
        int r;
        if ((r = dalloc(c, &q, frag_bytes(W.kind, W.rows, W.cols, width)))) return r;
        cudaError_t e = launch_frag_pack(W, width, pm, q, c->stream);
        if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "fragment repack: %s", cudaGetErrorString(e));
        out->kind = W.kind;
        out->rows = (W.cols / width) * ((W.rows + 15) / 16) * 16;
        out->cols = width;
        out->q = q;
        out->s = nullptr;
        return SD_OK;
    };
    // a norm gain or offset vector [d] in the padded activation layout (four zero floats after
    // every 32), as the kernel's matvec lanes read it next to their activations
    std::vector<float> hv(s.d), hpad((size_t)s.d + (s.d >> 3));
    auto padv = [&](const float* src, const float** out) -> int {
        *out = nullptr;
        if (!src) return SD_OK;
        CK(cudaMemcpy(hv.data(), src, sizeof(float) * s.d, cudaMemcpyDeviceToHost));
        std::fill(hpad.begin(), hpad.end(), 0.f);
        for (int k = 0; k < s.d; ++k) hpad[k + ((k >> 5) << 2)] = hv[k];
        float* dv = nullptr;
        int r;
        if ((r = dalloc(c, &dv, sizeof(float) * hpad.size()))) return r;
        CK(cudaMemcpy(dv, hpad.data(), sizeof(float) * hpad.size(), cudaMemcpyHostToDevice));
        *out = dv;
        return SD_OK;
    };
    if ((rc = padv(s.nfg, &a.nfg)) || (rc = padv(s.nfb, &a.nfb))) return rc;
    if ((rc = frag(c->head, c->head.cols, nullptr, &a.head))) return rc;
    std::vector<StepLayer> L(s.n_layer);
    std::vector<float> bh(R), bp(R);
    for (int l = 0; l < s.n_layer; ++l) {
        const DLayer& D = s.L[l];
        StepLayer& t = L[l];
        t.bo = D.bo; t.bfc = D.bfc; t.bproj = D.bproj;
        if ((rc = padv(D.n1g, &t.n1g)) || (rc = padv(D.n1b, &t.n1b)) || (rc = padv(D.n2g, &t.n2g)) ||
            (rc = padv(D.n2b, &t.n2b)))
            return rc;
        if ((rc = frag(D.wqkv, D.wqkv.cols, dperm, &t.wqkv)) || (rc = frag(D.wo, a.ko, nullptr, &t.wo)) ||
            (rc = frag(D.wfc, D.wfc.cols, nullptr, &t.wfc)) || (rc = frag(D.wproj, a.upc, nullptr, &t.wproj)))
            return rc;
        if (D.bqkv) {
            CK(cudaMemcpy(bh.data(), D.bqkv, sizeof(float) * R, cudaMemcpyDeviceToHost));
            for (int i = 0; i < R; ++i) bp[i] = bh[perm[i]];
            float* db = nullptr;
            if ((rc = dalloc(c, &db, sizeof(float) * R + 256))) return rc;  // bias windows widened to 16 bytes
            CK(cudaMemcpy(db, bp.data(), sizeof(float) * R, cudaMemcpyHostToDevice));
            t.bqkv = db;
        }
    }
    StepLayer* dl = nullptr;
    if ((rc = dalloc(c, &dl, sizeof(StepLayer) * s.n_layer))) return rc;
    CK(cudaMemcpy(dl, L.data(), sizeof(StepLayer) * s.n_layer, cudaMemcpyHostToDevice));
    a.layers = dl;
    const size_t w8 = sizeof(unsigned long long);
    if ((rc = dalloc(c, &a.ll_po, w8 * a.ncl * c->B * s.d)) || (rc = dalloc(c, &a.ll_pp, w8 * a.ncl * c->B * s.d)) ||
        (rc = dalloc(c, &a.ll_logits, w8 * c->B * m.vocab)) || (rc = dalloc(c, &a.ll_tok, w8 * 8 * 32)) ||
        (rc = dalloc(c, &a.gen, 256)))
        return rc;
    int clock_khz = 0;
    cudaDeviceGetAttribute(&clock_khz, cudaDevAttrClockRate, c->device);
    a.spin_budget = (long long)(clock_khz > 0 ? clock_khz : 2000000) * 200;  // 200 ms per wait
    // SD_L2_WEIGHTS=normal: weight copies without the evict-first policy (for measurement)
    if (const char* lw = getenv("SD_L2_WEIGHTS")) a.w_evict_first = strcmp(lw, "normal") != 0;
    // test hook: the first persistent launch lets one exchange-word wait run out after this many us
    if (const char* ts = getenv("SD_TEST_STALL_US"))
        c->test_stall = (long long)(clock_khz > 0 ? clock_khz : 2000000) * std::max(1, atoi(ts)) / 1000;
    if (const char* tp = getenv("SD_TRACE")) {
        c->trace_path = tp;
        if ((rc = dalloc(c, &a.trace_pub, sizeof(unsigned long long) * 2 * kTraceSteps * a.n_layer * kCTracePhases)) ||
            (rc = dalloc(c, &a.trace, sizeof(unsigned long long) * kCTraceSub)) ||
            (rc = dalloc(c, &a.trace_cta, sizeof(unsigned long long) * kCtaSteps * a.n_layer * kCTracePhases * grid)))
            return rc;
        if (const char* tg = getenv("SD_TRACE_CTA")) a.trace_gi = std::min(std::max(0, atoi(tg)), grid - 1);
    }
    CK(cudaStreamSynchronize(c->stream));
    c->step_grid = grid;
    c->cpersistent = true;
    c->persistent = true;
    return SD_OK;
}

// Persistent step plan for GPT-2/Llama with Q8_0/Q4_0 weights and B <= 2.
int setup_persistent(sd_ctx* c) {
    const sd_model_config& m = c->cfg;
    c->persistent = false;
    c->cpersistent = false;
    const int mode = persistent_mode(c->B);
    if (!mode || m.arch == SD_ARCH_QWEN_TTS || (m.quant != SD_Q8_0 && m.quant != SD_Q4_0) || c->B > 2) return SD_OK;
    if (mode == 1 || mode == 3) {
        int rc0 = setup_cstep(c);
        if (rc0 || c->cpersistent || mode == 3) return rc0;
    }
    DStack& s = c->main;
    std::vector<StepLayer> L(s.n_layer);
    for (int l = 0; l < s.n_layer; ++l) {
        const DLayer& D = s.L[l];
        L[l].n1g = D.n1g; L[l].n1b = D.n1b; L[l].bqkv = D.bqkv; L[l].bo = D.bo;
        L[l].n2g = D.n2g; L[l].n2b = D.n2b; L[l].bfc = D.bfc; L[l].bproj = D.bproj;
        L[l].wqkv = D.wqkv; L[l].wo = D.wo; L[l].wfc = D.wfc; L[l].wproj = D.wproj;
    }
    StepArgs& a = c->step;
    a.gpt2 = s.gpt2 ? 1 : 0; a.n_layer = s.n_layer; a.d = s.d; a.H = s.H; a.Hkv = s.Hkv; a.hd = s.hd; a.ff = s.ff;
    a.V = m.vocab; a.n_ctx = s.n_ctx; a.B = c->B; a.quant = m.quant; a.eps = s.eps;
    a.head = c->head; a.nfg = s.nfg; a.nfb = s.nfb; a.wte = c->wte; a.wpe = c->wpe; a.V_in = c->v_in;
    a.rope_cos = s.rope_cos; a.rope_sin = s.rope_sin; a.kc = s.kc; a.vc = s.vc;
    a.logits = c->logits;
    a.pos = &c->ds->pos; a.tok = c->ds->tok; a.u1 = c->ds->u1; a.sp = &c->ds->samp[0]; a.err = &c->ds->err;
    if (const char* sl = getenv("SD_SPLIT_LEN")) a.split_len = std::max(16, atoi(sl));
    c->step_grid = step_plan_grid(a, c->sm_count);
    cudaGetLastError();
    if (c->step_grid <= 0) return SD_OK;
    int rc;
    if ((rc = dalloc(c, &c->step_layers, sizeof(StepLayer) * s.n_layer))) return rc;
    CK(cudaMemcpy(c->step_layers, L.data(), sizeof(StepLayer) * s.n_layer, cudaMemcpyHostToDevice));
    a.layers = c->step_layers;
    // exchange words start at epoch 0, which no step uses
    const int B = c->B, qkv_rows = s.qkv_rows();
    const size_t W = sizeof(unsigned long long) * 4;  // four replicas of every exchange buffer
    if ((rc = dalloc(c, &a.ll_xa, W * B * s.d)) || (rc = dalloc(c, &a.ll_xb, W * B * s.d)) ||
        (rc = dalloc(c, &a.ll_qkv, W * B * qkv_rows)) ||
        (rc = dalloc(c, &a.ll_part, W * B * s.H * a.max_split * (s.hd + 2))) ||
        (rc = dalloc(c, &a.ll_u, W * B * s.ff)) || (rc = dalloc(c, &a.ll_logits, W * B * m.vocab)) ||
        (rc = dalloc(c, &a.ll_tok, W * 32)) || (rc = dalloc(c, &a.gen, 256)))
        return rc;
    int clock_khz = 0;
    cudaDeviceGetAttribute(&clock_khz, cudaDevAttrClockRate, c->device);
    a.spin_budget = (long long)(clock_khz > 0 ? clock_khz : 2000000) * 200;  // 200 ms per wait
    // SD_L2_WEIGHTS=normal: weight copies without the evict-first policy (for measurement)
    if (const char* lw = getenv("SD_L2_WEIGHTS")) a.w_evict_first = strcmp(lw, "normal") != 0;
    // test hook: the first persistent launch lets one exchange-word wait run out after this many us
    if (const char* ts = getenv("SD_TEST_STALL_US"))
        c->test_stall = (long long)(clock_khz > 0 ? clock_khz : 2000000) * std::max(1, atoi(ts)) / 1000;
    if (const char* tp = getenv("SD_TRACE")) {
        c->trace_path = tp;
        if ((rc = dalloc(c, &a.trace, sizeof(unsigned long long) * 64))) return rc;
        if ((rc = dalloc(c, &a.trace_pub, sizeof(unsigned long long) * 2 * kTraceSteps * a.n_layer * kTracePhases)))
            return rc;
    }
    c->persistent = true;
    return SD_OK;
}

// Per-phase times of CTA 0 over the last persistent launch, appended to
// SD_TRACE: for each phase kind the mean wait for its inputs and the mean work.
void write_ctrace(sd_ctx* c, int n_steps) {
    const CStepArgs& a = c->cstep;
    if (c->trace_path.empty() || !a.trace_pub || n_steps < 1 || a.n_layer < 2) return;
    const int L = a.n_layer, ns = std::min(n_steps, kTraceSteps);
    const size_t half = (size_t)kTraceSteps * L * kCTracePhases;
    std::vector<unsigned long long> tp(2 * half);
    if (cudaMemcpy(tp.data(), a.trace_pub, tp.size() * 8, cudaMemcpyDeviceToHost) != cudaSuccess) return;
    FILE* f = fopen(c->trace_path.c_str(), "a");
    if (!f) return;
    const char* pn[kCTracePhases] = {"x-ready", "qkv", "attn", "o-pub", "x'-sent", "fc", "proj-pub", "x''-sent"};
    double dl[kCTracePhases] = {}, sp[kCTracePhases] = {};
    int cnt = 0;
    for (int st = 0; st < ns; ++st)
        for (int l = 1; l < L; ++l) {
            const unsigned long long* mx = tp.data() + ((size_t)st * L + l) * kCTracePhases;
            const unsigned long long* mn = mx + half;
            const unsigned long long* prev = tp.data() + ((size_t)st * L + l - 1) * kCTracePhases;
            for (int ph = 0; ph < kCTracePhases; ++ph) {
                const unsigned long long ref = ph == 0 ? prev[kCTracePhases - 1] : mx[ph - 1];
                dl[ph] += (double)(long long)(mx[ph] - ref);
                sp[ph] += (double)(long long)(mx[ph] - mn[ph]);
            }
            ++cnt;
        }
    fprintf(f, "cluster step: steps=%d clusters=%d x %d ring=%d act=%d kkc=%d\n", n_steps, a.ncl, a.cs, a.ring_bytes,
            a.act_bytes, a.kkc);
    fprintf(f, "  critical path per layer (us): phase: latest stamp - previous latest | latest - earliest\n");
    double tot = 0;
    for (int ph = 0; ph < kCTracePhases; ++ph) {
        fprintf(f, "    %-9s %8.3f %8.3f\n", pn[ph], dl[ph] / 1e3 / cnt, sp[ph] / 1e3 / cnt);
        tot += dl[ph] / 1e3 / cnt;
    }
    fprintf(f, "    layer     %8.3f\n", tot);
    if (a.trace_cta) {
        // every CTA's stamps of the first steps, raw, beside the trace: int32 grid, layers, phases,
        // steps, then [steps][layers][phases][grid] uint64 global-timer ns
        const int G = a.ncl * a.cs, ns2 = std::min(n_steps, kCtaSteps);
        std::vector<unsigned long long> tc((size_t)kCtaSteps * L * kCTracePhases * G);
        if (cudaMemcpy(tc.data(), a.trace_cta, tc.size() * 8, cudaMemcpyDeviceToHost) == cudaSuccess) {
            FILE* fb = fopen((c->trace_path + ".cta.bin").c_str(), "wb");
            if (fb) {
                const int32_t hdr[4] = {G, L, kCTracePhases, ns2};
                fwrite(hdr, sizeof hdr, 1, fb);
                fwrite(tc.data(), 8, (size_t)ns2 * L * kCTracePhases * G, fb);
                fclose(fb);
            }
        }
    }
    unsigned long long t[kCTraceSub];
    if (a.trace && cudaMemcpy(t, a.trace, sizeof t, cudaMemcpyDeviceToHost) == cudaSuccess) {
        // CTA 0's cycles per sub-step (per layer, or per step for the last four)
        const char* nm[30] = {"wait x''", "rec qkv", "norm1", "mma qkv+send", "wait qkv", "attn keys",
                              "comb+send", "wait part", "combine", "rec o", "mma o+pub", "reduce o", "wait x'",
                              "rec fc", "norm2", "mma fc+send", "wait u", "rec proj", "mma proj+pub", "reduce proj",
                              "head*", "end*", "(q prep)", "(kv wait)", "(wp+bar)", "(send+bar)", "start*", "embed*", "gather*",
                              "sample*"};
        const double nl = (double)n_steps * L;
        fprintf(f, "  CTA %d cycles per layer (* per step):\n   ", a.trace_gi);
        for (int k = 0; k < 30; ++k) {
            if (!nm[k][0]) continue;
            fprintf(f, " %s %.0f |", nm[k], (double)t[k] / ((k >= 20 && k <= 21) || k >= 26 ? (double)n_steps : nl));
            if (k % 7 == 6) fprintf(f, "\n   ");
        }
        fprintf(f, "\n");
    }
    fclose(f);
}

void write_trace(sd_ctx* c, int n_steps) {
    if (c->cpersistent) return write_ctrace(c, n_steps);
    if (c->trace_path.empty() || !c->step.trace || n_steps < 1) return;
    unsigned long long t[64];
    if (cudaMemcpy(t, c->step.trace, sizeof t, cudaMemcpyDeviceToHost) != cudaSuccess) return;
    FILE* f = fopen(c->trace_path.c_str(), "a");
    if (!f) return;
    const char* names[8] = {"embed", "qkv", "attn", "o", "fc", "proj", "head", "sample"};
    const double per[8] = {1.0, (double)c->step.n_layer, (double)c->step.n_layer, (double)c->step.n_layer,
                           (double)c->step.n_layer, (double)c->step.n_layer, 1.0, 1.0};
    double tot = 0;
    for (int k = 0; k < 24; ++k) tot += (double)t[k];
    fprintf(f, "steps=%d grid=%d ring=%d act=%d max_split=%d | CTA 0 per step %.2f us | phase: input wait / "
               "weight wait / rest us\n",
            n_steps, c->step_grid, c->step.ring_bytes, c->step.act_bytes, c->step.max_split, tot / 1e3 / n_steps);
    for (int k = 0; k < 8; ++k)
        fprintf(f, "  %-6s %8.3f %8.3f %8.3f\n", names[k], (double)t[3 * k] / 1e3 / n_steps / per[k],
                (double)t[3 * k + 1] / 1e3 / n_steps / per[k], (double)t[3 * k + 2] / 1e3 / n_steps / per[k]);
    fprintf(f, "  qkv sub-phases us: slice %.3f record %.3f norm %.3f matvec %.3f publish %.3f\n",
            (double)t[24] / 1e3 / n_steps / per[1], (double)t[25] / 1e3 / n_steps / per[1],
            (double)t[26] / 1e3 / n_steps / per[1], (double)t[27] / 1e3 / n_steps / per[1],
            (double)t[28] / 1e3 / n_steps / per[1]);
    {
        // cycle stamps of CTA 0: FC phase sub-steps and attention item sub-steps, per layer
        const double nl = (double)n_steps * c->step.n_layer;
        fprintf(f, "  fc cycles/layer: inputs %.0f norm %.0f matvec %.0f publish %.0f release %.0f\n", t[32] / nl,
                t[33] / nl, t[34] / nl, t[35] / nl, t[36] / nl);
        fprintf(f, "  attn cycles/layer: qkv-wait %.0f rope+append %.0f stage-wait %.0f warps %.0f partials %.0f "
                   "combine+publish %.0f fence %.0f\n",
                t[40] / nl, t[41] / nl, t[42] / nl, t[43] / nl, t[44] / nl, t[45] / nl, t[46] / nl);
    }
    if (c->step.trace_pub) {
        // critical path: per phase, the latest publish minus the previous phase's latest publish,
        // and the spread between the earliest and the latest CTA (layers >= 1 of the first steps)
        const int L = c->step.n_layer, ns = std::min(n_steps, kTraceSteps);
        const size_t half = (size_t)kTraceSteps * L * kTracePhases;
        std::vector<unsigned long long> tp(2 * half);
        if (L > 1 && cudaMemcpy(tp.data(), c->step.trace_pub, tp.size() * 8, cudaMemcpyDeviceToHost) == cudaSuccess) {
            const char* pn[kTracePhases] = {"input", "qkv", "attn", "o", "fc", "proj"};
            double dl[kTracePhases] = {}, sp[kTracePhases] = {};
            int cnt = 0;
            for (int st = 0; st < ns; ++st)
                for (int l = 1; l < L; ++l) {
                    const unsigned long long* mx = tp.data() + ((size_t)st * L + l) * kTracePhases;
                    const unsigned long long* mn = mx + half;
                    const unsigned long long* prev = tp.data() + ((size_t)st * L + l - 1) * kTracePhases;
                    for (int ph = 0; ph < kTracePhases; ++ph) {
                        const unsigned long long ref = ph == 0 ? prev[kTracePhases - 1] : mx[ph - 1];
                        dl[ph] += (double)(long long)(mx[ph] - ref);
                        sp[ph] += (double)(long long)(mx[ph] - mn[ph]);
                    }
                    ++cnt;
                }
            fprintf(f, "  critical path per layer (us): phase: latest publish - previous latest | latest - earliest\n");
            double tot = 0;
            for (int ph = 0; ph < kTracePhases; ++ph) {
                fprintf(f, "    %-6s %8.3f %8.3f\n", pn[ph], dl[ph] / 1e3 / cnt, sp[ph] / 1e3 / cnt);
                tot += dl[ph] / 1e3 / cnt;
            }
            fprintf(f, "    layer  %8.3f\n", tot);
        }
    }
    fclose(f);
}

int upload_inputs(sd_ctx* c, bool full) {
    const size_t a = offsetof(DevState, prompt_on);
    const size_t e = full ? offsetof(DevState, codes) : offsetof(DevState, u);
    CK(cudaMemcpyAsync(reinterpret_cast<char*>(c->ds) + a, reinterpret_cast<char*>(c->hs) + a, e - a,
                       cudaMemcpyHostToDevice, c->stream));
    return SD_OK;
}

int check_device_err(sd_ctx* c) {
    if (c->hs->err) {
        const int code = c->hs->err;
        c->hs->err = 0;
        cudaMemsetAsync(&c->ds->err, 0, sizeof(int32_t), c->stream);
        if (code == 6) return fail(c, SD_ERR_TIMEOUT, "a grid barrier of the persistent step timed out");
        return fail(c, SD_ERR_DEVICE, "a kernel flagged an out-of-range index (code %d)", code);
    }
    return SD_OK;
}

int download_counters(sd_ctx* c, bool codes) {
    CK(cudaMemcpyAsync(c->hs, c->ds, kStepD2H, cudaMemcpyDeviceToHost, c->stream));
    if (codes)
        CK(cudaMemcpyAsync(c->hs->codes, c->ds->codes, sizeof(c->hs->codes), cudaMemcpyDeviceToHost, c->stream));
    CK(cudaStreamSynchronize(c->stream));
    return check_device_err(c);
}

// SD_OK, or the error code of an sd_sampler the decode sampler does not take
int sampler_check(const sd_sampler* s) {
    if (!(s->temperature >= 0.f) || s->top_k < 1 || !(s->top_p > 0.f && s->top_p <= 1.f)) return SD_ERR_INVALID_ARG;
    if (!(s->rep_penalty >= 0.f)) return SD_ERR_INVALID_ARG;
    if (s->rep_penalty != 0.f && s->rep_penalty != 1.f) return SD_ERR_UNSUPPORTED;
    return SD_OK;
}

// which: 0 the T3 / Talker sampler, 1 the code predictor's.  Only the Talker's sampler keeps a
// history (the codebook-0 tokens fed so far), so only it takes a repetition penalty.
int set_sampler(sd_ctx* c, int which, const sd_sampler* s) {
    if (!s) return fail(c, SD_ERR_INVALID_ARG, "sampler is NULL");
    int rc = sampler_check(s);
    if (rc == SD_ERR_UNSUPPORTED && c->cfg.arch == SD_ARCH_QWEN_TTS && which == 0) rc = SD_OK;
    if (rc)
        return fail(c, rc, "sampler %s (T=%g k=%d p=%g penalty=%g)",
                    rc == SD_ERR_UNSUPPORTED ? "asks for a repetition penalty, which only the Talker's sampler applies"
                                             : "out of range",
                    s->temperature, s->top_k, s->top_p, s->rep_penalty);
    c->hs->samp[which].temperature = s->temperature;
    c->hs->samp[which].top_k = s->top_k;
    c->hs->samp[which].top_p = s->top_p;
    c->hs->samp[which].greedy = s->greedy;
    c->hs->samp[which].rep_penalty = s->rep_penalty > 0.f ? s->rep_penalty : 1.0f;
    return SD_OK;
}

int check_draws(sd_ctx* c, const float* u, int n) {
    if (!u) return fail(c, SD_ERR_INVALID_ARG, "draws are NULL");
    for (int i = 0; i < n; ++i)
        if (!(u[i] >= 0.f && u[i] < 1.f)) return fail(c, SD_ERR_INVALID_ARG, "draw %d = %g outside [0,1)", i, u[i]);
    return SD_OK;
}

}  // namespace

void sd::set_last_error(const char* msg) { g_err = msg; }

// ======================================================================= C ABI

extern "C" {

const char* sd_last_error(const sd_ctx* c) { return c ? c->err.c_str() : g_err.c_str(); }

int sd_create(const sd_model_config* cfg, int device, void* stream, sd_ctx** out) {
    sd_ctx* c = nullptr;
    if (!cfg || !out) return fail(nullptr, SD_ERR_INVALID_ARG, "sd_create: NULL argument");
    *out = nullptr;
    if (!validate_cfg(*cfg)) return fail(nullptr, SD_ERR_INVALID_ARG, "sd_create: invalid model config");
    c = new sd_ctx();
    c->cfg = *cfg;
    c->device = device;
    c->B = cfg->batch;
    c->v_in = cfg->vocab + cfg->batch * cfg->max_ctx;
    auto bail = [&](int rc) { g_err = c->err; sd_destroy(c); return rc; };
    if (cudaSetDevice(device) != cudaSuccess) return bail(fail(c, SD_ERR_CUDA, "cudaSetDevice(%d) failed", device));
    if (cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return bail(fail(c, SD_ERR_CUDA, "device query failed"));
    {
        int clock_khz = 0;
        cudaDeviceGetAttribute(&clock_khz, cudaDevAttrClockRate, device);
        c->spin_budget = (long long)(clock_khz > 0 ? clock_khz : 2000000) * 200;
    }
    if (stream) {
        c->stream = reinterpret_cast<cudaStream_t>(stream);
    } else {
        if (cudaStreamCreateWithFlags(&c->stream, cudaStreamNonBlocking) != cudaSuccess)
            return bail(fail(c, SD_ERR_CUDA, "stream create failed"));
        c->own_stream = true;
    }
    if (cudaStreamCreateWithFlags(&c->cap, cudaStreamNonBlocking) != cudaSuccess)
        return bail(fail(c, SD_ERR_CUDA, "stream create failed"));
    const sd_model_config& m = *cfg;
    init_stack(c->main, m.arch == SD_ARCH_GPT2, m.n_layer, m.d_model, m.n_head, m.n_kv_head, m.head_dim, m.d_ff,
               m.max_ctx, m.norm_eps, m.rope_theta);
    int rc;
    if ((rc = alloc_stack(c, c->main))) return bail(rc);
    if (m.arch == SD_ARCH_QWEN_TTS) {
        init_stack(c->cp, false, m.cp_layer, m.cp_d_model, m.cp_n_head, m.cp_n_kv_head, m.cp_head_dim, m.cp_d_ff,
                   m.cp_max_ctx, m.norm_eps, m.rope_theta);
        if ((rc = alloc_stack(c, c->cp))) return bail(rc);
        c->vmax = std::max(m.vocab, m.cp_vocab);
        c->logits_ld = kMaxCodebooks * c->vmax;
        if ((rc = dalloc(c, &c->ebuf, sizeof(float) * c->B * m.d_model))) return bail(rc);
        if ((rc = dalloc(c, &c->seen0, (size_t)c->B * m.vocab))) return bail(rc);
    } else {
        c->vmax = m.vocab;
        c->logits_ld = m.vocab;
    }
    if ((rc = dalloc(c, &c->logits, sizeof(float) * c->B * c->logits_ld))) return bail(rc);
    if ((rc = dalloc(c, &c->nrm, sizeof(float) * c->B * std::max(m.d_model, m.arch == SD_ARCH_QWEN_TTS ? m.cp_d_model : 0))))
        return bail(rc);
    if ((rc = dalloc(c, &c->prompt, sizeof(int32_t) * c->B * m.max_ctx))) return bail(rc);
    if (c->B > 2) {
        const char* rg = getenv("SD_ROWS_GEMM");
        c->rows_gemm_mma = rg && strcmp(rg, "mma") == 0;
        c->rows_gemm_tc = rg && strcmp(rg, "tc") == 0;  // default: the mma.sync skinny GEMM (faster, measured)
        // skinny GEMM workspace: the largest partial-sum array and tile count over every matrix
        std::vector<std::pair<int, int>> nk;  // (rows, cols)
        auto stack_mats = [&](int d, int H, int Hkv, int hd, int ff, bool gpt2) {
            nk.push_back({(H + 2 * Hkv) * hd, d});
            nk.push_back({d, H * hd});
            nk.push_back({gpt2 ? ff : 2 * ff, d});
            nk.push_back({d, ff});
        };
        stack_mats(m.d_model, m.n_head, m.n_kv_head, m.head_dim, m.d_ff, m.arch == SD_ARCH_GPT2);
        nk.push_back({m.vocab, m.d_model});
        if (m.arch == SD_ARCH_QWEN_TTS) {
            stack_mats(m.cp_d_model, m.cp_n_head, m.cp_n_kv_head, m.cp_head_dim, m.cp_d_ff, false);
            nk.push_back({m.cp_d_model, m.d_model});
            nk.push_back({m.cp_vocab, m.cp_d_model});
        }
        size_t wsf = 0;
        int tiles = 0;
        for (const auto& p : nk) {
            wsf = std::max(wsf, gemm16_ws_floats(p.first, p.second, c->sm_count));
            if (m.quant == SD_A8G64 && p.second % 64 == 0)
                wsf = std::max(wsf, gemm16_tc_ws_floats(p.first, p.second, c->sm_count));
            tiles = std::max(tiles, gemm16_tiles(p.first));
        }
        if ((rc = dalloc(c, &c->g16_ws, sizeof(float) * wsf)) || (rc = dalloc(c, &c->g16_cnt, sizeof(int) * tiles)))
            return bail(rc);
    }
    {
        // GEMM prefill: SD_PREFILL=steps runs the prompt through the per-position step graphs instead
        const char* e = getenv("SD_PREFILL");
        c->gemm_prefill = !(e && strcmp(e, "steps") == 0);
        const DStack& s = c->main;
        c->pf_chunk = std::max(1, std::min(m.max_ctx, 512 / c->B));
        const size_t R = (size_t)c->B * c->pf_chunk;
        if ((rc = dalloc(c, &c->pf_x, sizeof(float) * R * s.d)) || (rc = dalloc(c, &c->pf_h, sizeof(float) * R * s.d)) ||
            (rc = dalloc(c, &c->pf_qkv, sizeof(float) * R * s.qkv_rows())) ||
            (rc = dalloc(c, &c->pf_o, sizeof(float) * R * s.H * s.hd)) ||
            (rc = dalloc(c, &c->pf_u, sizeof(float) * R * s.ff)))
            return bail(rc);
    }
    if ((rc = dalloc(c, &c->ds, sizeof(DevState)))) return bail(rc);
    if (cudaHostAlloc(&c->hs, sizeof(DevState), cudaHostAllocDefault) != cudaSuccess)
        return bail(fail(c, SD_ERR_OOM, "pinned staging allocation failed"));
    memset(c->hs, 0, sizeof(DevState));
    *out = c;
    return SD_OK;
}

int sd_load_weights(sd_ctx* c, const void* blob, size_t nbytes, int blob_on_device) {
    if (!c || !blob) return fail(c, SD_ERR_INVALID_ARG, "sd_load_weights: NULL argument");
    if (c->phase != Phase::Created) return fail(c, SD_ERR_STATE, "weights already loaded");
    CK(cudaSetDevice(c->device));
    // header + table on the host
    uint8_t hdr[16];
    if (nbytes < 16 + 4 * 32) return fail(c, SD_ERR_BLOB, "blob too small");
    if (blob_on_device) CK(cudaMemcpy(hdr, blob, 16, cudaMemcpyDeviceToHost));
    else memcpy(hdr, blob, 16);
    uint32_t magic, ver, n, toff;
    memcpy(&magic, hdr, 4); memcpy(&ver, hdr + 4, 4); memcpy(&n, hdr + 8, 4); memcpy(&toff, hdr + 12, 4);
    if (magic != kBlobMagic || ver != 1) return fail(c, SD_ERR_BLOB, "blob: bad magic or version");
    const size_t tend = (size_t)toff + (size_t)n * kEntryBytes;
    if (tend > nbytes || toff < 16 + 4 * 32) return fail(c, SD_ERR_BLOB, "blob: table out of range");
    std::vector<uint8_t> head(tend);
    if (blob_on_device) CK(cudaMemcpy(head.data(), blob, tend, cudaMemcpyDeviceToHost));
    else memcpy(head.data(), blob, tend);
    if (memcmp(head.data() + 16, &c->cfg, kConfigFields * 4) != 0)
        return fail(c, SD_ERR_BLOB, "blob: config echo does not match the context's config");
    Blob b;
    for (uint32_t i = 0; i < n; ++i) {
        const uint8_t* e = head.data() + toff + (size_t)i * kEntryBytes;
        char name[65] = {0};
        memcpy(name, e, 64);
        BlobTensor t;
        memcpy(&t.kind, e + 64, 4); memcpy(&t.rows, e + 68, 4); memcpy(&t.cols, e + 72, 4);
        memcpy(&t.off, e + 80, 8); memcpy(&t.nbytes, e + 88, 8);
        if (t.off + t.nbytes > nbytes || t.off % 16) return fail(c, SD_ERR_BLOB, "blob: tensor '%s' out of range", name);
        b.t[name] = t;
    }
    // blob bytes on the device (staging copy when the caller's blob is on the host)
    uint8_t* staging = nullptr;
    if (blob_on_device) {
        b.base = reinterpret_cast<const uint8_t*>(blob);
    } else {
        cudaError_t e = cudaMalloc(&staging, nbytes);
        if (e != cudaSuccess) return fail(c, SD_ERR_OOM, "staging cudaMalloc(%zu) failed", nbytes);
        e = cudaMemcpy(staging, blob, nbytes, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) { cudaFree(staging); return fail(c, SD_ERR_CUDA, "blob upload: %s", cudaGetErrorString(e)); }
        b.base = staging;
    }
    size_t total = 0;
    int rc = load_all(c, b, nullptr, &total);
    if (!rc) {
        // + 256: the persistent step copies scale and bias windows widened to 16 bytes
        cudaError_t e = cudaMalloc(&c->weights, total + 256);
        if (e != cudaSuccess) rc = fail(c, SD_ERR_OOM, "weight arena cudaMalloc(%zu) failed", total);
    }
    if (!rc) rc = load_all(c, b, c->weights, nullptr);
    cudaError_t se = cudaStreamSynchronize(c->stream);
    if (staging) cudaFree(staging);
    if (rc) return rc;
    if (se != cudaSuccess) return fail(c, SD_ERR_CUDA, "weight repack: %s", cudaGetErrorString(se));
    c->weight_bytes = (int64_t)total;
    if ((rc = setup_persistent(c))) return rc;
    if ((rc = setup_tc_prefill(c))) return rc;
    // graphs
    if (c->cfg.arch == SD_ARCH_QWEN_TTS) {
        if ((rc = capture(c, GraphKind::QwenFrame, &c->g_frame, &c->kernels_per_step))) return rc;
        if ((rc = capture(c, GraphKind::QwenBody, &c->g_body, nullptr))) return rc;
        if ((rc = capture(c, GraphKind::QwenPromptLast, &c->g_prompt_last, nullptr))) return rc;
    } else {
        if ((rc = capture(c, GraphKind::T3Step, &c->g_step, &c->kernels_per_step))) return rc;
        if ((rc = capture(c, GraphKind::T3Body, &c->g_body, nullptr))) return rc;
    }
    c->phase = Phase::Loaded;
    c->host_pos = 0;
    return SD_OK;
}

int sd_reset(sd_ctx* c) {
    if (!c) return fail(nullptr, SD_ERR_INVALID_ARG, "sd_reset: NULL context");
    if (cudaSetDevice(c->device) != cudaSuccess) return fail(c, SD_ERR_CUDA, "cudaSetDevice failed");
    cudaStreamSynchronize(c->stream);
    cudaGetLastError();
    if (c->ds) {
        cudaMemsetAsync(c->ds, 0, offsetof(DevState, prompt_on), c->stream);
        if (cudaStreamSynchronize(c->stream) != cudaSuccess) return fail(c, SD_ERR_CUDA, "reset failed");
    }
    if (c->hs) memset(c->hs, 0, sizeof(DevState));
    c->host_pos = 0;
    c->force_pending = false;
    if (c->phase == Phase::Running) c->phase = Phase::Loaded;
    return SD_OK;
}

int sd_set_ladder(sd_ctx* c, const sd_sampler_ladder* s) {
    if (!c) return fail(nullptr, SD_ERR_INVALID_ARG, "sd_set_ladder: NULL context");
    if (c->cfg.arch == SD_ARCH_QWEN_TTS || c->B != 2)
        return fail(c, SD_ERR_UNSUPPORTED, "the ladder needs a GPT-2/Llama context with a conditional and an unconditional row");
    if (c->phase != Phase::Loaded || c->host_pos != 0) return fail(c, SD_ERR_STATE, "sd_set_ladder needs a loaded, reset context");
    if (c->cfg.vocab > 16384) return fail(c, SD_ERR_UNSUPPORTED, "the ladder takes at most 16384 logits");
    if (s && (!(s->repetition_penalty > 0.f) || !(s->min_p >= 0.f) || !(s->top_p > 0.f && s->top_p <= 1.f) ||
              !(s->temperature == s->temperature) || !(s->cfg_weight == s->cfg_weight)))
        return fail(c, SD_ERR_INVALID_ARG, "sd_set_ladder: ladder out of range");
    CK(cudaSetDevice(c->device));
    int rc;
    if (s && !c->seen) {
        if ((rc = dalloc(c, &c->seen, (size_t)((c->cfg.vocab + 15) & ~15))) || (rc = dalloc(c, &c->lad_u, 16)) ||
            (rc = dalloc(c, &c->lad_t, 16)) || (rc = dalloc(c, &c->lad_in, 16)))
            return rc;
    }
    c->ladder_on = s != nullptr;
    if (s) {
        c->ladder.cfg_weight = s->cfg_weight; c->ladder.rep_penalty = s->repetition_penalty;
        c->ladder.temperature = s->temperature; c->ladder.min_p = s->min_p; c->ladder.top_p = s->top_p;
        c->ladder.top_k = s->top_k;
    }
    // the step graph takes the ladder (or the per-row sampler again)
    CK(cudaStreamSynchronize(c->stream));
    if (c->g_step) cudaGraphExecDestroy(c->g_step);
    c->g_step = nullptr;
    return capture(c, GraphKind::T3Step, &c->g_step, &c->kernels_per_step);
}

int sd_set_forced_codes(sd_ctx* c, const int32_t* codes) {
    if (!c) return fail(nullptr, SD_ERR_INVALID_ARG, "NULL context");
    if (c->cfg.arch != SD_ARCH_QWEN_TTS) return fail(c, SD_ERR_UNSUPPORTED, "forced codes need a Talker+CP model");
    if (!codes) { c->force_pending = false; return SD_OK; }
    for (int b = 0; b < c->B; ++b)
        for (int j = 0; j < c->cfg.n_codebooks; ++j) {
            const int v = codes[b * kMaxCodebooks + j], V = j ? c->cfg.cp_vocab : c->cfg.vocab;
            if (v < 0 || v >= V) return fail(c, SD_ERR_INVALID_ARG, "forced code [%d][%d]=%d out of range", b, j, v);
            c->hs->force[b * kMaxCodebooks + j] = v;
        }
    c->force_pending = true;
    return SD_OK;
}

// Row 0's KV cache at positions [0, npos) of the main stack copied into every other row (the
// cache is [row][layer * kv head][position][dim]: one 2-D copy per row and tensor).
int copy_prompt_kv(sd_ctx* c, int npos) {
    const DStack& s = c->main;
    const size_t rh = (size_t)s.n_layer * s.Hkv, pitch = (size_t)s.n_ctx * s.hd * sizeof(__half);
    for (int b = 1; b < c->B; ++b)
        for (__half* t : {s.kc, s.vc})
            CK(cudaMemcpy2DAsync(t + (size_t)b * rh * s.n_ctx * s.hd, pitch, t, pitch, (size_t)npos * s.hd * sizeof(__half),
                                 rh, cudaMemcpyDeviceToDevice, c->stream));
    return SD_OK;
}

// The prompt of every row (token indices below v_limit: the vocabulary, or the prompt-vector rows
// after it).  shared: every row's prompt is row 0's, and positions [0, n - 1) are computed for
// row 0 only and copied (on the GEMM prefill path).
int prefill_impl(sd_ctx* c, const int32_t* tokens, int32_t n, const sd_sampler* sampler, const float* u,
                 int32_t* out_tok, int v_limit, bool shared) {
    if (c->phase != Phase::Loaded || c->host_pos != 0) return fail(c, SD_ERR_STATE, "sd_prefill needs a loaded, reset context");
    if (n < 1 || n > c->cfg.max_ctx) return fail(c, SD_ERR_CTX_FULL, "prompt length %d outside [1, %d]", n, c->cfg.max_ctx);
    CK(cudaSetDevice(c->device));
    const bool qwen = c->cfg.arch == SD_ARCH_QWEN_TTS;
    const int B = c->B, ns = qwen ? c->cfg.n_codebooks : 1;
    for (int i = 0; i < B * n; ++i)
        if (tokens[i] < 0 || tokens[i] >= v_limit)
            return fail(c, SD_ERR_INVALID_ARG, "prompt token %d = %d outside [0, %d)", i, tokens[i], v_limit);
    int rc;
    if ((rc = set_sampler(c, 0, sampler))) return rc;
    if (qwen) {  // the prompt frame's code predictor takes the same settings without the Talker's penalty
        sd_sampler cp = *sampler;
        cp.rep_penalty = 1.0f;
        if ((rc = set_sampler(c, 1, &cp))) return rc;
    }
    if (!u) return fail(c, SD_ERR_INVALID_ARG, "draws are NULL");
    for (int b = 0; b < B; ++b) {
        if ((rc = check_draws(c, u + b * ns, ns))) return rc;
        for (int j = 0; j < ns; ++j) c->hs->u[b * kMaxCodebooks + j] = u[b * ns + j];
        c->hs->u1[b] = u[b * ns];
    }
    // prompt tokens, row-major with a max_ctx leading dimension
    for (int b = 0; b < B; ++b)
        CK(cudaMemcpyAsync(c->prompt + (size_t)b * c->cfg.max_ctx, tokens + (size_t)b * n, sizeof(int32_t) * n,
                           cudaMemcpyHostToDevice, c->stream));
    c->hs->prompt_on = 1;
    c->hs->force_on = c->force_pending ? 1 : 0;
    c->hs->u_seq = nullptr; c->hs->out_seq = nullptr;
    for (int b = 0; b < B; ++b) c->hs->tok[b] = tokens[(size_t)b * n + n - 1];  // read by the persistent step
    if ((rc = upload_inputs(c, qwen))) return rc;
    if (c->ladder_on) CK(cudaMemsetAsync(c->seen, 0, (size_t)c->cfg.vocab, c->stream));
    if (c->seen0) CK(cudaMemsetAsync(c->seen0, 0, (size_t)B * c->cfg.vocab, c->stream));
    if (c->gemm_prefill && n > 1) {
        if ((rc = enqueue_prefill_gemm(c, n - 1, shared ? 1 : B, c->stream))) return rc;
        if (shared && B > 1 && (rc = copy_prompt_kv(c, n - 1))) return rc;
    } else {
        for (int i = 0; i < n - 1; ++i) CK(cudaGraphLaunch(c->g_body, c->stream));
    }
    CK(cudaGraphLaunch(qwen ? c->g_prompt_last : c->g_step, c->stream));
    c->force_pending = false;
    rc = download_counters(c, qwen);   // synchronises: the staging mirror may change after this
    c->hs->prompt_on = 0;
    c->hs->force_on = 0;
    if (rc) return rc;
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < ns; ++j)
            out_tok[b * ns + j] = qwen ? c->hs->codes[b * kMaxCodebooks + j] : c->hs->tok[b];
    c->host_pos = n;
    c->phase = Phase::Running;
    return SD_OK;
}

int sd_prefill(sd_ctx* c, const int32_t* tokens, int32_t n, const sd_sampler* sampler, const float* u,
               int32_t* out_tok) {
    if (!c || !tokens || !out_tok) return fail(c, SD_ERR_INVALID_ARG, "sd_prefill: NULL argument");
    return prefill_impl(c, tokens, n, sampler, u, out_tok, c->cfg.vocab, false);
}

int sd_prefill_shared(sd_ctx* c, const int32_t* tokens, int32_t n, const sd_sampler* sampler, const float* u,
                      int32_t* out_tok) {
    if (!c || !tokens || !out_tok) return fail(c, SD_ERR_INVALID_ARG, "sd_prefill_shared: NULL argument");
    if (n < 1 || n > c->cfg.max_ctx) return fail(c, SD_ERR_CTX_FULL, "prompt length %d outside [1, %d]", n, c->cfg.max_ctx);
    std::vector<int32_t> all((size_t)c->B * n);
    for (int b = 0; b < c->B; ++b) memcpy(all.data() + (size_t)b * n, tokens, sizeof(int32_t) * n);
    return prefill_impl(c, all.data(), n, sampler, u, out_tok, c->cfg.vocab, true);
}

int sd_prefill_embeds(sd_ctx* c, const float* embeds, int32_t n, const sd_sampler* sampler, const float* u,
                      int32_t* out_tok) {
    if (!c || !embeds || !out_tok) return fail(c, SD_ERR_INVALID_ARG, "sd_prefill_embeds: NULL argument");
    if (c->phase != Phase::Loaded || c->host_pos != 0)
        return fail(c, SD_ERR_STATE, "sd_prefill_embeds needs a loaded, reset context");
    if (n < 1 || n > c->cfg.max_ctx) return fail(c, SD_ERR_CTX_FULL, "prompt length %d outside [1, %d]", n, c->cfg.max_ctx);
    const int d = c->cfg.d_model, V = c->cfg.vocab, ld = c->cfg.max_ctx;
    for (size_t i = 0; i < (size_t)c->B * n * d; ++i)
        if (!std::isfinite(embeds[i])) return fail(c, SD_ERR_INVALID_ARG, "prompt vector element %zu is not finite", i);
    CK(cudaSetDevice(c->device));
    float* table = const_cast<float*>(c->cfg.arch == SD_ARCH_QWEN_TTS ? c->emb[0] : c->wte);
    std::vector<int32_t> idx((size_t)c->B * n);
    for (int b = 0; b < c->B; ++b) {
        CK(cudaMemcpyAsync(table + ((size_t)V + (size_t)b * ld) * d, embeds + (size_t)b * n * d, sizeof(float) * n * d,
                           cudaMemcpyHostToDevice, c->stream));
        for (int p = 0; p < n; ++p) idx[(size_t)b * n + p] = V + b * ld + p;
    }
    return prefill_impl(c, idx.data(), n, sampler, u, out_tok, c->v_in, false);
}

int sd_step(sd_ctx* c, const int32_t* tok, const sd_sampler* sampler, const float* u, int32_t* out_tok) {
    if (!c || !tok || !out_tok) return fail(c, SD_ERR_INVALID_ARG, "sd_step: NULL argument");
    if (c->cfg.arch == SD_ARCH_QWEN_TTS) return fail(c, SD_ERR_UNSUPPORTED, "use sd_frame for a Talker+CP model");
    if (c->phase != Phase::Running) return fail(c, SD_ERR_STATE, "sd_step before sd_prefill");
    if (c->host_pos >= c->cfg.max_ctx) return fail(c, SD_ERR_CTX_FULL, "context full (%d)", c->host_pos);
    CK(cudaSetDevice(c->device));
    int rc;
    if ((rc = set_sampler(c, 0, sampler))) return rc;
    if ((rc = check_draws(c, u, c->B))) return rc;
    for (int b = 0; b < c->B; ++b) {
        if (tok[b] < 0 || tok[b] >= c->cfg.vocab)
            return fail(c, SD_ERR_INVALID_ARG, "token %d outside [0, %d)", tok[b], c->cfg.vocab);
        c->hs->tok[b] = tok[b];
        c->hs->u1[b] = u[b];
    }
    c->hs->prompt_on = 0; c->hs->u_seq = nullptr; c->hs->out_seq = nullptr;
    if ((rc = upload_inputs(c, false))) return rc;
    CK(cudaGraphLaunch(c->g_step, c->stream));
    if ((rc = download_counters(c, false))) return rc;
    for (int b = 0; b < c->B; ++b) out_tok[b] = c->hs->tok[b];
    c->host_pos++;
    return SD_OK;
}

int sd_decode_n(sd_ctx* c, int32_t n_steps, const sd_sampler* sampler, const float* u_dev, int32_t* out_dev) {
    if (!c || !u_dev || !out_dev) return fail(c, SD_ERR_INVALID_ARG, "sd_decode_n: NULL argument");
    if (c->cfg.arch == SD_ARCH_QWEN_TTS) return fail(c, SD_ERR_UNSUPPORTED, "sd_decode_n needs a GPT-2/Llama model");
    if (c->phase != Phase::Running) return fail(c, SD_ERR_STATE, "sd_decode_n before sd_prefill");
    if (n_steps < 0) return fail(c, SD_ERR_INVALID_ARG, "negative step count");
    if (c->host_pos + n_steps > c->cfg.max_ctx) return fail(c, SD_ERR_CTX_FULL, "context would overflow");
    CK(cudaSetDevice(c->device));
    int rc;
    if ((rc = set_sampler(c, 0, sampler))) return rc;
    c->hs->prompt_on = 0; c->hs->u_seq = u_dev; c->hs->out_seq = out_dev;
    if ((rc = upload_inputs(c, false))) return rc;
    CK(cudaMemsetAsync(&c->ds->step_idx, 0, sizeof(int32_t), c->stream));
    if (c->persistent && !c->ladder_on) {
        if (n_steps > 0 && (rc = enqueue_persistent(c, n_steps, u_dev, out_dev, c->stream))) return rc;
    } else {
        for (int i = 0; i < n_steps; ++i) CK(cudaGraphLaunch(c->g_step, c->stream));
    }
    rc = download_counters(c, false);  // synchronises before the staging mirror changes
    // later per-step calls upload null sequence pointers
    c->hs->u_seq = nullptr; c->hs->out_seq = nullptr;
    if (rc) return rc;
    if (c->persistent && !c->ladder_on) write_trace(c, n_steps);
    c->host_pos += n_steps;
    return SD_OK;
}

int sd_frame(sd_ctx* c, const int32_t* codes_in, const sd_sampler* talker, const sd_sampler* cp, const float* u,
             int32_t* codes_out) {
    if (!c || !codes_in || !u || !codes_out) return fail(c, SD_ERR_INVALID_ARG, "sd_frame: NULL argument");
    if (c->cfg.arch != SD_ARCH_QWEN_TTS) return fail(c, SD_ERR_UNSUPPORTED, "sd_frame needs a Talker+CP model");
    if (c->phase != Phase::Running) return fail(c, SD_ERR_STATE, "sd_frame before sd_prefill");
    if (c->host_pos >= c->cfg.max_ctx) return fail(c, SD_ERR_CTX_FULL, "context full (%d)", c->host_pos);
    CK(cudaSetDevice(c->device));
    const int B = c->B, ns = c->cfg.n_codebooks;
    int rc;
    if ((rc = set_sampler(c, 0, talker)) || (rc = set_sampler(c, 1, cp))) return rc;
    for (int b = 0; b < B; ++b) {
        if ((rc = check_draws(c, u + b * ns, ns))) return rc;
        for (int j = 0; j < ns; ++j) {
            const int v = codes_in[b * ns + j], V = j ? c->cfg.cp_vocab : c->cfg.vocab;
            if (v < 0 || v >= V) return fail(c, SD_ERR_INVALID_ARG, "code [%d][%d]=%d out of range", b, j, v);
            c->hs->codes_in[b * kMaxCodebooks + j] = v;
            c->hs->u[b * kMaxCodebooks + j] = u[b * ns + j];
        }
    }
    c->hs->prompt_on = 0;
    c->hs->force_on = c->force_pending ? 1 : 0;
    if ((rc = upload_inputs(c, true))) return rc;
    CK(cudaGraphLaunch(c->g_frame, c->stream));
    c->force_pending = false;
    rc = download_counters(c, true);
    c->hs->force_on = 0;
    if (rc) return rc;
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < ns; ++j) codes_out[b * ns + j] = c->hs->codes[b * kMaxCodebooks + j];
    c->host_pos++;
    return SD_OK;
}

int sd_get_logits(sd_ctx* c, float* host_out, size_t n_floats) {
    if (!c || !host_out) return fail(c, SD_ERR_INVALID_ARG, "sd_get_logits: NULL argument");
    const size_t need = (size_t)c->B * c->logits_ld;
    if (n_floats < need) return fail(c, SD_ERR_INVALID_ARG, "need %zu floats", need);
    CK(cudaSetDevice(c->device));
    CK(cudaMemcpyAsync(host_out, c->logits, need * sizeof(float), cudaMemcpyDeviceToHost, c->stream));
    CK(cudaStreamSynchronize(c->stream));
    return SD_OK;
}

int sd_get_info(const sd_ctx* c, sd_info* out) {
    if (!c || !out) return fail(nullptr, SD_ERR_INVALID_ARG, "sd_get_info: NULL argument");
    out->pos = c->host_pos;
    out->sm_count = c->sm_count;
    out->kernels_per_step = c->kernels_per_step;
    out->attn_splits = c->main.nsplit;
    out->persistent = c->persistent ? c->step_grid : 0;
    out->persistent_clusters = c->cpersistent ? c->cstep.ncl : 0;
    out->cluster_size = c->cpersistent ? c->cstep.cs : 0;
    out->prefill = !c->gemm_prefill ? 0 : (c->tc_prefill ? 2 : 1);
    out->weight_bytes = c->weight_bytes;
    out->kv_bytes = c->kv_bytes;
    const bool qwen = c->cfg.arch == SD_ARCH_QWEN_TTS;
    out->step_h2d_bytes = (int64_t)(qwen ? kFrameH2D : kStepH2D);
    out->step_d2h_bytes = (int64_t)(qwen ? kFrameD2H : kStepD2H);
    return SD_OK;
}

void sd_destroy(sd_ctx* c) {
    if (!c) return;
    cudaSetDevice(c->device);
    if (c->stream) cudaStreamSynchronize(c->stream);
    for (cudaGraphExec_t g : {c->g_step, c->g_body, c->g_frame, c->g_prompt_last})
        if (g) cudaGraphExecDestroy(g);
    for (void* p : c->allocs) cudaFree(p);
    if (c->weights) cudaFree(c->weights);
    if (c->hs) cudaFreeHost(c->hs);
    if (c->cap) cudaStreamDestroy(c->cap);
    if (c->own_stream && c->stream) cudaStreamDestroy(c->stream);
    delete c;
}

// ======================================================================= op-level ABI

struct sd_qmat {
    QMat m;
    void* buf = nullptr;
    int device = 0;
    __half* split = nullptr;  // dequantised fp16 hi [rows][cols] then lo, made on first tensor-core use
    float* g16_ws = nullptr;  // skinny GEMM partial sums, made on first use
    int* g16_cnt = nullptr;   // skinny GEMM column-tile counters (zero between launches)
};

int sd_qmat_create(int quant, const void* canon, int64_t rows, int64_t cols, int on_device, int device, sd_qmat** out) {
    sd_ctx* c = nullptr;
    if (!canon || !out) return fail(c, SD_ERR_INVALID_ARG, "sd_qmat_create: NULL argument");
    *out = nullptr;
    if (!q_valid(quant) || rows < 1 || cols < 1 || rows > (1 << 24) || cols > 65536 || cols % q_group(quant))
        return fail(c, SD_ERR_INVALID_ARG, "sd_qmat_create: bad shape or kind");
    CK(cudaSetDevice(device));
    const size_t canon_bytes = q_canon_bytes(quant, (size_t)rows, (size_t)cols);
    const uint8_t* src = reinterpret_cast<const uint8_t*>(canon);
    void* staging = nullptr;
    if (!on_device) {
        CK(cudaMalloc(&staging, canon_bytes));
        CK(cudaMemcpy(staging, canon, canon_bytes, cudaMemcpyHostToDevice));
        src = reinterpret_cast<const uint8_t*>(staging);
    }
    sd_qmat* q = new sd_qmat();
    q->device = device;
    const size_t total = qbytes(quant, (int)rows, (int)cols);
    if (cudaMalloc(&q->buf, total) != cudaSuccess) {
        delete q;
        if (staging) cudaFree(staging);
        return fail(c, SD_ERR_OOM, "sd_qmat_create: cudaMalloc failed");
    }
    const size_t qsz = q_code_bytes(quant, (size_t)rows, (size_t)cols);
    q->m.kind = quant; q->m.rows = (int)rows; q->m.cols = (int)cols;
    q->m.q = reinterpret_cast<uint8_t*>(q->buf);
    q->m.s = reinterpret_cast<uint8_t*>(q->buf) + (qsz + 255) / 256 * 256;
    cudaError_t e = launch_repack(quant, src, (int)rows, (int)cols, 0, const_cast<uint8_t*>(q->m.q),
                                  const_cast<void*>(q->m.s), nullptr);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (staging) cudaFree(staging);
    if (e != cudaSuccess) {
        cudaFree(q->buf);
        delete q;
        return fail(c, SD_ERR_CUDA, "sd_qmat_create: repack failed: %s", cudaGetErrorString(e));
    }
    *out = q;
    return SD_OK;
}

void sd_qmat_destroy(sd_qmat* m) {
    if (!m) return;
    cudaSetDevice(m->device);
    cudaFree(m->buf);
    if (m->split) cudaFree(m->split);
    if (m->g16_ws) cudaFree(m->g16_ws);
    if (m->g16_cnt) cudaFree(m->g16_cnt);
    delete m;
}

int sd_qmat_dequant(const sd_qmat* m, float* out_dev, void* stream) {
    sd_ctx* c = nullptr;
    if (!m || !out_dev) return fail(c, SD_ERR_INVALID_ARG, "sd_qmat_dequant: NULL argument");
    CK(launch_dequant(m->m, out_dev, reinterpret_cast<cudaStream_t>(stream)));
    return SD_OK;
}

int sd_qmat_gemv(const sd_qmat* m, const float* x_dev, int32_t nb, const float* bias_dev, float* y_dev, void* stream) {
    sd_ctx* c = nullptr;
    if (!m || !x_dev || !y_dev || (nb != 1 && nb != 2)) return fail(c, SD_ERR_INVALID_ARG, "sd_qmat_gemv: bad argument");
    if (m->m.cols > 8192) return fail(c, SD_ERR_UNSUPPORTED, "sd_qmat_gemv: cols > 8192");
    int sms = 0;
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, m->device));
    GemvArgs a;
    a.W = m->m; a.nb = nb; a.x = x_dev; a.x_stride = m->m.cols; a.pro = PRO_NONE;
    a.epi = EPI_LINEAR; a.bias = bias_dev; a.y = y_dev; a.y_stride = m->m.rows;
    CK(launch_gemv(a, sms, reinterpret_cast<cudaStream_t>(stream)));
    return SD_OK;
}

int sd_qmat_gemm(const sd_qmat* m, const float* x_dev, int32_t M, int32_t epilogue, const float* bias_dev,
                 const float* resid_dev, float* y_dev, void* stream) {
    sd_ctx* c = nullptr;
    if (!m || !x_dev || !y_dev || M < 1 || epilogue < SD_EPI_LINEAR || epilogue > SD_EPI_SWIGLU)
        return fail(c, SD_ERR_INVALID_ARG, "sd_qmat_gemm: bad argument");
    if (epilogue == SD_EPI_SWIGLU && (bias_dev || m->m.rows % 2))
        return fail(c, SD_ERR_INVALID_ARG, "sd_qmat_gemm: SwiGLU needs even rows and no bias");
    QGemmArgs a;
    a.W = m->m; a.M = M; a.x = x_dev; a.ldx = m->m.cols; a.epi = epilogue; a.bias = bias_dev;
    a.resid = resid_dev; a.y = y_dev; a.ldy = epilogue == SD_EPI_SWIGLU ? m->m.rows / 2 : m->m.rows;
    CK(cudaSetDevice(m->device));
    CK(launch_qgemm(a, reinterpret_cast<cudaStream_t>(stream)));
    return SD_OK;
}

int sd_qmat_gemm16(sd_qmat* m, const float* x_dev, int32_t M, int32_t epilogue, const float* bias_dev,
                   const float* resid_dev, float* y_dev, void* stream) {
    sd_ctx* c = nullptr;
    if (!m || !x_dev || !y_dev || M < 1 || M > 16 || epilogue < SD_EPI_LINEAR || epilogue > SD_EPI_SWIGLU ||
        reinterpret_cast<uintptr_t>(x_dev) % 16)
        return fail(c, SD_ERR_INVALID_ARG, "sd_qmat_gemm16: bad argument");
    if (epilogue == SD_EPI_SWIGLU && (bias_dev || m->m.rows % 2))
        return fail(c, SD_ERR_INVALID_ARG, "sd_qmat_gemm16: SwiGLU needs even rows and no bias");
    CK(cudaSetDevice(m->device));
    int sms = 0;
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, m->device));
    const char* rg = getenv("SD_ROWS_GEMM");
    const bool tc = gemm16_tc_supported(m->m) && rg && strcmp(rg, "tc") == 0;
    if (!m->g16_ws) {
        size_t wsf = gemm16_ws_floats(m->m.rows, m->m.cols, sms);
        if (gemm16_tc_supported(m->m)) wsf = std::max(wsf, gemm16_tc_ws_floats(m->m.rows, m->m.cols, sms));
        CK(cudaMalloc(&m->g16_ws, sizeof(float) * wsf));
        CK(cudaMalloc(&m->g16_cnt, sizeof(int) * gemm16_tiles(m->m.rows)));
        CK(cudaMemset(m->g16_cnt, 0, sizeof(int) * gemm16_tiles(m->m.rows)));
    }
    Gemm16Args a;
    a.W = m->m; a.M = M; a.x = x_dev; a.ldx = m->m.cols; a.epi = epilogue; a.bias = bias_dev;
    a.resid = resid_dev; a.y = y_dev; a.ldy = epilogue == SD_EPI_SWIGLU ? m->m.rows / 2 : m->m.rows;
    a.ws = m->g16_ws; a.cnt = m->g16_cnt;
    CK(tc ? launch_gemm16_tc(a, sms, nullptr, reinterpret_cast<cudaStream_t>(stream))
          : launch_gemm16(a, sms, reinterpret_cast<cudaStream_t>(stream)));
    return SD_OK;
}

int sd_qmat_gemm_tc(sd_qmat* m, const float* x_dev, int32_t M, int32_t epilogue, const float* bias_dev,
                    const float* resid_dev, float* y_dev, void* stream) {
    sd_ctx* c = nullptr;
    if (!m || !x_dev || !y_dev || M < 1 || epilogue < SD_EPI_LINEAR || epilogue > SD_EPI_SWIGLU)
        return fail(c, SD_ERR_INVALID_ARG, "sd_qmat_gemm_tc: bad argument");
    if (epilogue == SD_EPI_SWIGLU && (bias_dev || m->m.rows % 2))
        return fail(c, SD_ERR_INVALID_ARG, "sd_qmat_gemm_tc: SwiGLU needs even rows and no bias");
    if (m->m.cols % 64) return fail(c, SD_ERR_UNSUPPORTED, "sd_qmat_gemm_tc: cols must be a multiple of 64");
    CK(cudaSetDevice(m->device));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t wn = (size_t)m->m.rows * m->m.cols, xn = (size_t)M * m->m.cols;
    if (!m->split) {
        CK(cudaMalloc(&m->split, 2 * wn * sizeof(__half)));
        CK(launch_dequant_split(m->m, m->split, m->split + wn, st));
    }
    __half* xs = nullptr;
    int* err = nullptr;
    CK(cudaMalloc(&xs, 2 * xn * sizeof(__half) + 256));
    err = reinterpret_cast<int*>(reinterpret_cast<char*>(xs) + 2 * xn * sizeof(__half));
    TcGemmArgs a;
    bool ok = tc_map_fp16(&a.xh, xs, M, m->m.cols, false) && tc_map_fp16(&a.xl, xs + xn, M, m->m.cols, false) &&
              tc_map_fp16(&a.wh, m->split, m->m.rows, m->m.cols, true) &&
              tc_map_fp16(&a.wl, m->split + wn, m->m.rows, m->m.cols, true);
    cudaError_t e = ok ? cudaSuccess : cudaErrorInvalidValue;
    a.M = M; a.N = m->m.rows; a.K = m->m.cols; a.epi = epilogue; a.bias = bias_dev; a.resid = resid_dev;
    a.y = y_dev; a.ldy = epilogue == SD_EPI_SWIGLU ? m->m.rows / 2 : m->m.rows; a.err = err;
    int clock_khz = 0;
    cudaDeviceGetAttribute(&clock_khz, cudaDevAttrClockRate, m->device);
    a.spin_budget = (long long)(clock_khz > 0 ? clock_khz : 2000000) * 200;
    if (e == cudaSuccess) e = cudaMemsetAsync(err, 0, 4, st);
    if (e == cudaSuccess) e = launch_split_rows(x_dev, m->m.cols, M, m->m.cols, xs, xs + xn, st);
    if (e == cudaSuccess) e = launch_gemm_tc(a, st);
    int herr = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&herr, err, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    cudaFree(xs);
    if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "sd_qmat_gemm_tc: %s", cudaGetErrorString(e));
    if (herr) return fail(c, SD_ERR_TIMEOUT, "sd_qmat_gemm_tc: a wait of the kernel timed out");
    return SD_OK;
}

int sd_sample_rows(const float* logits_dev, int32_t rows, int32_t V, const sd_sampler* s, const float* u_dev,
                   int32_t* out_dev, void* stream) {
    sd_ctx* c = nullptr;
    if (!logits_dev || !s || !u_dev || !out_dev || rows < 1 || rows > 65535 || V < 1 || V > 16384)
        return fail(c, SD_ERR_INVALID_ARG, "sd_sample_rows: bad argument");
    if (const int rc = sampler_check(s)) return fail(c, rc, "sd_sample_rows: sampler out of range or unsupported");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    SampParams* sp = nullptr;
    int* err = nullptr;
    CK(cudaMalloc(&sp, sizeof(SampParams) + 16));
    err = reinterpret_cast<int*>(reinterpret_cast<char*>(sp) + sizeof(SampParams));
    SampParams h{s->temperature, s->top_k, s->top_p, s->greedy, 1.0f};
    cudaError_t e = cudaMemcpyAsync(sp, &h, sizeof h, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(err, 0, 4, st);
    SampleArgs a;
    a.logits = logits_dev; a.ld = V; a.V = V; a.sp = sp; a.u = u_dev; a.u_stride = 1; a.u_off = 0;
    a.out = out_dev; a.out_stride = 1; a.out_off = 0; a.err = err;
    if (e == cudaSuccess) e = launch_sample(a, rows, st);
    int herr = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&herr, err, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    cudaFree(sp);
    if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "sd_sample_rows: %s", cudaGetErrorString(e));
    if (herr) return fail(c, SD_ERR_DEVICE, "sd_sample_rows: kernel flagged code %d", herr);
    return SD_OK;
}

int sd_sample_rows_ladder(const float* logits_cond_dev, const float* logits_uncond_dev, int32_t rows, int32_t V,
                          const sd_sampler_ladder* s, const uint8_t* seen_dev, const float* u_dev, int32_t* out_dev,
                          void* stream) {
    sd_ctx* c = nullptr;
    if (!logits_cond_dev || !s || !u_dev || !out_dev || rows < 1 || rows > 65535 || V < 1 || V > 16384)
        return fail(c, SD_ERR_INVALID_ARG, "sd_sample_rows_ladder: bad argument");
    if (!(s->repetition_penalty > 0.f) || !(s->min_p >= 0.f) || !(s->top_p > 0.f && s->top_p <= 1.f) ||
        !(s->temperature == s->temperature) || !(s->cfg_weight == s->cfg_weight))
        return fail(c, SD_ERR_INVALID_ARG, "sd_sample_rows_ladder: sampler out of range");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    LadderParams p;
    p.cfg_weight = s->cfg_weight; p.rep_penalty = s->repetition_penalty; p.temperature = s->temperature;
    p.min_p = s->min_p; p.top_p = s->top_p; p.top_k = s->top_k;
    cudaError_t e = launch_sample_ladder(logits_cond_dev, logits_uncond_dev, rows, V, p, seen_dev, u_dev, out_dev, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "sd_sample_rows_ladder: %s", cudaGetErrorString(e));
    return SD_OK;
}

int sd_attend_rows(const float* q_dev, const uint16_t* k_dev, const uint16_t* v_dev, int32_t B, int32_t H, int32_t Hkv,
                   int32_t hd, int32_t n_ctx, int32_t n, int32_t nsplit, float* out_dev, void* stream) {
    sd_ctx* c = nullptr;
    if (!q_dev || !k_dev || !v_dev || !out_dev || B < 1 || H < 1 || Hkv < 1 || H % Hkv || H / Hkv > 4 ||
        (hd != 64 && hd != 128) || n < 1 || n > n_ctx || nsplit < 1 || nsplit > 64)
        return fail(c, SD_ERR_INVALID_ARG, "sd_attend_rows: bad argument");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float* part = nullptr;
    const size_t pbytes = sizeof(float) * B * H * nsplit * part_stride(hd);
    const size_t cbytes = sizeof(int) * (size_t)B * Hkv;
    CK(cudaMalloc(&part, pbytes + cbytes + 16));
    int* counters = reinterpret_cast<int*>(reinterpret_cast<char*>(part) + pbytes);
    int* pos = counters + (size_t)B * Hkv;
    const int pm1 = n - 1;
    cudaError_t e = cudaMemcpyAsync(pos, &pm1, 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(counters, 0, cbytes, st);
    AttnArgs a;
    a.q = q_dev; a.q_stride = H * hd; a.knew = nullptr; a.vnew = nullptr;
    a.kc = reinterpret_cast<__half*>(const_cast<uint16_t*>(k_dev));
    a.vc = reinterpret_cast<__half*>(const_cast<uint16_t*>(v_dev));
    a.row_heads = Hkv; a.head_off = 0; a.n_head = H; a.n_kv = Hkv; a.hd = hd; a.n_ctx = n_ctx; a.nsplit = nsplit;
    a.pos_ptr = pos; a.part = part; a.counters = counters; a.out = out_dev; a.out_stride = H * hd; a.max_len = n;
    if (e == cudaSuccess) e = launch_attention(a, B, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    cudaFree(part);
    if (e != cudaSuccess) return fail(c, SD_ERR_CUDA, "sd_attend_rows: %s", cudaGetErrorString(e));
    return SD_OK;
}

}  // extern "C"
