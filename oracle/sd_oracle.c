/*
 * Oracle of the speech-token decode step -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain C restatement of the decode step of three speech-token transformers:
 *   - GPT-2-Medium-style T3 ("Chatterbox -> ggml Port: Development Journal",
 *     section 3.2: prompt graph and step graph sharing one KV cache);
 *   - the Llama-style multilingual T3 (journal section 3.19: RMSNorm, SwiGLU,
 *     separate Q/K/V projections, NEOX RoPE);
 *   - the Qwen3-style Talker plus 15-pass code predictor ("Every Frame Is a
 *     Memory Read", section 1).
 * Weights are block-quantised (journal Tier A item A3, section 3.23 for the
 * Q4_0 byte layout, A3 for Q5_0; the blog's section 3 for affine group-64
 * 8-bit and section 5.8 for the 4-bit group-32 / group-64 code predictor).
 *
 * Nothing here is blocked, fused or reordered: each linear layer dequantises a
 * row and takes one double-precision dot product; attention scores, softmax and
 * the weighted value sum are plain loops.  Prefill is the same per-position
 * routine as decode.  The only concurrency is an optional OpenMP split over
 * independent output rows of a linear layer, which leaves every sum unchanged.
 *
 * Only the tests, the smoke entry and the benchmark's CPU-baseline leg load
 * this file's library.
 */
#include "sd_oracle.h"

#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { K_F32 = 0, K_Q8_0 = 1, K_Q4_0 = 2, K_A8G64 = 3, K_Q5_0 = 4, K_A4G32 = 5, K_A4G64 = 6 };
#define K_LAST K_A4G64
/* affine kinds (codes, then per-group fp16 scales, then per-group fp16 biases) and their group size */
static int is_affine(int kind) { return kind == K_A8G64 || kind == K_A4G32 || kind == K_A4G64; }
static int group_of(int kind) { return kind == K_A4G32 ? 32 : is_affine(kind) ? 64 : 32; }

/* Planted mistakes for the pin tests (tests/test_oracle_mutants.py): a build
 * with -DORC_MUTANT=n carries mistake n, and the pins must reject it.  Normal
 * builds leave ORC_MUTANT at 0 and none of these branches exist.
 *   1 fp16 rounding truncates          2 Q4_0 nibble halves swapped
 *   3 Q8_0 codes read unsigned         4 affine group bias dropped
 *   5 linear layer bias dropped        6 LayerNorm unbiased variance
 *   7 RMSNorm gain dropped             8 GELU with erf instead of tanh form
 *   9 RoPE rotates the wrong way      10 attention scores unscaled
 *  11 attention misses the newest key 12 sampler drops top-k ties
 *  13 top-p cut one element late      14 draw in probability order
 *  15 temperature multiplies          16 attention residual dropped
 *  17 SwiGLU gate and up swapped      18 query heads interleaved over KV heads
 *  19 RoPE skipped on keys         20 repetition penalty backwards
 *  21 ladder: top-k before top-p     22 margin ignores membership flips
 *  23 margin taken as if T were 1    24 top-p bound counts t before itself
 *  25 mass factor 1+r instead of its square root
 *  26 Q5_0 fifth bit taken from the wrong element
 *  27 4-bit affine codes read high nibble first
 *  28 plain sampler's penalty backwards                                   */
#ifndef ORC_MUTANT
#define ORC_MUTANT 0
#endif
enum { A_GPT2 = 1, A_LLAMA = 2, A_QWEN = 3 };

/* ------------------------------------------------------------------ fp16 */

float orc_half_to_float(uint16_t h) {
    int sign = (h >> 15) & 1, ex = (h >> 10) & 0x1f, man = h & 0x3ff;
    double v;
    if (ex == 0)
        v = ldexp((double)man, -24);                   /* subnormal: man * 2^-24 */
    else if (ex == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + man), ex - 25);      /* (1 + man/1024) * 2^(ex-15) */
    return (float)(sign ? -v : v);
}

uint16_t orc_float_to_half(float f) {
    double a = fabs((double)f);
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    if (isnan(f)) return 0x7e00;
    if (a >= 65520.0) return sign | 0x7c00;            /* rounds past the largest finite half */
    if (a < ldexp(1.0, -14)) {                          /* subnormal range: units of 2^-24 */
        double m = rint(a * ldexp(1.0, 24));            /* round half to even */
        return sign | (uint16_t)m;                      /* m == 1024 is the smallest normal */
    }
    int e;
    frexp(a, &e);                                       /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;                                             /* a in [2^e, 2^(e+1)) */
#if ORC_MUTANT == 1
    double m = floor(ldexp(a, 10 - e));
#else
    double m = rint(ldexp(a, 10 - e));                  /* in [1024, 2048] */
#endif
    if (m == 2048.0) { m = 1024.0; e += 1; }
    if (e + 15 >= 31) return sign | 0x7c00;
    return sign | (uint16_t)(((e + 15) << 10) | ((int)m - 1024));
}

/* ------------------------------------------------------------------ dequantisation */

static void dequant_row(int kind, const uint8_t* data, int64_t r, int64_t cols, float* out) {
    if (kind == K_Q8_0) {
        const uint8_t* row = data + r * (cols / 32) * 34;
        for (int64_t b = 0; b < cols / 32; ++b) {
            const uint8_t* blk = row + b * 34;
            float d = orc_half_to_float((uint16_t)(blk[0] | (blk[1] << 8)));
#if ORC_MUTANT == 3
            for (int j = 0; j < 32; ++j) out[b * 32 + j] = d * (float)blk[2 + j];
#else
            for (int j = 0; j < 32; ++j) out[b * 32 + j] = d * (float)(int8_t)blk[2 + j];
#endif
        }
    } else if (kind == K_Q4_0) {
        const uint8_t* row = data + r * (cols / 32) * 18;
        for (int64_t b = 0; b < cols / 32; ++b) {
            const uint8_t* blk = row + b * 18;
            float d = orc_half_to_float((uint16_t)(blk[0] | (blk[1] << 8)));
            for (int j = 0; j < 32; ++j) {
                int byte = blk[2 + (j % 16)];
#if ORC_MUTANT == 2
                int nib = j < 16 ? (byte >> 4) : (byte & 0xf);
#else
                int nib = j < 16 ? (byte & 0xf) : (byte >> 4);
#endif
                out[b * 32 + j] = d * (float)(nib - 8);
            }
        }
    } else if (kind == K_Q5_0) {
        /* 22-byte blocks: fp16 d, 32 fifth bits (bit j of the little-endian word = element j),
         * then the low nibbles as in Q4_0; value d * (q - 16) */
        const uint8_t* row = data + r * (cols / 32) * 22;
        for (int64_t b = 0; b < cols / 32; ++b) {
            const uint8_t* blk = row + b * 22;
            float d = orc_half_to_float((uint16_t)(blk[0] | (blk[1] << 8)));
            uint32_t qh = (uint32_t)blk[2] | ((uint32_t)blk[3] << 8) | ((uint32_t)blk[4] << 16) | ((uint32_t)blk[5] << 24);
            for (int j = 0; j < 32; ++j) {
                int byte = blk[6 + (j % 16)];
                int nib = j < 16 ? (byte & 0xf) : (byte >> 4);
#if ORC_MUTANT == 26
                int hi = (int)((qh >> (31 - j)) & 1u);
#else
                int hi = (int)((qh >> j) & 1u);
#endif
                out[b * 32 + j] = d * (float)((nib | (hi << 4)) - 16);
            }
        }
    }
}

typedef struct {
    int kind;
    int64_t rows, cols;
    const uint8_t* data;      /* quantised codes, or fp32 values */
    const uint16_t* scale;    /* affine kinds only */
    const uint16_t* bias;     /* affine kinds only */
} qmat;

static void qmat_row(const qmat* W, int64_t r, float* out) {
    if (is_affine(W->kind)) {
        /* value = scale * q + bias per group; 8-bit codes one per byte, 4-bit codes two per byte
         * (element 2i in the low nibble of byte i, element 2i+1 in the high nibble) */
        const int gs = group_of(W->kind), four = W->kind != K_A8G64;
        const uint8_t* q = W->data + r * (four ? W->cols / 2 : W->cols);
        const uint16_t* s = W->scale + r * (W->cols / gs);
        const uint16_t* b = W->bias + r * (W->cols / gs);
        for (int64_t g = 0; g < W->cols / gs; ++g) {
            const float sc = orc_half_to_float(s[g]), bi = orc_half_to_float(b[g]);
            for (int64_t k = g * gs; k < (g + 1) * gs; ++k) {
                int code;
                if (!four)
                    code = q[k];
#if ORC_MUTANT == 27
                else
                    code = (k & 1) ? (q[k / 2] & 0xf) : (q[k / 2] >> 4);
#else
                else
                    code = (k & 1) ? (q[k / 2] >> 4) : (q[k / 2] & 0xf);
#endif
#if ORC_MUTANT == 4
                out[k] = sc * (float)code + 0.0f * bi;
#else
                out[k] = fmaf(sc, (float)code, bi);
#endif
            }
        }
    } else if (W->kind == K_F32) {
        memcpy(out, (const float*)W->data + r * W->cols, (size_t)W->cols * sizeof(float));
    } else {
        dequant_row(W->kind, W->data, r, W->cols, out);
    }
}

static qmat make_qmat(int kind, const uint8_t* data, int64_t rows, int64_t cols) {
    qmat W = {kind, rows, cols, data, NULL, NULL};
    if (is_affine(kind)) {
        W.scale = (const uint16_t*)(data + rows * (kind == K_A8G64 ? cols : cols / 2));
        W.bias = W.scale + rows * (cols / group_of(kind));
    }
    return W;
}

int orc_dequant(int kind, const uint8_t* data, int64_t rows, int64_t cols, float* out) {
    if (kind < K_Q8_0 || kind > K_LAST || cols % group_of(kind)) return -1;
    qmat W = make_qmat(kind, data, rows, cols);
    for (int64_t r = 0; r < rows; ++r) qmat_row(&W, r, out + r * cols);
    return 0;
}

/* ------------------------------------------------------------------ linear */

static int g_threads = 1;

int orc_set_threads(int n) {
#ifdef _OPENMP
    g_threads = n > 0 ? n : 1;
    return g_threads;
#else
    (void)n;
    g_threads = 1;
    return 1;
#endif
}

static void linear_q(const qmat* W, const float* x, const float* bias, float* y) {
    int64_t rows = W->rows, cols = W->cols;
#ifdef _OPENMP
#pragma omp parallel num_threads(g_threads)
#endif
    {
        float* w = (float*)malloc((size_t)cols * sizeof(float));
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
        for (int64_t r = 0; r < rows; ++r) {
            qmat_row(W, r, w);
            double acc = 0.0;
            for (int64_t k = 0; k < cols; ++k) acc += (double)w[k] * (double)x[k];
#if ORC_MUTANT != 5
            if (bias) acc += (double)bias[r];
#else
            (void)bias;
#endif
            y[r] = (float)acc;
        }
        free(w);
    }
}

int orc_linear(int kind, const uint8_t* data, int64_t rows, int64_t cols,
               const float* x, const float* b, float* y) {
    if (kind < K_F32 || kind > K_LAST || (kind != K_F32 && cols % group_of(kind))) return -1;
    qmat W = make_qmat(kind, data, rows, cols);
    linear_q(&W, x, b, y);
    return 0;
}

/* ------------------------------------------------------------------ elementwise */

void orc_layernorm(const float* x, int n, const float* g, const float* b, float eps, float* out) {
    double mu = 0.0, var = 0.0;
    for (int i = 0; i < n; ++i) mu += x[i];
    mu /= n;
    for (int i = 0; i < n; ++i) var += ((double)x[i] - mu) * ((double)x[i] - mu);
#if ORC_MUTANT == 6
    var /= (n - 1);
#else
    var /= n;                                       /* biased variance */
#endif
    double r = 1.0 / sqrt(var + (double)eps);
    for (int i = 0; i < n; ++i) out[i] = (float)(((double)x[i] - mu) * r * (double)g[i] + (double)b[i]);
}

void orc_rmsnorm(const float* x, int n, const float* g, float eps, float* out) {
    double ms = 0.0;
    for (int i = 0; i < n; ++i) ms += (double)x[i] * (double)x[i];
    ms /= n;
    double r = 1.0 / sqrt(ms + (double)eps);
#if ORC_MUTANT == 7
    (void)g;
    for (int i = 0; i < n; ++i) out[i] = (float)((double)x[i] * r);
#else
    for (int i = 0; i < n; ++i) out[i] = (float)((double)x[i] * r * (double)g[i]);
#endif
}

float orc_gelu_tanh(float t) {
    double x = t;
#if ORC_MUTANT == 8
    return (float)(0.5 * x * (1.0 + erf(x / sqrt(2.0))));
#else
    return (float)(0.5 * x * (1.0 + tanh(sqrt(2.0 / 3.14159265358979323846) * (x + 0.044715 * x * x * x))));
#endif
}

float orc_silu(float t) {
    double x = t;
    return (float)(x / (1.0 + exp(-x)));
}

void orc_rope(float* x, int hd, int pos, float theta) {
    int half = hd / 2;
    for (int i = 0; i < half; ++i) {
        double freq = pow((double)theta, -2.0 * i / hd);
        double phi = (double)pos * freq;
#if ORC_MUTANT == 9
        double c = cos(phi), s = -sin(phi);
#else
        double c = cos(phi), s = sin(phi);
#endif
        double a = x[i], b = x[i + half];
        x[i] = (float)(a * c - b * s);
        x[i + half] = (float)(a * s + b * c);
    }
}

void orc_attend(const float* q, const uint16_t* k, const uint16_t* v, int n, int hd, float* out) {
    double* s = (double*)malloc((size_t)n * sizeof(double));
#if ORC_MUTANT == 10
    double scale = 1.0;
#else
    double scale = 1.0 / sqrt((double)hd);
#endif
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int d = 0; d < hd; ++d) acc += (double)q[d] * (double)orc_half_to_float(k[(size_t)j * hd + d]);
        s[j] = acc * scale;
        if (s[j] > m) m = s[j];
    }
    double z = 0.0;
    for (int j = 0; j < n; ++j) { s[j] = exp(s[j] - m); z += s[j]; }
    for (int d = 0; d < hd; ++d) {
        double acc = 0.0;
        for (int j = 0; j < n; ++j) acc += s[j] * (double)orc_half_to_float(v[(size_t)j * hd + d]);
        out[d] = (float)(acc / z);
    }
    free(s);
}

/* ------------------------------------------------------------------ sampler */

typedef struct { double z; int32_t i; } zi;

static int cmp_desc(const void* a, const void* b) {
    const zi* x = (const zi*)a; const zi* y = (const zi*)b;
    if (x->z > y->z) return -1;
    if (x->z < y->z) return 1;
    return (x->i > y->i) - (x->i < y->i);           /* ties: lower index first */
}

/* ------------------------------------------------------------------ decision margin
 *
 * The pages define no margin for a sampled decision.  Here it is the size of the
 * smallest change of the decision's inputs that can change the chosen token,
 * in one unit r:
 *   - the draw u moved by r (u is a normalised position on the kept mass);
 *   - every unnormalised probability multiplied by its own factor within
 *     [(1+r)^-1/2, (1+r)^1/2], i.e. every scaled logit z/T moved by at most
 *     log1p(r)/2 (a logit error d at temperature T is r = expm1(2d/T)).
 * Every selection stage (top-k, top-p, min_p) keeps a prefix of its input in
 * (scaled logit desc, index asc) order, so after all stages an element's
 * membership can flip under a change of size r only if it lies between the
 * prefix that surely stays and the prefix that possibly stays; both are
 * bounded stage by stage below.  Two facts bound the token's CDF edges:
 * changing every mass by a factor within [1/a, a] (a^2 = 1+r) moves a
 * normalised edge by at most r/4; adding or removing mass F moves it by at most
 * F over the remaining total.  So the token cannot change while
 *   r < its distance to the CDF edges between kept entries (u moved), and
 *   r/4 + (1+r)F/(zs - (1+r)F) < its distance to its interval's ends
 * (F = mass of the entries whose membership can flip, zs = kept mass).  The
 * margin is the largest such r, found by bisection: the condition is monotone
 * in r.  It never exceeds the smallest change that flips the token, and it is
 * the draw's distance itself when no membership flip can move the token's
 * edges that far. */

enum { SEL_TOPK = 1, SEL_TOPP = 2, SEL_MINP = 3 };
typedef struct { int kind; int32_t k; double p; } sel_stage;

/* positions t with zz[t] > x, and with zz[t] >= x (zz descending) */
static int32_t n_above(const double* zz, int32_t V, double x) {
    int32_t lo = 0, hi = V;
    while (lo < hi) { int32_t mid = lo + (hi - lo) / 2; if (zz[mid] > x) lo = mid + 1; else hi = mid; }
    return lo;
}
static int32_t n_at_or_above(const double* zz, int32_t V, double x) {
    int32_t lo = 0, hi = V;
    while (lo < hi) { int32_t mid = lo + (hi - lo) / 2; if (zz[mid] >= x) lo = mid + 1; else hi = mid; }
    return lo;
}

/* Lengths *nq <= *np of the sorted prefixes that surely / possibly survive all
 * stages under every change of size r.  zz: scaled logits sorted descending
 * (ties: lower index first); cw[t] = sum of exp(zz[i] - zz[0]) over i < t. */
static void kept_bounds(const double* zz, const double* cw, int32_t V, const sel_stage* st, int n_st, double r,
                        int32_t* nq_out, int32_t* np_out) {
    const double L = log1p(r);            /* largest change of a difference of two scaled logits */
#if ORC_MUTANT == 25
    const double a = 1.0 + r;
#else
    const double a = sqrt(1.0 + r);       /* largest factor on one mass */
#endif
    int32_t np = V, nq = V;                /* before the first stage every entry is present */
    for (int s = 0; s < n_st; ++s) {
        int32_t np2 = 0, nq2 = 0;
        if (st[s].kind == SEL_TOPK) {
            /* kept iff fewer than k present entries lie strictly above.  t can stay
             * if fewer than k surely-present entries surely lie above it; t surely
             * stays if fewer than k possibly-present others can lie above it. */
            const int32_t k = st[s].k;
            while (np2 < np) {
                int32_t above = n_above(zz, V, zz[np2] + L);
                if (above > nq) above = nq;
                if (above >= k) break;
                ++np2;
            }
            while (nq2 < nq) {
                int32_t above = n_at_or_above(zz, V, zz[nq2] - L);
                if (above > np) above = np;
                if (above - 1 >= k) break;     /* less t itself */
                ++nq2;
            }
        } else if (st[s].kind == SEL_TOPP) {
            /* kept iff the mass of the present entries ordered before t, over the
             * present total, is below p.  Least that share can be: only the
             * surely-present entries surely above t count before it, shrunk, and
             * every possibly-present entry not surely above t counts after it,
             * grown.  Most: every possibly-present entry that can be above t counts
             * before it, grown, and only t and the surely-present entries surely
             * below it count after it, shrunk. */
            const double p = st[s].p;
            while (np2 < np) {
                const int32_t t = np2;
                const int32_t m = n_above(zz, V, zz[t] + L);
                const int32_t mq = m < nq ? m : nq;
                const double B = cw[mq] / a, R = (cw[np] - cw[m]) * a;
                if (B / (B + R) >= p) break;
                ++np2;
            }
            while (nq2 < nq) {
                const int32_t t = nq2;
                const int32_t j = n_at_or_above(zz, V, zz[t] - L);
                const int32_t jp = j < np ? j : np;
                const double w_t = cw[t + 1] - cw[t];
#if ORC_MUTANT == 24
                const double B = cw[jp] * a;
#else
                const double B = (cw[jp] - w_t) * a;
#endif
                const double R = (w_t + (j < nq ? cw[nq] - cw[j] : 0.0)) / a;
                if (B / (B + R) >= p) break;
                ++nq2;
            }
        } else {
            /* min_p, the first stage: kept iff its probability is at least p times
             * the largest, i.e. zz[t] - zz[0] >= log p; the largest moves too */
            const double lp = log(st[s].p);
            while (np2 < np && zz[np2] - zz[0] + L >= lp) ++np2;
            while (nq2 < nq && zz[nq2] - zz[0] - L >= lp) ++nq2;
        }
        np = np2;
        nq = nq2 < np2 ? nq2 : np2;
    }
    *nq_out = nq;
    *np_out = np;
}

/* can membership flips under a change of size r move the token's edges by m_edge? */
static int flips_reach(const double* zz, const double* cw, int32_t V, const sel_stage* st, int n_st, double zs,
                       double m_edge, double r) {
    int32_t nq, np;
    kept_bounds(zz, cw, V, st, n_st, r, &nq, &np);
    const double F = cw[np] - cw[nq];
    if (!(F > 0.0)) return 0;
    const double rest = zs - (1.0 + r) * F;
    if (rest <= 0.0) return 1;
    return r / 4.0 + (1.0 + r) * F / rest >= m_edge;
}

/* The margin of a sampled draw.  s: every entry's scaled logit in (desc, index
 * asc) order; kept[i]: entry i survived every stage; the draw chose `tok`,
 * whose interval on the kept mass zs is [c_lo, c) and holds target = u zs. */
static double draw_margin(const zi* s, int32_t V, const sel_stage* st, int n_st, const char* kept, int32_t tok,
                          double target, double c_lo, double c, double zs) {
    int32_t first = -1, last = -1;
    for (int32_t i = 0; i < V; ++i) if (kept[i]) { if (first < 0) first = i; last = i; }
    double lo_d = target - c_lo, hi_d = c - target;
    if (lo_d < 0.0) lo_d = 0.0;
    if (hi_d < 0.0) hi_d = 0.0;
    /* distance to the interval's ends, and to the edges shared with another kept
     * entry (the ends of [0, 1) are not reachable by moving u) */
    const double m_edge = fmin(lo_d, hi_d) / zs;
    const double m_move = fmin(tok != first ? lo_d : INFINITY, tok != last ? hi_d : INFINITY) / zs;
#if ORC_MUTANT == 22
    (void)st; (void)n_st; (void)s; (void)m_edge; (void)flips_reach;
    return m_move;
#else
    double* zz = (double*)malloc((size_t)V * sizeof(double));
    double* cw = (double*)malloc((size_t)(V + 1) * sizeof(double));
    cw[0] = 0.0;
    for (int32_t t = 0; t < V; ++t) {
        zz[t] = s[t].z;
        cw[t + 1] = cw[t] + exp(s[t].z - s[0].z);
    }
    double m;
    double hi = m_move < 1e6 ? m_move : 1e6;
    if (!flips_reach(zz, cw, V, st, n_st, zs, m_edge, hi)) {
        m = m_move;
    } else if (flips_reach(zz, cw, V, st, n_st, zs, m_edge, 0.0)) {
        m = 0.0;
    } else {
        double lo = 0.0;
        for (int it = 0; it < 200; ++it) {
            const double mid = 0.5 * (lo + hi);
            if (flips_reach(zz, cw, V, st, n_st, zs, m_edge, mid)) hi = mid; else lo = mid;
        }
        m = lo;
    }
    free(zz);
    free(cw);
    return m;
#endif
}

int32_t orc_sample(const float* z, int32_t V, float temperature, int32_t top_k, float top_p,
                   int32_t greedy, double u, double* margin) {
    if (V <= 0) return -1;
    if (greedy || top_k == 1 || temperature <= 0.0f) {
        int32_t best = 0;
        for (int32_t i = 1; i < V; ++i) if (z[i] > z[best]) best = i;
        double second = -INFINITY;
        for (int32_t i = 0; i < V; ++i) if (i != best && (double)z[i] > second) second = z[i];
        if (margin) *margin = V > 1 ? (double)z[best] - second : INFINITY;
        return best;
    }
#if ORC_MUTANT == 15
    double inv_t = (double)temperature;
#else
    double inv_t = 1.0 / (double)temperature;
#endif
    zi* s = (zi*)malloc((size_t)V * sizeof(zi));
    for (int32_t i = 0; i < V; ++i) { s[i].z = (double)z[i] * inv_t; s[i].i = i; }
    qsort(s, (size_t)V, sizeof(zi), cmp_desc);
    /* top-k: keep every value >= the k-th largest (ties at the threshold kept) */
    int32_t k = top_k < 1 || top_k > V ? V : top_k;
    double thr = s[k - 1].z;
    int32_t n_keep = 0;
#if ORC_MUTANT == 12
    (void)thr;
    n_keep = k;
#else
    while (n_keep < V && s[n_keep].z >= thr) ++n_keep;
#endif
    /* softmax over the survivors (s is already in (p desc, index asc) order) */
    double zmax = s[0].z, Z = 0.0;
    double* p = (double*)malloc((size_t)V * sizeof(double));  /* indexed by vocabulary id */
    char* in_s = (char*)calloc((size_t)V, 1);
    for (int32_t t = 0; t < n_keep; ++t) p[s[t].i] = exp(s[t].z - zmax);
    for (int32_t t = 0; t < n_keep; ++t) in_s[s[t].i] = 1;
    for (int32_t i = 0; i < V; ++i) if (in_s[i]) Z += p[i];
    /* top-p: the shortest (p desc, index asc) prefix whose cumulative mass >= top_p */
    if (top_p < 1.0f) {
        double cum = 0.0;
        int32_t cut = n_keep - 1;
        for (int32_t t = 0; t < n_keep; ++t) {
            cum += p[s[t].i] / Z;
#if ORC_MUTANT == 13
            if (cum >= (double)top_p) { cut = t + 1 < n_keep ? t + 1 : t; break; }
#else
            if (cum >= (double)top_p) { cut = t; break; }
#endif
        }
        for (int32_t t = cut + 1; t < n_keep; ++t) in_s[s[t].i] = 0;
    }
    /* draw in vocabulary order */
    double zs = 0.0;
    for (int32_t i = 0; i < V; ++i) if (in_s[i]) zs += p[i];
    double target = u * zs, c = 0.0, c_lo = 0.0;
    int32_t tok = -1, last = -1;
#if ORC_MUTANT == 14
    for (int32_t t = 0; t < V; ++t) {
        const int32_t i = s[t].i;
#else
    for (int32_t i = 0; i < V; ++i) {
#endif
        if (!in_s[i]) continue;
        last = i;
        c_lo = c;
        c += p[i];
        if (c > target) { tok = i; break; }
    }
    if (tok < 0) { tok = last; c_lo = c - p[last]; }
    if (margin) {
        sel_stage st[2];
        int n_st = 0;
        st[n_st].kind = SEL_TOPK; st[n_st].k = k; st[n_st].p = 0.0; ++n_st;
        if (top_p < 1.0f) { st[n_st].kind = SEL_TOPP; st[n_st].k = 0; st[n_st].p = (double)top_p; ++n_st; }
#if ORC_MUTANT == 23
        for (int32_t t = 0; t < V; ++t) s[t].z = (double)z[s[t].i];   /* margin taken as if T were 1 */
#endif
        *margin = draw_margin(s, V, st, n_st, in_s, tok, target, c_lo, c, zs);
    }
    free(s); free(p); free(in_s);
    return tok;
}

/* The sampler with a repetition penalty over a history: every logit of a token
 * in seen[] is divided by the penalty when positive and multiplied by it
 * otherwise (the journal's HF rule; "Every Frame Is a Memory Read", section
 * 2: the Talker decodes with a penalty over the tokens it generated), then the
 * plain sampler runs on the penalised logits (rounded to fp32, the logits'
 * type).  seen may be NULL and rep_penalty 1: no penalty. */
int32_t orc_sample_pen(const float* z, int32_t V, const uint8_t* seen, float rep_penalty, float temperature,
                       int32_t top_k, float top_p, int32_t greedy, double u, double* margin) {
    if (V <= 0) return -1;
    float* zp = (float*)malloc((size_t)V * sizeof(float));
    for (int32_t i = 0; i < V; ++i) {
        double v = (double)z[i];
        if (seen && seen[i] && rep_penalty != 1.0f) {
#if ORC_MUTANT == 28
            v = v > 0.0 ? v * (double)rep_penalty : v / (double)rep_penalty;
#else
            v = v > 0.0 ? v / (double)rep_penalty : v * (double)rep_penalty;
#endif
        }
        zp[i] = (float)v;
    }
    int32_t tok = orc_sample(zp, V, temperature, top_k, top_p, greedy, u, margin);
    free(zp);
    return tok;
}

/* Sampler ladder of the multilingual T3 ("Chatterbox -> ggml Port:
 * Development Journal", the multilingual port's sampling path: CFG combine,
 * repetition penalty, temperature, min_p, top-p, top-k, multinomial).  Each
 * stage acts on the survivors of the previous one:
 *   z_i = c_i + w (c_i - u_i)                 (c conditional, u unconditional logits)
 *   seen i: z_i / penalty if z_i > 0, else z_i * penalty   (journal: the HF rule)
 *   z_i / T, p_i proportional to exp(z_i)
 *   min_p:  keep p_i >= min_p * max_j p_j
 *   top-p:  the shortest (p desc, index asc) prefix of the survivors whose
 *           renormalised mass reaches top_p
 *   top-k:  keep the survivors whose value is >= the k-th largest survivor's
 *   draw:   the smallest vocabulary index whose cumulative kept mass exceeds u
 *           times the kept total. */
int32_t orc_sample_ladder(const float* z_cond, const float* z_uncond, int32_t V, float cfg_weight,
                          const uint8_t* seen, float rep_penalty, float temperature, float min_p, float top_p,
                          int32_t top_k, double u, double* margin, double* draw_dist) {
    if (V <= 0) return -1;
    if (draw_dist) *draw_dist = INFINITY;
    double* z = (double*)malloc((size_t)V * sizeof(double));
    for (int32_t i = 0; i < V; ++i) {
        double c = z_cond[i];
        if (z_uncond && cfg_weight != 0.0f) c = c + (double)cfg_weight * (c - (double)z_uncond[i]);
        z[i] = c;
    }
    if (seen && rep_penalty != 1.0f)
        for (int32_t i = 0; i < V; ++i)
            if (seen[i]) {
#if ORC_MUTANT == 20
                z[i] = z[i] > 0.0 ? z[i] * (double)rep_penalty : z[i] / (double)rep_penalty;
#else
                z[i] = z[i] > 0.0 ? z[i] / (double)rep_penalty : z[i] * (double)rep_penalty;
#endif
            }
    if (temperature <= 0.0f) {
        int32_t best = 0;
        for (int32_t i = 1; i < V; ++i) if (z[i] > z[best]) best = i;
        double second = -INFINITY;
        for (int32_t i = 0; i < V; ++i) if (i != best && z[i] > second) second = z[i];
        if (margin) *margin = V > 1 ? z[best] - second : INFINITY;
        free(z);
        return best;
    }
    for (int32_t i = 0; i < V; ++i) z[i] /= (double)temperature;
    double mx = -INFINITY;
    for (int32_t i = 0; i < V; ++i) if (z[i] > mx) mx = z[i];
    double* p = (double*)malloc((size_t)V * sizeof(double));
    char* keep = (char*)malloc((size_t)V);
    for (int32_t i = 0; i < V; ++i) { p[i] = exp(z[i] - mx); keep[i] = 1; }
    /* min_p: relative to the largest probability, which is exp(0) = 1 here (the
     * largest always survives: min_p above 1 acts as 1) */
    if (min_p > 0.0f) {
        const double mp = min_p < 1.0f ? (double)min_p : 1.0;
        for (int32_t i = 0; i < V; ++i) if (p[i] < mp) keep[i] = 0;
    }
    /* survivors in (p desc, index asc) order: z desc, index asc */
    zi* s = (zi*)malloc((size_t)V * sizeof(zi));
    int32_t ns = 0;
    for (int32_t i = 0; i < V; ++i) if (keep[i]) { s[ns].z = z[i]; s[ns].i = i; ++ns; }
    qsort(s, (size_t)ns, sizeof(zi), cmp_desc);
#if ORC_MUTANT == 21
    /* top-k before top-p (the order of the first port) */
    {
        int32_t k = top_k < 1 || top_k > ns ? ns : top_k;
        int32_t n_keep = 0;
        while (n_keep < ns && s[n_keep].z >= s[k - 1].z) ++n_keep;
        for (int32_t t = n_keep; t < ns; ++t) keep[s[t].i] = 0;
        ns = n_keep;
    }
#endif
    if (top_p < 1.0f) {
        double mass = 0.0;
        for (int32_t t = 0; t < ns; ++t) mass += p[s[t].i];
        double cum = 0.0;
        int32_t cut = ns - 1;
        for (int32_t t = 0; t < ns; ++t) {
            cum += p[s[t].i] / mass;
            if (cum >= (double)top_p) { cut = t; break; }
        }
        for (int32_t t = cut + 1; t < ns; ++t) keep[s[t].i] = 0;
        ns = cut + 1;
    }
#if ORC_MUTANT != 21
    {
        int32_t k = top_k < 1 || top_k > ns ? ns : top_k;
        int32_t n_keep = 0;
        while (n_keep < ns && s[n_keep].z >= s[k - 1].z) ++n_keep;   /* ties at the k-th value kept */
        for (int32_t t = n_keep; t < ns; ++t) keep[s[t].i] = 0;
    }
#endif
    double zs = 0.0;
    for (int32_t i = 0; i < V; ++i) if (keep[i]) zs += p[i];
    double target = u * zs, c = 0.0, c_lo = 0.0;
    int32_t tok = -1, last = -1;
    for (int32_t i = 0; i < V; ++i) {
        if (!keep[i]) continue;
        last = i;
        c_lo = c;
        c += p[i];
        if (c > target) { tok = i; break; }
    }
    if (tok < 0) { tok = last; c_lo = c - p[last]; }
    if (draw_dist) *draw_dist = fmax(0.0, fmin(target - c_lo, c - target)) / zs;
    if (margin) {
        /* every entry in (desc, index asc) order, and the stages as applied */
        zi* a = (zi*)malloc((size_t)V * sizeof(zi));
        for (int32_t i = 0; i < V; ++i) { a[i].z = z[i]; a[i].i = i; }
        qsort(a, (size_t)V, sizeof(zi), cmp_desc);
        sel_stage st[3];
        int n_st = 0;
        if (min_p > 0.0f) { st[n_st].kind = SEL_MINP; st[n_st].k = 0; st[n_st].p = min_p < 1.0f ? (double)min_p : 1.0; ++n_st; }
        if (top_p < 1.0f) { st[n_st].kind = SEL_TOPP; st[n_st].k = 0; st[n_st].p = (double)top_p; ++n_st; }
        st[n_st].kind = SEL_TOPK; st[n_st].k = top_k < 1 ? V : top_k; st[n_st].p = 0.0; ++n_st;
        *margin = draw_margin(a, V, st, n_st, keep, tok, target, c_lo, c, zs);
        free(a);
    }
    free(z); free(p); free(keep); free(s);
    return tok;
}

/* ------------------------------------------------------------------ blob */

#define BLOB_MAGIC 0x31574453u
#define ENTRY_BYTES 96

typedef struct {
    char name[64];
    uint32_t kind, rows, cols;
    const uint8_t* data;
    uint64_t nbytes;
} otensor;

typedef struct {
    int32_t arch, n_layer, d_model, n_head, n_kv_head, head_dim, d_ff, vocab, max_ctx, batch, quant;
    float rope_theta, norm_eps;
    int32_t cp_layer, cp_d_model, cp_n_head, cp_n_kv_head, cp_head_dim, cp_d_ff, cp_vocab, n_codebooks, cp_max_ctx;
} ocfg;

typedef struct {
    const float *n1g, *n1b, *bqkv, *bo, *n2g, *n2b, *bfc, *bproj;
    qmat wqkv, wo, wfc, wproj;     /* wfc = stacked gate/up and wproj = down for SwiGLU stacks */
} olayer;

typedef struct {
    int gpt2;                      /* LayerNorm + biases + GELU, else RMSNorm + SwiGLU + RoPE */
    int n_layer, d, n_head, n_kv, hd, ff, max_ctx, batch;
    float eps, theta;
    olayer* L;
    const float *nfg, *nfb;
    uint16_t *kc, *vc;             /* [batch][layer][kv_head][max_ctx][hd] fp16 */
    int32_t* pos;                  /* [batch] */
    float *x, *h, *qkv, *o, *t, *u, *y;  /* scratch */
} ostack;

struct orc_model {
    ocfg c;
    uint32_t n_t;
    otensor* t;
    ostack s, cp;
    const float *wte, *wpe;
    qmat head, cp_proj;
    const float* emb[16];
    qmat cp_head[16];
};

static const otensor* find(const orc_model* m, const char* name) {
    for (uint32_t i = 0; i < m->n_t; ++i)
        if (strcmp(m->t[i].name, name) == 0) return &m->t[i];
    return NULL;
}

static int get_f32(const orc_model* m, const char* name, int64_t n, const float** out) {
    const otensor* t = find(m, name);
    if (!t || t->kind != K_F32 || (int64_t)t->rows * t->cols != n) {
        fprintf(stderr, "oracle: missing or mis-shaped fp32 tensor %s\n", name);
        return -1;
    }
    *out = (const float*)t->data;
    return 0;
}

static int get_q(const orc_model* m, const char* name, int64_t rows, int64_t cols, qmat* out) {
    const otensor* t = find(m, name);
    if (!t || t->kind == K_F32 || t->kind > K_LAST || t->rows != rows || t->cols != cols || cols % group_of((int)t->kind)) {
        fprintf(stderr, "oracle: missing or mis-shaped matrix %s\n", name);
        return -1;
    }
    *out = make_qmat((int)t->kind, t->data, rows, cols);
    return 0;
}

static uint32_t rd32(const uint8_t* p) { return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24); }
static uint64_t rd64(const uint8_t* p) { return (uint64_t)rd32(p) | ((uint64_t)rd32(p + 4) << 32); }

static int stack_alloc(ostack* s) {
    size_t kv = (size_t)s->batch * s->n_layer * s->n_kv * s->max_ctx * s->hd;
    int qkv_rows = (s->n_head + 2 * s->n_kv) * s->hd;
    int wide = s->ff * 2 > qkv_rows ? s->ff * 2 : qkv_rows;
    s->kc = (uint16_t*)calloc(kv, 2);
    s->vc = (uint16_t*)calloc(kv, 2);
    s->pos = (int32_t*)calloc((size_t)s->batch, 4);
    s->x = (float*)calloc((size_t)s->d, 4);
    s->h = (float*)calloc((size_t)s->d, 4);
    s->qkv = (float*)calloc((size_t)wide, 4);
    s->o = (float*)calloc((size_t)s->n_head * s->hd, 4);
    s->t = (float*)calloc((size_t)wide, 4);
    s->u = (float*)calloc((size_t)s->ff, 4);
    s->y = (float*)calloc((size_t)(s->d > s->ff ? s->d : s->ff), 4);
    return (s->kc && s->vc && s->pos && s->x && s->h && s->qkv && s->o && s->t && s->u && s->y) ? 0 : -1;
}

static void stack_free(ostack* s) {
    free(s->L); free(s->kc); free(s->vc); free(s->pos);
    free(s->x); free(s->h); free(s->qkv); free(s->o); free(s->t); free(s->u); free(s->y);
}

static int load_layers(orc_model* m, ostack* s, const char* pfx) {
    char nm[96];
    int d = s->d, qd = s->n_head * s->hd, qkv_rows = (s->n_head + 2 * s->n_kv) * s->hd;
    s->L = (olayer*)calloc((size_t)s->n_layer, sizeof(olayer));
    for (int l = 0; l < s->n_layer; ++l) {
        olayer* L = &s->L[l];
        int rc = 0;
#define F32(field, suffix, n) snprintf(nm, sizeof nm, "%s%d." suffix, pfx, l); rc |= get_f32(m, nm, n, &L->field)
#define QM(field, suffix, r, c) snprintf(nm, sizeof nm, "%s%d." suffix, pfx, l); rc |= get_q(m, nm, r, c, &L->field)
        if (s->gpt2) {
            F32(n1g, "ln1.g", d); F32(n1b, "ln1.b", d);
            QM(wqkv, "wqkv", qkv_rows, d); F32(bqkv, "bqkv", qkv_rows);
            QM(wo, "wo", d, qd); F32(bo, "bo", d);
            F32(n2g, "ln2.g", d); F32(n2b, "ln2.b", d);
            QM(wfc, "wfc", s->ff, d); F32(bfc, "bfc", s->ff);
            QM(wproj, "wproj", d, s->ff); F32(bproj, "bproj", d);
        } else {
            F32(n1g, "rms1.g", d); QM(wqkv, "wqkv", qkv_rows, d); QM(wo, "wo", d, qd);
            F32(n2g, "rms2.g", d); QM(wfc, "wgu", 2 * s->ff, d); QM(wproj, "wdown", d, s->ff);
        }
#undef F32
#undef QM
        if (rc) return -1;
    }
    return stack_alloc(s);
}

int orc_open(const uint8_t* blob, uint64_t nbytes, orc_model** out) {
    *out = NULL;
    if (nbytes < 144 || rd32(blob) != BLOB_MAGIC || rd32(blob + 4) != 1) return -1;
    orc_model* m = (orc_model*)calloc(1, sizeof(orc_model));
    memcpy(&m->c, blob + 16, sizeof(ocfg));
    m->n_t = rd32(blob + 8);
    uint32_t toff = rd32(blob + 12);
    if (toff + (uint64_t)m->n_t * ENTRY_BYTES > nbytes) { free(m); return -1; }
    m->t = (otensor*)calloc(m->n_t, sizeof(otensor));
    for (uint32_t i = 0; i < m->n_t; ++i) {
        const uint8_t* e = blob + toff + (uint64_t)i * ENTRY_BYTES;
        memcpy(m->t[i].name, e, 63);
        m->t[i].kind = rd32(e + 64); m->t[i].rows = rd32(e + 68); m->t[i].cols = rd32(e + 72);
        uint64_t off = rd64(e + 80), nb = rd64(e + 88);
        if (off + nb > nbytes) { orc_close(m); return -1; }
        m->t[i].data = blob + off; m->t[i].nbytes = nb;
    }
    ocfg* c = &m->c;
    ostack* s = &m->s;
    s->gpt2 = c->arch == A_GPT2;
    s->n_layer = c->n_layer; s->d = c->d_model; s->n_head = c->n_head; s->n_kv = c->n_kv_head;
    s->hd = c->head_dim; s->ff = c->d_ff; s->max_ctx = c->max_ctx; s->batch = c->batch;
    s->eps = c->norm_eps; s->theta = c->rope_theta;
    int rc = 0;
    if (c->arch == A_GPT2) {
        rc |= get_f32(m, "wte", (int64_t)c->vocab * c->d_model, &m->wte);
        rc |= get_f32(m, "wpe", (int64_t)c->max_ctx * c->d_model, &m->wpe);
        rc |= load_layers(m, s, "l");
        rc |= get_f32(m, "lnf.g", c->d_model, &s->nfg) | get_f32(m, "lnf.b", c->d_model, &s->nfb);
        rc |= get_q(m, "whead", c->vocab, c->d_model, &m->head);
    } else if (c->arch == A_LLAMA) {
        rc |= get_f32(m, "wte", (int64_t)c->vocab * c->d_model, &m->wte);
        rc |= load_layers(m, s, "l");
        rc |= get_f32(m, "normf.g", c->d_model, &s->nfg);
        rc |= get_q(m, "whead", c->vocab, c->d_model, &m->head);
    } else if (c->arch == A_QWEN) {
        char nm[64];
        if (c->n_codebooks < 2 || c->n_codebooks > 16) rc = -1;
        for (int j = 0; j < c->n_codebooks && !rc; ++j) {
            snprintf(nm, sizeof nm, "emb.%d", j);
            rc |= get_f32(m, nm, (int64_t)(j ? c->cp_vocab : c->vocab) * c->d_model, &m->emb[j]);
        }
        rc |= load_layers(m, s, "t");
        rc |= get_f32(m, "t.normf.g", c->d_model, &s->nfg);
        rc |= get_q(m, "t.head", c->vocab, c->d_model, &m->head);
        rc |= get_q(m, "cp.proj", c->cp_d_model, c->d_model, &m->cp_proj);
        ostack* p = &m->cp;
        p->gpt2 = 0;
        p->n_layer = c->cp_layer; p->d = c->cp_d_model; p->n_head = c->cp_n_head; p->n_kv = c->cp_n_kv_head;
        p->hd = c->cp_head_dim; p->ff = c->cp_d_ff; p->max_ctx = c->cp_max_ctx; p->batch = c->batch;
        p->eps = c->norm_eps; p->theta = c->rope_theta;
        rc |= load_layers(m, p, "c");
        rc |= get_f32(m, "cp.normf.g", c->cp_d_model, &p->nfg);
        for (int j = 1; j < c->n_codebooks && !rc; ++j) {
            snprintf(nm, sizeof nm, "cp.head.%d", j);
            rc |= get_q(m, nm, c->cp_vocab, c->cp_d_model, &m->cp_head[j]);
        }
    } else {
        rc = -1;
    }
    if (rc) { orc_close(m); return -1; }
    *out = m;
    return 0;
}

void orc_close(orc_model* m) {
    if (!m) return;
    stack_free(&m->s);
    stack_free(&m->cp);
    free(m->t);
    free(m);
}

void orc_reset(orc_model* m) {
    for (int b = 0; b < m->s.batch; ++b) m->s.pos[b] = 0;
    if (m->cp.pos) for (int b = 0; b < m->cp.batch; ++b) m->cp.pos[b] = 0;
}

int orc_pos(const orc_model* m, int row) { return m->s.pos[row]; }

int orc_copy_row(orc_model* m, int dst, int src) {
    ostack* s = &m->s;
    if (dst < 0 || src < 0 || dst >= s->batch || src >= s->batch) return -1;
    const size_t per_row = (size_t)s->n_layer * s->n_kv * s->max_ctx * s->hd;
    memcpy(s->kc + (size_t)dst * per_row, s->kc + (size_t)src * per_row, per_row * sizeof(uint16_t));
    memcpy(s->vc + (size_t)dst * per_row, s->vc + (size_t)src * per_row, per_row * sizeof(uint16_t));
    s->pos[dst] = s->pos[src];
    return 0;
}

/* ------------------------------------------------------------------ one transformer position */

/* Runs the stack on input x (d floats, overwritten) at the row's next position
 * and leaves the final-normed hidden state in s->h.  Returns -1 when full. */
static int stack_forward(ostack* s, int row, float* x) {
    int pos = s->pos[row];
    if (pos >= s->max_ctx) return -1;
    int d = s->d, hd = s->hd, H = s->n_head, Hk = s->n_kv, qd = H * hd, kd = Hk * hd;
    for (int l = 0; l < s->n_layer; ++l) {
        olayer* L = &s->L[l];
        /* attention block */
        if (s->gpt2) orc_layernorm(x, d, L->n1g, L->n1b, s->eps, s->h);
        else orc_rmsnorm(x, d, L->n1g, s->eps, s->h);
        linear_q(&L->wqkv, s->h, s->gpt2 ? L->bqkv : NULL, s->qkv);
        float *q = s->qkv, *k = s->qkv + qd, *v = s->qkv + qd + kd;
        if (!s->gpt2) {
            for (int h = 0; h < H; ++h) orc_rope(q + h * hd, hd, pos, s->theta);
#if ORC_MUTANT != 19
            for (int h = 0; h < Hk; ++h) orc_rope(k + h * hd, hd, pos, s->theta);
#endif
        }
        size_t layer_base = ((size_t)row * s->n_layer + l) * Hk;
        for (int g = 0; g < Hk; ++g) {
            size_t base = ((layer_base + g) * s->max_ctx + pos) * hd;
            for (int i = 0; i < hd; ++i) {
                s->kc[base + i] = orc_float_to_half(k[g * hd + i]);
                s->vc[base + i] = orc_float_to_half(v[g * hd + i]);
            }
        }
        for (int h = 0; h < H; ++h) {
#if ORC_MUTANT == 18
            int g = h % Hk;
#else
            int g = h / (H / Hk);                   /* contiguous query-head groups */
#endif
            size_t base = (layer_base + g) * s->max_ctx * hd;
#if ORC_MUTANT == 11
            orc_attend(q + h * hd, s->kc + base, s->vc + base, pos > 0 ? pos : 1, hd, s->o + h * hd);
#else
            orc_attend(q + h * hd, s->kc + base, s->vc + base, pos + 1, hd, s->o + h * hd);
#endif
        }
        linear_q(&L->wo, s->o, s->gpt2 ? L->bo : NULL, s->y);
#if ORC_MUTANT == 16
        for (int i = 0; i < d; ++i) x[i] = s->y[i];
#else
        for (int i = 0; i < d; ++i) x[i] = (float)((double)x[i] + (double)s->y[i]);
#endif
        /* MLP block */
        if (s->gpt2) {
            orc_layernorm(x, d, L->n2g, L->n2b, s->eps, s->h);
            linear_q(&L->wfc, s->h, L->bfc, s->t);
            for (int i = 0; i < s->ff; ++i) s->u[i] = orc_gelu_tanh(s->t[i]);
        } else {
            orc_rmsnorm(x, d, L->n2g, s->eps, s->h);
            linear_q(&L->wfc, s->h, NULL, s->t);    /* rows [0, ff) gate, [ff, 2ff) up */
            for (int i = 0; i < s->ff; ++i)
#if ORC_MUTANT == 17
                s->u[i] = (float)((double)orc_silu(s->t[s->ff + i]) * (double)s->t[i]);
#else
                s->u[i] = (float)((double)orc_silu(s->t[i]) * (double)s->t[s->ff + i]);
#endif
        }
        linear_q(&L->wproj, s->u, s->gpt2 ? L->bproj : NULL, s->y);
        for (int i = 0; i < d; ++i) x[i] = (float)((double)x[i] + (double)s->y[i]);
    }
    if (s->gpt2) orc_layernorm(x, d, s->nfg, s->nfb, s->eps, s->h);
    else orc_rmsnorm(x, d, s->nfg, s->eps, s->h);
    s->pos[row] = pos + 1;
    return 0;
}

int orc_token_forward(orc_model* m, int row, int32_t tok, float* logits) {
    ostack* s = &m->s;
    if (m->c.arch == A_QWEN || row < 0 || row >= s->batch || tok < 0 || tok >= m->c.vocab) return -1;
    int pos = s->pos[row], d = s->d;
    if (pos >= s->max_ctx) return -1;
    for (int i = 0; i < d; ++i) {
        float e = m->wte[(size_t)tok * d + i];
        s->x[i] = m->c.arch == A_GPT2 ? e + m->wpe[(size_t)pos * d + i] : e;
    }
    if (stack_forward(s, row, s->x)) return -1;
    if (logits) linear_q(&m->head, s->h, NULL, logits);
    return 0;
}

/* One position of a GPT-2 / Llama row whose input is the vector e[d] instead of a
 * token's embedding row (a conditioning prefix: text, speaker and conditioning
 * embeddings, journal section 3.19); GPT-2 adds its learned position as for a
 * token. */
int orc_embed_forward(orc_model* m, int row, const float* e, float* logits) {
    ostack* s = &m->s;
    if (m->c.arch == A_QWEN || row < 0 || row >= s->batch || !e) return -1;
    int pos = s->pos[row], d = s->d;
    if (pos >= s->max_ctx) return -1;
    for (int i = 0; i < d; ++i) s->x[i] = m->c.arch == A_GPT2 ? e[i] + m->wpe[(size_t)pos * d + i] : e[i];
    if (stack_forward(s, row, s->x)) return -1;
    if (logits) linear_q(&m->head, s->h, NULL, logits);
    return 0;
}

int orc_talker_embed(orc_model* m, int32_t tok, float* e) {
    if (m->c.arch != A_QWEN || tok < 0 || tok >= m->c.vocab) return -1;
    memcpy(e, m->emb[0] + (size_t)tok * m->c.d_model, (size_t)m->c.d_model * 4);
    return 0;
}

int orc_talker_forward(orc_model* m, int row, const float* e, float* logits0, float* hidden) {
    ostack* s = &m->s;
    if (m->c.arch != A_QWEN || row < 0 || row >= s->batch) return -1;
    memcpy(s->x, e, (size_t)s->d * 4);
    if (stack_forward(s, row, s->x)) return -1;
    if (logits0) linear_q(&m->head, s->h, NULL, logits0);
    if (hidden) memcpy(hidden, s->h, (size_t)s->d * 4);
    return 0;
}

int orc_cp_forward(orc_model* m, int row, const float* v, int head, float* logits) {
    ostack* p = &m->cp;
    if (m->c.arch != A_QWEN || row < 0 || row >= p->batch || head >= m->c.n_codebooks) return -1;
    linear_q(&m->cp_proj, v, NULL, p->x);
    if (stack_forward(p, row, p->x)) return -1;
    if (head >= 1 && logits) linear_q(&m->cp_head[head], p->h, NULL, logits);
    return 0;
}

void orc_cp_reset(orc_model* m, int row) {
    if (m->cp.pos && row >= 0 && row < m->cp.batch) m->cp.pos[row] = 0;
}

int orc_code_embed(orc_model* m, int j, int32_t code, float* out) {
    if (m->c.arch != A_QWEN || j < 0 || j >= m->c.n_codebooks) return -1;
    int32_t V = j ? m->c.cp_vocab : m->c.vocab;
    if (code < 0 || code >= V) return -1;
    memcpy(out, m->emb[j] + (size_t)code * m->c.d_model, (size_t)m->c.d_model * 4);
    return 0;
}

int orc_code_embed_sum(orc_model* m, const int32_t* codes, float* e) {
    if (m->c.arch != A_QWEN) return -1;
    int d = m->c.d_model;
    for (int j = 0; j < m->c.n_codebooks; ++j) {
        int32_t V = j ? m->c.cp_vocab : m->c.vocab;
        if (codes[j] < 0 || codes[j] >= V) return -1;
    }
    for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int j = 0; j < m->c.n_codebooks; ++j) acc += (double)m->emb[j][(size_t)codes[j] * d + i];
        e[i] = (float)acc;
    }
    return 0;
}
