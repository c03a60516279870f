/*
 * Oracle of the speech-token decode step -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-pass CPU restatement of what one decode step of the
 * GPT-2-style T3, the Llama-style T3 and the Qwen3-style Talker + code
 * predictor computes, used to check the CUDA library.  Only the tests, the
 * package's smoke entry and the CPU-baseline leg of the benchmark may load it;
 * the product path never does.  It shares no source with the CUDA library.
 *
 * Arithmetic convention: every activation is stored as fp32 after each
 * operation; every reduction (dot products, norm statistics, softmax sums,
 * attention) accumulates in double and is rounded once; transcendental
 * functions are the C library's double versions.  The KV cache holds fp16
 * (round-to-nearest-even) values, widened to double when read.
 */
#ifndef SD_ORACLE_H
#define SD_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct orc_model orc_model;

/* fp16 <-> fp32 conversions written from the IEEE 754 binary16 definition. */
float    orc_half_to_float(uint16_t h);
uint16_t orc_float_to_half(float f);

/* Dequantise rows x cols weights stored in blob kind `kind` (1 Q8_0, 2 Q4_0,
 * 3 A8G64) to fp32. */
int orc_dequant(int kind, const uint8_t* data, int64_t rows, int64_t cols, float* out);

/* y[r] = fp32( sum_k w[r][k] * x[k] (+ b[r]) ), the sum in double. b may be NULL. */
int orc_linear(int kind, const uint8_t* data, int64_t rows, int64_t cols,
               const float* x, const float* b, float* y);

void orc_layernorm(const float* x, int n, const float* g, const float* b, float eps, float* out);
void orc_rmsnorm(const float* x, int n, const float* g, float eps, float* out);
float orc_gelu_tanh(float t);
float orc_silu(float t);
/* NEOX (half-split) rotary embedding of one head vector, in place. */
void orc_rope(float* x, int hd, int pos, float theta);
/* One query against n cached fp16 keys/values (stride hd): softmax(q.K/sqrt(hd)) V. */
void orc_attend(const float* q, const uint16_t* k, const uint16_t* v, int n, int hd, float* out);

/* Sampler: temperature -> top-k -> top-p -> draw in vocabulary order with u.
 * margin (may be NULL) receives the decision margin.  Greedy (or top_k 1, or
 * temperature <= 0): the gap between the two largest logits.  A sampled draw:
 * the largest r such that neither moving u by less than r nor multiplying
 * every unnormalised probability by factors within [(1+r)^-1/2, (1+r)^1/2]
 * can change the token (a lower bound of the true value, found by bisection;
 * it equals the draw's distance to the token's CDF edges when no membership
 * flip at the top-k / top-p boundaries can move those edges that far). */
int32_t orc_sample(const float* z, int32_t V, float temperature, int32_t top_k, float top_p,
                   int32_t greedy, double u, double* margin);

/* orc_sample on the logits after a repetition penalty over seen[] (NULL: none):
 * a seen token's logit is divided by rep_penalty when positive, else multiplied. */
int32_t orc_sample_pen(const float* z, int32_t V, const uint8_t* seen, float rep_penalty, float temperature,
                       int32_t top_k, float top_p, int32_t greedy, double u, double* margin);

/* Sampler ladder of the multilingual T3: classifier-free-guidance combine ->
 * repetition penalty -> temperature -> min_p -> top-p -> top-k -> draw in
 * vocabulary order with u.  z_uncond may be NULL (no combine); seen may be
 * NULL (no penalty); top_k < 1 or > V keeps every survivor; temperature <= 0
 * returns the argmax of the combined, penalised logits.  margin (may be NULL)
 * receives the decision margin as orc_sample defines it, over the combined,
 * penalised and scaled logits and the min_p, top-p and top-k stages;
 * draw_dist (may be NULL) the draw's distance alone: u to the nearer end of the
 * chosen token's interval on the kept mass (normalised; infinite for argmax). */
int32_t orc_sample_ladder(const float* z_cond, const float* z_uncond, int32_t V, float cfg_weight,
                          const uint8_t* seen, float rep_penalty, float temperature, float min_p, float top_p,
                          int32_t top_k, double u, double* margin, double* draw_dist);

/* Model.  The blob must outlive the model. */
int  orc_open(const uint8_t* blob, uint64_t nbytes, orc_model** out);
void orc_close(orc_model* m);
void orc_reset(orc_model* m);
int  orc_set_threads(int n);
int  orc_pos(const orc_model* m, int row);
/* Row dst takes a copy of row src's (Talker / T3) cache and position: the state
 * that row src's inputs so far produced, for a row that received the same inputs. */
int  orc_copy_row(orc_model* m, int dst, int src);

/* GPT-2 / Llama: process token `tok` at row `row`'s next position; logits may be NULL. */
int orc_token_forward(orc_model* m, int row, int32_t tok, float* logits);

/* Qwen Talker: process input vector e (d_model) at the row's next Talker
 * position; logits0 (codebook-0 vocab) and hidden (final-normed state) may be NULL. */
int orc_talker_forward(orc_model* m, int row, const float* e, float* logits0, float* hidden);
/* Talker input for a prompt token: row `tok` of the codebook-0 embedding. */
/* A GPT-2 / Llama position whose input is e[d] in place of a token's embedding
 * row (GPT-2 still adds its learned position); logits may be NULL. */
int orc_embed_forward(orc_model* m, int row, const float* e, float* logits);
int orc_talker_embed(orc_model* m, int32_t tok, float* e);
/* Code predictor: project v (Talker width) with Pr, run the CP stack at the
 * row's next CP position, and if head >= 1 write head `head`'s logits. */
int orc_cp_forward(orc_model* m, int row, const float* v, int head, float* logits);
void orc_cp_reset(orc_model* m, int row);
/* Row `code` of codebook j's embedding (Talker width). */
int orc_code_embed(orc_model* m, int j, int32_t code, float* out);
/* e = sum_{j=0..n_codebooks-1} E_j[codes[j]], summed in j order in double, rounded once. */
int orc_code_embed_sum(orc_model* m, const int32_t* codes, float* e);

#ifdef __cplusplus
}
#endif
#endif
