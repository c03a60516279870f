/*
 * sd.h -- C ABI of the single-stream speech-token decode library (libsd.so).
 *
 * The library runs, on one GB300 (sm_103a), the autoregressive decode step of
 * three speech-token transformers:
 *   - the GPT-2-Medium-style T3 of "Chatterbox -> ggml Port: Development
 *     Journal" (section 3.2: a prompt graph and a step graph sharing one
 *     persistent KV cache; section 3.13: the cache laid out the way the
 *     attention reads it);
 *   - the Llama-style T3 of the journal's section 3.19 (RMSNorm, SwiGLU, NEOX
 *     RoPE; section 3.21: two rows decoded in one batched step);
 *   - the Qwen3-style Talker plus code predictor of "Every Frame Is a Memory
 *     Read" (section 1: the Talker predicts codebook 0, the code predictor runs
 *     15 sequential passes for codebooks 1-15, and the sum of the 16 code
 *     embeddings is the next Talker input).
 * Weights are block quantised (Q8_0, Q5_0, Q4_0: journal Tier A item A3 and
 * section 3.23; 8-bit affine groups of 64: the blog's section 3; 4-bit affine
 * groups of 32 or 64: its section 5.8).  `quant` in the config names the format
 * of every matrix, except that a Talker + code-predictor blob may store the
 * code predictor's matrices in another format (each tensor records its own).
 * The persistent decode step kernels take Q8_0 and Q4_0; the other formats
 * decode through the per-operation step graph.
 *
 * Conventions shared by every entry point:
 *   - Return value: SD_OK (0) or a negative SD_ERR_* code.  Nothing aborts or
 *     exits; after an error sd_last_error() describes it, and sd_reset() or
 *     sd_destroy() are always allowed.
 *   - Pointers named *_dev are device pointers; every other pointer is host
 *     memory.  The caller owns every pointer it passes; the library copies
 *     what it keeps.
 *   - A context is bound to one CUDA device and one stream (the caller's, or
 *     one the library creates when `stream` is NULL).  Calls on one context
 *     must not overlap.
 *   - Rows: `batch` independent sequences decoded in lockstep (B <= 16); all
 *     rows share one position counter.
 */
#ifndef SD_H
#define SD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SD_OK 0
#define SD_ERR_INVALID_ARG (-1)  /* null pointer, token out of [0, vocab), bad sampler, bad size */
#define SD_ERR_STATE (-2)        /* call out of order (e.g. sd_step before sd_prefill) */
#define SD_ERR_CTX_FULL (-3)     /* the position would reach max_ctx */
#define SD_ERR_OOM (-4)          /* device or pinned allocation failed */
#define SD_ERR_CUDA (-5)         /* a CUDA runtime call failed */
#define SD_ERR_TIMEOUT (-6)      /* a device-side bounded wait expired */
#define SD_ERR_UNSUPPORTED (-7)  /* valid request the library does not implement */
#define SD_ERR_BLOB (-8)         /* weight blob malformed or not matching the config */
#define SD_ERR_DEVICE (-9)       /* a kernel flagged an out-of-range index and skipped it */

enum { SD_ARCH_GPT2 = 1, SD_ARCH_LLAMA = 2, SD_ARCH_QWEN_TTS = 3 };
enum { SD_Q8_0 = 1, SD_Q4_0 = 2, SD_A8G64 = 3, SD_Q5_0 = 4, SD_A4G32 = 5, SD_A4G64 = 6 };

#define SD_MAX_ROWS 16
#define SD_MAX_CODEBOOKS 16

/* Model shape.  The field order equals the config echo stored in the weight
 * blob header.  GPT-2 uses LayerNorm, biases, tanh GELU and learned positions;
 * Llama and the Qwen Talker/code predictor use RMSNorm, no biases, SwiGLU and
 * NEOX RoPE with base rope_theta.  The cp_* fields describe the code
 * predictor and are zero for the other architectures. */
typedef struct sd_model_config {
    int32_t arch, n_layer, d_model, n_head, n_kv_head, head_dim, d_ff, vocab, max_ctx, batch, quant;
    float rope_theta, norm_eps;
    int32_t cp_layer, cp_d_model, cp_n_head, cp_n_kv_head, cp_head_dim, cp_d_ff, cp_vocab, n_codebooks,
        cp_max_ctx;
} sd_model_config;

/* Sampler (journal section 3.2: temperature -> top-k -> top-p).  greedy != 0,
 * top_k == 1 or temperature == 0 selects argmax (ties: lowest index).
 * Otherwise: keep every logit >= the top_k-th largest (ties kept); softmax of
 * logit/temperature over the kept set; if top_p < 1 keep the shortest prefix,
 * in (probability desc, index asc) order, whose mass reaches top_p; draw the
 * smallest vocabulary index whose cumulative kept mass (index order) exceeds
 * u times the kept total.  Valid: temperature >= 0, top_k >= 1,
 * 0 < top_p <= 1.  rep_penalty: 1, or 0 (read as 1), applies none.  The
 * Talker's sampler of a Talker + code-predictor context (sd_prefill, and the
 * `talker` argument of sd_frame) takes any positive penalty: before sampling
 * codebook 0, the logit of every codebook-0 token fed to the Talker since
 * sd_prefill (the prompt's own tokens excluded) is divided by it when positive
 * and multiplied by it otherwise ("Every Frame Is a Memory Read", sections 2
 * and 8: the penalty, kept per row on the device; the journal's HF sign rule).
 * sd_prefill gives the prompt frame's code predictor the same settings without
 * the penalty.  Elsewhere (GPT-2 / Llama steps, the code predictor's sampler)
 * a penalty other than 1 returns SD_ERR_UNSUPPORTED -- the multilingual T3's
 * penalty is part of its ladder (sd_set_ladder) -- and a negative or NaN value
 * SD_ERR_INVALID_ARG. */
typedef struct sd_sampler {
    float temperature;
    int32_t top_k;
    float top_p;
    int32_t greedy;
    float rep_penalty;
} sd_sampler;

/* Parameters of the multilingual T3's sampler ladder ("Chatterbox -> ggml Port:
 * Development Journal", section 3.19, "Sampling path"): classifier-free-guidance
 * combine -> repetition penalty -> temperature -> min_p -> top-p -> top-k -> draw
 * in vocabulary order (sd_set_ladder here, sd_sample_rows_ladder in sd_ops.h). */
typedef struct sd_sampler_ladder {
    float cfg_weight;          /* guidance weight w: z = c + w (c - u); 0 = conditional logits only */
    float repetition_penalty;  /* > 0; 1 = off */
    float temperature;         /* <= 0: argmax of the combined, penalised logits */
    float min_p;               /* keep p >= min_p * max p; 0 = off (values above 1 act as 1) */
    float top_p;               /* (0, 1]; 1 = off */
    int32_t top_k;             /* < 1 or >= the survivors: off */
} sd_sampler_ladder;

typedef struct sd_ctx sd_ctx;

/* Create a context on CUDA device `device` (journal section 3.2: the prompt
 * graph and the step graph share one KV cache, allocated here; section 3.13:
 * laid out [row][layer][kv_head][pos][dim] fp16, the order the attention reads).
 * `stream` is a cudaStream_t or NULL.  Allocates the cache, activations and
 * pinned staging; weights come later.  Errors: SD_ERR_INVALID_ARG (bad
 * config), SD_ERR_UNSUPPORTED (a shape the kernels do not take), SD_ERR_OOM,
 * SD_ERR_CUDA; *out is NULL then. */
int sd_create(const sd_model_config* cfg, int device, void* stream, sd_ctx** out);

/* Load the weight blob (the flat format written by the seeded generator:
 * header + config echo + tensor table + canonical tensors; the block formats
 * of journal Tier A item A3 and section 3.23, and the blog's section 3 for
 * affine groups).  `blob` is host memory, or device memory when
 * blob_on_device != 0.  The tensors are repacked into the library's device
 * layout; the blob may be freed after the call.  The config echo must equal
 * the context's config (else SD_ERR_BLOB). */
int sd_load_weights(sd_ctx* ctx, const void* blob, size_t nbytes, int blob_on_device);

/* The prompt graph (journal section 3.2; "Every Frame Is a Memory Read",
 * section 1 for the Talker's prompt frame).
 * Process a prompt of n tokens per row (tokens [batch][n], host) at positions
 * 0..n-1 and sample the first generated token of each row with draw u[row].
 * GPT-2/Llama: out_tok[batch].  Qwen Talker+CP: u and out_tok are
 * [batch][16]: the codes of frame 0 (code 0 from the Talker's last prompt
 * position, codes 1..15 from the code predictor).  Requires a reset context
 * (position 0). */
int sd_prefill(sd_ctx* ctx, const int32_t* tokens, int32_t n, const sd_sampler* sampler, const float* u,
               int32_t* out_tok);

/* sd_prefill with one prompt for every row (tokens [n], host): the G rollouts
 * of one prompt ("Every Frame Is a Memory Read", section 8: G rows share each
 * weight read; the rows differ only by their draws).  On the GEMM prefill path
 * positions 0..n-2 are computed for row 0 alone and row 0's KV cache is copied
 * to the other rows (a snapshot of the prompt state restored into each row);
 * the last position runs for every row with its own draws.  Results equal
 * sd_prefill with every row given `tokens`. */
int sd_prefill_shared(sd_ctx* ctx, const int32_t* tokens, int32_t n, const sd_sampler* sampler, const float* u,
                      int32_t* out_tok);

/* sd_prefill whose prompt is given as input vectors: embeds [batch][n][d_model]
 * fp32, host (a conditioning prefix: text, speaker and conditioning embeddings
 * assembled by the caller, journal section 3.19 and Tier A item A1).  Vector p
 * of a row takes the place of a prompt token's embedding row; GPT-2 still adds
 * its learned position p.  The vectors are kept in B * max_ctx rows of the
 * input embedding table that follow the vocabulary.  Errors as sd_prefill, and
 * SD_ERR_INVALID_ARG for a non-finite element. */
int sd_prefill_embeds(sd_ctx* ctx, const float* embeds, int32_t n, const sd_sampler* sampler, const float* u,
                      int32_t* out_tok);

/* One decode step (GPT-2/Llama; the step graph of journal section 3.2, two
 * rows in one step per section 3.21): consume tok[row] at the current
 * position, sample the next token with draw u[row] into out_tok[row],
 * advance.  Errors: SD_ERR_STATE before sd_prefill, SD_ERR_CTX_FULL at
 * max_ctx, SD_ERR_TIMEOUT / SD_ERR_DEVICE from the kernels (sd_reset
 * recovers). */
int sd_step(sd_ctx* ctx, const int32_t* tok, const sd_sampler* sampler, const float* u, int32_t* out_tok);

/* One frame (Qwen Talker+CP; "Every Frame Is a Memory Read", section 1 and
 * section 5.2, the code-predictor frame): the Talker consumes the sum of the 16 code
 * embeddings of codes_in[row][0..15] (the previous frame), samples code 0 with
 * `talker`; the code predictor then samples codes 1..15 with `cp`.  Draws
 * u[row][j] feed code j.  Output codes_out[row][16]. */
int sd_frame(sd_ctx* ctx, const int32_t* codes_in, const sd_sampler* talker, const sd_sampler* cp,
             const float* u, int32_t* codes_out);

/* The multilingual T3's guided decode (journal section 3.19, "Sampling path",
 * and section 3.21: the conditional and the unconditional sequence decoded as
 * two rows of one step).  For a GPT-2/Llama context of batch 2 -- row 0 the
 * conditional, row 1 the unconditional sequence -- a non-NULL ladder makes
 * every sd_prefill / sd_step / sd_decode_n step draw ONE token: the ladder above
 * on row 0's and row 1's logits, the repetition penalty over the tokens drawn
 * since the last sd_prefill (a device-side mask), with row 0's draw; the token
 * is returned for, and fed to, both rows.  The sampler argument of those calls
 * is then only checked.  The steps run on the per-operation step graph (the
 * persistent kernels do not implement the ladder).  NULL restores per-row
 * sampling.  Needs a loaded or reset context (position 0) and vocab <= 16384;
 * SD_ERR_UNSUPPORTED for other models or batch sizes, SD_ERR_INVALID_ARG for
 * a ladder out of range. */
int sd_set_ladder(sd_ctx* ctx, const sd_sampler_ladder* ladder);

/* Teacher forcing (a test aid for the parity of "Every Frame Is a Memory
 * Read", section 1's frame) for the next sd_prefill/sd_frame of a Qwen context: within
 * the frame the code fed to the next code-predictor pass is codes[row][j]
 * instead of the sampled one (the sampled codes are still returned).  NULL
 * clears it.  Applies to one call only. */
int sd_set_forced_codes(sd_ctx* ctx, const int32_t* codes);

/* n_steps decode steps with device-side token feedback (GPT-2/Llama; "Every
 * Frame Is a Memory Read", section 3: no host round trip in the loop): step i
 * samples with u_dev[i][row] and writes out_dev[i][row]; its input is the
 * previous step's token (the last sd_prefill/sd_step output for i = 0).  No
 * host round trip between steps. */
int sd_decode_n(sd_ctx* ctx, int32_t n_steps, const sd_sampler* sampler, const float* u_dev, int32_t* out_dev);

/* The head's output of journal section 3.2's step graph, for parity checks.
 * Copy the last step's logits to host: [batch][vocab] (GPT-2/Llama) or
 * [batch][16][max(vocab, cp_vocab)] (Qwen, pass j in slot j).  n_floats must
 * be at least that size. */
int sd_get_logits(sd_ctx* ctx, float* host_out, size_t n_floats);

/* Back to position 0 (journal section 3.2: a new utterance reuses the graphs
 * and the cache); weights are kept, cache contents become undefined.  Clears
 * a recorded kernel error. */
int sd_reset(sd_ctx* ctx);

/* Free the context and everything it allocated (NULL is ignored). */
void sd_destroy(sd_ctx* ctx);

/* Last error message of the context (never NULL); with ctx == NULL the last
 * error of a failed sd_create or of an op-level call on this thread. */
const char* sd_last_error(const sd_ctx* ctx);

/* Introspection for benchmarks and tests ("Every Frame Is a Memory Read",
 * section 3: bytes per step against the bandwidth). */
typedef struct sd_info {
    int32_t pos;               /* current position (Talker position for Qwen) */
    int32_t sm_count;          /* streaming multiprocessors of the device */
    int32_t kernels_per_step;  /* kernel launches in one decode step or frame */
    int32_t attn_splits;       /* split-KV chunks per (row, kv head) */
    int64_t weight_bytes;      /* repacked weight bytes resident on the device */
    int64_t kv_bytes;          /* KV cache bytes allocated */
    int64_t step_h2d_bytes;    /* host->device bytes one sd_step (Talker+CP: one sd_frame) copies (pinned staging) */
    int64_t step_d2h_bytes;    /* device->host bytes one sd_step (Talker+CP: one sd_frame) copies back */
    int32_t persistent;        /* CTAs of the persistent step kernel (0: per-operation kernels) */
    int32_t prefill;           /* prompt path: 0 per-position step graphs, 1 mma.sync GEMMs, 2 tcgen05 GEMMs */
    int32_t persistent_clusters; /* thread-block clusters of the persistent step (0: the flat kernel or none) */
    int32_t cluster_size;      /* CTAs per cluster of the persistent step (0: the flat kernel or none) */
} sd_info;
int sd_get_info(const sd_ctx* ctx, sd_info* out);

#ifdef __cplusplus
}
#endif
#endif /* SD_H */
