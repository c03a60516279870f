/*
 * sd_ops.h -- op-level C ABI of libsd.so: the individual decode-step kernels,
 * exposed so that each can be checked on its own at full workload shapes.
 * Same conventions as sd.h (SD_* return codes; *_dev pointers are device
 * memory owned by the caller; `stream` is a cudaStream_t or NULL for the
 * legacy default stream).  Errors are reported through sd_last_error(NULL).
 */
#ifndef SD_OPS_H
#define SD_OPS_H

#include "sd.h"

#ifdef __cplusplus
extern "C" {
#endif

/* A block-quantised matrix [rows][cols] (one row per output feature, cols
 * contiguous: the orientation of "Chatterbox -> ggml Port: Development
 * Journal", section 3.2, issue 5) repacked into the device layout the GEMV
 * streams: codes of a row contiguous (16-byte units) and the fp16 scales (and
 * affine biases) in a separate array.  `canon` holds the canonical blob
 * bytes of one tensor: Q8_0 34-byte blocks, Q4_0 18-byte blocks (journal
 * section 3.23), Q5_0 22-byte blocks (fp16 d, 32 fifth bits, 16 nibble
 * bytes), or affine codes (8-bit: one per byte; 4-bit: element 2i in the low
 * nibble of byte i) + fp16 scales + fp16 biases; host memory, or device memory
 * when on_device != 0.  cols must be a multiple of 32 (64 for SD_A8G64 and
 * SD_A4G64). */
typedef struct sd_qmat sd_qmat;
int sd_qmat_create(int quant, const void* canon, int64_t rows, int64_t cols, int on_device, int device,
                   sd_qmat** out);
void sd_qmat_destroy(sd_qmat* m);

/* Dequantise to fp32 out_dev[rows][cols]: Q8_0 d*q, Q4_0 d*(q-8), Q5_0
 * d*(q-16), affine fma(scale, q, bias) -- bit-exact definitions of the formats. */
int sd_qmat_dequant(const sd_qmat* m, float* out_dev, void* stream);

/* y_dev[b][r] = sum_k W[r][k] x_dev[b][k] (+ bias_dev[r]) for b < nb (nb 1 or
 * 2), fp32 accumulation.  bias_dev may be NULL. */
int sd_qmat_gemv(const sd_qmat* m, const float* x_dev, int32_t nb, const float* bias_dev, float* y_dev,
                 void* stream);

/* Epilogues of sd_qmat_gemm. */
enum { SD_EPI_LINEAR = 0, SD_EPI_GELU = 1, SD_EPI_SWIGLU = 2 };

/* Tensor-core GEMM for prompt prefill and batched rows ("Chatterbox -> ggml
 * Port: Development Journal", section 3.2: the prompt graph applies every
 * layer to all prompt positions at once):
 *   t[i][r] = sum_k W[r][k] x_dev[i][k] for i < M (x_dev [M][cols], fp32);
 *   SD_EPI_LINEAR: y_dev[i][r] = t[i][r] (+ bias_dev[r]) (+ resid_dev[i][r]);
 *   SD_EPI_GELU:   y_dev[i][r] = gelu_tanh(t[i][r] (+ bias_dev[r])) (+ resid_dev[i][r]);
 *   SD_EPI_SWIGLU: rows are interleaved gate/up pairs (row 2j gate j, row
 *     2j+1 up j), y_dev[i][j] = silu(t[i][2j]) * t[i][2j+1] (+ resid_dev[i][j]),
 *     j < rows/2; bias_dev must be NULL; rows must be even.
 * y_dev and resid_dev have leading dimension rows (rows/2 for SwiGLU); resid_dev
 * may equal y_dev; bias_dev and resid_dev may be NULL.  The codes of a
 * quantisation block enter the tensor cores exactly (fp16 integers), the
 * fp32 activations as an fp16 high + low pair, and the block scale (and
 * affine bias times the group's activation sum) is applied in fp32.
 * Device pointers; enqueued on `stream`; returns SD_ERR_INVALID_ARG on a NULL
 * pointer, M < 1 or a bad epilogue. */
int sd_qmat_gemm(const sd_qmat* m, const float* x_dev, int32_t M, int32_t epilogue, const float* bias_dev,
                 const float* resid_dev, float* y_dev, void* stream);

/* As sd_qmat_gemm, on the 5th-generation tensor cores (tcgen05 MMA with a
 * tensor-memory accumulator, operands loaded by TMA), the form the prompt
 * prefill uses.  The weights are dequantised once (kept with the matrix,
 * device memory rows*cols*4 bytes, allocated on the first call) and, like the
 * activations, split into fp16 high and low parts; three fp16 products per
 * K step (hi*hi + hi*lo + lo*hi) accumulate in fp32.  cols must be a multiple
 * of 64 (else SD_ERR_UNSUPPORTED).  Synchronises `stream` before returning;
 * allocates and frees a scratch buffer of M*cols*4 bytes per call.  A kernel
 * wait that runs out of its time budget returns SD_ERR_TIMEOUT. */
int sd_qmat_gemm_tc(sd_qmat* m, const float* x_dev, int32_t M, int32_t epilogue, const float* bias_dev,
                    const float* resid_dev, float* y_dev, void* stream);

/* As sd_qmat_gemm for 1 <= M <= 16 rows (the G rollouts of "Every Frame Is a
 * Memory Read", section 8, which share one read of the weights per step):
 * the form the decode step uses for more than two rows.  The weights stream
 * once from memory straight into the tensor cores (mma.sync m16n8k16, the same
 * exact-code / fp16 hi+lo / fp32-scale arithmetic); K is split over CTAs and
 * the partial sums are added in a fixed order, so results are reproducible.
 * x_dev must be 16-byte aligned.  A workspace of partial sums and column-tile
 * counters is kept with the matrix (allocated on the first call, at most
 * 16 * rows * cols / 32 floats).  Calls on one matrix must not run
 * concurrently on different streams.  Returns SD_ERR_INVALID_ARG on a NULL
 * pointer, M outside [1, 16], a bad epilogue or a misaligned x_dev. */
int sd_qmat_gemm16(sd_qmat* m, const float* x_dev, int32_t M, int32_t epilogue, const float* bias_dev,
                   const float* resid_dev, float* y_dev, void* stream);

/* Sample one token per row from logits_dev[rows][V] with draws u_dev[rows];
 * tokens to out_dev[rows].  Sampler semantics as in sd.h.  V <= 16384. */
int sd_sample_rows(const float* logits_dev, int32_t rows, int32_t V, const sd_sampler* sampler,
                   const float* u_dev, int32_t* out_dev, void* stream);

/* (sd_sampler_ladder, the ladder's parameters, is declared in sd.h.) */

/* Sampler ladder of the multilingual T3 ("Chatterbox -> ggml Port: Development
 * Journal", the multilingual port's sampling path): classifier-free-guidance
 * combine -> repetition penalty -> temperature -> min_p -> top-p -> top-k ->
 * draw in vocabulary order.  Per row b:
 *   z_i = c_i + w (c_i - u_i)      (c = logits_cond_dev[b], u = logits_uncond_dev[b]; w ignored when NULL)
 *   seen_dev[b][i] != 0: z_i / penalty if z_i > 0, else z_i * penalty   (seen_dev may be NULL)
 *   z_i / T; p_i proportional to exp(z_i); min_p keeps p_i >= min_p * max p;
 *   top-p keeps the shortest (p desc, index asc) prefix of those whose
 *   renormalised mass reaches top_p; top-k keeps the ones whose value is >= the
 *   k-th largest remaining (ties kept); the token is the smallest vocabulary
 *   index whose cumulative kept mass exceeds u_dev[b] times the kept total.
 * Layouts: logits [rows][V] fp32, seen [rows][V] bytes, u [rows], out [rows] int32;
 * device pointers; 1 <= V <= 16384.  Double-precision arithmetic, one CTA per row.
 * This entry is an op-level form of the ladder: the decode step's own sampler
 * is temperature -> top-k -> top-p (sd.h).  Synchronises `stream`; returns
 * SD_ERR_INVALID_ARG on a NULL required pointer or a parameter out of range. */
int sd_sample_rows_ladder(const float* logits_cond_dev, const float* logits_uncond_dev, int32_t rows, int32_t V,
                          const sd_sampler_ladder* sampler, const uint8_t* seen_dev, const float* u_dev,
                          int32_t* out_dev, void* stream);

/* Decode attention for one query per head against n cached positions
 * (journal section 3.13 flash attention over a cache laid out
 * [head][pos][dim]): out[b][h] = softmax(q[b][h] . K[b][g][0:n] / sqrt(hd))
 * V[b][g][0:n] with g = h / (H / Hkv).  q_dev [B][H][hd] fp32, k_dev/v_dev
 * [B][Hkv][n_ctx][hd] fp16, out_dev [B][H][hd] fp32.  Split-KV over
 * `nsplit` chunks per (row, kv head) then a log-sum-exp combine.  hd is 64 or
 * 128; 1 <= n <= n_ctx. */
int sd_attend_rows(const float* q_dev, const uint16_t* k_dev, const uint16_t* v_dev, int32_t B, int32_t H,
                   int32_t Hkv, int32_t hd, int32_t n_ctx, int32_t n, int32_t nsplit, float* out_dev,
                   void* stream);

/* The decode attention of sd_attend_rows for callers that may not allocate
 * device memory while they run -- for instance a host thread with a hard
 * latency budget (cudaMalloc can synchronise the whole device) or a host
 * framework that owns all device memory through its own pool.  This entry has
 * no counterpart in the pages; it exists for those callers.  Arguments,
 * layouts and the values written to out_dev are those of sd_attend_rows.
 *
 * Unlike sd_attend_rows, the call is stream-ordered: it queues a counter clear
 * (cudaMemsetAsync) and the attention kernel on `stream` and returns without
 * waiting.  out_dev is ready, and the inputs may be released, only after the
 * caller synchronises the stream (or orders later work after it); an error
 * raised by the kernel appears at that synchronisation, not in this call's
 * return value, which reports only argument and launch errors.
 *
 * Instead of allocating, the split-KV partial results and one counter per
 * (row, kv head) go to one fixed array of 1048576 floats (4 MiB) that every
 * device loading the library keeps until the process exits.  A call needs
 * B * H * nsplit * (hd + 4) + B * Hkv floats of it; a larger request returns
 * SD_ERR_INVALID_ARG.  The call allocates nothing: no cudaMalloc, cudaFree or
 * allocating library routine.  The first call on each device (with that device
 * current) looks up the array's device address; make that first call before
 * any stream capture.  All calls share the one array: calls that overlap on
 * the GPU (different streams, or different threads on the same device) race on
 * it and must be serialised by the caller.  Every partial record a call reads
 * is written earlier in the same call; the counters, which must start at zero,
 * are cleared by the call itself on `stream` before the kernel runs. */
int sd_attend_rows_static(const float* q_dev, const uint16_t* k_dev, const uint16_t* v_dev, int32_t B, int32_t H,
                          int32_t Hkv, int32_t hd, int32_t n_ctx, int32_t n, int32_t nsplit, float* out_dev,
                          void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SD_OPS_H */
