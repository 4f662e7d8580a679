/*
 * lt_compress.h -- C ABI of the fused KV compressor (GB300, sm_103a).
 *
 * The operation. Compressed sparse attention keeps one KV entry per block of
 * `ratio` consecutive tokens (4:1 for CSA, 128:1 for HCA: AICon 2026 Shenzhen
 * speaker page, outline section 1.1). The SGLang DeepSeek-V4 inference talk
 * notes (section 3.1, fusion of the KV compression operators) describe the
 * compressor as a chain that touches memory five times -- read, add, softmax,
 * dot product, store -- and fuse the three compute steps into one operator so
 * that only the read and the store remain; the AICon page (outline section
 * 3.1) names the fused kernel FlashCompressor. Per complete block g of a row
 * and per channel c (the plainest reading of those step names):
 *
 *   v[t][c] = score[t][c] + bias[t mod ratio][c]
 *   w[t][c] = exp(v[t][c]) / sum over the block's tokens t' of exp(v[t'][c])
 *   out[g][c] = sum over the block's tokens t of w[t][c] * kv[t][c]
 *
 * A score per token rather than per channel is a score repeated across the
 * channels. The softmax runs in fp32 whatever the storage type.
 *
 * Memory. Every pointer is DEVICE memory owned by the caller; the library
 * allocates nothing and never synchronises the stream. Calls are asynchronous
 * on `stream` (a cudaStream_t passed as void*) and use programmatic dependent
 * launch like the top-k calls.
 *
 * Errors. Argument errors return LT_ERR_INVALID_ARG / LT_ERR_UNSUPPORTED
 * synchronously and launch nothing; a failed launch returns LT_ERR_CUDA.
 * Inputs are expected finite; NaN or infinite inputs propagate as IEEE
 * arithmetic does.
 */
#ifndef LT_COMPRESS_H
#define LT_COMPRESS_H

#include "lt_topk.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Largest compression ratio accepted. */
#define LT_MAX_RATIO 4096

/*
 * lt_compress -- the compressor over whole rows (prefill).
 *
 *   kv, score   [rows][row_tokens][dim] of `dtype` (LT_DTYPE_F32 float or
 *               LT_DTYPE_BF16 uint16_t bf16 bits); both of the same type
 *   bias        float [ratio][dim]
 *   lengths     int32 [rows] or NULL: tokens of row r are [0, L_r),
 *               L_r = clamp(lengths[r], 0, row_tokens); NULL means row_tokens
 *   rows >= 0, row_tokens >= 1, dim >= 1, 1 <= ratio <= LT_MAX_RATIO
 *   out         [rows][row_tokens / ratio][dim] of `dtype`: block g of row r
 *               (tokens g*ratio .. g*ratio + ratio - 1) is written when
 *               g < L_r / ratio (integer division); the other entries are not
 *               touched (an incomplete trailing block waits for its tokens)
 * bf16 outputs are the fp32 result rounded to nearest even. When kv, score
 * and bias are 16-byte aligned, dim * size is a multiple of 16 bytes and out
 * allows vector stores, bulk copies stream the rows through shared memory
 * (the fast path); other layouts take register loads (vector loads when
 * aligned with dim % 4 == 0, else scalar). Same results up to rounding.
 */
lt_status lt_compress(const void* kv, const void* score, const float* bias, const int32_t* lengths,
                      int32_t rows, int64_t row_tokens, int32_t dim, int32_t ratio, void* out,
                      int32_t dtype, void* stream);

/*
 * lt_compress_decode -- one decode step of the same compressor for a batch of
 * sequences, with the state kept in two caller-owned ring buffers (the AICon
 * page, outline section 2.3, keeps the compressor's intermediate state of the
 * preceding tokens in two ring buffers).
 *
 *   kv_new, score_new     [seqs][dim] of `dtype`: the new token of each sequence
 *   ring_kv, ring_score   [seqs][ratio][dim] of `dtype`, read and written: the
 *                         new token is stored in slot pos[s] mod ratio
 *   pos                   int32 [seqs]: position of the new token (>= 0)
 *   out                   [seqs][dim] of `dtype`: written for the sequences
 *                         whose new token completes a block
 *                         (pos[s] mod ratio == ratio - 1), from the ring's
 *                         ratio tokens: the same function as lt_compress (the
 *                         same bits whenever a block fits one stage of
 *                         lt_compress's ring, ratio * dim * size <= 16 KB);
 *                         the other rows are not touched
 * A sequence with a negative pos is skipped.
 */
lt_status lt_compress_decode(const void* kv_new, const void* score_new, const float* bias,
                             void* ring_kv, void* ring_score, const int32_t* pos, int32_t seqs,
                             int32_t dim, int32_t ratio, void* out, int32_t dtype, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LT_COMPRESS_H */
