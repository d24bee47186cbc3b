/*
 * pkv_prefill.h - prefill over the shared KV page pool: a chunk of prompt
 * tokens per sequence is written into its pages, then every token of the
 * chunk attends causally to all tokens up to and including itself, reading
 * K/V from the pages.
 *   [samir-vllm: Build LLM Inference From Scratch in C++ and CUDA,
 *    "Architecture walkthrough", Prefill and KV cache paragraphs; 6 Hours of
 *    YouTube and 85 handtyped pages of notes on LLM Inference - Start here,
 *    README feature list, dense causal prefill and shared BF16 KV page pool
 *    bullets]
 *
 * Geometry and pool layout are those of pkv.h (32 query heads over 8 KV
 * heads, head_dim 64, 16-token pages, pools [num_pages][8][16][64] BF16,
 * block tables [num_layers][max_batch][max_seq_len / 16] int32).
 *
 * A call covers `batch` sequences. Sequence b contributes a chunk of
 * n_b = cu_tokens[b+1] - cu_tokens[b] tokens, packed at rows cu_tokens[b] ..
 * cu_tokens[b+1] - 1 of the token-major inputs, at absolute positions
 * start_pos[b] .. start_pos[b] + n_b - 1. start_pos[b] > 0 continues a
 * prompt whose earlier positions are already in the pages (chunked
 * prefill); the pages the whole length needs must be in the block table.
 *
 *   q     BF16 [total_tokens][32][64]    (rotary embedding already applied)
 *   k, v  BF16 [total_tokens][8][64]     (k already rotated)
 *   out   FP32 [total_tokens][32][64]
 *   cu_tokens int32 [batch + 1] (device), cu_tokens[0] = 0, non-decreasing,
 *             cu_tokens[batch] = total_tokens
 *   start_pos int32 [batch] (device)
 *
 * total_tokens (the rows of q, k, v and out) and max_chunk_tokens (>= every
 * n_b, <= max_seq_len) are host integers that size the launch; a sequence
 * whose rows fall outside [0, total_tokens) is skipped and flagged. All
 * pointers: device memory owned by the caller, 16-byte aligned.
 * Asynchronous on `stream`. Host-detectable errors return INVALID_ARG and
 * launch nothing; positions, lengths and page ids found invalid on the
 * device are skipped and recorded in the pool's sticky error flag
 * (pkv_get_error), as in pkv.h. A chunk longer than max_chunk_tokens is not
 * fully computed and is flagged.
 *
 * Arithmetic: scores and outputs accumulate in FP32 on the tensor cores
 * (BF16 operands); the softmax probabilities enter the value product as
 * the sum of two BF16 terms (a high and a low part), so the result meets
 * the same tolerance as the FP32 decode path.
 */
#ifndef PKV_PREFILL_H
#define PKV_PREFILL_H

#include <stdint.h>

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Writes k[i], v[i] of every chunk token to
 * k_pool / v_pool [block_tables[layer][b][p / 16]][h][p % 16][:], p its
 * position. Bit copy. */
pkv_status pkv_prefill_fill(pkv_pool_t pool, int layer, const void* k, const void* v,
                            void* k_pool, void* v_pool, const int32_t* block_tables,
                            const int32_t* cu_tokens, const int32_t* start_pos, int batch,
                            int total_tokens, int max_chunk_tokens, void* stream);

/* out[i][h][:] = sum_{t <= p_i} softmax_t(q[i][h] . K_t / 8) V_t for every
 * chunk token i at position p_i, K_t, V_t read through block_tables[layer]
 * (kv head h / 4). The chunk's own K/V must be in the pages already
 * (pkv_prefill_fill, earlier on the stream). */
pkv_status pkv_prefill_attention(pkv_pool_t pool, int layer, const void* q, const void* k_pool,
                                 const void* v_pool, const int32_t* block_tables,
                                 const int32_t* cu_tokens, const int32_t* start_pos, float* out,
                                 int batch, int total_tokens, int max_chunk_tokens,
                                 void* stream);

/* pkv_prefill_fill, then pkv_prefill_attention, on the stream. */
pkv_status pkv_prefill(pkv_pool_t pool, int layer, const void* q, const void* k, const void* v,
                       void* k_pool, void* v_pool, const int32_t* block_tables,
                       const int32_t* cu_tokens, const int32_t* start_pos, float* out,
                       int batch, int total_tokens, int max_chunk_tokens, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_PREFILL_H */
