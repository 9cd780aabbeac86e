/*
 * CPU oracle for the candidate-block sparse MQA-logits top-k indexer.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library. The CUDA library never links,
 * includes or calls it, and it shares no code with the CUDA library.
 *
 * Every function is the plain definition, in double precision:
 *  - decode Q, K and the head weights from their codes,
 *  - score every position of the row's context,
 *  - mask to the candidate blocks,
 *  - sort to take the top-k.
 * Sources are the three pages on the vLLM DeepSeek-V4.1 sparse indexer:
 *  - "vllm.model_executor.layers.sparse_mqa_indexer" (API docs),
 *  - "vllm/v1/attention/backends/mla/sparse_indexer.py" (source listing),
 *  - "vllm.model_executor.layers.rocm_paged_mxfp4_indexer" (API docs).
 * The score formula, sum_h w[h] * ReLU(q[h] . k), is the DeepSeek
 * "lightning indexer" score that those pages' MQA-logits kernels compute.
 * The pages name that score but do not print it.
 *
 * Layouts are the ones the CUDA library's header documents:
 *  - Q is [H][D] E4M3 bytes per row, with one float scale per row.
 *  - weights are [H] bfloat16 bits per row.
 *  - a cache page holds values [page_size][D/2], two E2M1 codes per byte
 *    (element 2i in the low nibble), followed by scales [page_size][D/32] of
 *    UE8M0 codes, one per 32 elements.
 *
 * All functions return 0 on success, or -1 on an out-of-range index or a
 * non-finite decoded input. Non-finite inputs are never generated.
 */
#ifndef SMQ_ORACLE_H
#define SMQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element decoders (OCP OFP8 E4M3 "fn", OCP MX v1.0 E2M1 and E8M0, bfloat16). */
double smq_oracle_e4m3(uint8_t code);
double smq_oracle_e2m1(uint8_t nibble);
double smq_oracle_ue8m0(uint8_t code);
double smq_oracle_bf16(uint16_t bits);

/* Dense logits of one paged (decode) row over positions [p0, p1) of its
 * sequence.
 *  - Position p is stored in page bt_row[p / page_size], at token p % page_size.
 *  - q8 is [H*D] E4M3, weights is [H] bf16, and out is [p1 - p0]. */
int smq_oracle_logits_paged(int H, int D, int page_size, const uint8_t *q8,
                            float q_scale, const uint16_t *weights,
                            const uint8_t *k_cache, int64_t num_pages,
                            const int32_t *bt_row, int64_t bt_cols, int64_t p0,
                            int64_t p1, double *out);

/* Dense logits of one contiguous (prefill) row.
 *  - Position p (relative to ks) is workspace row ks + p.
 *  - k_values is [total_len][D/2] and k_scales is [total_len][D/32]. */
int smq_oracle_logits_contig(int H, int D, const uint8_t *q8, float q_scale,
                             const uint16_t *weights, const uint8_t *k_values,
                             const uint8_t *k_scales, int64_t total_len,
                             int64_t ks, int64_t p0, int64_t p1, double *out);

/* Candidate mask of one row over positions [0, L).
 *  - valid[p] = 1 if p lies in a block b of cand[0..ncb) with b >= 0, that is
 *    b*cbs <= p < (b+1)*cbs. Otherwise valid[p] = 0. */
int smq_oracle_candidate_mask(int cbs, int ncb, const int32_t *cand, int64_t L,
                              uint8_t *valid);

/* Top-k of one row.
 *  - Sorts the valid positions by (logit descending, position ascending).
 *  - Writes the first min(k, #valid) positions to out[0..k), then -1. */
int smq_oracle_topk(int64_t L, const double *logits, const uint8_t *valid,
                    int k, int32_t *out);

/* Canonical candidate expansion of one row, in units of sbkv tokens.
 *  - Keeps the in-range blocks, ascending and deduplicated.
 *  - Splits each kept block into cbs/sbkv sub-blocks and drops sub-blocks that
 *    start at or past L.
 *  - Writes sub-block ids to sparse_indices[0..nsb), padded with -1.
 *  - Sets *end to the number of valid positions they cover. */
int smq_oracle_expand(int cbs, int sbkv, int ncb, const int32_t *cand,
                      int64_t L, int nsb, int32_t *sparse_indices,
                      int32_t *end);

/* Paged -> contiguous copy of one sequence's first seq_len positions.
 *  - values_out is [seq_len][D/2] and scales_out is [seq_len][D/32]. */
int smq_oracle_gather(int D, int page_size, const uint8_t *k_cache,
                      int64_t num_pages, const int32_t *bt_row,
                      int64_t bt_cols, int64_t seq_len, uint8_t *values_out,
                      uint8_t *scales_out);

/* Producers (the pages fix the formats, not the rounding; the readings are
 * in smq_oracle.c):
 *  - element encoders: nearest value, ties to the even code, saturating
 *    (E2M1 at 6, E4M3 at 448); bfloat16 round to nearest even;
 *  - one token's key [D] bf16 -> packed E2M1 values [D/2], UE8M0 scales [D/32];
 *  - ntok keys into the paged cache through slot_mapping (negative: skipped);
 *  - one query row [H*D] bf16 + weights [H] float -> E4M3 codes, float
 *    scale, bf16 weights. */
uint8_t smq_oracle_encode_e2m1(double v);
uint8_t smq_oracle_encode_e4m3(double v);
uint16_t smq_oracle_encode_bf16(float f);
int smq_oracle_quantize_k_token(int D, const uint16_t *k, uint8_t *values, uint8_t *scales);
int smq_oracle_write_k_cache(int D, int page_size, const uint16_t *k, const int64_t *slot_mapping, int64_t ntok,
                             uint8_t *cache, int64_t num_pages);
int smq_oracle_quantize_q(int H, int D, const uint16_t *q, const float *w, uint8_t *q8, float *scale,
                          uint16_t *w_bf16);

/* Candidate source: the ncb blocks (of cbs positions) of a row's dense
 * logits [L] with the largest maximum logit, ties to the lower block id, in
 * that order, then -1. block_scores [ceil(L / cbs)] (may be NULL) receives
 * each block's maximum. */
int smq_oracle_source_blocks(int64_t L, const double *logits, int cbs, int ncb, double *block_scores,
                             int32_t *cand);

#ifdef __cplusplus
}
#endif
#endif
