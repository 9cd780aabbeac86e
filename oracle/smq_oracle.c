/*
 * CPU oracle for the candidate-block sparse MQA-logits top-k indexer.
 *
 * TEST INFRASTRUCTURE ONLY: it is loaded by the tests, the smoke check and
 * the benchmark's CPU-baseline leg. It is plain, slow and double precision,
 * and it shares no code with the CUDA library. See smq_oracle.h for layouts
 * and sources.
 *
 * What is computed is the dense definition that the sparse path must equal.
 * The candidate-source indexer publishes candidate blocks. A consumer
 * indexer scores every position of the row's context, masks everything
 * outside those blocks, and takes the top-k. ("sparse_mqa_indexer" docs,
 * module docstring: the dense SparseAttnIndexer computes logits over the
 * whole context and masks, and the sparse layer must pick the same top-k
 * while scoring only the candidate blocks.)
 */
#include "smq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------------
 * Element formats
 * ------------------------------------------------------------------------- */

/* OCP OFP8 E4M3 ("fn"): sign, 4 exponent bits with bias 7, 3 mantissa bits.
 * It has no infinities, and S.1111.111 is NaN. Q values arrive as these
 * bytes ("sparse_mqa_indexer" docs, SparseMQAIndexer.forward: the Q values
 * are viewed as int8). */
double smq_oracle_e4m3(uint8_t code) {
  int sign = code >> 7;
  int e = (code >> 3) & 15;
  int m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6); /* subnormal: 0.mmm * 2^(1-7) */
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* OCP MX v1.0 FP4 E2M1: sign, 2 exponent bits with bias 1, 1 mantissa bit.
 * Every code is finite. */
double smq_oracle_e2m1(uint8_t nibble) {
  int sign = (nibble >> 3) & 1;
  int e = (nibble >> 1) & 3;
  int m = nibble & 1;
  double v;
  if (e == 0)
    v = 0.5 * (double)m; /* subnormal: 0.m * 2^(1-1) */
  else
    v = ldexp(1.0 + (double)m / 2.0, e - 1);
  return sign ? -v : v;
}

/* OCP MX v1.0 E8M0 scale: 2^(code - 127), and 0xFF is NaN. The K cache
 * carries one per 32 elements ("sparse_indexer.py", builder __init__:
 * UE8M0-packed granularity-32 scales). */
double smq_oracle_ue8m0(uint8_t code) {
  if (code == 0xFF) return NAN;
  return ldexp(1.0, (int)code - 127);
}

/* bfloat16: the upper half of an IEEE binary32. The per-head weights are
 * bf16 ("sparse_mqa_indexer" docs, weights_dtype). */
double smq_oracle_bf16(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* ---------------------------------------------------------------------------
 * Keys
 * ------------------------------------------------------------------------- */

/* Decode one token's key from its packed values and scales. */
static int decode_key(int D, const uint8_t *vals, const uint8_t *scales,
                      double *k) {
  for (int d = 0; d < D; ++d) {
    uint8_t byte = vals[d / 2];
    uint8_t nib = (d % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
    k[d] = smq_oracle_e2m1(nib) * smq_oracle_ue8m0(scales[d / 32]);
    if (!isfinite(k[d])) return -1;
  }
  return 0;
}

/* Key of sequence position p of a paged request. The page comes from the
 * request's block-table row ("sparse_mqa_indexer" docs, forward: the decode
 * call takes the paged cache, block_table and row_indices). */
static int key_paged(int D, int page_size, const uint8_t *k_cache,
                     int64_t num_pages, const int32_t *bt_row, int64_t bt_cols,
                     int64_t p, double *k) {
  int64_t slot = p / page_size;
  int64_t tok = p % page_size;
  int64_t page_bytes = (int64_t)page_size * (D / 2 + D / 32);
  if (p < 0 || slot >= bt_cols) return -1;
  int64_t page = bt_row[slot];
  if (page < 0 || page >= num_pages) return -1;
  const uint8_t *base = k_cache + page * page_bytes;
  const uint8_t *vals = base + tok * (D / 2);
  const uint8_t *scales = base + (int64_t)page_size * (D / 2) + tok * (D / 32);
  return decode_key(D, vals, scales, k);
}

/* ---------------------------------------------------------------------------
 * Score
 * ------------------------------------------------------------------------- */

/* Dequantised query of one row: Q[h][d] = e4m3(q8[h][d]) * q_scale, the
 * per-row scale applied to the FP8 query; w[h] = bf16(weights[h]). */
static int decode_query(int H, int D, const uint8_t *q8, float q_scale,
                        const uint16_t *weights, double *q, double *w) {
  for (int i = 0; i < H * D; ++i) {
    q[i] = smq_oracle_e4m3(q8[i]) * (double)q_scale;
    if (!isfinite(q[i])) return -1;
  }
  for (int h = 0; h < H; ++h) {
    w[h] = smq_oracle_bf16(weights[h]);
    if (!isfinite(w[h])) return -1;
  }
  return 0;
}

/* logit = sum_h w[h] * max(0, sum_d Q[h][d] * K[d]). */
static double score(int H, int D, const double *q, const double *w,
                    const double *k) {
  double logit = 0.0;
  for (int h = 0; h < H; ++h) {
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += q[h * D + d] * k[d];
    double relu = dot > 0.0 ? dot : 0.0;
    logit += w[h] * relu;
  }
  return logit;
}

/* Scratch for one row: key [D], query [H*D], weights [H]. */
typedef struct {
  double *k, *q, *w;
} row_scratch;

static int scratch_init(row_scratch *s, int H, int D, const uint8_t *q8,
                        float q_scale, const uint16_t *weights) {
  s->k = (double *)malloc(sizeof(double) * (size_t)D);
  s->q = (double *)malloc(sizeof(double) * (size_t)H * (size_t)D);
  s->w = (double *)malloc(sizeof(double) * (size_t)H);
  if (!s->k || !s->q || !s->w) return -1;
  return decode_query(H, D, q8, q_scale, weights, s->q, s->w);
}

static void scratch_free(row_scratch *s) {
  free(s->k);
  free(s->q);
  free(s->w);
}

int smq_oracle_logits_paged(int H, int D, int page_size, const uint8_t *q8,
                            float q_scale, const uint16_t *weights,
                            const uint8_t *k_cache, int64_t num_pages,
                            const int32_t *bt_row, int64_t bt_cols, int64_t p0,
                            int64_t p1, double *out) {
  row_scratch s;
  int rc = scratch_init(&s, H, D, q8, q_scale, weights);
  for (int64_t p = p0; p < p1 && rc == 0; ++p) {
    rc = key_paged(D, page_size, k_cache, num_pages, bt_row, bt_cols, p, s.k);
    if (rc == 0) out[p - p0] = score(H, D, s.q, s.w, s.k);
    if (rc == 0 && !isfinite(out[p - p0])) rc = -1;
  }
  scratch_free(&s);
  return rc;
}

int smq_oracle_logits_contig(int H, int D, const uint8_t *q8, float q_scale,
                             const uint16_t *weights, const uint8_t *k_values,
                             const uint8_t *k_scales, int64_t total_len,
                             int64_t ks, int64_t p0, int64_t p1, double *out) {
  row_scratch s;
  int rc = scratch_init(&s, H, D, q8, q_scale, weights);
  for (int64_t p = p0; p < p1 && rc == 0; ++p) {
    int64_t row = ks + p; /* the workspace row of sequence position p */
    if (row < 0 || row >= total_len) {
      rc = -1;
      break;
    }
    rc = decode_key(D, k_values + row * (D / 2), k_scales + row * (D / 32), s.k);
    if (rc == 0) out[p - p0] = score(H, D, s.q, s.w, s.k);
    if (rc == 0 && !isfinite(out[p - p0])) rc = -1;
  }
  scratch_free(&s);
  return rc;
}

/* ---------------------------------------------------------------------------
 * Mask, top-k
 * ------------------------------------------------------------------------- */

/* A position is a candidate if some published block covers it. Blocks are
 * in units of candidate_block_size, and -1 or any negative id names no
 * block. Positions at or past the row's end L are not keys at all. */
int smq_oracle_candidate_mask(int cbs, int ncb, const int32_t *cand, int64_t L,
                              uint8_t *valid) {
  memset(valid, 0, (size_t)L);
  for (int i = 0; i < ncb; ++i) {
    int64_t b = cand[i];
    if (b < 0) continue;
    for (int64_t j = 0; j < cbs; ++j) {
      int64_t p = b * cbs + j;
      if (p < L) valid[p] = 1;
    }
  }
  return 0;
}

typedef struct {
  double v;
  int64_t p;
} scored_pos;

static int by_logit_desc_pos_asc(const void *a, const void *b) {
  const scored_pos *x = (const scored_pos *)a;
  const scored_pos *y = (const scored_pos *)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->p > y->p) - (x->p < y->p);
}

/* The k best valid positions. A row with fewer valid positions keeps -1 in
 * the rest ("sparse_mqa_indexer" docs, forward: the output rows are filled
 * with -1 before any kernel runs). */
int smq_oracle_topk(int64_t L, const double *logits, const uint8_t *valid,
                    int k, int32_t *out) {
  int64_t n = 0;
  for (int64_t p = 0; p < L; ++p) n += valid[p] ? 1 : 0;
  scored_pos *s = (scored_pos *)malloc(sizeof(scored_pos) * (size_t)(n ? n : 1));
  if (!s) return -1;
  int64_t i = 0;
  for (int64_t p = 0; p < L; ++p)
    if (valid[p]) {
      s[i].v = logits[p];
      s[i].p = p;
      ++i;
    }
  qsort(s, (size_t)n, sizeof(scored_pos), by_logit_desc_pos_asc);
  for (int j = 0; j < k; ++j) out[j] = (j < n) ? (int32_t)s[j].p : -1;
  free(s);
  return 0;
}

/* ---------------------------------------------------------------------------
 * Candidate expansion
 * ------------------------------------------------------------------------- */

static int int64_asc(const void *a, const void *b) {
  int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
  return (x > y) - (x < y);
}

/* The per-row state is sparse_indices [rows, num_sparse_blocks] of sparse
 * block ids plus end [rows], the valid sparse-column count. Here
 * num_sparse_blocks = candidate_topk_blocks * (candidate_block_size /
 * sparse_block_kv). ("sparse_indexer.py", SparseMQARowsMetadata and the
 * builder __init__.) Its canonical form:
 *  - the in-range candidate blocks, ascending and without repeats;
 *  - each split into cbs/sbkv sub-blocks;
 *  - sub-blocks that start at or past L dropped;
 *  - -1 after the last.
 * end counts the positions below L that the kept sub-blocks cover. */
int smq_oracle_expand(int cbs, int sbkv, int ncb, const int32_t *cand,
                      int64_t L, int nsb, int32_t *sparse_indices,
                      int32_t *end) {
  if (sbkv <= 0 || cbs % sbkv != 0) return -1;
  int64_t *kept = (int64_t *)malloc(sizeof(int64_t) * (size_t)(ncb ? ncb : 1));
  if (!kept) return -1;
  int nk = 0;
  for (int i = 0; i < ncb; ++i) {
    int64_t b = cand[i];
    if (b >= 0 && b * cbs < L) kept[nk++] = b;
  }
  qsort(kept, (size_t)nk, sizeof(int64_t), int64_asc);
  int nu = 0;
  for (int i = 0; i < nk; ++i)
    if (nu == 0 || kept[nu - 1] != kept[i]) kept[nu++] = kept[i];
  int per = cbs / sbkv;
  int out = 0;
  int64_t cols = 0;
  for (int i = 0; i < nu; ++i) {
    for (int j = 0; j < per; ++j) {
      int64_t sub = kept[i] * per + j;
      int64_t start = sub * sbkv;
      if (start >= L) continue;
      if (out >= nsb) {
        free(kept);
        return -1;
      }
      sparse_indices[out++] = (int32_t)sub;
      cols += (L - start < sbkv) ? (L - start) : sbkv;
    }
  }
  for (int i = out; i < nsb; ++i) sparse_indices[i] = -1;
  *end = (int32_t)cols;
  free(kept);
  return 0;
}

/* ---------------------------------------------------------------------------
 * Gather
 * ------------------------------------------------------------------------- */

/* Copy a sequence's paged K into the packed (values, scales) workspace
 * ("sparse_mqa_indexer" docs, _gather_prefill_chunk_k and
 * _prefill_k_workspaces). */
int smq_oracle_gather(int D, int page_size, const uint8_t *k_cache,
                      int64_t num_pages, const int32_t *bt_row,
                      int64_t bt_cols, int64_t seq_len, uint8_t *values_out,
                      uint8_t *scales_out) {
  int64_t page_bytes = (int64_t)page_size * (D / 2 + D / 32);
  for (int64_t p = 0; p < seq_len; ++p) {
    int64_t slot = p / page_size, tok = p % page_size;
    if (slot >= bt_cols) return -1;
    int64_t page = bt_row[slot];
    if (page < 0 || page >= num_pages) return -1;
    const uint8_t *base = k_cache + page * page_bytes;
    memcpy(values_out + p * (D / 2), base + tok * (D / 2), (size_t)(D / 2));
    memcpy(scales_out + p * (D / 32),
           base + (int64_t)page_size * (D / 2) + tok * (D / 32),
           (size_t)(D / 32));
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * Producers: the MXFP4 K-cache writer and the FP8 query quantiser
 * ------------------------------------------------------------------------- */

/* The model writes the MXFP4 indexer K cache, and a fused query kernel emits
 * the FP8 query, its per-row scale and the bf16 head weights
 * ("sparse_mqa_indexer" docs, SparseMQAIndexer and weights_dtype;
 * "sparse_indexer.py", builder __init__: MXFP4 with UE8M0-packed
 * granularity-32 scales). The pages give no rounding rules; the readings
 * taken here are:
 *  - K: per group of 32, the scale exponent e is the smallest integer with
 *    amax <= 6 * 2^e (no element saturates), the UE8M0 code e + 127 clamped
 *    to [1, 254]; each element x * 2^-e rounds to the nearest E2M1 value,
 *    ties to the even code, clamped to +-6. A group of zeros has code 127.
 *  - Q: scale = amax / 448 in float (1 for a zero row); each element
 *    x / scale, divided in float, rounds to the nearest E4M3 value, ties to
 *    the even code, clamped to +-448.
 *  - weights: float to bfloat16, round to nearest, ties to even.
 * The sign of an element that rounds to zero is kept (IEEE rounding). */

/* Nearest value of a table of non-negative values (codes 0..n-1 in
 * increasing order), ties to the even code, saturating at the last. */
static int nearest_code(double a, const double *table, int n) {
  if (a > table[n - 1]) a = table[n - 1]; /* saturation */
  int best = 0;
  for (int c = 1; c < n; ++c) {
    double dc = fabs(a - table[c]), db = fabs(a - table[best]);
    if (dc < db || (dc == db && (c % 2) == 0)) best = c;
  }
  return best;
}

uint8_t smq_oracle_encode_e2m1(double v) {
  double table[8];
  for (int c = 0; c < 8; ++c) table[c] = smq_oracle_e2m1((uint8_t)c);
  int c = nearest_code(fabs(v), table, 8);
  return (uint8_t)(signbit(v) ? (c | 8) : c);
}

uint8_t smq_oracle_encode_e4m3(double v) {
  double table[127]; /* codes 0x00..0x7E; 0x7F is NaN */
  for (int c = 0; c < 127; ++c) table[c] = smq_oracle_e4m3((uint8_t)c);
  int c = nearest_code(fabs(v), table, 127);
  return (uint8_t)(signbit(v) ? (c | 0x80) : c);
}

uint16_t smq_oracle_encode_bf16(float f) {
  /* the bfloat16 nearest to f: compare the two neighbours that truncation
   * and truncation plus one ulp give (f finite) */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint16_t lo = (uint16_t)(u >> 16), hi = (uint16_t)(lo + 1);
  double dlo = fabs((double)f - smq_oracle_bf16(lo));
  double dhi = fabs((double)f - smq_oracle_bf16(hi));
  if (dhi < dlo || (dhi == dlo && (hi & 1) == 0)) return hi;
  return lo;
}

/* One token's key (D bf16 values) to its packed E2M1 values [D/2] and
 * UE8M0 scales [D/32]. */
int smq_oracle_quantize_k_token(int D, const uint16_t *k, uint8_t *values, uint8_t *scales) {
  for (int g = 0; g < D / 32; ++g) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) {
      double x = smq_oracle_bf16(k[32 * g + i]);
      if (!isfinite(x)) return -1;
      if (fabs(x) > amax) amax = fabs(x);
    }
    int e = 0;
    if (amax > 0.0) {
      e = ilogb(amax) - 3; /* 6 * 2^e < amax here; step up to the first e that covers it */
      while (6.0 * ldexp(1.0, e) < amax) ++e;
    }
    int code = e + 127;
    if (code < 1) code = 1;
    if (code > 254) code = 254;
    e = code - 127;
    scales[g] = (uint8_t)code;
    for (int i = 0; i < 32; i += 2) {
      uint8_t lo = smq_oracle_encode_e2m1(ldexp(smq_oracle_bf16(k[32 * g + i]), -e));
      uint8_t hi = smq_oracle_encode_e2m1(ldexp(smq_oracle_bf16(k[32 * g + i + 1]), -e));
      values[(32 * g + i) / 2] = (uint8_t)(lo | (hi << 4));
    }
  }
  return 0;
}

/* Quantise ntok tokens' keys [ntok][D] into the paged cache: token t goes to
 * slot slot_mapping[t] = page * page_size + offset (negative: skipped). */
int smq_oracle_write_k_cache(int D, int page_size, const uint16_t *k, const int64_t *slot_mapping, int64_t ntok,
                             uint8_t *cache, int64_t num_pages) {
  int64_t page_bytes = (int64_t)page_size * (D / 2 + D / 32);
  for (int64_t t = 0; t < ntok; ++t) {
    int64_t s = slot_mapping[t];
    if (s < 0) continue;
    int64_t page = s / page_size, off = s % page_size;
    if (page >= num_pages) return -1;
    uint8_t *base = cache + page * page_bytes;
    if (smq_oracle_quantize_k_token(D, k + t * D, base + off * (D / 2),
                                    base + (int64_t)page_size * (D / 2) + off * (D / 32)) != 0)
      return -1;
  }
  return 0;
}

/* One query row: q [H*D] bf16 and weights [H] float to the E4M3 codes
 * [H*D], the float scale and the bf16 weights [H]. */
int smq_oracle_quantize_q(int H, int D, const uint16_t *q, const float *w, uint8_t *q8, float *scale,
                          uint16_t *w_bf16) {
  float amax = 0.0f;
  for (int i = 0; i < H * D; ++i) {
    float x = (float)smq_oracle_bf16(q[i]);
    if (!isfinite(x)) return -1;
    if (fabsf(x) > amax) amax = fabsf(x);
  }
  float s = amax > 0.0f ? amax / 448.0f : 1.0f;
  *scale = s;
  for (int i = 0; i < H * D; ++i) {
    float v = (float)smq_oracle_bf16(q[i]) / s;
    q8[i] = smq_oracle_encode_e4m3((double)v);
  }
  for (int h = 0; h < H; ++h) {
    if (!isfinite(w[h])) return -1;
    w_bf16[h] = smq_oracle_encode_bf16(w[h]);
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * Candidate source
 * ------------------------------------------------------------------------- */

/* The candidate-source indexer of two-level selection: a dense indexer over
 * the row's whole context that publishes its top candidate blocks
 * ("sparse_mqa_indexer" docs, module docstring; "rocm_paged_mxfp4_indexer"
 * docs, RocmSparseAttnIndexer: the source layer publishes its candidate
 * pool, candidate_write). The pages do not define a block's score. The
 * reading taken here: the score of block b (positions [b*cbs, (b+1)*cbs)
 * below L) is the largest dense logit among its positions; the ncb blocks of
 * highest score are published, ties to the lower block id, in that order,
 * then -1 when the context has fewer blocks. */
typedef struct {
  double v;
  int64_t b;
} scored_block;

static int by_score_desc_id_asc(const void *a, const void *b) {
  const scored_block *x = (const scored_block *)a;
  const scored_block *y = (const scored_block *)b;
  if (x->v != y->v) return x->v > y->v ? -1 : 1;
  return (x->b > y->b) - (x->b < y->b);
}

int smq_oracle_source_blocks(int64_t L, const double *logits, int cbs, int ncb, double *block_scores,
                             int32_t *cand) {
  int64_t nb = L > 0 ? (L + cbs - 1) / cbs : 0;
  scored_block *s = (scored_block *)malloc(sizeof(scored_block) * (size_t)(nb ? nb : 1));
  if (!s) return -1;
  for (int64_t b = 0; b < nb; ++b) {
    double m = -INFINITY;
    for (int64_t p = b * cbs; p < (b + 1) * cbs && p < L; ++p)
      if (logits[p] > m) m = logits[p];
    s[b].v = m;
    s[b].b = b;
    if (block_scores) block_scores[b] = m;
  }
  qsort(s, (size_t)nb, sizeof(scored_block), by_score_desc_id_asc);
  for (int i = 0; i < ncb; ++i) cand[i] = i < nb ? (int32_t)s[i].b : -1;
  free(s);
  return 0;
}
