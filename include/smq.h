/*
 * smq.h: C ABI of the GB300 candidate-block sparse MQA-logits top-k indexer.
 *
 * DeepSeek-V4.1 two-level selection works like this. A candidate-source
 * indexer publishes, for every query row, its top candidate blocks. Each
 * later consumer indexer then scores only the key positions inside those
 * blocks and keeps its top-k token ids, so its work is O(candidate blocks)
 * rather than O(context). Source: the "vllm.model_executor.layers.
 * sparse_mqa_indexer" API docs, module docstring and SparseMQAIndexer.
 *
 * For a row with FP8 query q[h][d] (H heads, D = 128), per-row scale s,
 * bf16 head weights w[h] and key k[d], the score of a position is
 *     logit = sum_h w[h] * ReLU(s * q[h] . k).
 * This is the DeepSeek indexer score that the pages' MQA-logits kernels
 * compute. The pages name it but do not print it.
 *
 * Positions outside the row's key range [ks, ke), and positions in no
 * valid candidate block, are masked. The top-k token ids per row are
 * written relative to ks, padded with -1.
 *
 * Conventions of every entry point
 *  - Every pointer named "device" is CUDA device memory owned by the caller.
 *    The library allocates nothing in any call. Only smq_plan_create and
 *    smq_plan_destroy allocate or free host memory for the plan itself.
 *    (Source: "vllm/v1/attention/backends/mla/sparse_indexer.py", module
 *    docstring: the layer op allocates nothing per step.)
 *  - Every call is asynchronous on the caller's stream (a cudaStream_t
 *    passed as void*; NULL is the legacy default stream). Exceptions:
 *    smq_plan_create, smq_plan_destroy and smq_get_status.
 *  - Every call returns an smq_status code. A non-zero return means nothing
 *    was enqueued.
 *  - Errors the GPU detects are OR-ed into a status word at the start of
 *    the workspace: an out-of-range page, block-table row or block id
 *    (SMQ_ERR_BOUNDS), or a pipeline wait that gave up (SMQ_ERR_TIMEOUT).
 *    The outputs of a call that raised one are unspecified.
 *    smq_get_status reads the word and clears it.
 *  - The arguments are checked once, at plan creation ("engine start").
 *    Calls only re-check pointers, alignment and sizes. (Source:
 *    sparse_indexer.py, DeepseekV41SparseIndexerMetadataBuilder: every
 *    requirement of the sparse kernels is checked at engine start rather
 *    than by falling back per step.)
 *  - Argument structs begin with struct_size. Set it to sizeof(the struct)
 *    so that later versions can append fields.
 *
 * Formats (the pages fix the element formats; the byte layout is this
 * library's)
 *  - Q: [rows][H][D] bytes, OCP FP8 E4M3 ("fn"). q_scale: [rows] float,
 *    positive and finite.
 *  - weights: [rows][H] bfloat16 (as uint16 bits).
 *  - Paged MXFP4 K cache: pages of page_size tokens. page_bytes =
 *    page_size * (D/2 + D/32), and the cache base must be 16-byte aligned.
 *    A page is
 *      values [page_size][D/2]: OCP MX FP4 E2M1, element 2i in the low
 *        nibble of byte i and element 2i+1 in the high nibble;
 *      scales [page_size][D/32]: OCP MX E8M0 exponents, byte g scaling
 *        elements [32g, 32g+32). 0xFF (NaN) must not occur.
 *    (Source: sparse_indexer.py, builder __init__: the MXFP4 indexer cache
 *    with UE8M0-packed granularity-32 scales.)
 *  - Contiguous K workspace (prefill): values [total_len][D/2] and scales
 *    [total_len][D/32] with the same encodings. This is the layout the
 *    gather writes. (Source: sparse_mqa_indexer docs,
 *    _prefill_k_workspaces.)
 *  - Candidate blocks: [rows][candidate_topk_blocks] int32 block ids, in
 *    units of candidate_block_size tokens, relative to the row's ks.
 *    Negative ids name no block. Blocks at or past the row's end are
 *    masked.
 */
#ifndef SMQ_H
#define SMQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SMQ_API __attribute__((visibility("default")))

typedef enum smq_status {
  SMQ_OK = 0,
  SMQ_ERR_INVALID_ARG = 1,         /* null or misaligned pointer, bad size */
  SMQ_ERR_UNSUPPORTED = 2,         /* shape or device this library cannot run */
  SMQ_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < smq_workspace_size() */
  SMQ_ERR_CUDA = 4,                /* a CUDA runtime or driver call failed */
  SMQ_ERR_BOUNDS = 8,              /* device: page / row / block id out of range */
  SMQ_ERR_TIMEOUT = 16             /* device: a pipeline wait gave up */
} smq_status;

typedef struct smq_plan smq_plan;

/* Geometry fixed at engine start. (Source: sparse_indexer.py, builder
 * __init__: the hf config's candidate_block_size, candidate_topk_blocks and
 * index_topk; the page size of the indexer cache spec; and
 * pick_sparse_block_kv / check_deep_select_layout.) */
typedef struct smq_plan_desc {
  uint32_t struct_size;
  int32_t num_heads;             /* H: a multiple of 8 in [8, 128] */
  int32_t head_dim;              /* D: must be 128 */
  int32_t page_size;             /* tokens per cache page: a multiple of sparse_block_kv */
  int32_t candidate_block_size;  /* cbs > 0 */
  int32_t candidate_topk_blocks; /* ncb > 0 candidate blocks per row */
  int32_t topk;                  /* k: 1 <= k <= num_sparse_cols, k <= 16384 */
  int32_t sparse_block_kv;       /* sub-block size in tokens: 16, 32, 64 or 128 (else
                                    SMQ_ERR_UNSUPPORTED); 0 picks the largest of
                                    128/64/32/16 dividing both page_size and cbs */
  int32_t max_rows;              /* upper bound on rows per call (workspace sizing), <= 8192 */
  int32_t device;                /* CUDA device ordinal the plan runs on */
} smq_plan_desc;

/* Values derived at plan creation. */
typedef struct smq_plan_info {
  uint32_t struct_size;
  int32_t sparse_block_kv;   /* tokens per sparse sub-block */
  int32_t num_sparse_blocks; /* per row: ncb * (cbs / sparse_block_kv) */
  int32_t num_sparse_cols;   /* S = num_sparse_blocks * sparse_block_kv */
  int32_t page_bytes;        /* bytes per K-cache page */
  int32_t num_sms;           /* SM count of the plan's device */
} smq_plan_info;

/* Validate the descriptor and create a plan. It reads the device's SM
 * count and does no GPU work. The plan is host memory owned by the caller
 * until smq_plan_destroy. Returns SMQ_ERR_INVALID_ARG or
 * SMQ_ERR_UNSUPPORTED for a geometry this library does not run. */
SMQ_API int smq_plan_create(const smq_plan_desc *desc, smq_plan **plan);
SMQ_API int smq_plan_destroy(smq_plan *plan);
SMQ_API int smq_plan_get_info(const smq_plan *plan, smq_plan_info *info);

/* Failure-path controls of later calls with this plan (host side; not
 * thread-safe with calls in flight on other threads).
 *  - smq_plan_set_wait_limit: every pipeline wait gives up after ns
 *    nanoseconds (default 2e9) and raises SMQ_ERR_TIMEOUT; the kernel then
 *    winds down: it waits, bounded, for its own copies in flight, drains its
 *    MMAs and frees its TMEM.
 *  - smq_plan_inject_stall: for tests of that path. The loaders of the first
 *    CTA of the score kernel withhold the hand-off of its tile `tile` to the
 *    MMA, so that the MMA's wait runs out. -1 (the default) withholds
 *    nothing. The outputs of a stalled call are unspecified; zero the
 *    workspace (smq_workspace_init) before the next call. */
SMQ_API int smq_plan_set_wait_limit(smq_plan *plan, int64_t ns);
SMQ_API int smq_plan_inject_stall(smq_plan *plan, int32_t tile);

/* Device workspace bytes for calls of up to `rows` rows (<= max_rows).
 * It holds the status word, one tile counter per plan row (decode calls that
 * expand their rows in the score kernel also select their top-k there; the
 * counters find the CTA that finishes a row) and the fp32 logits scratch
 * [rows][S]. Allocate it once, then zero it with smq_workspace_init. A call
 * leaves the counters at zero; after a call whose status reports an error,
 * zero the workspace again before the next call. */
SMQ_API int smq_workspace_size(const smq_plan *plan, int32_t rows, size_t *bytes);

/* Device workspace bytes for prefill chunks of up to `rows` rows and
 * `total_len` workspace rows. It adds to smq_workspace_size(plan, rows) the
 * scratch of the window-major prefill path: per workspace position a window
 * count and a cursor (int32 each), per row a record count and its 64 head
 * weights and q_scale as float, per (row, window) pair a record (8 bytes) and
 * a group slot (32 bytes per two records). The path applies to 64-head plans
 * and total_len <= 2^20; otherwise the size equals smq_workspace_size.
 * A prefill call whose workspace is smaller than this (but at least
 * smq_workspace_size) runs the row-major path instead; both give the same
 * logits, bit for bit, and the same top-k. Errors: SMQ_ERR_INVALID_ARG for a
 * null plan or bytes, rows < 0 or > max_rows, total_len < 0. */
SMQ_API int smq_prefill_workspace_size(const smq_plan *plan, int32_t rows, int64_t total_len, size_t *bytes);

/* Zero the workspace status word and tile counters (async on stream). */
SMQ_API int smq_workspace_init(const smq_plan *plan, void *workspace, size_t workspace_bytes,
                               void *stream);

/* Synchronise `stream`, read the workspace status word into *code (a
 * bitwise OR of SMQ_ERR_BOUNDS / SMQ_ERR_TIMEOUT, or 0), then clear it. */
SMQ_API int smq_get_status(const void *workspace, void *stream, int32_t *code);

SMQ_API const char *smq_error_string(int code);

/* Shared per-step candidate expansion. (Source: sparse_indexer.py,
 * SparseMQARowsMetadata and the module docstring: the first consumer layer
 * of a step fills sparse_indices / end, and later consumer layers reuse
 * them.)
 * For each row, with L = row_ke - row_ks:
 *  - drop negative blocks and blocks starting at or past L;
 *  - sort the rest ascending without repeats;
 *  - split each into cbs/sbkv sub-blocks, dropping sub-blocks that start at
 *    or past L.
 * Outputs (device memory):
 *  - sparse_indices [rows][num_sparse_blocks] int32: sub-block ids in units
 *    of sbkv tokens, relative to row_ks, then -1 padding.
 *  - end [rows] int32: the number of valid sparse columns. Every sparse
 *    column c < end is a key position, and only the last kept sub-block
 *    can be partial.
 * Inputs (device memory):
 *  - candidate_blocks [rows][ncb] int32;
 *  - row_ks [rows] int32, or NULL for all zeros (paged decode);
 *  - row_ke [rows] int32.
 * rows may be 0, which enqueues nothing. */
SMQ_API int sparse_mqa_candidate_expand(const smq_plan *plan, const int32_t *candidate_blocks,
                                        const int32_t *row_ks, const int32_t *row_ke,
                                        int32_t rows, int32_t *sparse_indices, int32_t *end,
                                        void *workspace, size_t workspace_bytes, void *stream);

/* Paged decode: one query row per decode token. (Source: sparse_mqa_indexer
 * docs, SparseMQAIndexer.forward, the sparse_mqa_logits_paged_decode call;
 * sparse_indexer.py, SparseMQARowsMetadata and build(): row_ks is zero for
 * paged decode, row_ke is the compressed context length, block_table is
 * [rows, pages], and row_indices maps row -> request.) */
typedef struct smq_decode_args {
  uint32_t struct_size;
  int32_t rows;                   /* R >= 0 */
  const uint8_t *q;               /* device [R][H][D] E4M3 */
  const float *q_scale;           /* device [R] */
  const uint16_t *weights;        /* device [R][H] bf16 */
  const uint8_t *k_cache;         /* device [num_pages][page_bytes], 16-byte aligned (32-byte
                                    aligned lets rows that share pages use tensor copies) */
  int64_t num_pages;
  const int32_t *block_table;     /* device [bt_rows][bt_stride] page ids */
  int32_t bt_rows;
  int32_t bt_stride;              /* columns of block_table */
  const int32_t *row_indices;     /* device [R] row -> block-table row, or NULL = identity */
  const int32_t *row_ke;          /* device [R] context length of the row */
  const int32_t *candidate_blocks;/* device [R][ncb] */
  int32_t *topk_out;              /* device [R][topk_ld]; columns [0, topk) are written */
  int32_t topk_ld;                /* >= topk */
  int32_t *sparse_indices;        /* device [R][num_sparse_blocks]: written if !expansion_ready */
  int32_t *end;                   /* device [R]: written if !expansion_ready */
  int32_t expansion_ready;        /* 1: sparse_indices / end already hold this step's expansion */
  int32_t *col_indices;           /* device [R][topk] selected sparse columns, or NULL */
  float *logits_out;              /* device [R][S] fp32 logits by sparse column (columns >= end
                                     are -inf), or NULL */
  void *workspace;                /* device, >= smq_workspace_size(plan, R) bytes */
  size_t workspace_bytes;
  void *profile_events[4];        /* optional cudaEvent_t, recorded on the stream before the
                                     expansion, before the gather+score kernel, before the top-k
                                     and after it; NULL entries are skipped */
  uint16_t *logits_out_bf16;      /* device [R][S] bf16 logits by sparse column, each the fp32
                                     logit rounded to the nearest-even bf16 (columns >= end are
                                     -inf), or NULL. The top-k still selects on the fp32 logits.
                                     Read only when struct_size covers it. (Source:
                                     sparse_indexer.py, builder __init__: DeepSelect takes bf16
                                     logits.) */
} smq_decode_args;

SMQ_API int sparse_mqa_logits_topk_decode(const smq_plan *plan, const smq_decode_args *args,
                                          void *stream);

/* Paged decode for callers that cannot allocate device memory, for
 * example code running where cudaMalloc is forbidden or where memory is
 * owned by another allocator (a graph-replay engine or a runtime that hands
 * out only its own tensors). The pages have no counterpart to this call.
 *
 * It does what sparse_mqa_logits_topk_decode does, with the same arguments,
 * except that args->workspace must be NULL and args->workspace_bytes 0. The
 * library uses its own scratch instead: a static device array of 256 bytes
 * plus 8 MiB (SMQ_NOALLOC_SCRATCH_BYTES) for the tile counters and the fp32
 * logits, held on every GPU that loads the library until the process exits.
 *  - The counters (4 bytes per plan row, rounded up to 256) plus
 *    rows * num_sparse_cols * 4 must not exceed 8 MiB, for example 200 rows
 *    of 8192 columns. A larger call returns SMQ_ERR_WORKSPACE_TOO_SMALL and
 *    enqueues nothing. The limit holds whether or not logits_out is given.
 *  - The first call on a device looks up the scratch's device address
 *    (cudaGetSymbolAddress) with that device current. Make that first call
 *    before any stream capture.
 *  - Every call shares the one scratch: calls that overlap on the GPU (on
 *    different streams without ordering) race. Each call zeroes the scratch
 *    status word and counters first.
 *  - Device-detected errors (bad page or row ids, timeouts) are recorded in
 *    the scratch and not returned. Callers who need them use
 *    sparse_mqa_logits_topk_decode with a workspace.
 * It calls no cudaMalloc, cudaFree or allocating routine. */
#define SMQ_NOALLOC_SCRATCH_BYTES (8u << 20)
SMQ_API int sparse_mqa_logits_topk_decode_noalloc(const smq_plan *plan, const smq_decode_args *args,
                                                  void *stream);

/* One prefill chunk on a contiguous K workspace. (Source: sparse_mqa_indexer
 * docs, SparseMQAIndexer.forward, the sparse_mqa_logits_prefill_chunk call
 * with cu_seqlen_ks / cu_seqlen_ke.) Row r's keys are workspace rows
 * [cu_seqlen_ks[r], cu_seqlen_ke[r]). Its candidate blocks and output ids
 * are relative to cu_seqlen_ks[r].
 * With a workspace of smq_prefill_workspace_size(plan, R, total_len) bytes
 * (64-head plans) the chunk runs window-major: the rows are indexed by the
 * 128-key windows [ks + 128 u, ks + 128 u + 128) their sparse sub-blocks fall
 * in, and each window's keys stay in shared memory while the query tiles of
 * the rows that selected it stream past. Four kernels then run before the
 * top-k: record, plan and fill of the index, and the score (plus one memset
 * of the window counts); profile_events[1] is recorded after the index. */
typedef struct smq_prefill_args {
  uint32_t struct_size;
  int32_t rows;
  const uint8_t *q;               /* device [R][H][D] E4M3 */
  const float *q_scale;           /* device [R] */
  const uint16_t *weights;        /* device [R][H] bf16 */
  const uint8_t *k_values;        /* device [total_len][D/2], 32-byte aligned */
  const uint8_t *k_scales;        /* device [total_len][D/32], 4-byte aligned */
  int64_t total_len;
  const int32_t *cu_seqlen_ks;    /* device [R] */
  const int32_t *cu_seqlen_ke;    /* device [R] */
  const int32_t *candidate_blocks;/* device [R][ncb] */
  int32_t *topk_out;
  int32_t topk_ld;
  int32_t *sparse_indices;
  int32_t *end;
  int32_t expansion_ready;
  int32_t *col_indices;
  float *logits_out;
  void *workspace;
  size_t workspace_bytes;
  void *profile_events[4];        /* as in smq_decode_args */
  uint16_t *logits_out_bf16;      /* as in smq_decode_args */
} smq_prefill_args;

SMQ_API int sparse_mqa_logits_topk_prefill_chunk(const smq_plan *plan, const smq_prefill_args *args,
                                                 void *stream);

/* Paged -> contiguous K gather for a prefill chunk. (Source:
 * sparse_mqa_indexer docs, _gather_prefill_chunk_k:
 * cp_gather_indexer_k_quant_cache with the chunk's block_table and
 * local_cu_seq_lens.) Sequence s occupies workspace rows
 * [cu_seq_lens[s], cu_seq_lens[s+1]). Its position p comes from page
 * block_table[s][p / page_size].
 *  - block_table: device [num_seqs][bt_stride].
 *  - cu_seq_lens: device [num_seqs + 1], non-decreasing, with
 *    cu_seq_lens[num_seqs] == total_len.
 *  - k_values: device [total_len][D/2]. k_scales: device [total_len][D/32].
 * An out-of-range page raises SMQ_ERR_BOUNDS in the workspace status word,
 * and that position is left unwritten. */
SMQ_API int sparse_mqa_gather_k(const smq_plan *plan, const uint8_t *k_cache, int64_t num_pages,
                                const int32_t *block_table, int32_t bt_stride,
                                const int32_t *cu_seq_lens, int32_t num_seqs, int64_t total_len,
                                uint8_t *k_values, uint8_t *k_scales, void *workspace,
                                size_t workspace_bytes, void *stream);

/* The candidate source of two-level selection, on paged decode rows: a
 * dense indexer over each row's whole context [0, row_ke) that publishes the
 * row's best candidate blocks for the consumer calls above. (Source:
 * sparse_mqa_indexer docs, module docstring: the candidate-source indexer
 * publishes the top candidate blocks and later indexers pick their top-k
 * inside them; rocm_paged_mxfp4_indexer docs, RocmSparseAttnIndexer: the
 * source layer publishes its candidate pool, candidate_write.) The pages do
 * not define a block's score. This library's: block b (positions
 * [b * cbs, (b + 1) * cbs) below row_ke) scores its largest logit, the
 * logit being the one the consumer calls compute. Each row publishes its
 * candidate_topk_blocks best blocks, best first, ties to the lower block id,
 * then -1 when the context has fewer blocks. */
typedef struct smq_source_args {
  uint32_t struct_size;
  int32_t rows;                   /* R >= 0 */
  const uint8_t *q;               /* device [R][H][D] E4M3 */
  const float *q_scale;           /* device [R] */
  const uint16_t *weights;        /* device [R][H] bf16 */
  const uint8_t *k_cache;         /* device [num_pages][page_bytes], 16-byte aligned */
  int64_t num_pages;
  const int32_t *block_table;     /* device [bt_rows][bt_stride] */
  int32_t bt_rows;
  int32_t bt_stride;
  const int32_t *row_indices;     /* device [R] row -> block-table row, or NULL = identity */
  const int32_t *row_ke;          /* device [R] context length; a longer context than max_context
                                     raises SMQ_ERR_BOUNDS and is cut there */
  int32_t max_context;            /* the longest context of the call, 1 .. 1048576 */
  int32_t *candidate_blocks;      /* device [R][candidate_topk_blocks] out */
  float *block_scores;            /* device [R][ceil(max_context / cbs)] out (-inf past a row's
                                     blocks), or NULL */
  void *workspace;                /* device, >= smq_source_workspace_size(plan, R, max_context) */
  size_t workspace_bytes;
} smq_source_args;

/* Workspace bytes of a candidate-source call: the status word, the dense
 * layout of the rows and their fp32 logits [rows][max_context rounded up
 * to whole blocks]. Zero it with smq_workspace_init before the first call.
 * ceil(max_context / cbs) may not exceed 8192. */
SMQ_API int smq_source_workspace_size(const smq_plan *plan, int32_t rows, int32_t max_context, size_t *bytes);

SMQ_API int sparse_mqa_candidate_source_decode(const smq_plan *plan, const smq_source_args *args,
                                               void *stream);

/* Producers of the indexer's inputs. (Source: sparse_mqa_indexer docs,
 * SparseMQAIndexer and weights_dtype: the model writes the MXFP4 indexer K
 * cache, and a fused query kernel writes the FP8 query, its scale and the
 * bf16 weights; sparse_indexer.py, builder __init__: MXFP4 with UE8M0-packed
 * granularity-32 scales.) The pages fix the formats but not the rounding.
 * This library's rounding:
 *  - K, per group of 32 elements: the scale exponent e is the smallest
 *    integer with amax <= 6 * 2^e, stored as the UE8M0 code e + 127 clamped
 *    to [1, 254] (a group of zeros: 127). Each element x * 2^-e rounds to the
 *    nearest E2M1 value, ties to even, saturating at 6.
 *  - Q, per row: scale = amax / 448 (1 for a row of zeros). Each element
 *    x / scale (float division) rounds to the nearest E4M3 value, ties to
 *    even, saturating at 448.
 *  - weights: float to the nearest-even bfloat16.
 * The sign of an element that rounds to zero is kept. Inputs must be finite.
 * RoPE, which the pages' fused query kernel also applies, is not defined on
 * the pages and is not part of this call. */

/* Write ntok keys into the paged K cache (layout at the top of this file).
 *  - k: device [ntok][D] bfloat16 bits, 16-byte aligned.
 *  - slot_mapping: device [ntok] int64. Token t goes to page
 *    slot_mapping[t] / page_size, row slot_mapping[t] % page_size; a negative
 *    slot skips the token.
 *  - k_cache: device [num_pages][page_bytes], 16-byte aligned.
 * A slot past the cache raises SMQ_ERR_BOUNDS in the workspace status word
 * (at least smq_workspace_size(plan, 0) bytes), and that token is skipped.
 * Tokens that share a slot race. ntok may be 0. */
SMQ_API int sparse_mqa_write_k_cache(const smq_plan *plan, const uint16_t *k, const int64_t *slot_mapping,
                                     int64_t ntok, uint8_t *k_cache, int64_t num_pages, void *workspace,
                                     size_t workspace_bytes, void *stream);

/* Quantise `rows` query rows and their head weights.
 *  - q: device [rows][H][D] bfloat16 bits, 16-byte aligned.
 *  - weights: device [rows][H] float.
 *  - q_fp8: device [rows][H][D] E4M3 out, 16-byte aligned. q_scale: device
 *    [rows] float out. weights_bf16: device [rows][H] bfloat16 bits out.
 * These are the q, q_scale and weights of the decode and prefill calls.
 * rows may be 0. */
SMQ_API int sparse_mqa_quantize_q(const smq_plan *plan, const uint16_t *q, const float *weights, int32_t rows,
                                  uint8_t *q_fp8, float *q_scale, uint16_t *weights_bf16, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SMQ_H */
