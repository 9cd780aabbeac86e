// Kernel parameter blocks and launchers shared by the C ABI (smq_api.cu) and
// the kernels (smq_kernels.cu). Internal to the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace smq {

constexpr int kHeadDim = 128;       // D
constexpr int kMmaM = 128;          // key positions per MMA (its M)
constexpr int kTileM = 256;         // key positions per pipeline stage: two MMA halves
constexpr int kHalves = kTileM / kMmaM;
constexpr int kMaxSubsPerTile = kTileM / 16;  // sparse sub-blocks per stage (they hold at least 16 positions)
constexpr int kRowBytes = 128;      // smem bytes per K row (padded FP4) and per Q row (E4M3)
constexpr int kScaleWordBytes = 4;  // D/32 UE8M0 bytes per key position
constexpr int kScoreThreads = 384;  // scheduler, 2 MMA, 4 epilogue, 4 loader and 1 query-loader warps
constexpr int kQueryWarp = 10;
constexpr int kMmaWarp1 = 11;       // second MMA issuer (odd tiles); warp 1 issues the even tiles
constexpr int kEpilogueThreads = 128;
constexpr int kLoaderThreads = 128;
constexpr int kLoadAhead = 2;       // tiles each register-path loader thread keeps in flight
constexpr int kScoreStages = 4;     // key stages resident in shared memory (32 KB each)
constexpr int kMaxAccBuffers = 3;
constexpr int kDescRing = 16;       // tiles whose source addresses may be published ahead of the loaders
constexpr int kMaxFusedBlocks = 64; // candidate blocks per row the score kernel expands itself

// TMEM accumulators in flight between the MMA and the epilogue, each two
// halves of n_mma fp32 columns: 3 for 64-wide heads, 1 for 128. With more
// than one the two MMA threads take alternate stages. A parity wait on an
// accumulator cannot pass a phase early: issuing stage it needs stage it to
// be full, hence the epilogue past stage it - kScoreStages, hence (it works
// in order) done reading stage it - 2 NA as long as kScoreStages < 2 NA. With
// one accumulator a single thread issues every stage.
__host__ __device__ constexpr int acc_buffers(int n_mma) { return n_mma <= 64 ? 3 : 1; }

static_assert(kScoreStages < 2 * acc_buffers(64), "accumulator parity waits need kScoreStages < 2 NA");

// TMEM columns per CTA: accumulators, then 4 scale columns per stage half, then 4 for the query scales.
__host__ __device__ constexpr int score_tmem_columns(int n_mma) {
  return acc_buffers(n_mma) * kHalves * n_mma + 4 * kHalves * kScoreStages + 4 <= 256 ? 256 : 512;
}
constexpr int kFusedTopkCols = kScoreThreads * 22;  // widest row the score kernel selects itself
constexpr int kExpandWarps = 8;
constexpr int kMaxRowsPerCall = 8192;
constexpr int kMaxSparseCols = 16384;
constexpr int kStatusBounds = 8;    // SMQ_ERR_BOUNDS
constexpr int kStatusTimeout = 16;  // SMQ_ERR_TIMEOUT

// Tracing build (-DSMQ_TRACE, a separate library; see include/smq_trace.h):
// the score kernel stamps %globaltimer at its phase boundaries into a device
// array of kTraceSlots stamps per CTA. In the product build every mark
// compiles to nothing.
#ifdef SMQ_TRACE
constexpr int kTraceSlots = 32;
constexpr int kTraceCtas = 1024;
cudaError_t trace_read(uint64_t* host, size_t count);
cudaError_t trace_clear();
#define SMQ_MARK(slot) ::smq::trace_mark(slot)
#else
#define SMQ_MARK(slot) ((void)0)
#endif

// Everything the fused gather + score kernel reads besides its tensor maps.
struct ScoreParams {
  int32_t rows;
  int32_t heads;          // H
  int32_t n_mma;          // MMA N: H rounded up to 64 or 128
  int32_t sbkv;           // tokens per sparse sub-block
  int32_t subs_per_tile;  // kTileM / sbkv
  int32_t nsb;            // sparse sub-blocks per row
  int32_t num_cols;       // S = nsb * sbkv
  int32_t tmem_cols;      // TMEM columns allocated per CTA
  const float* q_scale;
  const uint16_t* weights;
  const int32_t* sparse_indices;
  const int32_t* end;
  // paged cache (decode)
  const uint8_t* k_cache;
  int64_t num_pages;
  int64_t page_bytes;
  int32_t page_size;
  int32_t bt_rows;
  int32_t bt_stride;
  const int32_t* block_table;
  const int32_t* row_indices;  // may be null (identity)
  // contiguous workspace (prefill)
  const int32_t* row_ks;
  const uint8_t* k_values;
  const uint8_t* k_scales;
  int64_t total_len;
  // in-kernel candidate expansion (paged decode, at most kMaxFusedBlocks candidate blocks):
  // tiles are spread over rows by an upper bound from row_ke alone, ceil(min(row_ke, num_cols) / kTileM),
  // and each CTA expands its own rows, writing sparse_indices_out / end_out
  int32_t fused;
  int32_t ncb;            // candidate blocks per row
  int32_t cbs;            // candidate block size
  const int32_t* candidate_blocks;
  const int32_t* row_ke;
  int32_t* sparse_indices_out;
  int32_t* end_out;
  // top-k selected in the score kernel (rows expanded here, num_cols <= kFusedTopkCols): the CTA
  // that finishes a row's last tile, counted in row_done, selects that row after its pipeline
  int32_t fused_topk;
  int32_t topk;
  int32_t topk_ld;
  int32_t* row_done;     // [rows] finished tiles per row; zero before a call, left zero after it
  int32_t* topk_out;     // [rows][topk_ld]
  int32_t* col_indices;  // [rows][topk], may be null
  float* logits_fill;    // when non-null: -inf into columns >= end (the caller's logits_out)
  // row-cluster kernel: CTAs per row (the cluster size); logits_out, or null
  int32_t cluster;
  float* logits_out;
  uint16_t* logits_bf16;  // when non-null: the logits rounded to bf16, -inf past end (the caller's logits_out_bf16)
  // outputs
  float* logits;     // [rows][num_cols]
  int32_t* status;   // workspace status word
  // failure path: every wait gives up after wait_ns; with stall_tile >= 0 the
  // loaders of CTA 0 withhold the hand-off of that tile (counted in CTA 0) to
  // the MMA, whose wait then runs out (tests of the failure path only)
  int64_t wait_ns;
  int32_t stall_tile;
};

struct TopkParams {
  int32_t rows;
  int32_t num_sms;  // CTAs of the warp-per-row kernel: at most one per SM
  int32_t topk;
  int32_t topk_ld;
  int32_t sbkv;
  int32_t nsb;
  int32_t num_cols;
  const float* logits;
  float* logits_fill;  // when non-null: write -inf to columns >= end (the caller's logits_out)
  uint16_t* logits_fill_bf16;  // the same for the caller's bf16 logits
  const int32_t* sparse_indices;
  const int32_t* end;
  int32_t* topk_out;
  int32_t* col_indices;  // may be null
};

struct ExpandParams {
  int32_t rows;
  int32_t ncb;
  int32_t cbs;
  int32_t sbkv;
  int32_t nsb;
  const int32_t* candidate_blocks;
  const int32_t* row_ks;  // may be null
  const int32_t* row_ke;
  int32_t* sparse_indices;
  int32_t* end;
};

struct GatherParams {
  int32_t num_seqs;
  int32_t page_size;
  int32_t bt_stride;
  int64_t total_len;
  int64_t num_pages;
  int64_t page_bytes;
  const uint8_t* k_cache;
  const int32_t* block_table;
  const int32_t* cu_seq_lens;
  uint8_t* k_values;
  uint8_t* k_scales;
  int32_t* status;
};

// The MXFP4 K-cache writer: bf16 keys [ntok][128] to slots of the paged cache.
struct KWriteParams {
  const uint16_t* k;
  const int64_t* slot_mapping;  // [ntok] page * page_size + offset; negative: skipped
  int64_t ntok;
  int32_t page_size;
  int64_t num_pages;
  int64_t page_bytes;
  uint8_t* k_cache;
  int32_t* status;  // SMQ_ERR_BOUNDS for a slot past the cache
};

// The query quantiser: bf16 rows [rows][heads][128] to E4M3 and a float
// scale per row; float weights [rows][heads] to bf16.
struct QQuantParams {
  const uint16_t* q;
  const float* weights_in;
  int64_t rows;
  int32_t heads;
  uint8_t* q_fp8;
  float* q_scale;
  uint16_t* weights_out;
};

// The candidate source: every position of a row as a sparse column, then
// each block's maximum logit and the row's best blocks.
struct SourceParams {
  int32_t rows;
  int32_t sbkv;
  int32_t nsb;          // sub-blocks per row of the dense layout
  int32_t num_cols;     // nsb * sbkv
  int32_t cbs;
  int32_t ncb;          // blocks published per row
  int32_t max_blocks;   // num_cols / cbs
  const int32_t* row_ke;
  int32_t* sparse_indices;  // [rows][nsb] the dense layout: sub-block j, or -1 past the row
  int32_t* end;             // [rows]
  const float* logits;      // [rows][num_cols]
  int32_t* candidate_blocks;  // [rows][ncb]
  float* block_scores;        // [rows][max_blocks], may be null
  int32_t* status;
};

constexpr int kSourceMaxBlocks = 8192;  // blocks per row the selection sorts in shared memory
cudaError_t launch_source_layout(const SourceParams& p, cudaStream_t stream);
cudaError_t launch_source_select(const SourceParams& p, cudaStream_t stream);

cudaError_t launch_write_k_cache(const KWriteParams& p, cudaStream_t stream);
cudaError_t launch_quantize_q(const QQuantParams& p, cudaStream_t stream);

// Shared-memory bytes of the score kernel for a geometry.
size_t score_smem_bytes(int n_mma, int heads, int rows);

// The row-cluster decode kernel: one cluster of at most kRowClusterMaxCtas
// CTAs per row, for rows of at most kRowClusterMaxCols sparse columns. Its
// shared-memory bytes:
constexpr int kRowClusterMaxCols = 8192;
constexpr int kRowClusterMaxCtas = 8;
size_t row_cluster_smem_bytes(int n_mma, int heads, int nsb, int num_cols);

cudaError_t launch_expand(const ExpandParams& p, cudaStream_t stream);
cudaError_t launch_score(const ScoreParams& p, bool paged, bool copy, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                         int grid, size_t smem, cudaStream_t stream);  // paged with p.fused: rows expanded in the kernel
cudaError_t launch_row_cluster(const ScoreParams& p, const CUtensorMap& tm_q, size_t smem,
                               cudaStream_t stream);  // grid = rows x p.cluster
cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream);
cudaError_t launch_gather(const GatherParams& p, cudaStream_t stream);
cudaError_t prepare_kernels(int n_mma);  // raise the dynamic-smem limits once per device

// ---------------------------------------------------------------------------
// Window-major prefill (smq_prefill.cu). Rows of a chunk select the same key
// windows many times over, so the score runs per 128-key window of the
// contiguous workspace: the window's keys stay in shared memory while the
// query tiles of the rows that selected it stream past, two rows per MMA
// (N = 128). A window is the 128 positions from P = ks + 128 u (u >= 0) of a
// row's own coordinates, so a sub-block never straddles two windows.
//
// A record is one (row, window) pair: a run of consecutive entries of the
// row's sparse list inside one window with ascending slots (slot = offset in
// the window / sbkv). It holds P and the column of its first entry c0, with
// the slot mask in the top byte (c0m = c0 | mask << 24); the column of key m
// of the window (slot s = m / sbkv, present when mask bit s is set) is
// c0 + popc(mask & ((1 << s) - 1)) * sbkv + m % sbkv.
// A group is two records of the same window (row[1] = -1 when the window's
// record count is odd); groups are numbered window by window.
constexpr int kBmThreads = 896;           // window loader, 3 MMA issuers, 6 x 4 epilogue warps
constexpr int kBmStages = 9;              // query stages of two rows (16 KB each), 3 per MMA issuer
constexpr int kBmRowParams = 68;          // floats per row: 64 head weights, q_scale, 3 pad
constexpr int64_t kBmMaxTotalLen = 1 << 20;  // windows are counted per workspace position

struct BmGroup {
  int32_t P;        // first workspace position of the window
  int32_t row[2];   // row of each column half; row[1] = -1 for a lone record
  int32_t wo;       // window ordinal: the nonempty windows at lower positions
  int32_t c0m[2];   // column of the record's first entry | slot mask << 24
  int32_t end[2];   // the row's valid column count
};
static_assert(sizeof(BmGroup) == 32, "one group descriptor is 32 bytes (a bulk copy unit)");

struct BmIndexParams {
  int rows;
  int nsb;
  int sbkv;
  int num_cols;  // S
  int64_t total_len;
  const int32_t* sparse_indices;  // [rows][nsb]
  const int32_t* end;             // [rows]
  const int32_t* row_ks;          // [rows]
  const uint16_t* weights;        // [rows][64] bf16
  const float* q_scale;           // [rows]
  int2* rec;                      // [rows][nsb] (P, c0m)
  int32_t* nrec;                  // [rows]
  int32_t* cnt;                   // [total_len], zero on entry
  int32_t* cursor;                // [total_len]
  float* rowparams;               // [rows][kBmRowParams]
  BmGroup* groups;                // [rows * nsb]
  int32_t* ngroups;               // [1]
  int32_t* tile_groups;           // [ceil(total_len / 2048)] groups per tile of positions
  int32_t* tile_windows;          // [ceil(total_len / 2048)] nonempty windows per tile
  int32_t* status;
};

struct BmScoreParams {
  const BmGroup* groups;
  const int32_t* ngroups;
  const float* rowparams;
  const uint8_t* k_scales;  // [total_len][4]
  int64_t total_len;
  int num_cols;
  int sbkv;
  float* logits;            // [rows][S]
  uint16_t* logits_bf16;    // optional copy
  int32_t* status;
  uint64_t wait_ns;
  int32_t stall_group;      // failure-path tests: CTA 0 withholds this group's stage, -1: none
};

size_t bm_score_smem_bytes();
cudaError_t launch_bm_index(const BmIndexParams& p, cudaStream_t stream);  // zeroes cnt, then 4 kernels
cudaError_t launch_bm_score(const BmScoreParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kw, int grid,
                            cudaStream_t stream);
cudaError_t prepare_bm_kernels();

}  // namespace smq
