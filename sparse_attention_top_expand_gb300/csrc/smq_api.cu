// Host side of the C ABI declared in include/smq.h: argument validation, the
// plan, TMA tensor-map encoding and kernel launches. Nothing here allocates
// device memory; every tensor is the caller's.
#include "smq.h"
#include "smq_trace.h"
#include "smq_kernels.cuh"

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

using smq::kHeadDim;
using smq::kTileM;

struct smq_plan {
  smq_plan_desc desc;
  int64_t wait_ns;     // every pipeline wait gives up after this (smq_plan_set_wait_limit)
  int32_t stall_tile;  // failure-path tests: a withheld hand-off (smq_plan_inject_stall), -1: none
  int32_t sbkv;
  int32_t nsb;
  int32_t num_cols;
  int32_t page_bytes;
  int32_t num_sms;
  int32_t n_mma;
  bool prepared;
};

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int pick_sbkv(int page_size, int cbs) {
  for (int s : {128, 64, 32, 16})
    if (page_size % s == 0 && cbs % s == 0) return s;
  return 0;
}

// Q viewed as [rows * H][128] bytes; one box = one row's H heads, padded to the MMA N.
int encode_q(CUtensorMap* m, const uint8_t* q, int64_t qrows, int n_mma) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return SMQ_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(qrows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kHeadDim), static_cast<cuuint32_t>(n_mma)};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(q), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SMQ_OK : SMQ_ERR_CUDA;
}

// Key values as a 3-D tensor [pages][rows][128 FP4 values]: the copy of one
// sub-block unpacks each 16 values (8 bytes) into a 16-byte container, with
// the 128-byte swizzle the MMA descriptors use. The contiguous prefill
// workspace is one page of total_len rows.
int encode_k(CUtensorMap* m, const uint8_t* values, int64_t rows, int64_t page_stride, int64_t pages, int sbkv) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return SMQ_ERR_CUDA;
  if (!aligned(values, 32) || page_stride % 32 != 0 || rows > (int64_t(1) << 31) - 1 || pages > (int64_t(1) << 31) - 1)
    return SMQ_ERR_INVALID_ARG;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(pages)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim / 2), static_cast<cuuint64_t>(page_stride)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kHeadDim), static_cast<cuuint32_t>(sbkv), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<uint8_t*>(values), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SMQ_OK : SMQ_ERR_CUDA;
}

constexpr size_t kStatusBytes = 256;

// Workspace: [status word, 256 B][per-row tile counters, max_rows int32][fp32 logits, rows x num_cols].
size_t counter_bytes(const smq_plan* p) {
  return (static_cast<size_t>(p->desc.max_rows) * sizeof(int32_t) + 255) / 256 * 256;
}

size_t workspace_bytes_for(const smq_plan* p, int64_t rows) {
  return kStatusBytes + counter_bytes(p) + static_cast<size_t>(rows) * p->num_cols * sizeof(float);
}

int check_device(smq_plan* p) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SMQ_ERR_CUDA;
  if (dev != p->desc.device) return SMQ_ERR_INVALID_ARG;
  if (!p->prepared) {
    if (smq::prepare_kernels(p->n_mma) != cudaSuccess || smq::prepare_bm_kernels() != cudaSuccess)
      return SMQ_ERR_CUDA;
    p->prepared = true;
  }
  return SMQ_OK;
}

// Whether the score kernel's shared memory fits the opt-in limit for this many rows.
bool smem_fits(const smq_plan* p, int rows) {
  return smq::score_smem_bytes(p->n_mma, p->desc.num_heads, rows) <= 232448;
}

// Record a caller's profiling event. Inside a stream capture it becomes an
// external event-record node, so that graph replays stamp it.
void record(void* ev, cudaStream_t s) {
  if (!ev) return;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev), s, cudaEventRecordExternal);
  else
    cudaEventRecord(static_cast<cudaEvent_t>(ev), s);
}

// The bf16 logits pointer of an argument struct, or null when the caller's
// struct_size predates the field.
template <typename A>
uint16_t* bf16_logits(const A* a) {
  return a->struct_size >= offsetof(A, logits_out_bf16) + sizeof(a->logits_out_bf16) ? a->logits_out_bf16 : nullptr;
}

// The smallest struct_size accepted: the struct without its last field.
template <typename A>
bool struct_ok(const A* a) {
  return a->struct_size >= offsetof(A, logits_out_bf16);
}

struct CommonRows {
  int32_t rows;
  const uint8_t* q;
  const float* q_scale;
  const uint16_t* weights;
  const int32_t* candidate_blocks;
  int32_t* topk_out;
  int32_t topk_ld;
  int32_t* sparse_indices;
  int32_t* end;
  int32_t expansion_ready;
  int32_t* col_indices;
  float* logits_out;
  void* workspace;
  size_t workspace_bytes;
  uint16_t* logits_out_bf16;
};

int check_common(const smq_plan* p, const CommonRows& a) {
  if (a.rows < 0 || a.rows > p->desc.max_rows) return SMQ_ERR_INVALID_ARG;
  if (a.rows == 0) return SMQ_OK;
  if (!a.q || !a.q_scale || !a.weights || !a.topk_out || !a.sparse_indices || !a.end || !a.workspace)
    return SMQ_ERR_INVALID_ARG;
  if (!a.expansion_ready && !a.candidate_blocks) return SMQ_ERR_INVALID_ARG;
  if (a.topk_ld < p->desc.topk) return SMQ_ERR_INVALID_ARG;
  if (!aligned(a.q, 16) || !aligned(a.weights, 16) || !aligned(a.workspace, 16) || !aligned(a.q_scale, 4) ||
      !aligned(a.topk_out, 4) || !aligned(a.sparse_indices, 4) || !aligned(a.end, 4))
    return SMQ_ERR_INVALID_ARG;
  if (a.logits_out && !aligned(a.logits_out, 4)) return SMQ_ERR_INVALID_ARG;
  if (a.logits_out_bf16 && !aligned(a.logits_out_bf16, 2)) return SMQ_ERR_INVALID_ARG;
  if (a.workspace_bytes < workspace_bytes_for(p, a.rows)) return SMQ_ERR_WORKSPACE_TOO_SMALL;
  return SMQ_OK;
}

smq::ScoreParams score_params(const smq_plan* p, const CommonRows& a) {
  smq::ScoreParams s;
  std::memset(&s, 0, sizeof s);
  s.rows = a.rows;
  s.heads = p->desc.num_heads;
  s.n_mma = p->n_mma;
  s.sbkv = p->sbkv;
  s.subs_per_tile = kTileM / p->sbkv;
  s.nsb = p->nsb;
  s.num_cols = p->num_cols;
  s.tmem_cols = smq::score_tmem_columns(p->n_mma);
  s.q_scale = a.q_scale;
  s.weights = a.weights;
  s.sparse_indices = a.sparse_indices;
  s.end = a.end;
  s.status = static_cast<int32_t*>(a.workspace);
  s.wait_ns = p->wait_ns;
  s.stall_tile = p->stall_tile;
  s.row_done = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(a.workspace) + kStatusBytes);
  s.logits_bf16 = a.logits_out_bf16;
  s.logits = a.logits_out ? a.logits_out
                          : reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + kStatusBytes +
                                                     counter_bytes(p));
  return s;
}

int run_expand(const smq_plan* p, const int32_t* cand, const int32_t* ks, const int32_t* ke, int rows, int32_t* si,
               int32_t* end, cudaStream_t stream) {
  smq::ExpandParams e;
  e.rows = rows;
  e.ncb = p->desc.candidate_topk_blocks;
  e.cbs = p->desc.candidate_block_size;
  e.sbkv = p->sbkv;
  e.nsb = p->nsb;
  e.candidate_blocks = cand;
  e.row_ks = ks;
  e.row_ke = ke;
  e.sparse_indices = si;
  e.end = end;
  return smq::launch_expand(e, stream) == cudaSuccess ? SMQ_OK : SMQ_ERR_CUDA;
}

int run_topk(const smq_plan* p, const CommonRows& a, const smq::ScoreParams& s, cudaStream_t stream) {
  smq::TopkParams t;
  t.rows = a.rows;
  t.num_sms = p->num_sms;
  t.topk = p->desc.topk;
  t.topk_ld = a.topk_ld;
  t.sbkv = p->sbkv;
  t.nsb = p->nsb;
  t.num_cols = p->num_cols;
  t.logits = s.logits;
  t.logits_fill = a.logits_out;
  t.logits_fill_bf16 = a.logits_out_bf16;
  t.sparse_indices = a.sparse_indices;
  t.end = a.end;
  t.topk_out = a.topk_out;
  t.col_indices = a.col_indices;
  return smq::launch_topk(t, stream) == cudaSuccess ? SMQ_OK : SMQ_ERR_CUDA;
}

// CTAs per row of the row-cluster kernel for a decode call of `rows` rows, or
// 0 where it does not apply: more rows than SMs, rows wider than its limit, or
// shared memory that does not fit.
int row_cluster_size(const smq_plan* p, int rows) {
  if (rows <= 0 || rows > p->num_sms || p->num_cols > smq::kRowClusterMaxCols) return 0;
  if (smq::row_cluster_smem_bytes(p->n_mma, p->desc.num_heads, p->nsb, p->num_cols) > 232448) return 0;
  int c = p->num_sms / rows;
  if (c > smq::kRowClusterMaxCtas) c = smq::kRowClusterMaxCtas;
  const int tiles = (p->num_cols + kTileM - 1) / kTileM;
  return c > tiles ? tiles : c;  // a CTA without a tile would only wait
}

// Window-major prefill scratch, after the common part of the workspace:
// per-position window counts and cursors, then per-row record counts, the
// group count, groups and windows per tile of 2048 positions, the (row, window) records,
// the rows' float params and the groups (at most one per record).
struct BmScratch {
  size_t cnt, cursor, nrec, ngroups, tile_groups, tile_windows, rec, rowparams, groups, end;
};

BmScratch bm_scratch(const smq_plan* p, int64_t rows, int64_t total_len) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t records = static_cast<size_t>(rows) * p->nsb;
  BmScratch w;
  w.cnt = up(workspace_bytes_for(p, rows));
  w.cursor = w.cnt + up(static_cast<size_t>(total_len) * 4);
  w.nrec = w.cursor + up(static_cast<size_t>(total_len) * 4);
  w.ngroups = w.nrec + up(static_cast<size_t>(rows) * 4);
  w.tile_groups = w.ngroups + 256;
  w.tile_windows = w.tile_groups + up(static_cast<size_t>((total_len + 2047) / 2048) * 4);
  w.rec = w.tile_windows + up(static_cast<size_t>((total_len + 2047) / 2048) * 4);
  w.rowparams = w.rec + up(records * 8);
  w.groups = w.rowparams + up(static_cast<size_t>(rows) * smq::kBmRowParams * 4);
  w.end = w.groups + up(records * sizeof(smq::BmGroup));
  return w;
}

// The window-major prefill path: 64 heads (two rows per MMA of N = 128) and
// a workspace short enough to count windows per position.
bool bm_applies(const smq_plan* p, int64_t total_len) {
  return p->desc.num_heads == 64 && total_len > 0 && total_len <= smq::kBmMaxTotalLen;
}

int score_grid(const smq_plan* p, int rows) {
  const int64_t max_tiles = static_cast<int64_t>(rows) * ((p->num_cols + kTileM - 1) / kTileM);
  return static_cast<int>(max_tiles < p->num_sms ? max_tiles : p->num_sms);
}

}  // namespace

// Scratch of sparse_mqa_logits_topk_decode_noalloc: a status header, then
// the fp32 logits. Some callers cannot hand the library a workspace: a
// runtime whose device memory all belongs to its own pool and is not lent
// out, or a plugin that may touch only the buffers it was handed. For them
// the scratch is part of the loaded module, one copy on every device the
// library is loaded on. Only the status word and the per-row tile counters
// must start at zero (each call clears them); the score kernel writes every
// logits column it covers before top-k reads it.
static __device__ __align__(256) uint8_t smq_noalloc_scratch[kStatusBytes + SMQ_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch on device `dev`, which must be current. In
// host code the array's name is only a stand-in, so the address comes from
// cudaGetSymbolAddress, once per device.
int noalloc_scratch(int dev, void** out) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return SMQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, smq_noalloc_scratch) != cudaSuccess || !p) return SMQ_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return SMQ_OK;
}

}  // namespace

extern "C" {

SMQ_API const char* smq_error_string(int code) {
  switch (code) {
    case SMQ_OK: return "ok";
    case SMQ_ERR_INVALID_ARG: return "invalid argument";
    case SMQ_ERR_UNSUPPORTED: return "unsupported geometry or device";
    case SMQ_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case SMQ_ERR_CUDA: return "CUDA error";
    case SMQ_ERR_BOUNDS: return "device: index out of range";
    case SMQ_ERR_TIMEOUT: return "device: pipeline wait timed out";
    case SMQ_ERR_BOUNDS | SMQ_ERR_TIMEOUT: return "device: index out of range and pipeline wait timed out";
    default: return "unknown status";
  }
}

SMQ_API int smq_plan_create(const smq_plan_desc* desc, smq_plan** plan) {
  if (!desc || !plan || desc->struct_size < sizeof(smq_plan_desc)) return SMQ_ERR_INVALID_ARG;
  *plan = nullptr;
  const smq_plan_desc& d = *desc;
  if (d.num_heads < 8 || d.num_heads > 128 || d.num_heads % 8 != 0) return SMQ_ERR_UNSUPPORTED;
  if (d.head_dim != kHeadDim) return SMQ_ERR_UNSUPPORTED;
  if (d.page_size <= 0 || d.candidate_block_size <= 0 || d.candidate_topk_blocks <= 0 || d.topk <= 0 ||
      d.max_rows <= 0 || d.device < 0)
    return SMQ_ERR_INVALID_ARG;
  if (d.candidate_topk_blocks > 512 || d.max_rows > smq::kMaxRowsPerCall) return SMQ_ERR_UNSUPPORTED;
  int sbkv = d.sparse_block_kv;
  if (sbkv == 0) sbkv = pick_sbkv(d.page_size, d.candidate_block_size);
  if (sbkv != 16 && sbkv != 32 && sbkv != 64 && sbkv != 128) return SMQ_ERR_UNSUPPORTED;
  // the cache pages must be a multiple of the sub-block, and a candidate block splits into sub-blocks
  if (d.page_size % sbkv != 0 || d.candidate_block_size % sbkv != 0) return SMQ_ERR_INVALID_ARG;
  const int64_t nsb = static_cast<int64_t>(d.candidate_topk_blocks) * (d.candidate_block_size / sbkv);
  const int64_t cols = nsb * sbkv;
  if (cols > smq::kMaxSparseCols) return SMQ_ERR_UNSUPPORTED;
  if (d.topk > cols) return SMQ_ERR_INVALID_ARG;  // the top-k must fit the sparse columns
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || d.device >= count) return SMQ_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d.device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d.device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d.device) != cudaSuccess)
    return SMQ_ERR_CUDA;
  if (major != 10 || minor != 3) return SMQ_ERR_UNSUPPORTED;  // built for sm_103a only
  smq_plan* p = new (std::nothrow) smq_plan;
  if (!p) return SMQ_ERR_INVALID_ARG;
  p->desc = d;
  p->desc.sparse_block_kv = sbkv;
  p->sbkv = sbkv;
  p->nsb = static_cast<int32_t>(nsb);
  p->num_cols = static_cast<int32_t>(cols);
  p->page_bytes = d.page_size * (kHeadDim / 2 + kHeadDim / 32);
  p->num_sms = sms;
  p->n_mma = d.num_heads <= 64 ? 64 : 128;
  p->prepared = false;
  p->wait_ns = 2000000000ll;  // 2 s: far beyond any legitimate wait
  p->stall_tile = -1;
  if (!smem_fits(p, d.max_rows)) {
    delete p;
    return SMQ_ERR_UNSUPPORTED;
  }
  *plan = p;
  return SMQ_OK;
}

SMQ_API int smq_plan_destroy(smq_plan* plan) {
  delete plan;
  return SMQ_OK;
}

SMQ_API int smq_plan_get_info(const smq_plan* plan, smq_plan_info* info) {
  if (!plan || !info || info->struct_size < sizeof(smq_plan_info)) return SMQ_ERR_INVALID_ARG;
  info->sparse_block_kv = plan->sbkv;
  info->num_sparse_blocks = plan->nsb;
  info->num_sparse_cols = plan->num_cols;
  info->page_bytes = plan->page_bytes;
  info->num_sms = plan->num_sms;
  return SMQ_OK;
}

SMQ_API int smq_plan_set_wait_limit(smq_plan* plan, int64_t ns) {
  if (!plan || ns <= 0) return SMQ_ERR_INVALID_ARG;
  plan->wait_ns = ns;
  return SMQ_OK;
}

SMQ_API int smq_plan_inject_stall(smq_plan* plan, int32_t tile) {
  if (!plan || tile < -1) return SMQ_ERR_INVALID_ARG;
  plan->stall_tile = tile;
  return SMQ_OK;
}

SMQ_API int smq_workspace_size(const smq_plan* plan, int32_t rows, size_t* bytes) {
  if (!plan || !bytes || rows < 0 || rows > plan->desc.max_rows) return SMQ_ERR_INVALID_ARG;
  *bytes = workspace_bytes_for(plan, rows);
  return SMQ_OK;
}

SMQ_API int smq_prefill_workspace_size(const smq_plan* plan, int32_t rows, int64_t total_len, size_t* bytes) {
  if (!plan || !bytes || rows < 0 || rows > plan->desc.max_rows || total_len < 0) return SMQ_ERR_INVALID_ARG;
  *bytes = bm_applies(plan, total_len) ? bm_scratch(plan, rows, total_len).end : workspace_bytes_for(plan, rows);
  return SMQ_OK;
}

SMQ_API int smq_workspace_init(const smq_plan* plan, void* workspace, size_t workspace_bytes, void* stream) {
  if (!plan || !workspace || workspace_bytes < kStatusBytes + counter_bytes(plan)) return SMQ_ERR_INVALID_ARG;
  return cudaMemsetAsync(workspace, 0, kStatusBytes + counter_bytes(plan), static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? SMQ_OK
             : SMQ_ERR_CUDA;
}

SMQ_API int smq_get_status(const void* workspace, void* stream, int32_t* code) {
  if (!workspace || !code) return SMQ_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return SMQ_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, workspace, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return SMQ_ERR_CUDA;
  if (cudaMemset(const_cast<void*>(workspace), 0, sizeof v) != cudaSuccess) return SMQ_ERR_CUDA;
  *code = v;
  return SMQ_OK;
}

SMQ_API int sparse_mqa_candidate_expand(const smq_plan* plan, const int32_t* candidate_blocks,
                                        const int32_t* row_ks, const int32_t* row_ke, int32_t rows,
                                        int32_t* sparse_indices, int32_t* end, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  if (!plan || rows < 0 || rows > plan->desc.max_rows) return SMQ_ERR_INVALID_ARG;
  if (rows == 0) return SMQ_OK;
  if (!candidate_blocks || !row_ke || !sparse_indices || !end || !workspace) return SMQ_ERR_INVALID_ARG;
  if (workspace_bytes < kStatusBytes) return SMQ_ERR_WORKSPACE_TOO_SMALL;
  int rc = check_device(const_cast<smq_plan*>(plan));
  if (rc != SMQ_OK) return rc;
  return run_expand(plan, candidate_blocks, row_ks, row_ke, rows, sparse_indices, end,
                    static_cast<cudaStream_t>(stream));
}

SMQ_API int sparse_mqa_logits_topk_decode(const smq_plan* plan, const smq_decode_args* args, void* stream) {
  if (!plan || !args || !struct_ok(args)) return SMQ_ERR_INVALID_ARG;
  const smq_decode_args& a = *args;
  CommonRows c{a.rows, a.q, a.q_scale, a.weights, a.candidate_blocks, a.topk_out, a.topk_ld, a.sparse_indices,
               a.end, a.expansion_ready, a.col_indices, a.logits_out, a.workspace, a.workspace_bytes,
               bf16_logits(args)};
  int rc = check_common(plan, c);
  if (rc != SMQ_OK || a.rows == 0) return rc;
  if (!a.k_cache || !a.block_table || !a.row_ke || a.num_pages <= 0 || a.bt_rows <= 0 || a.bt_stride <= 0)
    return SMQ_ERR_INVALID_ARG;
  if (!aligned(a.k_cache, 16) || !aligned(a.block_table, 4)) return SMQ_ERR_INVALID_ARG;
  rc = check_device(const_cast<smq_plan*>(plan));
  if (rc != SMQ_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!smem_fits(plan, a.rows)) return SMQ_ERR_UNSUPPORTED;
  CUtensorMap tm_q, tm_k;
  rc = encode_q(&tm_q, a.q, static_cast<int64_t>(a.rows) * plan->desc.num_heads, plan->n_mma);
  if (rc != SMQ_OK) return rc;
  // A paged cache is read through registers (coalesced loads two tiles ahead
  // buffer DRAM latency best), unless many rows share each block-table row (a
  // prefill chunk run in place): then the pages are re-read from L2 and
  // unpacking tensor copies are faster. Copies need a 32-byte aligned cache.
  std::memset(&tm_k, 0, sizeof(tm_k));
  bool copy = a.rows >= 8 * a.bt_rows && plan->n_mma == 64 && aligned(a.k_cache, 32);
  // up to 64 candidate blocks per row the score kernel expands the rows itself
  const bool fused = !a.expansion_ready && plan->desc.candidate_topk_blocks <= smq::kMaxFusedBlocks;
  // A narrow batch (no more rows than SMs) takes one cluster of CTAs per row,
  // which keeps the row's logits and top-k on chip.
  const int cluster = row_cluster_size(plan, a.rows);
  if (cluster > 0 && !copy) {
    const size_t smem = smq::row_cluster_smem_bytes(plan->n_mma, plan->desc.num_heads, plan->nsb, plan->num_cols);
    record(a.profile_events[0], s);
    if (!a.expansion_ready && !fused) {
      rc = run_expand(plan, a.candidate_blocks, nullptr, a.row_ke, a.rows, a.sparse_indices, a.end, s);
      if (rc != SMQ_OK) return rc;
    }
    record(a.profile_events[1], s);
    smq::ScoreParams sp = score_params(plan, c);
    sp.fused = fused ? 1 : 0;
    sp.cluster = cluster;
    sp.logits_out = a.logits_out;
    sp.topk = plan->desc.topk;
    sp.topk_ld = a.topk_ld;
    sp.topk_out = a.topk_out;
    sp.col_indices = a.col_indices;
    sp.ncb = plan->desc.candidate_topk_blocks;
    sp.cbs = plan->desc.candidate_block_size;
    sp.candidate_blocks = a.candidate_blocks;
    sp.row_ke = a.row_ke;
    sp.sparse_indices_out = a.sparse_indices;
    sp.end_out = a.end;
    sp.k_cache = a.k_cache;
    sp.num_pages = a.num_pages;
    sp.page_bytes = plan->page_bytes;
    sp.page_size = plan->desc.page_size;
    sp.bt_rows = a.bt_rows;
    sp.bt_stride = a.bt_stride;
    sp.block_table = a.block_table;
    sp.row_indices = a.row_indices;
    if (smq::launch_row_cluster(sp, tm_q, smem, s) != cudaSuccess) return SMQ_ERR_CUDA;
    record(a.profile_events[2], s);
    record(a.profile_events[3], s);
    return SMQ_OK;
  }
  record(a.profile_events[0], s);
  if (!a.expansion_ready && !fused) {
    rc = run_expand(plan, a.candidate_blocks, nullptr, a.row_ke, a.rows, a.sparse_indices, a.end, s);
    if (rc != SMQ_OK) return rc;
  }
  record(a.profile_events[1], s);
  smq::ScoreParams sp = score_params(plan, c);
  sp.fused = fused ? 1 : 0;
  copy = copy && fused &&
         encode_k(&tm_k, a.k_cache, plan->desc.page_size, plan->page_bytes, a.num_pages, plan->sbkv) == SMQ_OK;
  // the score kernel also selects the top-k of the rows it expands when they are narrow enough
  // and few enough that the CTA finishing a row rarely has a second one to select (a wide
  // batch of rows is faster in the separate kernel, one CTA per row over every SM)
  const bool fuse_topk = fused && plan->num_cols <= smq::kFusedTopkCols && 2 * a.rows <= plan->num_sms;
  if (fuse_topk) {
    sp.fused_topk = 1;
    sp.topk = plan->desc.topk;
    sp.topk_ld = a.topk_ld;
    sp.topk_out = a.topk_out;
    sp.col_indices = a.col_indices;
    sp.logits_fill = a.logits_out;
  }
  sp.ncb = plan->desc.candidate_topk_blocks;
  sp.cbs = plan->desc.candidate_block_size;
  sp.candidate_blocks = a.candidate_blocks;
  sp.row_ke = a.row_ke;
  sp.sparse_indices_out = a.sparse_indices;
  sp.end_out = a.end;
  sp.k_cache = a.k_cache;
  sp.num_pages = a.num_pages;
  sp.page_bytes = plan->page_bytes;
  sp.page_size = plan->desc.page_size;
  sp.bt_rows = a.bt_rows;
  sp.bt_stride = a.bt_stride;
  sp.block_table = a.block_table;
  sp.row_indices = a.row_indices;
  const size_t smem = smq::score_smem_bytes(plan->n_mma, plan->desc.num_heads, a.rows);
  if (smq::launch_score(sp, true, copy, tm_q, tm_k, score_grid(plan, a.rows), smem, s) != cudaSuccess) return SMQ_ERR_CUDA;
  record(a.profile_events[2], s);
  if (!fuse_topk) rc = run_topk(plan, c, sp, s);
  record(a.profile_events[3], s);
  return rc;
}

SMQ_API int sparse_mqa_logits_topk_prefill_chunk(const smq_plan* plan, const smq_prefill_args* args,
                                                 void* stream) {
  if (!plan || !args || !struct_ok(args)) return SMQ_ERR_INVALID_ARG;
  const smq_prefill_args& a = *args;
  CommonRows c{a.rows, a.q, a.q_scale, a.weights, a.candidate_blocks, a.topk_out, a.topk_ld, a.sparse_indices,
               a.end, a.expansion_ready, a.col_indices, a.logits_out, a.workspace, a.workspace_bytes,
               bf16_logits(args)};
  int rc = check_common(plan, c);
  if (rc != SMQ_OK || a.rows == 0) return rc;
  if (!a.k_values || !a.k_scales || !a.cu_seqlen_ks || !a.cu_seqlen_ke || a.total_len <= 0 ||
      a.total_len > (int64_t(1) << 31) - 1)
    return SMQ_ERR_INVALID_ARG;
  if (!aligned(a.k_values, 32) || !aligned(a.k_scales, 4)) return SMQ_ERR_INVALID_ARG;
  rc = check_device(const_cast<smq_plan*>(plan));
  if (rc != SMQ_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool window_major =
      bm_applies(plan, a.total_len) && a.workspace_bytes >= bm_scratch(plan, a.rows, a.total_len).end;
  if (!window_major && !smem_fits(plan, a.rows)) return SMQ_ERR_UNSUPPORTED;
  CUtensorMap tm_q, tm_k;
  rc = encode_q(&tm_q, a.q, static_cast<int64_t>(a.rows) * plan->desc.num_heads, plan->n_mma);
  if (rc != SMQ_OK) return rc;
  // key tiles: 128-row windows (window-major) or one sub-block per copy
  rc = encode_k(&tm_k, a.k_values, a.total_len, a.total_len * (kHeadDim / 2), 1, window_major ? 128 : plan->sbkv);
  if (rc != SMQ_OK) return rc;
  record(a.profile_events[0], s);
  if (!a.expansion_ready) {
    rc = run_expand(plan, a.candidate_blocks, a.cu_seqlen_ks, a.cu_seqlen_ke, a.rows, a.sparse_indices, a.end, s);
    if (rc != SMQ_OK) return rc;
  }
  smq::ScoreParams sp = score_params(plan, c);
  sp.row_ks = a.cu_seqlen_ks;
  sp.k_values = a.k_values;
  sp.k_scales = a.k_scales;
  sp.total_len = a.total_len;
  if (window_major) {
    // the (row, window) index, then the score per window
    const BmScratch w = bm_scratch(plan, a.rows, a.total_len);
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    smq::BmIndexParams ip;
    ip.rows = a.rows;
    ip.nsb = plan->nsb;
    ip.sbkv = plan->sbkv;
    ip.num_cols = plan->num_cols;
    ip.total_len = a.total_len;
    ip.sparse_indices = a.sparse_indices;
    ip.end = a.end;
    ip.row_ks = a.cu_seqlen_ks;
    ip.weights = a.weights;
    ip.q_scale = a.q_scale;
    ip.rec = reinterpret_cast<int2*>(ws + w.rec);
    ip.nrec = reinterpret_cast<int32_t*>(ws + w.nrec);
    ip.cnt = reinterpret_cast<int32_t*>(ws + w.cnt);
    ip.cursor = reinterpret_cast<int32_t*>(ws + w.cursor);
    ip.rowparams = reinterpret_cast<float*>(ws + w.rowparams);
    ip.groups = reinterpret_cast<smq::BmGroup*>(ws + w.groups);
    ip.ngroups = reinterpret_cast<int32_t*>(ws + w.ngroups);
    ip.tile_groups = reinterpret_cast<int32_t*>(ws + w.tile_groups);
    ip.tile_windows = reinterpret_cast<int32_t*>(ws + w.tile_windows);
    ip.status = sp.status;
    if (smq::launch_bm_index(ip, s) != cudaSuccess) return SMQ_ERR_CUDA;
    record(a.profile_events[1], s);
    smq::BmScoreParams bp;
    bp.groups = ip.groups;
    bp.ngroups = ip.ngroups;
    bp.rowparams = ip.rowparams;
    bp.k_scales = a.k_scales;
    bp.total_len = a.total_len;
    bp.num_cols = plan->num_cols;
    bp.sbkv = plan->sbkv;
    bp.logits = sp.logits;
    bp.logits_bf16 = a.logits_out_bf16;
    bp.status = sp.status;
    bp.wait_ns = static_cast<uint64_t>(plan->wait_ns);
    bp.stall_group = plan->stall_tile;
    if (smq::launch_bm_score(bp, tm_q, tm_k, plan->num_sms, s) != cudaSuccess) return SMQ_ERR_CUDA;
    record(a.profile_events[2], s);
    rc = run_topk(plan, c, sp, s);
    record(a.profile_events[3], s);
    return rc;
  }
  record(a.profile_events[1], s);
  const size_t smem = smq::score_smem_bytes(plan->n_mma, plan->desc.num_heads, a.rows);
  if (smq::launch_score(sp, false, true, tm_q, tm_k, score_grid(plan, a.rows), smem, s) != cudaSuccess) return SMQ_ERR_CUDA;
  record(a.profile_events[2], s);
  rc = run_topk(plan, c, sp, s);
  record(a.profile_events[3], s);
  return rc;
}

SMQ_API int sparse_mqa_gather_k(const smq_plan* plan, const uint8_t* k_cache, int64_t num_pages,
                                const int32_t* block_table, int32_t bt_stride, const int32_t* cu_seq_lens,
                                int32_t num_seqs, int64_t total_len, uint8_t* k_values, uint8_t* k_scales,
                                void* workspace, size_t workspace_bytes, void* stream) {
  if (!plan || num_seqs < 0 || total_len < 0) return SMQ_ERR_INVALID_ARG;
  if (num_seqs == 0 || total_len == 0) return SMQ_OK;
  if (!k_cache || !block_table || !cu_seq_lens || !k_values || !k_scales || !workspace || num_pages <= 0 ||
      bt_stride <= 0)
    return SMQ_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(k_values, 16) || !aligned(k_scales, 4)) return SMQ_ERR_INVALID_ARG;
  if (workspace_bytes < kStatusBytes) return SMQ_ERR_WORKSPACE_TOO_SMALL;
  int rc = check_device(const_cast<smq_plan*>(plan));
  if (rc != SMQ_OK) return rc;
  smq::GatherParams g;
  g.num_seqs = num_seqs;
  g.page_size = plan->desc.page_size;
  g.bt_stride = bt_stride;
  g.total_len = total_len;
  g.num_pages = num_pages;
  g.page_bytes = plan->page_bytes;
  g.k_cache = k_cache;
  g.block_table = block_table;
  g.cu_seq_lens = cu_seq_lens;
  g.k_values = k_values;
  g.k_scales = k_scales;
  g.status = static_cast<int32_t*>(workspace);
  return smq::launch_gather(g, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SMQ_OK : SMQ_ERR_CUDA;
}

SMQ_API int sparse_mqa_logits_topk_decode_noalloc(const smq_plan* plan, const smq_decode_args* args,
                                                  void* stream) {
  if (!plan || !args || !struct_ok(args)) return SMQ_ERR_INVALID_ARG;
  if (args->workspace || args->workspace_bytes) return SMQ_ERR_INVALID_ARG;  // the library's scratch replaces it
  if (args->rows < 0 || args->rows > plan->desc.max_rows) return SMQ_ERR_INVALID_ARG;
  if (workspace_bytes_for(plan, args->rows) > kStatusBytes + SMQ_NOALLOC_SCRATCH_BYTES)
    return SMQ_ERR_WORKSPACE_TOO_SMALL;
  if (args->rows == 0) return SMQ_OK;
  int rc = check_device(const_cast<smq_plan*>(plan));  // the plan's device is current
  if (rc != SMQ_OK) return rc;
  void* scratch = nullptr;
  rc = noalloc_scratch(plan->desc.device, &scratch);
  if (rc != SMQ_OK) return rc;
  // the kernels OR device-detected errors into the status word and count finished
  // tiles per row: start both at zero (a call that gave up may have left counts)
  if (cudaMemsetAsync(scratch, 0, kStatusBytes + counter_bytes(plan), static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return SMQ_ERR_CUDA;
  smq_decode_args a;  // the caller's fields (as many as its struct_size holds), then the scratch
  std::memset(&a, 0, sizeof a);
  std::memcpy(&a, args, args->struct_size < sizeof a ? args->struct_size : sizeof a);
  a.struct_size = sizeof a;
  a.workspace = scratch;
  a.workspace_bytes = kStatusBytes + SMQ_NOALLOC_SCRATCH_BYTES;
  return sparse_mqa_logits_topk_decode(plan, &a, stream);
}

namespace {

// The candidate source's dense layout: whole blocks covering max_context.
struct SourceLayout {
  int32_t num_cols, nsb, max_blocks;
  size_t si_off, end_off, logits_off, total;
};

bool source_layout(const smq_plan* p, int64_t rows, int64_t max_context, SourceLayout* out) {
  if (max_context <= 0 || max_context > (int64_t(1) << 20) || rows < 0) return false;
  const int64_t cbs = p->desc.candidate_block_size;
  const int64_t blocks = (max_context + cbs - 1) / cbs;
  if (blocks > smq::kSourceMaxBlocks) return false;
  out->max_blocks = static_cast<int32_t>(blocks);
  out->num_cols = static_cast<int32_t>(blocks * cbs);
  out->nsb = out->num_cols / p->sbkv;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  out->si_off = kStatusBytes + counter_bytes(p);
  out->end_off = out->si_off + up(static_cast<size_t>(rows) * out->nsb * 4);
  out->logits_off = out->end_off + up(static_cast<size_t>(rows) * 4);
  out->total = out->logits_off + static_cast<size_t>(rows) * out->num_cols * 4;
  return true;
}

}  // namespace

SMQ_API int smq_source_workspace_size(const smq_plan* plan, int32_t rows, int32_t max_context, size_t* bytes) {
  if (!plan || !bytes || rows < 0 || rows > plan->desc.max_rows) return SMQ_ERR_INVALID_ARG;
  SourceLayout l;
  if (!source_layout(plan, rows, max_context, &l)) return SMQ_ERR_UNSUPPORTED;
  *bytes = l.total;
  return SMQ_OK;
}

SMQ_API int sparse_mqa_candidate_source_decode(const smq_plan* plan, const smq_source_args* args, void* stream) {
  if (!plan || !args || args->struct_size < sizeof(smq_source_args)) return SMQ_ERR_INVALID_ARG;
  const smq_source_args& a = *args;
  if (a.rows < 0 || a.rows > plan->desc.max_rows) return SMQ_ERR_INVALID_ARG;
  if (a.rows == 0) return SMQ_OK;
  SourceLayout l;
  if (!source_layout(plan, a.rows, a.max_context, &l)) return SMQ_ERR_UNSUPPORTED;
  if (!a.q || !a.q_scale || !a.weights || !a.k_cache || !a.block_table || !a.row_ke || !a.candidate_blocks ||
      !a.workspace || a.num_pages <= 0 || a.bt_rows <= 0 || a.bt_stride <= 0)
    return SMQ_ERR_INVALID_ARG;
  if (!aligned(a.q, 16) || !aligned(a.weights, 16) || !aligned(a.k_cache, 16) || !aligned(a.workspace, 16) ||
      !aligned(a.q_scale, 4) || !aligned(a.block_table, 4) || !aligned(a.candidate_blocks, 4) ||
      (a.block_scores && !aligned(a.block_scores, 4)))
    return SMQ_ERR_INVALID_ARG;
  if (a.workspace_bytes < l.total) return SMQ_ERR_WORKSPACE_TOO_SMALL;
  int rc = check_device(const_cast<smq_plan*>(plan));
  if (rc != SMQ_OK) return rc;
  if (!smem_fits(plan, a.rows)) return SMQ_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  smq::SourceParams sp;
  std::memset(&sp, 0, sizeof sp);
  sp.rows = a.rows;
  sp.sbkv = plan->sbkv;
  sp.nsb = l.nsb;
  sp.num_cols = l.num_cols;
  sp.cbs = plan->desc.candidate_block_size;
  sp.ncb = plan->desc.candidate_topk_blocks;
  sp.max_blocks = l.max_blocks;
  sp.row_ke = a.row_ke;
  sp.sparse_indices = reinterpret_cast<int32_t*>(ws + l.si_off);
  sp.end = reinterpret_cast<int32_t*>(ws + l.end_off);
  sp.logits = reinterpret_cast<float*>(ws + l.logits_off);
  sp.candidate_blocks = a.candidate_blocks;
  sp.block_scores = a.block_scores;
  sp.status = static_cast<int32_t*>(a.workspace);
  if (smq::launch_source_layout(sp, s) != cudaSuccess) return SMQ_ERR_CUDA;
  // the dense rows through the score kernel, its sub-blocks read from the layout
  CUtensorMap tm_q, tm_k;
  std::memset(&tm_k, 0, sizeof tm_k);
  rc = encode_q(&tm_q, a.q, static_cast<int64_t>(a.rows) * plan->desc.num_heads, plan->n_mma);
  if (rc != SMQ_OK) return rc;
  smq::ScoreParams p;
  std::memset(&p, 0, sizeof p);
  p.rows = a.rows;
  p.heads = plan->desc.num_heads;
  p.n_mma = plan->n_mma;
  p.sbkv = plan->sbkv;
  p.subs_per_tile = kTileM / plan->sbkv;
  p.nsb = l.nsb;
  p.num_cols = l.num_cols;
  p.tmem_cols = smq::score_tmem_columns(plan->n_mma);
  p.q_scale = a.q_scale;
  p.weights = a.weights;
  p.sparse_indices = sp.sparse_indices;
  p.end = sp.end;
  p.k_cache = a.k_cache;
  p.num_pages = a.num_pages;
  p.page_bytes = plan->page_bytes;
  p.page_size = plan->desc.page_size;
  p.bt_rows = a.bt_rows;
  p.bt_stride = a.bt_stride;
  p.block_table = a.block_table;
  p.row_indices = a.row_indices;
  p.logits = const_cast<float*>(sp.logits);
  p.status = sp.status;
  p.row_done = reinterpret_cast<int32_t*>(ws + kStatusBytes);
  p.wait_ns = plan->wait_ns;
  p.stall_tile = plan->stall_tile;
  const int64_t tiles = static_cast<int64_t>(a.rows) * ((l.num_cols + kTileM - 1) / kTileM);
  const int grid = static_cast<int>(tiles < plan->num_sms ? tiles : plan->num_sms);
  const size_t smem = smq::score_smem_bytes(plan->n_mma, plan->desc.num_heads, a.rows);
  if (smq::launch_score(p, true, false, tm_q, tm_k, grid, smem, s) != cudaSuccess) return SMQ_ERR_CUDA;
  return smq::launch_source_select(sp, s) == cudaSuccess ? SMQ_OK : SMQ_ERR_CUDA;
}

SMQ_API int sparse_mqa_write_k_cache(const smq_plan* plan, const uint16_t* k, const int64_t* slot_mapping,
                                     int64_t ntok, uint8_t* k_cache, int64_t num_pages, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  if (!plan || ntok < 0) return SMQ_ERR_INVALID_ARG;
  if (ntok == 0) return SMQ_OK;
  if (!k || !slot_mapping || !k_cache || !workspace || num_pages <= 0) return SMQ_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(slot_mapping, 8) || !aligned(k_cache, 16) || !aligned(workspace, 16))
    return SMQ_ERR_INVALID_ARG;
  if (workspace_bytes < kStatusBytes) return SMQ_ERR_WORKSPACE_TOO_SMALL;
  int rc = check_device(const_cast<smq_plan*>(plan));
  if (rc != SMQ_OK) return rc;
  smq::KWriteParams w;
  w.k = k;
  w.slot_mapping = slot_mapping;
  w.ntok = ntok;
  w.page_size = plan->desc.page_size;
  w.num_pages = num_pages;
  w.page_bytes = plan->page_bytes;
  w.k_cache = k_cache;
  w.status = static_cast<int32_t*>(workspace);
  return smq::launch_write_k_cache(w, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SMQ_OK : SMQ_ERR_CUDA;
}

SMQ_API int sparse_mqa_quantize_q(const smq_plan* plan, const uint16_t* q, const float* weights, int32_t rows,
                                  uint8_t* q_fp8, float* q_scale, uint16_t* weights_bf16, void* stream) {
  if (!plan || rows < 0) return SMQ_ERR_INVALID_ARG;
  if (rows == 0) return SMQ_OK;
  if (!q || !weights || !q_fp8 || !q_scale || !weights_bf16) return SMQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(q_fp8, 16) || !aligned(weights, 4) || !aligned(q_scale, 4) ||
      !aligned(weights_bf16, 2))
    return SMQ_ERR_INVALID_ARG;
  int rc = check_device(const_cast<smq_plan*>(plan));
  if (rc != SMQ_OK) return rc;
  smq::QQuantParams p;
  p.q = q;
  p.weights_in = weights;
  p.rows = rows;
  p.heads = plan->desc.num_heads;
  p.q_fp8 = q_fp8;
  p.q_scale = q_scale;
  p.weights_out = weights_bf16;
  return smq::launch_quantize_q(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SMQ_OK : SMQ_ERR_CUDA;
}

#ifdef SMQ_TRACE
SMQ_API int smq_trace_read(uint64_t* host, size_t count) {
  if (!host) return SMQ_ERR_INVALID_ARG;
  return smq::trace_read(host, count) == cudaSuccess ? SMQ_OK : SMQ_ERR_CUDA;
}

SMQ_API int smq_trace_clear(void) { return smq::trace_clear() == cudaSuccess ? SMQ_OK : SMQ_ERR_CUDA; }
#endif

}  // extern "C"
