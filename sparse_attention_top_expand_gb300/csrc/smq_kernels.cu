// GB300 (sm_103a) kernels of the candidate-block sparse MQA-logits indexer.
//
//   expand_kernel  candidate blocks -> sorted, deduplicated sparse sub-blocks
//                  (sparse_indices, end), one warp per row
//   score_kernel   fused K gather + block-scaled tcgen05 MMA + epilogue:
//                  logit[c] = q_scale * sum_h w[h] * max(0, sum_d K[c,d] Q[h,d])
//                  for every valid sparse column c, written to an fp32 row
//   topk_kernel    radix select of the k largest logits per row, ids mapped
//                  back to token positions, -1 padded
//   gather_kernel  paged MXFP4 cache -> contiguous (values, scales) workspace
//
// The score kernel is a persistent, warp-specialised pipeline with one CTA
// per SM. A tile (stage) is 256 positions, two MMA halves of 128.
//  - warp 0 (scheduler): it resolves each tile's sub-blocks to source
//    addresses (sparse id, block-table page, bounds) and publishes them into a
//    ring. For decode rows with at most 64 candidate blocks it first expands
//    the row itself.
//  - warp 10 (query loader): when the row changes it TMA-loads the row's Q
//    tile (E4M3, 128-byte swizzle) and bf16 head weights.
//  - warps 6..9 (loaders): paged caches go through registers (512-byte
//    coalesced warp loads two tiles ahead, then stores into the padded 16-byte
//    containers that kind::mxf8f6f4 reads for E2M1: 8 data bytes per 16
//    elements, 128-byte swizzle). The contiguous prefill workspace goes through
//    tensor copies that unpack into those containers themselves. Thread m
//    writes the scale words of key rows m and m + 128 into the stage's
//    512-byte scale blocks.
//  - warps 1 and 11 (MMA, alternate tiles): one thread copies a half's scale
//    block to TMEM (tcgen05.cp; row m of A reads lane m, column base + m/32,
//    byte = scale id) and issues 4 x tcgen05.mma kind::mxf8f6f4 with UE8M0
//    block scales, M = 128 positions, N = heads, K = 32 each. The fp32
//    accumulators live in TMEM, three in flight.
//  - warps 2..5 (epilogue): one TMEM lane (= one position) per thread; they
//    reduce over heads with ReLU and the weights. For narrow decode batches
//    the CTA that completes a row then selects its top-k.
// Every wait is bounded. A wait that gives up sets SMQ_ERR_TIMEOUT in the
// status word and the CTA winds down. Out-of-range page / row / block ids set
// SMQ_ERR_BOUNDS, and the load is skipped.
#include "smq_kernels.cuh"
#include "smq_ptx.cuh"

#include <cfloat>
#include <cuda_bf16.h>

namespace smq {

namespace {

constexpr uint32_t kFullMask = 0xffffffffu;
constexpr uint32_t kE2M1 = 5, kE4M3 = 0;
constexpr int32_t kRowDone = 0x40000000;  // flag on a row's end: this CTA selects the row's top-k

__host__ __device__ constexpr uint32_t round_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// One sub-block of a tile as the scheduler warp publishes it to the loaders.
struct SubBlockSrc {
  const uint8_t* values;  // FP4 values of its first position (64 B per position)
  const uint8_t* scales;  // UE8M0 word of its first position (4 B per position)
  int32_t row, page;      // the values' tensor-copy coordinates (row in the page, page)
  int32_t positions;      // positions that may be read; 0: nothing is loaded
  int32_t pad;
};

// Byte offsets inside the score kernel's dynamic shared memory (base aligned to 1024).
struct ScoreLayout {
  uint32_t kv, q, sf, desc, w, w_stride, meta, bars, misc, scan, sched, prefix, rend, total;
  __host__ __device__ ScoreLayout(int n_mma, int heads, int rows) {
    uint32_t o = 0;
    kv = o;  // [stages][256 rows][128 B] padded FP4 keys, 128-byte swizzle (two 128-row MMA halves)
    o += static_cast<uint32_t>(kScoreStages) * kTileM * kRowBytes;
    q = o;  // [2][n_mma rows][128 B] E4M3 queries, 128-byte swizzle
    o += 2u * static_cast<uint32_t>(n_mma) * kRowBytes;
    sf = o;  // [stages][halves][32 rows][16 B] key scale words, copied to TMEM by the MMA thread; then one block of 2^0
    o += static_cast<uint32_t>(kScoreStages * kHalves + 1) * 512u;
    desc = o;  // [ring][8 sub-blocks] source addresses published by the scheduler warp
    o += static_cast<uint32_t>(kDescRing) * kMaxSubsPerTile * sizeof(SubBlockSrc);
    w_stride = round_up(static_cast<uint32_t>(heads) * 2u, 16);
    w = o;  // [2][heads] bf16 weights
    o += 2u * w_stride;
    meta = o;  // [2] {row, end, q_scale, unused}
    o += 2u * 16u;
    bars = o;  // full, empty [stages]; acc_full, acc_empty [accumulators]; q_full, q_empty [2]; drain [2]; (then, below)
               // desc_full, desc_empty [ring]; setup copy; row stored
    o += round_up((2u * kScoreStages + 2u * kMaxAccBuffers + 6u + 2u * kDescRing + 2u + kScoreStages) * 8u, 16);
    misc = o;  // tmem base, abort flag
    o += 16u;
    scan = o;  // per-warp partial sums of the prologue scan
    o += 64u;
    sched = o;  // the scheduler's sorted candidate blocks of its current row
    o += kMaxFusedBlocks * 4u;
    prefix = o;  // [rows + 1] exclusive prefix of tiles per row
    o += round_up((static_cast<uint32_t>(rows) + 1u) * 4u, 16);
    rend = o;  // [rows] the end of each row this CTA expands, by local row index
    o += round_up(static_cast<uint32_t>(rows) * 4u, 16);
    total = o;
  }
};

struct RowMeta {
  int32_t row;
  int32_t end;
  float q_scale;
  int32_t pad;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Row owning flat tile t: the last r with prefix[r] <= t (prefix[rows] > t).
__device__ __forceinline__ int find_row(const int32_t* prefix, int rows, int64_t t) {
  int lo = 0, hi = rows;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

__device__ __forceinline__ void set_status(int32_t* status, int code) { atomicOr(status, code); }

// float to the nearest-even bfloat16 bits
__device__ __forceinline__ uint16_t to_bf16(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
constexpr uint16_t kBf16NegInf = 0xFF80;

}  // namespace

#ifdef SMQ_TRACE
__device__ uint64_t g_trace[kTraceCtas * kTraceSlots];

__device__ __forceinline__ void trace_mark(int slot) {
  if (blockIdx.x < kTraceCtas) g_trace[blockIdx.x * kTraceSlots + slot] = global_ns();
}

cudaError_t trace_read(uint64_t* host, size_t count) {
  if (count > sizeof(g_trace) / sizeof(uint64_t)) count = sizeof(g_trace) / sizeof(uint64_t);
  return cudaMemcpyFromSymbol(host, g_trace, count * sizeof(uint64_t));
}

cudaError_t trace_clear() {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_trace);
  return e == cudaSuccess ? cudaMemset(p, 0, sizeof(g_trace)) : e;
}
#endif


size_t score_smem_bytes(int n_mma, int heads, int rows) {
  return ScoreLayout(n_mma, heads, rows).total + 1024;
}

__device__ int expand_row_in_warp(int ncb, int64_t cbs, int64_t L, int c0, int c1, int32_t* sorted, int* nkept_out,
                                   int lane);

// ===========================================================================
// Candidate expansion: one warp per row.
// ===========================================================================
__global__ void __launch_bounds__(kExpandWarps * 32) expand_kernel(const __grid_constant__ ExpandParams p) {
  extern __shared__ int32_t expand_smem[];
  griddep_launch_dependents();
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kExpandWarps + warp;
  if (r >= p.rows) return;
  int32_t* cand = expand_smem + warp * 2 * p.ncb;
  int32_t* kept = cand + p.ncb;
  const int64_t ks = p.row_ks ? p.row_ks[r] : 0;
  int64_t L = static_cast<int64_t>(p.row_ke[r]) - ks;
  if (L < 0) L = 0;
  const int spb = p.cbs / p.sbkv;
  int32_t* si = p.sparse_indices + static_cast<int64_t>(r) * p.nsb;
  if (p.ncb <= kMaxFusedBlocks) {  // one or two ids per lane: the warp's sorting network
    const int32_t* cbr = p.candidate_blocks + static_cast<int64_t>(r) * p.ncb;
    const int c0 = lane < p.ncb ? cbr[lane] : -1, c1 = lane + 32 < p.ncb ? cbr[lane + 32] : -1;
    int nkept = 0;
    const int cols = expand_row_in_warp(p.ncb, p.cbs, L, c0, c1, cand, &nkept, lane);
    for (int slot = lane; slot < p.nsb; slot += 32) {
      const int k = slot / spb;
      int v = -1;
      if (k < nkept) {
        const int sub = cand[k] * spb + slot % spb;
        if (static_cast<int64_t>(sub) * p.sbkv < L) v = sub;
      }
      si[slot] = v;
    }
    if (lane == 0) p.end[r] = cols;
    return;
  }
  for (int i = lane; i < p.ncb; i += 32) cand[i] = p.candidate_blocks[static_cast<int64_t>(r) * p.ncb + i];
  __syncwarp();
  // keep a block if it is in range and its first occurrence; others -> INT_MAX
  // (branch-free scans: every lane reads the same cand[j], a broadcast)
  for (int i = lane; i < p.ncb; i += 32) {
    const int32_t b = cand[i];
    bool dup = false;
    for (int j = 0; j < p.ncb; ++j) dup |= (j < i) & (cand[j] == b);
    const bool keep = b >= 0 && static_cast<int64_t>(b) * p.cbs < L && !dup;
    kept[i] = keep ? b : INT_MAX;
  }
  __syncwarp();
  int64_t cols = 0;
  int nkept = 0;
  for (int i = lane; i < p.ncb; i += 32) {
    const int32_t b = kept[i];
    if (b == INT_MAX) continue;
    int rank = 0;
    for (int j = 0; j < p.ncb; ++j) rank += kept[j] < b;
    ++nkept;
    for (int u = 0; u < spb; ++u) {
      const int64_t sub = static_cast<int64_t>(b) * spb + u;
      const int64_t start = sub * p.sbkv;
      const int slot = rank * spb + u;
      if (start < L) {
        si[slot] = static_cast<int32_t>(sub);
        cols += (L - start < p.sbkv) ? (L - start) : p.sbkv;
      } else {
        si[slot] = -1;
      }
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    nkept += __shfl_xor_sync(kFullMask, nkept, o);
    cols += __shfl_xor_sync(kFullMask, cols, o);
  }
  for (int slot = nkept * spb + lane; slot < p.nsb; slot += 32) si[slot] = -1;
  if (lane == 0) p.end[r] = static_cast<int32_t>(cols);
}

// ===========================================================================
// Fused gather + score.
// ===========================================================================
// Global -> shared loads on the LSU path (the key rows of a tile come from
// scattered pages; many independent 16-byte loads keep far more bytes in
// flight per SM than the tensor-copy engine did for 64-byte rows).
// The same loads under a predicate (no branch): where pred is false nothing
// is read and v keeps its value.
__device__ __forceinline__ void ldg_stream_v4_if(uint4& v, const void* p, bool pred) {
  asm volatile(
      "{\n .reg .pred q;\n setp.ne.b32 q, %5, 0;\n @q ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];\n}"
      : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
      : "l"(p), "r"(pred ? 1 : 0));
}

__device__ __forceinline__ void ldg_stream_u32_if(uint32_t& v, const void* p, bool pred) {
  asm volatile("{\n .reg .pred q;\n setp.ne.b32 q, %2, 0;\n @q ld.global.nc.L1::no_allocate.u32 %0, [%1];\n}"
               : "+r"(v)
               : "l"(p), "r"(pred ? 1 : 0));
}

__device__ __forceinline__ void sts_u32(uint32_t addr, uint32_t a) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(a) : "memory");
}

__device__ __forceinline__ void sts_v2(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

// The address ring is shared between warps that hand entries back and forth
// through mbarriers. Writes are volatile shared stores. Reads are plain loads
// between the reader's mbarrier wait and its hand-back arrival: both are
// compiler memory barriers, so no read moves out of that window, and the
// compiler is free to merge and schedule the reads inside it.
__device__ __forceinline__ void put_src(SubBlockSrc* e, const uint8_t* values, const uint8_t* scales, int row, int page,
                                        int positions) {
  const uint32_t a = smem_addr(e);
  asm volatile("st.volatile.shared.v2.u64 [%0], {%1, %2};" ::"r"(a), "l"(values), "l"(scales) : "memory");
  asm volatile("st.volatile.shared.v2.s32 [%0], {%1, %2};" ::"r"(a + 16), "r"(row), "r"(page) : "memory");
  asm volatile("st.volatile.shared.s32 [%0], %1;" ::"r"(a + 24), "r"(positions) : "memory");
}

__device__ __forceinline__ SubBlockSrc get_src(const SubBlockSrc* e) {
  return *e;
}

__device__ __forceinline__ void st_volatile_s32(int32_t* a, int32_t v) {
  asm volatile("st.volatile.shared.s32 [%0], %1;" ::"r"(smem_addr(a)), "r"(v) : "memory");
}

__device__ __forceinline__ int32_t ld_volatile_s32(const int32_t* a) {
  int32_t v;
  asm volatile("ld.volatile.shared.s32 %0, [%1];" : "=r"(v) : "r"(smem_addr(a)) : "memory");
  return v;
}

// Loads one word and drops it. Issued early for buffers that are written
// much later, so that their address translation is cached by then (a cold
// miss stalls the stores that hit it for microseconds).
__device__ __forceinline__ void touch_global(const void* p) {
  asm volatile("{\n .reg .b32 t;\n ld.global.cg.b32 t, [%0];\n}" ::"l"(p));
}

// Adds with release and acquire semantics at GPU scope: this thread's
// earlier writes (and those it acquired) are visible before the add, and
// writes released by the adds it observes are visible after it.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Candidate expansion of row r by one warp, for at most 64 candidate blocks
// (the same result as expand_kernel): a block is kept if it lies in [0, L)
// and no earlier candidate has the same id; the kept blocks are sorted into
// sorted[0 .. *nkept_out). Returns the row's column count.
__device__ int expand_row_in_warp(int ncb, int64_t cbs, int64_t L, int c0, int c1, int32_t* sorted, int* nkept_out,
                                   int lane);

__device__ int expand_row_in_warp(const ScoreParams& p, int r, int64_t L, int32_t* sorted, int* nkept_out, int lane) {
  const int32_t* cb = p.candidate_blocks + static_cast<int64_t>(r) * p.ncb;
  return expand_row_in_warp(p.ncb, p.cbs, L, lane < p.ncb ? cb[lane] : -1, lane + 32 < p.ncb ? cb[lane + 32] : -1,
                            sorted, nkept_out, lane);
}

// The same with the row's candidates already loaded: lane l holds ids l (c0)
// and l + 32 (c1), -1 past the row's ncb.
// The ids that are in range go through a bitonic sorting network across the
// warp (one id per lane, or two for more than 32 candidates; out-of-range ids
// sort last as INT_MAX). A sorted id equal to its predecessor is a repeat and is
// dropped; the rest land in `sorted` at their rank, counted by ballots. Block b
// holds min(cbs, L - b cbs) columns below L.
__device__ int expand_row_in_warp(int ncb, int64_t cbs, int64_t L, int c0, int c1, int32_t* sorted, int* nkept_out,
                                   int lane) {
  auto key = [&](int b, bool live) { return live && b >= 0 && static_cast<int64_t>(b) * cbs < L ? b : INT_MAX; };
  auto block_cols = [&](int b, bool keep) {
    const int64_t rest = keep ? L - static_cast<int64_t>(b) * cbs : 0;
    return static_cast<int>(rest < cbs ? rest : cbs);
  };
  int v0 = key(c0, lane < ncb);
  int v1 = key(c1, lane + 32 < ncb);
  const uint32_t lt = (1u << lane) - 1u;
  if (ncb <= 32) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1) {
        const int o = __shfl_xor_sync(kFullMask, v0, j);
        v0 = (((lane & k) == 0) == ((lane & j) == 0)) ? min(v0, o) : max(v0, o);
      }
    const int prev = __shfl_up_sync(kFullMask, v0, 1);
    const bool keep = v0 != INT_MAX && (lane == 0 || prev != v0);
    const uint32_t bal = __ballot_sync(kFullMask, keep);
    if (keep) sorted[__popc(bal & lt)] = v0;
    const int cols = __reduce_add_sync(kFullMask, block_cols(v0, keep));
    __syncwarp();
    *nkept_out = __popc(bal);
    return cols;
  }
  // 64 entries: entry i is (lane i % 32, register i / 32)
#pragma unroll
  for (int k = 2; k <= 64; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j == 32) {  // partners in the same lane
        const int a = min(v0, v1), b = max(v0, v1);
        v0 = a;
        v1 = b;
      } else {
        const int o0 = __shfl_xor_sync(kFullMask, v0, j);
        const int o1 = __shfl_xor_sync(kFullMask, v1, j);
        const bool lower = (lane & j) == 0;
        const bool up0 = k == 64 || (lane & k) == 0;
        const bool up1 = k == 64 || (k < 32 && (lane & k) == 0);
        v0 = (up0 == lower) ? min(v0, o0) : max(v0, o0);
        v1 = (up1 == lower) ? min(v1, o1) : max(v1, o1);
      }
    }
  const int p0 = __shfl_up_sync(kFullMask, v0, 1);
  const int p1 = __shfl_up_sync(kFullMask, v1, 1);
  const int last0 = __shfl_sync(kFullMask, v0, 31);
  const bool keep0 = v0 != INT_MAX && (lane == 0 || p0 != v0);
  const bool keep1 = v1 != INT_MAX && (lane == 0 ? last0 != v1 : p1 != v1);
  const uint32_t b0 = __ballot_sync(kFullMask, keep0), b1 = __ballot_sync(kFullMask, keep1);
  if (keep0) sorted[__popc(b0 & lt)] = v0;
  if (keep1) sorted[__popc(b0) + __popc(b1 & lt)] = v1;
  const int cols = __reduce_add_sync(kFullMask, block_cols(v0, keep0) + block_cols(v1, keep1));
  __syncwarp();
  *nkept_out = __popc(b0) + __popc(b1);
  return cols;
}

// The expansion of row r (sorted[0 .. nkept), `cols` columns below L) to
// global memory: sparse_indices and end. The fence makes them visible to the
// CTA that selects the row's top-k.
__device__ void write_row_expansion(const ScoreParams& p, int r, int64_t L, const int32_t* sorted, int nkept,
                                    int cols, int lane) {
  const int sbkv = p.sbkv, spb = p.cbs / p.sbkv;
  int32_t* si = p.sparse_indices_out + static_cast<int64_t>(r) * p.nsb;
  for (int slot = lane; slot < p.nsb; slot += 32) {
    const int k = slot / spb;
    int v = -1;
    if (k < nkept) {
      const int sub = sorted[k] * spb + slot % spb;
      if (static_cast<int64_t>(sub) * sbkv < L) v = sub;
    }
    si[slot] = v;
  }
  if (lane == 0) p.end_out[r] = cols;
  __threadfence();
}

// ---------------------------------------------------------------------------
// Top-k selection of one row by one CTA (used by topk_kernel and by the score
// kernel for the rows it completes).
// ---------------------------------------------------------------------------
// Thread t holds the keys of columns t, t + T, t + 2T, ... in registers (T
// threads). Digit passes (most significant first) count the keys that still
// match the selected prefix; the bin holding the k-th largest key is found by
// a descending scan. Two schemes:
//  - 12, 12 and 8 bits in a 4096-bin histogram, thread t scanning a run of
//    consecutive bins and clearing them once read. Logits spread over the top
//    12 bits (sign, exponent, three mantissa bits), so a warp's increments
//    rarely meet in one bin, and two passes usually suffice (the score
//    kernel's own selection).
//  - four 8-bit passes over 256 bins with one copy per lane, which needs fewer
//    registers (the separate kernel, where occupancy matters).
// The passes stop once every key of the selected bin is taken.
// Then every key above the selected prefix, and the first `need` keys inside
// it in column order, are written by one ordered compaction: a single scan
// over the per-32-column counts gives each warp its output offsets.
__device__ __forceinline__ uint32_t ordered_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kTopkBins = 4096;

// Shared memory of one row's selection.
struct TopkScratch {
  uint32_t* hist;    // [kTopkBins] (12-bit digits) or [256 * 32] (8-bit digits, a copy per lane), 16-byte aligned
  int* bsum;         // [256] (8-bit digits)
  int* wsum;         // [threads / 32]
  uint32_t* chunk;   // [threads / 32 * kJ]
  int32_t* sidx;     // [nsb]
  int* sel;          // [12]
};

// Top-k of one row by the whole CTA. L: the row's S logits; end_src: where
// the row's end is read (after the key loads are issued); sparse_row: the
// row's sparse sub-block ids. Logits and ids may have been written by other
// CTAs of the same kernel, so they are read from L2.
// kShared: L and the ids (sm.sidx, sparse_row unused) are already in this
// CTA's shared memory.
// Value-range first pass (kRange): one block reduction gives the row's
// minimum and maximum, a 1024-bin histogram over that value range (a
// monotone map, so every key in a higher bin is strictly greater) finds the
// bin holding the k-th key, and one warp sorts that bin's keys (at most
// kRangeBin; key descending, column ascending) to give the exact threshold
// key and how many keys equal to it are taken. A row whose bin holds more
// keys (ties, spikes) falls back to the digit passes on the same registers.
constexpr int kRangeBins = 1024;
constexpr int kRangeBin = 64;

template <int kThreads, int kJ, bool kWide, bool kShared = false, bool kRange = false>
__device__ void select_topk(const float* L, int S, const int32_t* end_src, int k, const int32_t* sparse_row, int nsb,
                            int sbkv, int32_t* out, int32_t* colo, float* fill, uint16_t* fill16,
                            const TopkScratch& sm) {
  constexpr int kWarps = kThreads / 32;
  constexpr int kChunks = kWarps * kJ;  // 32-column chunks of the row, chunk j * kWarps + warp
  constexpr int kPerThread = (kTopkBins + kThreads - 1) / kThreads;  // bins a thread scans
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* hist = sm.hist;
  int* sel_bin = sm.sel;
  int* sel_above = sm.sel + 4;
  int* sel_cnt = sm.sel + 8;
  // the logits row has S columns whatever `end` is: load every key at once
  float raw[kJ];
#pragma unroll
  for (int j = 0; j < kJ; ++j) {
    const int c = tid + j * kThreads;
    raw[j] = c < S ? (kShared ? L[c] : __ldcg(L + c)) : 0.f;
  }
  int e = *end_src;
  e = e < 0 ? 0 : (e > S ? S : e);
  if constexpr (!kShared)
    for (int i = tid; i < nsb; i += kThreads) sm.sidx[i] = __ldcg(sparse_row + i);
  uint4* hist4 = reinterpret_cast<uint4*>(hist);
  for (int i = tid; i < (kWide ? kTopkBins : 256 * 32) / 4; i += kThreads) hist4[i] = make_uint4(0, 0, 0, 0);
  if (fill)
    for (int c = e + tid; c < S; c += kThreads) fill[c] = -INFINITY;
  if (fill16)
    for (int c = e + tid; c < S; c += kThreads) fill16[c] = kBf16NegInf;
  const int32_t* sidx = sm.sidx;
  const int sb_shift = 31 - __clz(sbkv);  // the sub-block size is a power of two (16..128)
  auto token = [&](int c) { return (sidx[c >> sb_shift] << sb_shift) | (c & (sbkv - 1)); };
  __syncthreads();
  if (kShared && tid == 0) SMQ_MARK(23);
  if (e <= k) {
    for (int c = tid; c < k; c += kThreads) {
      out[c] = c < e ? token(c) : -1;
      if (colo) colo[c] = c < e ? c : -1;
    }
    return;
  }
  uint32_t key[kJ];
#pragma unroll
  for (int j = 0; j < kJ; ++j) key[j] = tid + j * kThreads < e ? ordered_key(raw[j]) : 0u;
  uint32_t prefix = 0;  // selected high bits so far
  int need = k;         // keys still to take among those matching the prefix
  int done_bits = 0;
  bool ranged = false;  // the value-range pass found the threshold
  if constexpr (kRange) {
    // -- minimum and maximum of the valid keys
    float vmin = INFINITY, vmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < kJ; ++j)
      if (tid + j * kThreads < e) {
        vmin = fminf(vmin, raw[j]);
        vmax = fmaxf(vmax, raw[j]);
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      vmin = fminf(vmin, __shfl_xor_sync(kFullMask, vmin, o));
      vmax = fmaxf(vmax, __shfl_xor_sync(kFullMask, vmax, o));
    }
    float* red = reinterpret_cast<float*>(hist + kRangeBins + 2 * kRangeBin + 8);  // [2 * kWarps]
    if (lane == 0) {
      red[warp] = vmin;
      red[kWarps + warp] = vmax;
    }
    __syncthreads();
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) {
      vmin = fminf(vmin, red[w2]);
      vmax = fmaxf(vmax, red[kWarps + w2]);
    }
    if (!(vmax > vmin) || !(vmax - vmin < INFINITY)) {
      // every valid key equal (take the first k), or a range too wide for the map: the digit passes decide
      if (vmin == vmax) {
        prefix = ordered_key(vmin);
        done_bits = 32;
        ranged = true;
      }
    } else {
      const float scale = static_cast<float>(kRangeBins) / (vmax - vmin);
      auto bin_of = [&](float x) { return static_cast<int>(fminf((x - vmin) * scale, kRangeBins - 1.f)); };
#pragma unroll
      for (int j = 0; j < kJ; ++j)
        if (tid + j * kThreads < e) atomicAdd(&hist[bin_of(raw[j])], 1u);
      __syncthreads();
      // descending scan: thread t owns bins kRangeBins - 1 - per t - b for b < per
      constexpr int per = (kRangeBins + kThreads - 1) / kThreads;
      int cnt[per];
      int local = 0;
#pragma unroll
      for (int b = 0; b < per; ++b) {
        const int bin = kRangeBins - 1 - per * tid - b;
        cnt[b] = bin >= 0 ? static_cast<int>(hist[bin]) : 0;
        local += cnt[b];
      }
      int incl = local;
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl += v;
      }
      if (lane == 31) sm.wsum[warp] = incl;
      __syncthreads();
      int cum = incl - local;
#pragma unroll
      for (int w2 = 0; w2 < kWarps; ++w2) cum += w2 < warp ? sm.wsum[w2] : 0;
#pragma unroll
      for (int b = 0; b < per; ++b) {
        if (cnt[b] > 0 && cum < need && need <= cum + cnt[b]) {
          sel_bin[0] = kRangeBins - 1 - per * tid - b;
          sel_above[0] = cum;
          sel_cnt[0] = cnt[b];
        }
        cum += cnt[b];
      }
      uint32_t* list = hist + kRangeBins;  // [kRangeBin] (key, column) of the threshold bin
      int* list_n = reinterpret_cast<int*>(hist + kRangeBins + 2 * kRangeBin);
      if (tid == 0) *list_n = 0;
      __syncthreads();
      const int tb = sel_bin[0], tcount = sel_cnt[0], above = sel_above[0];
      if (tcount <= kRangeBin) {
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
          const int c = tid + j * kThreads;
          if (c < e && bin_of(raw[j]) == tb) {
            const int at = atomicAdd(list_n, 1);
            list[2 * at] = ordered_key(raw[j]);
            list[2 * at + 1] = static_cast<uint32_t>(c);
          }
        }
        __syncthreads();
        if (warp == 0) {
          // bitonic sort of kRangeBin = 64 composites (key, ~column), descending:
          // lane l holds elements l and l + 32
          uint64_t x[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int i = lane + 32 * h;
            x[h] = i < tcount ? (static_cast<uint64_t>(list[2 * i]) << 32) | (0xFFFFFFFFu - list[2 * i + 1]) : 0ull;
          }
#pragma unroll
          for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int i = lane + 32 * h;
                const bool desc = (i & size) == 0;  // this element's block sorts descending
                if (stride == 32) {
                  if (h == 0) {  // the pair (i, i + 32) sits in this lane
                    const bool swap = desc ? (x[0] < x[1]) : (x[0] > x[1]);
                    if (swap) {
                      const uint64_t tmp = x[0];
                      x[0] = x[1];
                      x[1] = tmp;
                    }
                  }
                } else {
                  const uint64_t y = __shfl_xor_sync(kFullMask, x[h], stride);
                  const bool lower = (i & stride) == 0;
                  const bool take_max = lower == desc;
                  x[h] = take_max ? (x[h] > y ? x[h] : y) : (x[h] < y ? x[h] : y);
                }
              }
            }
          }
          // the (need - above)-th largest is the threshold; how many equal keys are taken
          const int want = need - above;  // 1 .. tcount
          const int src = want - 1;
          const uint64_t tsel = __shfl_sync(kFullMask, x[src >> 5], src & 31);
          const uint32_t tkey = static_cast<uint32_t>(tsel >> 32);
          int eq = 0;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int i = lane + 32 * h;
            eq += (i < want && static_cast<uint32_t>(x[h] >> 32) == tkey) ? 1 : 0;
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) eq += __shfl_xor_sync(kFullMask, eq, o);
          if (lane == 0) {
            sel_bin[1] = static_cast<int>(tkey);
            sel_cnt[1] = eq;
          }
        }
        __syncthreads();
        prefix = static_cast<uint32_t>(sel_bin[1]);
        need = sel_cnt[1];
        done_bits = 32;
        ranged = true;
      }
    }
    if (!ranged) {  // back to the digit passes: clear what the range pass used
      __syncthreads();
      for (int i = tid; i < (kWide ? kTopkBins : 256 * 32) / 4; i += kThreads) hist4[i] = make_uint4(0, 0, 0, 0);
      __syncthreads();
    }
  }
  if (ranged) {
    // the threshold is known: straight to the compaction
  } else if constexpr (kWide) {
  for (int pass = 0; pass < 3; ++pass) {
    const int wbits = pass < 2 ? 12 : 8;
    const int nb = 1 << wbits;
    const int shift = 32 - done_bits - wbits;
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int c = tid + j * kThreads;
      const bool match = c < e && (done_bits == 0 || (key[j] >> (32 - done_bits)) == prefix);
      if (match) atomicAdd(&hist[(key[j] >> shift) & (nb - 1)], 1u);
    }
    __syncthreads();
    // descending scan: thread t owns bins nb - 1 - per t - b for b < per
    const int per = (nb + kThreads - 1) / kThreads;
    int cnt[kPerThread];
    int local = 0;
#pragma unroll
    for (int b = 0; b < kPerThread; ++b) {
      const int bin = nb - 1 - per * tid - b;
      cnt[b] = 0;
      if (b < per && bin >= 0) {
        cnt[b] = static_cast<int>(hist[bin]);
        hist[bin] = 0;  // read once, cleared for the next pass
      }
      local += cnt[b];
    }
    int incl = local;
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) sm.wsum[warp] = incl;
    __syncthreads();
    int cum = incl - local;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) cum += w2 < warp ? sm.wsum[w2] : 0;  // independent loads
#pragma unroll
    for (int b = 0; b < kPerThread; ++b) {
      if (cnt[b] > 0 && cum < need && need <= cum + cnt[b]) {
        sel_bin[pass] = nb - 1 - per * tid - b;
        sel_above[pass] = cum;
        sel_cnt[pass] = cnt[b];
      }
      cum += cnt[b];
    }
    __syncthreads();
    prefix = (prefix << wbits) | static_cast<uint32_t>(sel_bin[pass]);
    need -= sel_above[pass];
    done_bits += wbits;
    if (kShared && tid == 0) SMQ_MARK(24 + pass);
    if (need == sel_cnt[pass]) break;  // the whole bin is taken
  }
  } else {
  // four 8-bit passes over a 256-bin histogram with one copy per lane (bin b,
  // copy l at word 32 b + l, bank l): a warp's increments never meet
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - done_bits;
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int c = tid + j * kThreads;
      const bool match = c < e && (done_bits == 0 || (key[j] >> (32 - done_bits)) == prefix);
      if (match) atomicAdd(&hist[((key[j] >> shift) & 255) * 32 + lane], 1u);
    }
    __syncthreads();
    for (int b = tid; b < 256; b += kThreads) {  // bin totals, copies read in a rotated order
      int sum = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) sum += static_cast<int>(hist[b * 32 + ((i + b) & 31)]);
      sm.bsum[b] = sum;
    }
    __syncthreads();
    int cnt = 0, incl = 0;  // descending scan: thread t < 256 owns bin 255 - t
    if (tid < 256) {
      cnt = sm.bsum[255 - tid];
      incl = cnt;
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl += v;
      }
      if (lane == 31) sm.wsum[warp] = incl;
    }
    for (int i = tid; i < 256 * 8; i += kThreads) hist4[i] = make_uint4(0, 0, 0, 0);  // read: clear for the next pass
    __syncthreads();
    if (tid < 256) {
      int cum = incl - cnt;
#pragma unroll
      for (int w2 = 0; w2 < 8; ++w2) cum += w2 < warp ? sm.wsum[w2] : 0;
      if (cnt > 0 && cum < need && need <= cum + cnt) {
        sel_bin[pass] = 255 - tid;
        sel_above[pass] = cum;
        sel_cnt[pass] = cnt;
      }
    }
    __syncthreads();
    prefix = (prefix << 8) | static_cast<uint32_t>(sel_bin[pass]);
    need -= sel_above[pass];
    done_bits += 8;
    if (need == sel_cnt[pass]) break;  // the whole bin is taken
  }
  }
  // selected: keys whose top done_bits bits are above the prefix, and the
  // first `need` of those equal to it, in column order
  const uint32_t mask = ~0u << (32 - done_bits);
  const uint32_t pfx = prefix << (32 - done_bits);
  const int need_eq = need;
  uint32_t bg[kJ], be[kJ];
#pragma unroll
  for (int j = 0; j < kJ; ++j) {
    const int c = tid + j * kThreads;
    bg[j] = __ballot_sync(kFullMask, c < e && (key[j] & mask) > pfx);
    be[j] = __ballot_sync(kFullMask, c < e && (key[j] & mask) == pfx);
    if (lane == 0) sm.chunk[j * kWarps + warp] = (static_cast<uint32_t>(__popc(bg[j])) << 16) | __popc(be[j]);
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the packed counts (each half stays below 2^16)
    constexpr int kPer = (kChunks + 31) / 32;
    uint32_t v[kPer];
    uint32_t sum = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int c = lane * kPer + i;
      v[i] = c < kChunks ? sm.chunk[c] : 0u;
      sum += v[i];
    }
    uint32_t inc = sum;
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(kFullMask, inc, o);
      if (lane >= o) inc += t;
    }
    uint32_t run = inc - sum;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int c = lane * kPer + i;
      if (c < kChunks) sm.chunk[c] = run;
      run += v[i];
    }
  }
  __syncthreads();
  if (kShared && tid == 0) SMQ_MARK(27);
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < kJ; ++j) {
    const uint32_t pre = sm.chunk[j * kWarps + warp];
    const int c = tid + j * kThreads;
    const bool gt = (bg[j] >> lane) & 1u, eq = (be[j] >> lane) & 1u;
    const int pg = static_cast<int>(pre >> 16) + __popc(bg[j] & lt);
    const int pe = static_cast<int>(pre & 0xffffu) + __popc(be[j] & lt);
    int slot = -1;
    if (gt) slot = pg + min(pe, need_eq);
    else if (eq && pe < need_eq) slot = pg + pe;
    if (slot >= 0 && slot < k) {
      out[slot] = token(c);
      if (colo) colo[slot] = c;
    }
  }
}

// kCopy: key values by tensor copies (the contiguous workspace always; a paged
// cache whose pages many rows re-read from L2) rather than through registers.
template <bool kPaged, int kN, bool kFused, bool kCopy = !kPaged>
__global__ void __launch_bounds__(kScoreThreads, 1)
    score_kernel(const __grid_constant__ ScoreParams p, const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_k) {
  extern __shared__ uint8_t score_smem_raw[];
  uint8_t* smem = align1024(score_smem_raw);
  const ScoreLayout lay(kN, p.heads, p.rows);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int NS = kScoreStages;
  const int S = p.num_cols;
  const int R = p.rows;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
  auto bar_full = [&](int s) { return smem_addr(&bars[s]); };
  auto bar_empty = [&](int s) { return smem_addr(&bars[NS + s]); };
  constexpr int NA = acc_buffers(kN);
  constexpr int NB = 2 * NS + 2 * kMaxAccBuffers;
  auto bar_acc_full = [&](int a) { return smem_addr(&bars[2 * NS + a]); };
  auto bar_acc_empty = [&](int a) { return smem_addr(&bars[2 * NS + kMaxAccBuffers + a]); };
  auto bar_q_full = [&](int b) { return smem_addr(&bars[NB + b]); };
  auto bar_q_empty = [&](int b) { return smem_addr(&bars[NB + 2 + b]); };
  const uint32_t bar_drain = smem_addr(&bars[NB + 4]);
  auto bar_desc_full = [&](int d) { return smem_addr(&bars[NB + 6 + d]); };
  auto bar_desc_empty = [&](int d) { return smem_addr(&bars[NB + 6 + kDescRing + d]); };
  const uint32_t bar_setup = smem_addr(&bars[NB + 6 + 2 * kDescRing]);
  const uint32_t bar_row_stored = smem_addr(&bars[NB + 7 + 2 * kDescRing]);  // epilogue warps, per row end
  // tensor-copy path: the value copies of a stage complete here (the `full`
  // barrier then counts the loader warps' scale words only)
  auto bar_copy = [&](int st) { return smem_addr(&bars[NB + 8 + 2 * kDescRing + st]); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + lay.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + lay.misc + 4);
  int32_t* scan = reinterpret_cast<int32_t*>(smem + lay.scan);
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + lay.prefix);
  RowMeta* meta = reinterpret_cast<RowMeta*>(smem + lay.meta);
  SubBlockSrc* desc = reinterpret_cast<SubBlockSrc*>(smem + lay.desc);

  // ---- prologue: barriers, per-row tile counts and their prefix ---------
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      // one arrival per loader warp, and (tensor-copy path) the value copies' expect
      mbar_init(bar_full(s), kLoaderThreads / 32);
      mbar_init(bar_empty(s), 1);
      if (kCopy) mbar_init(bar_copy(s), 1);  // warp 6's expected bytes
    }
    for (int d = 0; d < kDescRing; ++d) {
      mbar_init(bar_desc_full(d), 1);
      mbar_init(bar_desc_empty(d), kLoaderThreads / 32);
    }
    for (int a = 0; a < NA; ++a) {
      mbar_init(bar_acc_full(a), 1);
      mbar_init(bar_acc_empty(a), kEpilogueThreads / 32);  // one arrival per epilogue warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_q_full(b), 1);
      mbar_init(bar_q_empty(b), 2 + kEpilogueThreads / 32);  // both MMA issuers, the epilogue warps
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_drain + 8, 1);
    mbar_init(bar_setup, 1);
    mbar_init(bar_row_stored, kEpilogueThreads / 32);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (tid == 32 * kQueryWarp) prefetch_tmap(&tm_q);
  if (kCopy && tid == 32 * 6) prefetch_tmap(&tm_k);
  if (tid == 0) SMQ_MARK(0);
  // with programmatic dependent launch the prologue above overlaps the
  // previous kernel; everything below reads what earlier kernels wrote
  griddep_launch_dependents();
  griddep_wait();
  if (tid == 0) SMQ_MARK(1);
  // tiles of row r: from its end, or (rows expanded here) the bound ceil(min(row_ke, S) / 256)
  const int per = (R + kScoreThreads - 1) / kScoreThreads;
  const int r0 = min(R, tid * per), r1 = min(R, r0 + per);
  auto tiles_of = [&](int r) {
    int e = kFused ? p.row_ke[r] : p.end[r];
    e = e < 0 ? 0 : (e > S ? S : e);
    return (e + kTileM - 1) / kTileM;
  };
  int mine = 0;
  for (int r = r0; r < r1; ++r) {
    const int nt = tiles_of(r);
    mine += nt;
    if (kFused && nt == 0 && blockIdx.x == 0) {  // no column at all: CTA 0 writes the empty expansion
      for (int slot = 0; slot < p.nsb; ++slot) p.sparse_indices_out[static_cast<int64_t>(r) * p.nsb + slot] = -1;
      p.end_out[r] = 0;
      if (p.fused_topk) {  // and the empty top-k
        for (int c = 0; c < p.topk; ++c) {
          p.topk_out[static_cast<int64_t>(r) * p.topk_ld + c] = -1;
          if (p.col_indices) p.col_indices[static_cast<int64_t>(r) * p.topk + c] = -1;
        }
        if (p.logits_fill)
          for (int c = 0; c < S; ++c) p.logits_fill[static_cast<int64_t>(r) * S + c] = -INFINITY;
        if (p.logits_bf16)
          for (int c = 0; c < S; ++c) p.logits_bf16[static_cast<int64_t>(r) * S + c] = kBf16NegInf;
      }
    }
  }
  int incl = mine;
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(kFullMask, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) scan[warp] = incl;
  __syncthreads();
  int run = incl - mine;
  for (int w = 0; w < warp; ++w) run += scan[w];
  for (int r = r0; r < r1; ++r) {
    prefix[r] = run;
    run += tiles_of(r);
  }
  if (tid == kScoreThreads - 1) prefix[R] = run;
  __syncthreads();
  const int64_t T = prefix[R];
  const int64_t t_begin = T * blockIdx.x / gridDim.x;
  const int64_t t_end = T * (blockIdx.x + 1) / gridDim.x;
  const int n = static_cast<int>(t_end - t_begin);
  if (tid == 0) SMQ_MARK(2);
  if (n <= 0) return;

  // ---- TMEM: [acc 0 .. acc NA-1 | SF-A per stage (4 cols) | SF-B (4 cols)] ----
  if (warp == 1) tmem_alloc(smem_addr(tmem_slot), p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tm_sfa = tmem + NA * kHalves * kN;
  const uint32_t tm_sfb = tm_sfa + 4 * kHalves * NS;
  // B (query) scales are all 2^0: one 512-byte block of 0x7F copied to the
  // SF-B columns by the first MMA thread, complete before any MMA is issued
  uint32_t* sf_one = reinterpret_cast<uint32_t*>(smem + lay.sf + kScoreStages * kHalves * 512);
  if (tid < 128) sf_one[tid] = 0x7F7F7F7Fu;
  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 32) {
    tmem_cp_32x128b_x4(tm_sfb, rows16_desc(smem_addr(sf_one)));
    mma_commit(bar_setup);
    if (!mbar_wait(bar_setup, 0, abort_flag, static_cast<uint64_t>(p.wait_ns))) {
      set_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int spt = p.subs_per_tile;
  const int sbkv = p.sbkv;
  const int H = p.heads;
  if (tid == 0) SMQ_MARK(3);

  if (warp == 0 && kFused) {
    // ======================= scheduler (rows expanded here) =======================
    // Row by row: expand the row (sorted candidate blocks and end), then
    // resolve its tiles in this CTA in batches of 32 / spt, each lane one
    // sub-block to its page. Tiles past the row's end are published empty.
    const int tiles_per_batch = 32 / spt;
    const int spb = p.cbs / sbkv;
    const int spp = p.page_size / sbkv;  // sub-blocks per cache page
    int32_t* sorted = reinterpret_cast<int32_t*>(smem + lay.sched);
    int32_t* rend = reinterpret_cast<int32_t*>(smem + lay.rend);
    const int r_first = find_row(prefix, R, t_begin);
    int it = 0;
    bool ok = true;
    for (int r = r_first; ok && r < R && prefix[r] < t_end; ++r) {
      const int64_t row0 = prefix[r];
      const int64_t rz = prefix[r + 1];
      if (rz == row0) continue;  // no tiles (written by CTA 0)
      const int brow = p.row_indices ? p.row_indices[r] : r;
      const int ke = p.row_ke[r];
      int nkept = 0;
      const int cols = expand_row_in_warp(p, r, ke > 0 ? ke : 0, sorted, &nkept, lane);
      if (lane == 0 && r == r_first) SMQ_MARK(4);
      // the CTA with the row's first tile writes its expansion, after the first
      // block-table loads are out so that the fence overlaps them
      bool pending_owner = row0 >= t_begin;
      int e = cols < 0 ? 0 : (cols > S ? S : cols);
      // read by the epilogue once it sees this row's first accumulator
      if (lane == 0) st_volatile_s32(rend + (r - r_first), e);
      __syncwarp();
      const int64_t ta = row0 > t_begin ? row0 : t_begin;
      const int64_t tz = rz < t_end ? rz : t_end;
      for (int64_t tb = ta; tb < tz && ok; tb += tiles_per_batch) {
        const int64_t t = tb + lane / spt;
        const int sub = lane % spt;
        const int col_sub = static_cast<int>(t - row0) * spt + sub;
        int ntok = 0, trow = 0, tpage = 0;
        const uint8_t* vsrc = nullptr;
        const uint8_t* ssrc = nullptr;
        const bool want = t < tz && col_sub * sbkv < e;  // columns below end are valid sub-blocks
        int tok = 0;
        int pg = -1;
        if (want) {
          const int sb = sorted[col_sub / spb] * spb + col_sub % spb;
          const int slot = sb / spp;
          tok = (sb - slot * spp) * sbkv;
          if (brow >= 0 && brow < p.bt_rows && slot < p.bt_stride)
            pg = p.block_table[static_cast<int64_t>(brow) * p.bt_stride + slot];
        }
        if (pending_owner) {
          write_row_expansion(p, r, ke > 0 ? ke : 0, sorted, nkept, cols, lane);
          pending_owner = false;
        }
        if (want) {
          if (pg >= 0 && pg < p.num_pages) {
            const uint8_t* base = p.k_cache + static_cast<int64_t>(pg) * p.page_bytes;
            vsrc = base + tok * (kHeadDim / 2);
            ssrc = base + p.page_size * (kHeadDim / 2) + tok * kScaleWordBytes;
            trow = tok;
            tpage = pg;
            ntok = sbkv;
          } else {
            set_status(p.status, kStatusBounds);
          }
        }
        for (int k = 0; k < tiles_per_batch; ++k) {
          if (tb + k >= tz) break;
          const int base = k * spt;
          const int dslot = it % kDescRing;
          bool e_ok = true;
          if (lane == 0)
            e_ok = mbar_wait(bar_desc_empty(dslot), ((it / kDescRing) & 1) ^ 1, abort_flag, static_cast<uint64_t>(p.wait_ns));
          ok = __shfl_sync(kFullMask, e_ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          if (lane >= base && lane < base + spt) put_src(&desc[dslot * kMaxSubsPerTile + (lane - base)], vsrc, ssrc, trow, tpage, ntok);
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_desc_full(dslot));
          if (lane == 0 && it == 0) SMQ_MARK(5);
          if (lane == 0 && it == n - 1) SMQ_MARK(6);
          ++it;
        }
      }
      __syncwarp();  // `sorted` is rewritten for the next row
    }
    if (!ok) {
      set_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    __syncwarp();
  } else if (warp == 0) {
    // ======================= scheduler =======================
    // Resolves each tile's sub-blocks to source addresses (row, sparse id,
    // block-table page, bounds), publishes them per stage, and loads the
    // row's query tile and weights when the row changes.
    const int tiles_per_batch = 32 / spt;
    int it = 0;
    bool ok = true;
    for (int64_t tb = t_begin; tb < t_end && ok; tb += tiles_per_batch) {
      const int64_t t = tb + lane / spt;
      const int sub = lane % spt;
      int ntok = 0, trow = 0, tpage = 0;
      const uint8_t* vsrc = nullptr;
      const uint8_t* ssrc = nullptr;
      if (t < t_end) {
        const int r = find_row(prefix, R, t);
        const int j = static_cast<int>(t - prefix[r]);
        const int col_sub = j * spt + sub;
        // the row's end, sparse id and block-table row do not depend on each
        // other: issue the three loads together
        const bool in_row = col_sub < p.nsb;
        int e = p.end[r];
        const int sb = in_row ? p.sparse_indices[static_cast<int64_t>(r) * p.nsb + col_sub] : -1;
        const int brow = kPaged ? (p.row_indices ? p.row_indices[r] : r) : 0;
        e = e < 0 ? 0 : (e > S ? S : e);
        if (in_row && col_sub * sbkv < e) {
          bool valid = false;
          if (sb >= 0) {
            if constexpr (kPaged) {
              const int spp = p.page_size / sbkv;
              const int slot = sb / spp;
              if (brow >= 0 && brow < p.bt_rows && slot < p.bt_stride) {
                const int pg = p.block_table[static_cast<int64_t>(brow) * p.bt_stride + slot];
                if (pg >= 0 && pg < p.num_pages) {
                  const int tok = (sb - slot * spp) * sbkv;
                  const uint8_t* base = p.k_cache + static_cast<int64_t>(pg) * p.page_bytes;
                  vsrc = base + tok * (kHeadDim / 2);
                  ssrc = base + p.page_size * (kHeadDim / 2) + tok * kScaleWordBytes;
                  trow = tok;
                  tpage = pg;
                  ntok = sbkv;
                  valid = true;
                }
              }
            } else {
              const int64_t pos = static_cast<int64_t>(p.row_ks[r]) + static_cast<int64_t>(sb) * sbkv;
              if (pos >= 0 && pos < p.total_len) {
                vsrc = p.k_values + pos * (kHeadDim / 2);
                ssrc = p.k_scales + pos * kScaleWordBytes;
                trow = static_cast<int>(pos);  // the contiguous workspace is one page of total_len rows
                ntok = static_cast<int>(p.total_len - pos < sbkv ? p.total_len - pos : sbkv);
                valid = true;
              }
            }
          }
          if (!valid) set_status(p.status, kStatusBounds);
        }
      }
      for (int k = 0; k < tiles_per_batch; ++k) {
        if (tb + k >= t_end) break;
        const int base = k * spt;
        // publish into the address ring; it does not wait for pipeline stages,
        // only for the loaders to have read the entry published kDescRing tiles ago
        const int dslot = it % kDescRing;
        bool e_ok = true;
        if (lane == 0)
          e_ok = mbar_wait(bar_desc_empty(dslot), ((it / kDescRing) & 1) ^ 1, abort_flag, static_cast<uint64_t>(p.wait_ns));
        ok = __shfl_sync(kFullMask, e_ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        // the lanes that resolved this tile's sub-blocks publish them
        if (lane >= base && lane < base + spt) put_src(&desc[dslot * kMaxSubsPerTile + (lane - base)], vsrc, ssrc, trow, tpage, ntok);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_desc_full(dslot));
        if (lane == 0 && it == 0) SMQ_MARK(5);
        if (lane == 0 && it == n - 1) SMQ_MARK(6);
        ++it;
      }
    }
    if (!ok) {
      set_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    __syncwarp();
  } else if (warp == kQueryWarp) {
    // ======================= query loader =======================
    // On every row change: wait until the row two back released its buffer,
    // then TMA the row's Q tile and copy its bf16 weights; end and q_scale go
    // along in shared memory. Kept apart from the scheduler so that address
    // publishing never waits on a query buffer.
    if (lane == 0) {
      int r = find_row(prefix, R, t_begin);
      int cur = -1;
      uint32_t quse = 0;
      bool ok = true;
      for (int it = 0; it < n && ok; ++it) {
        const int64_t t = t_begin + it;
        while (prefix[r + 1] <= t) ++r;
        if (r == cur) continue;
        cur = r;
        const int qb = quse & 1;
        ok = mbar_wait(bar_q_empty(qb), ((quse >> 1) & 1) ^ 1, abort_flag, static_cast<uint64_t>(p.wait_ns));
        if (!ok) break;
        meta[qb].row = r;
        if constexpr (!kFused) {  // expanded rows' ends come from the scheduler
          const int e = p.end[r];
          meta[qb].end = e < 0 ? 0 : (e > S ? S : e);
        }
        meta[qb].q_scale = p.q_scale[r];
        const uint32_t q_dst = smem_addr(smem + lay.q + qb * kN * kRowBytes);
        const uint32_t w_dst = smem_addr(smem + lay.w + qb * lay.w_stride);
        mbar_arrive_expect_tx(bar_q_full(qb), kN * kRowBytes + H * 2);
        tma_load_2d(q_dst, &tm_q, 0, r * H, bar_q_full(qb));
        bulk_load(w_dst, p.weights + static_cast<int64_t>(r) * H, H * 2, bar_q_full(qb));
        ++quse;
      }
      if (!ok) {
        set_status(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      // the last query load must land before the CTA exits (it has, unless a wait gave up)
      if (quse > 0) {
        const volatile int never = 0;
        mbar_wait(bar_q_full((quse - 1) & 1), ((quse - 1) >> 1) & 1, &never, static_cast<uint64_t>(p.wait_ns));
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == kMmaWarp1) {
    // ======================= MMA issuers =======================
    // Issuing a tcgen05 instruction costs a thread ~100 cycles, so two
    // threads share the work: warp 1 takes the even tiles, the other warp the
    // odd ones. Each commits its own tiles' accumulators; at the end of every
    // row both commit to the row's query buffer, which is free once the MMAs
    // of both have finished.
    const int par = warp == 1 ? 0 : 1;
    if (lane == 0) {
      uint32_t idesc[4];
      for (int g = 0; g < 4; ++g) idesc[g] = mxf8f6f4_idesc(kE2M1, kE4M3, kMmaM, kN, g, g);
      int r = find_row(prefix, R, t_begin);
      int cur = -1, qb = 0;
      uint32_t quse = 0;
      bool ok = true;
      for (int it = 0; it < n && ok; ++it) {
        const int64_t t = t_begin + it;
        while (prefix[r + 1] <= t) ++r;
        if (r != cur) {
          cur = r;
          qb = quse & 1;
          ++quse;
          // both threads wait for every row's query, so that neither can skip a
          // phase of a buffer and later match its parity too early
          ok = mbar_wait(bar_q_full(qb), ((quse - 1) >> 1) & 1, abort_flag, static_cast<uint64_t>(p.wait_ns));
          if (!ok) break;
        }
        const bool last_of_row = (t + 1 >= t_end) || (t + 1 >= prefix[r + 1]);
        // several accumulators: alternate stages; one: the first thread issues all
        if (NA > 1 ? ((it & 1) == par) : (par == 0)) {
          const int s = it % NS;
          const int a = it % NA;
          ok = mbar_wait(bar_full(s), (it / NS) & 1, abort_flag, static_cast<uint64_t>(p.wait_ns)) &&
               (!kCopy || mbar_wait(bar_copy(s), (it / NS) & 1, abort_flag, static_cast<uint64_t>(p.wait_ns))) &&
               mbar_wait(bar_acc_empty(a), ((it / NA) & 1) ^ 1, abort_flag, static_cast<uint64_t>(p.wait_ns));
          if (!ok) break;
          tc_fence_after();
          const uint32_t stage_addr = smem_addr(smem + lay.kv + s * (kTileM * kRowBytes));
          const uint64_t bdesc = sw128_desc(smem_addr(smem + lay.q + qb * kN * kRowBytes));
          for (int h = 0; h < kHalves; ++h) {
            // this half's key scales: shared memory -> TMEM, in order before its MMAs
            const uint32_t sfa = tm_sfa + 4 * (s * kHalves + h);
            tmem_cp_32x128b_x4(sfa, rows16_desc(smem_addr(smem + lay.sf + (s * kHalves + h) * 512)));
            const uint64_t adesc = sw128_desc(stage_addr + h * (kMmaM * kRowBytes));
            for (int g = 0; g < 4; ++g)  // K = 32 per MMA; advance 32 bytes along the swizzled rows
              mma_mxf8f6f4(tmem + (a * kHalves + h) * kN, adesc + 2 * g, bdesc + 2 * g, idesc[g], sfa, tm_sfb,
                           g > 0);
          }
          mma_commit(bar_acc_full(a));
          if (it == 0) SMQ_MARK(9);
          if (it == n - 1) SMQ_MARK(10);
        }
        if (last_of_row) mma_commit(bar_q_empty(qb));
      }
      if (!ok) {
        set_status(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      const uint32_t drain = bar_drain + 8 * par;
      mma_commit(drain);  // every MMA this thread issued has finished once this arrives
      const volatile int never = 0;
      mbar_wait(drain, 0, &never, static_cast<uint64_t>(p.wait_ns));
    }
    __syncwarp();
  } else if (warp < 6) {
    // ======================= epilogue (warps 2..5) =======================
    const int q4 = warp & 3;  // TMEM lane quarter this warp may access
    const int m = 32 * q4 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
    int r = find_row(prefix, R, t_begin);
    const int r_first = r;
    if constexpr (kFused) {
      if (p.fused_topk) {  // rows this CTA may select: warm the translations of their outputs
        const int rr = r_first + (tid - 2 * 32);
        if (rr < R && prefix[rr] < t_end && prefix[rr + 1] > prefix[rr]) {
          touch_global(p.topk_out + static_cast<int64_t>(rr) * p.topk_ld);
          touch_global(p.sparse_indices_out + static_cast<int64_t>(rr) * p.nsb);
          touch_global(p.logits + static_cast<int64_t>(rr) * S);
          touch_global(p.row_done + rr);
        }
      }
    }
    int cur = -1, qb = 0, row = 0, e = 0;
    uint32_t nrow_ends = 0;
    bool need_end = false;
    uint32_t quse = 0;
    float qs = 0.f;
    // head weights: packed pairs (2j, 2j + 1) for the packed FMA at 64 heads;
    // scalars at 128 heads (pairs would not fit the registers)
    constexpr bool kPacked = kN == 64;
    uint64_t w2[kPacked ? kN / 2 : 1];
    float w[kPacked ? 1 : kN];
    bool ok = true;
    for (int ie = 0; ie < n && ok; ++ie) {
      const int64_t t = t_begin + ie;
      while (prefix[r + 1] <= t) ++r;
      if (r != cur) {
        need_end = kFused;
        cur = r;
        qb = quse & 1;
        ok = warp_wait(bar_q_full(qb), (quse >> 1) & 1, abort_flag, static_cast<uint64_t>(p.wait_ns));
        ++quse;
        if (!ok) break;
        row = meta[qb].row;
        if constexpr (!kFused) e = meta[qb].end;
        qs = meta[qb].q_scale;
        const uint16_t* wsm = reinterpret_cast<const uint16_t*>(smem + lay.w + qb * lay.w_stride);
        if constexpr (kPacked) {
#pragma unroll
          for (int j = 0; j < kN / 2; ++j)
            w2[j] = pack2(2 * j < H ? bf16_to_f32(wsm[2 * j]) : 0.f, 2 * j + 1 < H ? bf16_to_f32(wsm[2 * j + 1]) : 0.f);
        } else {
#pragma unroll
          for (int h = 0; h < kN; ++h) w[h] = h < H ? bf16_to_f32(wsm[h]) : 0.f;
        }
      }
      const bool last_of_row = (t + 1 >= t_end) || (t + 1 >= prefix[r + 1]);
      const int a = ie % NA;
      ok = warp_wait(bar_acc_full(a), (ie / NA) & 1, abort_flag, static_cast<uint64_t>(p.wait_ns));
      if (!ok) break;
      if (need_end) {  // written by the scheduler before it published this row's first tile
        e = ld_volatile_s32(reinterpret_cast<const int32_t*>(smem + lay.rend) + (r - r_first)) & ~kRowDone;
        need_end = false;
      }
      // the MMAs of this tile have finished: its key stage and scale columns are free
      if (warp == 2 && lane == 0) mbar_arrive(bar_empty(ie % NS));
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < kHalves; ++h) {
        // four independent partial sums (heads h mod 4; two packed pairs at 64
        // heads) keep the FMA pipe busy instead of one 64-deep dependent chain
        uint64_t lo = 0, hi = 0;
        float acc4[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t tacc = tmem + (a * kHalves + h) * kN + lane_base;
#pragma unroll
        for (int c = 0; c < kN; c += 32) {
          uint32_t v0[16], v1[16];
          tmem_ld16(tacc + c, v0);
          tmem_ld16(tacc + c + 16, v1);
          tmem_wait_ld();
          if (h == kHalves - 1 && c + 32 >= kN) {  // every column read: hand the accumulator back, one arrival per warp
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_acc_empty(a));
          }
          if constexpr (kPacked) {
#pragma unroll
            for (int hh = 0; hh < 16; hh += 4) {
              relu2_fma2(lo, w2[(c + hh) / 2], __uint_as_float(v0[hh]), __uint_as_float(v0[hh + 1]));
              relu2_fma2(hi, w2[(c + hh) / 2 + 1], __uint_as_float(v0[hh + 2]), __uint_as_float(v0[hh + 3]));
            }
#pragma unroll
            for (int hh = 0; hh < 16; hh += 4) {
              relu2_fma2(lo, w2[(c + 16 + hh) / 2], __uint_as_float(v1[hh]), __uint_as_float(v1[hh + 1]));
              relu2_fma2(hi, w2[(c + 16 + hh) / 2 + 1], __uint_as_float(v1[hh + 2]), __uint_as_float(v1[hh + 3]));
            }
          } else {
#pragma unroll
            for (int hh = 0; hh < 16; ++hh)
              acc4[hh & 3] = fmaf(w[c + hh], fmaxf(__uint_as_float(v0[hh]), 0.f), acc4[hh & 3]);
#pragma unroll
            for (int hh = 0; hh < 16; ++hh)
              acc4[hh & 3] = fmaf(w[c + 16 + hh], fmaxf(__uint_as_float(v1[hh]), 0.f), acc4[hh & 3]);
          }
        }
        // the head sums (twice them, exactly, from the packed form)
        const float2 l2 = kPacked ? unpack2(lo) : make_float2(acc4[0], acc4[1]);
        const float2 h2 = kPacked ? unpack2(hi) : make_float2(acc4[2], acc4[3]);
        const float qscale = kPacked ? 0.5f * qs : qs;
        const float logit = ((l2.x + l2.y) + (h2.x + h2.y)) * qscale;
        const int col = static_cast<int>(t - prefix[r]) * kTileM + h * kMmaM + m;
        if (col < e) {
          p.logits[static_cast<int64_t>(row) * S + col] = logit;
          if (p.logits_bf16) p.logits_bf16[static_cast<int64_t>(row) * S + col] = to_bf16(logit);
        }
      }
      if (warp == 2 && lane == 0 && ie == 0) SMQ_MARK(11);
      if (warp == 2 && lane == 0 && ie == n - 1) SMQ_MARK(12);
      if (last_of_row) {
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_q_empty(qb));
        if constexpr (kFused) {
          if (p.fused_topk) {
            // this CTA's tiles of the row are stored: count them; the CTA that
            // completes the row selects its top-k after the pipeline
            if (lane == 0) mbar_arrive(bar_row_stored);
            if (warp == 2 && lane == 0) {
              if (mbar_wait(bar_row_stored, nrow_ends & 1, abort_flag, static_cast<uint64_t>(p.wait_ns))) {
                const int64_t lo = prefix[r] > t_begin ? prefix[r] : t_begin;
                const int64_t hi = prefix[r + 1] < t_end ? prefix[r + 1] : t_end;
                const int mine = static_cast<int>(hi - lo), total = prefix[r + 1] - prefix[r];
                // release: the logits the epilogue warps stored (acquired through the barrier);
                // acquire: those of the CTAs whose counts this add observes
                if (atom_add_acq_rel_gpu(p.row_done + r, mine) + mine == total) {
                  p.row_done[r] = 0;  // ready for the next call
                  st_volatile_s32(reinterpret_cast<int32_t*>(smem + lay.rend) + (r - r_first), e | kRowDone);
                }
              } else {
                set_status(p.status, kStatusTimeout);
                *abort_flag = 1;
              }
            }
            ++nrow_ends;
          }
        }
      }
    }
    if (!ok) {
      set_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
  } else if (warp >= 6 && warp < 10) {
    // ======================= loaders (warps 6..9) =======================
    // A paged cache is read through registers (coalesced 16-byte loads two
    // tiles ahead of the stage, then stores into the MMA's containers): with
    // few tiles per CTA and keys in DRAM, the register slots add two tiles of
    // buffering to the stages. The contiguous prefill workspace, read many
    // times from L2, goes through tensor copies that unpack into the
    // containers themselves.
    bool ok = true;
    if constexpr (!kCopy) {
      // Key values: loader thread t owns the 16-byte chunk t % 4 of key rows
      // t / 4 + 32 k (k = 0..7), so that each warp load reads 512 contiguous
      // bytes (8 rows of one sub-block). Scale words: thread t owns key rows t
      // and t + 128. Both are loaded kLoadAhead tiles before they are needed.
      // The values are stored into the 16-byte containers the MMA reads (8 data
      // bytes per 16 elements, 128-byte swizzle); the scale words go to the
      // stage half's scale block.
      constexpr int kChunks = kTileM / 32;
      const int q4 = warp & 3;
      const int m = 32 * q4 + lane;
      const uint32_t sf_base = smem_addr(smem + lay.sf);
      const int vch = m & 3;
      int vu[kChunks], vtk[kChunks];
  #pragma unroll
      for (int k8 = 0; k8 < kChunks; ++k8) {
        const int pos = (m >> 2) + 32 * k8;
        vu[k8] = pos / sbkv;
        vtk[k8] = pos % sbkv;
      }
      int su[kHalves], stk[kHalves];
  #pragma unroll
      for (int h = 0; h < kHalves; ++h) {
        su[h] = (m + h * kMmaM) / sbkv;
        stk[h] = (m + h * kMmaM) % sbkv;
      }
      const uint32_t kv_base = smem_addr(smem + lay.kv);
      uint4 v[kLoadAhead][kChunks];
      uint32_t sw[kLoadAhead][kHalves];
  #pragma unroll
      for (int k = 0; k < kLoadAhead; ++k) {
  #pragma unroll
        for (int k8 = 0; k8 < kChunks; ++k8) v[k][k8] = make_uint4(0u, 0u, 0u, 0u);
      }
      // Tiles go in pairs: slot k holds tile i0 + k. A wait costs a warp about
      // as much as a tile's stores, so each pair takes one `empty` wait (stages
      // are freed in tile order: the later one implies the earlier) and, once
      // the ring runs ahead, one descriptor wait (published in tile order).
      static_assert(kLoadAhead == 2, "the loader works on pairs of tiles");
      auto store_tile = [&](const uint4 (&vv)[kChunks], const uint32_t (&ss)[kHalves], int j) {
        const int s = j % NS;
        const uint32_t stage = kv_base + s * (kTileM * kRowBytes);
  #pragma unroll
        for (int k8 = 0; k8 < kChunks; ++k8) {
          // stored whether or not the chunk was loaded: an unloaded chunk holds
          // an older key's bytes (finite E2M1 values, scale 1) in a position the
          // epilogue never stores
          const int pos = (m >> 2) + 32 * k8;
          const uint32_t dst = stage + static_cast<uint32_t>(pos) * kRowBytes;
          const uint32_t swz = static_cast<uint32_t>(pos & 7);
          sts_v2(dst + (((2 * vch) ^ swz) << 4), vv[k8].x, vv[k8].y);
          sts_v2(dst + (((2 * vch + 1) ^ swz) << 4), vv[k8].z, vv[k8].w);
        }
        // scale word of key row m of each half: word 4 (m % 32) + m / 32 of the
        // half's block, which the copy to TMEM places at lane m, column base + m / 32
  #pragma unroll
        for (int h = 0; h < kHalves; ++h) sts_u32(sf_base + (s * kHalves + h) * 512 + 16 * lane + 4 * q4, ss[h]);
        fence_proxy_async_smem();  // make this thread's stores visible to the tensor core's reads
        __syncwarp();              // one arrival per warp
        if (lane == 0 && !(j == p.stall_tile && blockIdx.x == 0)) mbar_arrive(bar_full(s));
        if (warp == 6 && lane == 0 && j == 0) SMQ_MARK(7);
        if (warp == 6 && lane == 0 && j == n - 1) SMQ_MARK(8);
      };
      auto load_tile = [&](uint4 (&vv)[kChunks], uint32_t (&ss)[kHalves], int i) {
        const SubBlockSrc* dring = desc + (i % kDescRing) * kMaxSubsPerTile;
        // predicated loads: a branch per chunk costs more than the load
  #pragma unroll
        for (int k8 = 0; k8 < kChunks; ++k8) {
          const SubBlockSrc d = get_src(dring + vu[k8]);
          ldg_stream_v4_if(vv[k8], d.values + static_cast<int64_t>(vtk[k8]) * (kHeadDim / 2) + 16 * vch,
                           d.values != nullptr && vtk[k8] < d.positions);
        }
  #pragma unroll
        for (int h = 0; h < kHalves; ++h) {
          const SubBlockSrc ds = get_src(dring + su[h]);
          ss[h] = 0x7F7F7F7Fu;  // scale 1 where no key is loaded
          ldg_stream_u32_if(ss[h], ds.scales + static_cast<int64_t>(stk[h]) * kScaleWordBytes,
                            ds.values != nullptr && stk[h] < ds.positions);
        }
      };
      // Two register slots: each slot's tile is stored, then the slot takes
      // its next tile at once, so that the next load is out before the other
      // slot's stores.
      for (int i0 = 0; i0 < n + 2; i0 += 2) {
        const int j0 = i0 - 2;  // the pair whose data sits in the slots
        if (j0 >= 0 && j0 < n) {
          const int jl = j0 + 1 < n ? j0 + 1 : j0;
          // the stages are free once the MMAs of tiles j0 - NS and jl - NS have finished
          ok = warp_wait(bar_empty(jl % NS), ((jl / NS) & 1) ^ 1, abort_flag, static_cast<uint64_t>(p.wait_ns));
          if (!ok) break;
          store_tile(v[0], sw[0], j0);
        }
        if (i0 < n) {
          ok = warp_wait(bar_desc_full(i0 % kDescRing), (i0 / kDescRing) & 1, abort_flag, static_cast<uint64_t>(p.wait_ns));
          if (!ok) break;
          load_tile(v[0], sw[0], i0);
        }
        if (j0 >= 0 && j0 + 1 < n) store_tile(v[1], sw[1], j0 + 1);
        if (i0 + 1 < n) {
          ok = warp_wait(bar_desc_full((i0 + 1) % kDescRing), ((i0 + 1) / kDescRing) & 1, abort_flag,
                         static_cast<uint64_t>(p.wait_ns));
          if (!ok) break;
          load_tile(v[1], sw[1], i0 + 1);
        }
        if (i0 < n) {
          __syncwarp();  // every lane has read the entries before they are handed back
          if (lane == 0) {
            mbar_arrive(bar_desc_empty(i0 % kDescRing));
            if (i0 + 1 < n) mbar_arrive(bar_desc_empty((i0 + 1) % kDescRing));
          }
        }
      }
    } else {
      // Key values: tensor copies issued by warp 6, one per sub-block (lane l
      // copies sub-block l). The copy unpacks each 16 FP4 values (8 bytes) into
      // the 16-byte container the MMA reads (16U4_ALIGN16B) with the 128-byte
      // swizzle, and completes on the stage's `full` barrier.
      // Scale words: thread t owns key rows t and t + 128; it loads them into
      // registers two tiles ahead and stores them into the stage half's scale
      // block once the stage is free.
      // Step i: store the scale words of tile i - 2 (the slot is reloaded next);
      // read tile i's descriptors and load its scale words; wait for its stage
      // and issue its value copies.
      const int q4 = warp & 3;
      const int m = 32 * q4 + lane;
      const uint32_t sf_base = smem_addr(smem + lay.sf);
      const uint32_t kv_base = smem_addr(smem + lay.kv);
      const bool copier = warp == 6 && lane < spt;
      const uint32_t sub_bytes = static_cast<uint32_t>(sbkv) * kRowBytes;  // one sub-block in the stage
      // the copy's transaction count is the packed source size (half its footprint in the stage)
      const uint32_t sub_tx = static_cast<uint32_t>(sbkv) * (kHeadDim / 2);
      int su[kHalves], stk[kHalves];
  #pragma unroll
      for (int h = 0; h < kHalves; ++h) {
        su[h] = (m + h * kMmaM) / sbkv;
        stk[h] = (m + h * kMmaM) % sbkv;
      }
      uint32_t sw[2][kHalves];
      int issued = 0;  // (warp 6) tiles whose value copies are out
      for (int i0 = 0; i0 < n + 2 && ok; i0 += 2) {
  #pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int i = i0 + k;
          const int j = i - 2;  // its scale words sit in slot k: store them before slot k is reloaded
          if (j >= 0 && j < n) {
            // scale word of key row m of each half: word 4 (m % 32) + m / 32 of the
            // half's block, which the copy to TMEM places at lane m, column base + m / 32
            const int s = j % NS;
  #pragma unroll
            for (int h = 0; h < kHalves; ++h) sts_u32(sf_base + (s * kHalves + h) * 512 + 16 * lane + 4 * q4, sw[k][h]);
            fence_proxy_async_smem();  // make this thread's stores visible to the tensor core's reads
            __syncwarp();              // one arrival per warp
            if (lane == 0 && !(j == p.stall_tile && blockIdx.x == 0)) mbar_arrive(bar_full(s));
          }
          if (i < n) {
            const int dslot = i % kDescRing;
            ok = warp_wait(bar_desc_full(dslot), (i / kDescRing) & 1, abort_flag, static_cast<uint64_t>(p.wait_ns));
            if (!ok) break;
            const SubBlockSrc* dring = desc + dslot * kMaxSubsPerTile;
  #pragma unroll
            for (int h = 0; h < kHalves; ++h) {
              const SubBlockSrc ds = get_src(dring + su[h]);
              sw[k][h] = 0x7F7F7F7Fu;  // scale 1 where no key is loaded
              ldg_stream_u32_if(sw[k][h], ds.scales + static_cast<int64_t>(stk[h]) * kScaleWordBytes,
                                stk[h] < ds.positions);
            }
            SubBlockSrc dv;
            dv.positions = 0;
            if (copier) dv = get_src(dring + lane);
            __syncwarp();  // every lane has read the entries before they are handed back
            if (lane == 0) mbar_arrive(bar_desc_empty(dslot));
            // the stage is free once the MMAs of tile i - NS have finished
            const int s = i % NS;
            ok = warp_wait(bar_empty(s), ((i / NS) & 1) ^ 1, abort_flag, static_cast<uint64_t>(p.wait_ns));
            if (!ok) break;
            if (warp == 6) {
              const bool live = copier && dv.positions > 0;
              const uint32_t nlive = __popc(__ballot_sync(kFullMask, live));
              if (lane == 0) mbar_arrive_expect_tx(bar_copy(s), nlive * sub_tx);
              if (live) tma_load_3d(kv_base + s * (kTileM * kRowBytes) + lane * sub_bytes, &tm_k, 0, dv.row, dv.page,
                                    bar_copy(s));
              issued = i + 1;
            }
          }
        }
      }
      if (warp == 6 && lane == 0) {
        // the copies of the last NS tiles may still be in flight (each earlier
        // stage was reused, so its copies had landed), also when a wait of
        // another warp gives up later: wait, bounded, for them before the CTA
        // and its shared memory can go away
        const volatile int never = 0;
        for (int t = issued > NS ? issued - NS : 0; t < issued; ++t)
          mbar_wait(bar_copy(t % NS), (t / NS) & 1, &never, static_cast<uint64_t>(p.wait_ns));
      }
      __syncwarp();
    }
    if (!ok) {
      set_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
  }

  // ---- teardown (TMEM is freed at the very end, so the top-k tail need not wait for it) ----
  tc_fence_before();
  __syncthreads();
  if (tid == 0) SMQ_MARK(13);

  // ---- top-k of the rows this CTA completed (their logits are in L2) ----
  if constexpr (kFused) {
    if (p.fused_topk && *abort_flag == 0) {
      fence_proxy_async_smem();      // the tensor copies wrote these bytes; plain accesses follow
      uint8_t* scr = smem + lay.kv;  // the key stages are free now
      TopkScratch sm;
      sm.hist = reinterpret_cast<uint32_t*>(scr);
      sm.bsum = nullptr;
      sm.wsum = reinterpret_cast<int*>(scr + kTopkBins * 4);
      sm.chunk = reinterpret_cast<uint32_t*>(sm.wsum + 32);
      sm.sel = reinterpret_cast<int*>(sm.chunk + 32 * 32);
      sm.sidx = sm.sel + 16;
      const int32_t* rend = reinterpret_cast<const int32_t*>(smem + lay.rend);
      const int r_first = find_row(prefix, R, t_begin);
      for (int r = r_first; r < R && prefix[r] < t_end; ++r) {
        if (prefix[r + 1] == prefix[r]) continue;
        const int32_t* end_src = rend + (r - r_first);
        if ((*end_src & kRowDone) == 0) continue;
        int32_t* e_clean = sm.sel + 12;  // the end without the flag
        if (tid == 0) *e_clean = *end_src & ~kRowDone;
        if (tid == 0) SMQ_MARK(14);
        __syncthreads();
        const float* L = p.logits + static_cast<int64_t>(r) * S;
        int32_t* out = p.topk_out + static_cast<int64_t>(r) * p.topk_ld;
        int32_t* colo = p.col_indices ? p.col_indices + static_cast<int64_t>(r) * p.topk : nullptr;
        float* fill = p.logits_fill ? p.logits_fill + static_cast<int64_t>(r) * S : nullptr;
        uint16_t* fill16 = p.logits_bf16 ? p.logits_bf16 + static_cast<int64_t>(r) * S : nullptr;
        const int32_t* srow = p.sparse_indices_out + static_cast<int64_t>(r) * p.nsb;
        if (S <= kScoreThreads * 11)
          select_topk<kScoreThreads, 11, true>(L, S, e_clean, p.topk, srow, p.nsb, sbkv, out, colo, fill, fill16, sm);
        else
          select_topk<kScoreThreads, 22, true>(L, S, e_clean, p.topk, srow, p.nsb, sbkv, out, colo, fill, fill16, sm);
        __syncthreads();  // the scratch is reused by the next row
        if (tid == 0) SMQ_MARK(15);
      }
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
  if (tid == 0) SMQ_MARK(16);
}

// ===========================================================================
// Top-k: radix select over order-preserving keys, one CTA per row.
// ===========================================================================
// One CTA per row (rows whose top-k the score kernel does not select itself).
// Rows are many and each CTA is latency bound: rows of up to 4096 columns take
// 256 threads, wider ones 512, and the launch bound keeps as many CTAs per SM
// resident as 64 (or, 32 keys a thread, 128) registers a thread allow.
template <int kThreads, int kJ>
__global__ void __launch_bounds__(kThreads, kThreads == 256 ? (kJ <= 8 ? 6 : 4) : (kJ <= 16 ? 2 : 1))
    topk_kernel(const __grid_constant__ TopkParams p) {
  constexpr int kWarps = kThreads / 32;
  static_assert(kThreads >= 256, "the 8-bit passes give each of the 256 bins a thread");
  extern __shared__ int32_t sidx[];  // [nsb] sparse sub-block ids of the row
  __shared__ __align__(16) uint32_t hist[256 * 32];
  __shared__ int bsum[256];
  __shared__ int wsum[kWarps];
  __shared__ uint32_t chunk[kWarps * kJ];
  __shared__ int sel[12];
  griddep_launch_dependents();
  griddep_wait();
  const int r = blockIdx.x;
  const int S = p.num_cols;
  const TopkScratch sm{hist, bsum, wsum, chunk, sidx, sel};
  select_topk<kThreads, kJ, false, false, true>(p.logits + static_cast<int64_t>(r) * S, S, p.end + r, p.topk,
                                p.sparse_indices + static_cast<int64_t>(r) * p.nsb, p.nsb, p.sbkv,
                                p.topk_out + static_cast<int64_t>(r) * p.topk_ld,
                                p.col_indices ? p.col_indices + static_cast<int64_t>(r) * p.topk : nullptr,
                                p.logits_fill ? p.logits_fill + static_cast<int64_t>(r) * S : nullptr,
                                p.logits_fill_bf16 ? p.logits_fill_bf16 + static_cast<int64_t>(r) * S : nullptr, sm);
}

// ---------------------------------------------------------------------------
// Top-k of a row by one warp: the selection
// of select_topk (the value range, a 1024-bin histogram over it, the threshold
// bin's keys sorted; four 8-bit digit passes where that bin holds more than
// kRangeBin keys; one ordered compaction), with shuffles in place of block
// barriers, so that a row's chain of steps stays inside one warp, and few
// instructions per key (the kernel is issue bound). Each pass reads the row
// again through L2; lane l takes columns 4 (l + 32 i) + q, q < 4, of chunk i
// (128 columns) as one float4. Chunks wholly below `end` skip the per-column
// checks. The histogram's bins differ from select_topk's (a sampled range),
// the selection does not: it is exact either way.
// ---------------------------------------------------------------------------
__device__ void select_topk_warp(const float* L, int S, int e, int k, const int32_t* sidx, int sbkv, int32_t* out,
                                 int32_t* colo, uint32_t* hist, uint32_t* list, int* list_n) {
  const int lane = threadIdx.x & 31;
  const int sb_shift = 31 - __clz(sbkv);
  if (e <= k) {  // every valid column is selected, in column order
    for (int c = lane; c < k; c += 32) {
      out[c] = c < e ? (sidx[c >> sb_shift] << sb_shift) | (c & (sbkv - 1)) : -1;
      if (colo) colo[c] = c < e ? c : -1;
    }
    return;
  }
  const float4* L4 = reinterpret_cast<const float4*>(L);
  const int nfull = e >> 7;            // chunks whose 128 columns are all below e
  const int nchunks = (e + 127) >> 7;  // chunks with a column below e
  auto fetch = [&](int i) { return __ldcg(L4 + lane + 32 * i); };
  auto fetch_tail = [&](int i) {  // a chunk that crosses e: nothing at or past S is read
    return 4 * (lane + 32 * i) < S ? fetch(i) : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  // -- value range of the histogram: from a sample (each lane's first four
  // columns); keys outside it fall into the end bins. Any monotone binning
  // finds the threshold exactly (its bin's keys are sorted next); a row whose
  // sample has no spread takes the exact range (one more pass).
  float vmin = INFINITY, vmax = -INFINITY;
  {
    const float4 f = fetch_tail(0);
    const float v[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (4 * lane + q < e) {
        vmin = fminf(vmin, v[q]);
        vmax = fmaxf(vmax, v[q]);
      }
  }
  auto warp_range = [&]() {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      vmin = fminf(vmin, __shfl_xor_sync(kFullMask, vmin, o));
      vmax = fmaxf(vmax, __shfl_xor_sync(kFullMask, vmax, o));
    }
  };
  warp_range();
  if (!(vmax > vmin) || !(vmax - vmin < INFINITY)) {
#pragma unroll 8
    for (int i = 0; i < nfull; ++i) {
      const float4 f = fetch(i);
      vmin = fminf(vmin, fminf(fminf(f.x, f.y), fminf(f.z, f.w)));
      vmax = fmaxf(vmax, fmaxf(fmaxf(f.x, f.y), fmaxf(f.z, f.w)));
    }
    for (int i = nfull; i < nchunks; ++i) {
      const int c = 4 * (lane + 32 * i);
      const float4 f = fetch_tail(i);
      const float v[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (c + q < e) {
          vmin = fminf(vmin, v[q]);
          vmax = fmaxf(vmax, v[q]);
        }
    }
    warp_range();
  }
  uint32_t prefix = 0;  // selected high bits so far
  int need = k;         // keys still to take among those matching the prefix
  int done_bits = 0;
  bool ranged = false;
  uint4* hist4 = reinterpret_cast<uint4*>(hist);
  if (!(vmax > vmin) || !(vmax - vmin < INFINITY)) {
    if (vmin == vmax) {  // every valid key equal: the first k
      prefix = ordered_key(vmin);
      done_bits = 32;
      ranged = true;
    }
  } else {
    // bin = clamp((v - vmin) scale, 0, kRangeBins - 1): non-decreasing in v
    // (the conversion saturates below 0; NaN goes to the top bin)
    const float scale = static_cast<float>(kRangeBins) / (vmax - vmin);
    const float offset = -vmin * scale;
    auto bin_of = [&](float v) { return static_cast<int>(__float2uint_rz(fminf(fmaf(v, scale, offset), kRangeBins - 1.f))); };
    for (int w = lane; w < kRangeBins / 4; w += 32) hist4[w] = make_uint4(0u, 0u, 0u, 0u);
    if (lane == 0) *list_n = 0;
    __syncwarp();
#pragma unroll 4
    for (int i = 0; i < nfull; ++i) {
      const float4 f = fetch(i);
      atomicAdd(&hist[bin_of(f.x)], 1u);
      atomicAdd(&hist[bin_of(f.y)], 1u);
      atomicAdd(&hist[bin_of(f.z)], 1u);
      atomicAdd(&hist[bin_of(f.w)], 1u);
    }
    for (int i = nfull; i < nchunks; ++i) {
      const int c = 4 * (lane + 32 * i);
      const float4 f = fetch_tail(i);
      const float v[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (c + q < e) atomicAdd(&hist[bin_of(v[q])], 1u);
    }
    __syncwarp();
    // descending scan: lane l owns bins kRangeBins - 32 (l + 1) + b, b < 32, the highest first
    const int b0 = kRangeBins - 32 * (lane + 1);
    int local = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const uint4 v = hist4[b0 / 4 + w];
      local += static_cast<int>(v.x + v.y + v.z + v.w);
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl += v;
    }
    int cum = incl - local, tb = 0, above = 0, tcount = 0;
    const bool owner = cum < need && need <= incl;
    if (owner)  // the lane whose run of bins holds the k-th key reads them again
      for (int b = 31; b >= 0; --b) {
        const int c = static_cast<int>(hist[b0 + b]);
        if (c > 0 && cum < need && need <= cum + c) {
          tb = b0 + b;
          above = cum;
          tcount = c;
        }
        cum += c;
      }
    const int src = __ffs(__ballot_sync(kFullMask, owner)) - 1;
    tb = __shfl_sync(kFullMask, tb, src);
    above = __shfl_sync(kFullMask, above, src);
    tcount = __shfl_sync(kFullMask, tcount, src);
    if (tcount > 0 && tcount <= kRangeBin) {
      // the bin's (key, column) pairs, in any order (they are sorted next)
      auto take = [&](float v, int c) {
        if (bin_of(v) == tb) {
          const int at = atomicAdd(list_n, 1);
          if (at < kRangeBin) {
            list[2 * at] = ordered_key(v);
            list[2 * at + 1] = static_cast<uint32_t>(c);
          }
        }
      };
#pragma unroll 8
      for (int i = 0; i < nfull; ++i) {
        const int c = 4 * (lane + 32 * i);
        const float4 f = fetch(i);
        take(f.x, c);
        take(f.y, c + 1);
        take(f.z, c + 2);
        take(f.w, c + 3);
      }
      for (int i = nfull; i < nchunks; ++i) {
        const int c = 4 * (lane + 32 * i);
        const float4 f = fetch_tail(i);
        const float v[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (c + q < e) take(v[q], c + q);
      }
      __syncwarp();
      // bitonic sort of kRangeBin = 64 composites (key, ~column), descending:
      // lane l holds elements l and l + 32
      uint64_t y[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        y[h] = i < tcount ? (static_cast<uint64_t>(list[2 * i]) << 32) | (0xFFFFFFFFu - list[2 * i + 1]) : 0ull;
      }
#pragma unroll
      for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int i = lane + 32 * h;
            const bool desc = (i & size) == 0;
            if (stride == 32) {
              if (h == 0 && (desc ? (y[0] < y[1]) : (y[0] > y[1]))) {
                const uint64_t t = y[0];
                y[0] = y[1];
                y[1] = t;
              }
            } else {
              const uint64_t z = __shfl_xor_sync(kFullMask, y[h], stride);
              const bool take_max = ((i & stride) == 0) == desc;
              y[h] = take_max ? (y[h] > z ? y[h] : z) : (y[h] < z ? y[h] : z);
            }
          }
        }
      }
      // the (need - above)-th largest is the threshold; how many equal keys are taken
      const int want = need - above;
      const int at = want - 1;
      const uint32_t tkey = static_cast<uint32_t>(__shfl_sync(kFullMask, y[at >> 5], at & 31) >> 32);
      int eq = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) eq += (lane + 32 * h < want && static_cast<uint32_t>(y[h] >> 32) == tkey) ? 1 : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) eq += __shfl_xor_sync(kFullMask, eq, o);
      prefix = tkey;
      need = eq;
      done_bits = 32;
      ranged = true;
    }
  }
  if (!ranged) {
    // four 8-bit digit passes over a 256-bin histogram; lane l owns bins 255 - 8 l - b
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - done_bits;
      __syncwarp();
      for (int w = lane; w < 256 / 4; w += 32) hist4[w] = make_uint4(0u, 0u, 0u, 0u);
      __syncwarp();
      for (int i = 0; i < nchunks; ++i) {
        const int c = 4 * (lane + 32 * i);
        const float4 f = fetch_tail(i);
        const float v[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t key = ordered_key(v[q]);
          if (c + q < e && (done_bits == 0 || (key >> (32 - done_bits)) == prefix))
            atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
      }
      __syncwarp();
      const int b0 = 256 - 8 * (lane + 1);
      int local = 0;
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const uint4 v = hist4[b0 / 4 + w];
        local += static_cast<int>(v.x + v.y + v.z + v.w);
      }
      int incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl += v;
      }
      int cum = incl - local, sb = 0, above = 0, scount = 0;
      const bool owner = cum < need && need <= incl;
      if (owner)
        for (int b = 7; b >= 0; --b) {
          const int c = static_cast<int>(hist[b0 + b]);
          if (c > 0 && cum < need && need <= cum + c) {
            sb = b0 + b;
            above = cum;
            scount = c;
          }
          cum += c;
        }
      const int src = __ffs(__ballot_sync(kFullMask, owner)) - 1;
      sb = __shfl_sync(kFullMask, sb, src);
      above = __shfl_sync(kFullMask, above, src);
      scount = __shfl_sync(kFullMask, scount, src);
      prefix = (prefix << 8) | static_cast<uint32_t>(sb);
      need -= above;
      done_bits += 8;
      if (need == scount) break;  // the whole bin is taken
    }
  }
  // selected: keys whose top done_bits bits are above the prefix, and the
  // first `need` of those equal to it, in column order. A selected column's
  // slot is the number of selected columns before it; a lane's four columns
  // are consecutive, so its selected ones take consecutive slots.
  const uint32_t mask = ~0u << (32 - done_bits);
  const uint32_t pfx = prefix << (32 - done_bits);
  int base_g = 0, base_e = 0;
  auto compact = [&](int i, const float4& f, bool check, bool masked) {
    const int c = 4 * (lane + 32 * i);
    const float v[4] = {f.x, f.y, f.z, f.w};
    bool g[4], eq[4];
    uint32_t packed = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t kk = masked ? ordered_key(v[q]) & mask : ordered_key(v[q]);
      const bool ok = !check || c + q < e;
      g[q] = ok && kk > pfx;
      eq[q] = ok && kk == pfx;
      packed += (g[q] ? 0x10000u : 0u) + (eq[q] ? 1u : 0u);
    }
    uint32_t incl = packed;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl += t;
    }
    const uint32_t tot = __shfl_sync(kFullMask, incl, 31);
    const uint32_t pre = incl - packed;
    int pe = base_e + static_cast<int>(pre & 0xffffu);
    int slot = base_g + static_cast<int>(pre >> 16) + min(pe, need);
    base_g += static_cast<int>(tot >> 16);
    base_e += static_cast<int>(tot & 0xffffu);
    if (packed == 0) return;
    const int tok = (sidx[c >> sb_shift] << sb_shift) | (c & (sbkv - 1));  // a lane's columns share a sub-block
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const bool sel = g[q] || (eq[q] && pe < need);
      pe += eq[q] ? 1 : 0;
      if (sel && slot < k) {
        out[slot] = tok + q;
        if (colo) colo[slot] = c + q;
        ++slot;
      }
    }
  };
  if (done_bits == 32) {
#pragma unroll 2
    for (int i = 0; i < nfull; ++i) compact(i, fetch(i), false, false);
  } else {
#pragma unroll 2
    for (int i = 0; i < nfull; ++i) compact(i, fetch(i), false, true);
  }
  for (int i = nfull; i < nchunks; ++i) compact(i, fetch_tail(i), true, true);
}

// One row per warp at a time; one CTA of kTopkWarps warps per SM (at most
// #SM CTAs), rows dealt round robin: CTA b, warp w takes rows b + G (w + 32 j).
// Rows, not CTAs, balance the SMs: the kernel is issue bound, and CTAs that
// start early (on the SMs the previous kernel frees first) would otherwise
// stack up there. No block barrier. Dynamic shared memory per warp: a
// 1024-bin histogram, the threshold bin's list and its count, the row's
// sparse sub-block ids.
constexpr int kTopkWarps = 32;
constexpr int kTopkWarpMaxCols = 4096;  // rows this wide or narrower take the warp kernel

__host__ __device__ constexpr int topk_warp_words(int nsb) { return kRangeBins + 2 * kRangeBin + 4 + ((nsb + 3) & ~3); }

__global__ void __launch_bounds__(32 * kTopkWarps, 1) topk_warp_kernel(const __grid_constant__ TopkParams p) {
  extern __shared__ __align__(16) uint32_t topk_warp_smem_raw[];
  griddep_launch_dependents();
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.num_cols;
  uint32_t* hist = topk_warp_smem_raw + static_cast<size_t>(warp) * topk_warp_words(p.nsb);
  uint32_t* list = hist + kRangeBins;
  int* list_n = reinterpret_cast<int*>(list + 2 * kRangeBin);
  int32_t* sidx = reinterpret_cast<int32_t*>(list + 2 * kRangeBin + 4);
  for (int r = blockIdx.x + gridDim.x * warp; r < p.rows; r += gridDim.x * kTopkWarps) {
    __syncwarp();  // the previous row's reads of the scratch are done
    const int32_t* srow = p.sparse_indices + static_cast<int64_t>(r) * p.nsb;
    for (int i = lane; i < p.nsb; i += 32) sidx[i] = __ldcg(srow + i);
    int e = __ldcg(p.end + r);
    e = e < 0 ? 0 : (e > S ? S : e);
    if (p.logits_fill)
      for (int c = e + lane; c < S; c += 32) p.logits_fill[static_cast<int64_t>(r) * S + c] = -INFINITY;
    if (p.logits_fill_bf16)
      for (int c = e + lane; c < S; c += 32) p.logits_fill_bf16[static_cast<int64_t>(r) * S + c] = kBf16NegInf;
    __syncwarp();
    select_topk_warp(p.logits + static_cast<int64_t>(r) * S, S, e, p.topk, sidx, p.sbkv,
                     p.topk_out + static_cast<int64_t>(r) * p.topk_ld,
                     p.col_indices ? p.col_indices + static_cast<int64_t>(r) * p.topk : nullptr, hist, list, list_n);
  }
}

size_t topk_warp_smem(int nsb) { return static_cast<size_t>(kTopkWarps) * topk_warp_words(nsb) * 4; }

// ===========================================================================
// Paged -> contiguous K gather: one thread per workspace row.
// ===========================================================================
__global__ void __launch_bounds__(256) gather_kernel(const __grid_constant__ GatherParams p) {
  griddep_launch_dependents();
  griddep_wait();
  const int64_t wrow = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (wrow >= p.total_len) return;
  int lo = 0, hi = p.num_seqs;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.cu_seq_lens[mid] <= wrow) lo = mid; else hi = mid;
  }
  const int64_t start = p.cu_seq_lens[lo];
  const int64_t stop = p.cu_seq_lens[lo + 1];
  if (wrow < start || wrow >= stop) {
    set_status(p.status, kStatusBounds);
    return;
  }
  const int pos = static_cast<int>(wrow - start);  // a position within one sequence (int32 lengths)
  const int slot = pos / p.page_size;
  if (slot >= p.bt_stride) {
    set_status(p.status, kStatusBounds);
    return;
  }
  const int page = p.block_table[static_cast<int64_t>(lo) * p.bt_stride + slot];
  if (page < 0 || page >= p.num_pages) {
    set_status(p.status, kStatusBounds);
    return;
  }
  const int tok = pos - slot * p.page_size;
  const uint8_t* base = p.k_cache + static_cast<int64_t>(page) * p.page_bytes;
  const uint4* src = reinterpret_cast<const uint4*>(base + tok * (kHeadDim / 2));
  uint4* dst = reinterpret_cast<uint4*>(p.k_values + wrow * (kHeadDim / 2));
#pragma unroll
  for (int i = 0; i < kHeadDim / 32; ++i) dst[i] = src[i];
  const uint32_t* ssrc = reinterpret_cast<const uint32_t*>(base + p.page_size * (kHeadDim / 2) + tok * kScaleWordBytes);
  reinterpret_cast<uint32_t*>(p.k_scales)[wrow] = *ssrc;
}

// ===========================================================================
// Decode rows of a narrow batch: one thread-block cluster per row.
// ===========================================================================
// A cluster of C CTAs scores one row. Every CTA expands the row's candidate
// blocks (the same result in each), and the row's tiles (the bound
// ceil(min(row_ke, S) / 256), or ceil(end / 256) for an expansion passed in)
// are split into C contiguous ranges, one per CTA. Each CTA runs the score
// pipeline of the persistent kernel on its range, with the same warp roles,
// and keeps its logits in shared memory. The other CTAs then store their
// logits into CTA 0 (asynchronous stores through distributed shared memory,
// one exchange), and CTA 0 selects the row's top-k there. No logits, counters
// or atomics go through global memory.
struct RowLayout {
  uint32_t kv, q, sf, desc, w, bars, misc, sorted, sidx, lg, total;
  __host__ __device__ RowLayout(int n_mma, int heads, int nsb, int num_cols) {
    uint32_t o = 0;
    kv = o;  // [stages][256 rows][128 B] keys; after the pipeline, top-k scratch
    o += static_cast<uint32_t>(kScoreStages) * kTileM * kRowBytes;
    q = o;  // [n_mma rows][128 B] E4M3 queries, 128-byte swizzle
    o += static_cast<uint32_t>(n_mma) * kRowBytes;
    sf = o;  // [stages][halves] key scale blocks of 512 B, then one block of 2^0
    o += static_cast<uint32_t>(kScoreStages * kHalves + 1) * 512u;
    desc = o;  // [ring][16 sub-blocks] source addresses
    o += static_cast<uint32_t>(kDescRing) * kMaxSubsPerTile * sizeof(SubBlockSrc);
    w = o;  // [heads] bf16 weights
    o += round_up(static_cast<uint32_t>(heads) * 2u, 16);
    bars = o;  // full, empty [stages]; acc_full, acc_empty [3]; q_full; drain [2]; setup; desc_full, desc_empty [ring];
               // recv (the other CTAs' logits, in CTA 0)
    o += round_up((2u * kScoreStages + 2u * kMaxAccBuffers + 4u + 2u * kDescRing + 1u) * 8u, 16);
    misc = o;  // tmem base, abort flag, end, q_scale
    o += 32u;
    sorted = o;  // the row's kept candidate blocks, ascending
    o += kMaxFusedBlocks * 4u;
    sidx = o;  // [nsb] the row's sparse sub-block ids
    o += round_up(static_cast<uint32_t>(nsb) * 4u, 16);
    lg = o;  // [row columns] fp32 logits by sparse column: this CTA's, and in CTA 0 the whole row's
    o += round_up(static_cast<uint32_t>(num_cols) * 4u, 16);
    total = o;
  }
};

size_t row_cluster_smem_bytes(int n_mma, int heads, int nsb, int num_cols) {
  return RowLayout(n_mma, heads, nsb, num_cols).total + 1024;
}

template <int kN, int kJ>
__global__ void __launch_bounds__(kScoreThreads, 1)
    row_cluster_kernel(const __grid_constant__ ScoreParams p, const __grid_constant__ CUtensorMap tm_q) {
  extern __shared__ uint8_t rc_smem_raw[];
  uint8_t* smem = align1024(rc_smem_raw);
  constexpr int NS = kScoreStages;
  constexpr int NA = acc_buffers(kN);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = p.cluster;
  const int r = blockIdx.x / C;
  const int rank = static_cast<int>(cluster_ctarank());
  const int S = p.num_cols;
  const int sbkv = p.sbkv, spt = p.subs_per_tile;
  const int H = p.heads;
  const RowLayout lay(kN, H, p.nsb, S);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
  auto bar_full = [&](int s) { return smem_addr(&bars[s]); };
  auto bar_empty = [&](int s) { return smem_addr(&bars[NS + s]); };
  auto bar_acc_full = [&](int a) { return smem_addr(&bars[2 * NS + a]); };
  auto bar_acc_empty = [&](int a) { return smem_addr(&bars[2 * NS + kMaxAccBuffers + a]); };
  constexpr int NB = 2 * NS + 2 * kMaxAccBuffers;
  const uint32_t bar_q_full = smem_addr(&bars[NB]);
  const uint32_t bar_drain = smem_addr(&bars[NB + 1]);  // and the next one
  const uint32_t bar_setup = smem_addr(&bars[NB + 3]);
  auto bar_desc_full = [&](int d) { return smem_addr(&bars[NB + 4 + d]); };
  auto bar_desc_empty = [&](int d) { return smem_addr(&bars[NB + 4 + kDescRing + d]); };
  auto bar_recv = [&](int pass) { return smem_addr(&bars[NB + 4 + 2 * kDescRing + pass]); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + lay.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + lay.misc + 4);
  int32_t* end_sm = reinterpret_cast<int32_t*>(smem + lay.misc + 8);
  float* qscale_sm = reinterpret_cast<float*>(smem + lay.misc + 12);
  SubBlockSrc* desc = reinterpret_cast<SubBlockSrc*>(smem + lay.desc);
  int32_t* sorted = reinterpret_cast<int32_t*>(smem + lay.sorted);
  int32_t* sidx = reinterpret_cast<int32_t*>(smem + lay.sidx);
  float* lg = reinterpret_cast<float*>(smem + lay.lg);

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_full(s), kLoaderThreads / 32);
      mbar_init(bar_empty(s), 1);
    }
    for (int d = 0; d < kDescRing; ++d) {
      mbar_init(bar_desc_full(d), 1);
      mbar_init(bar_desc_empty(d), kLoaderThreads / 32);
    }
    for (int a = 0; a < NA; ++a) {
      mbar_init(bar_acc_full(a), 1);
      mbar_init(bar_acc_empty(a), kEpilogueThreads / 32);
    }
    mbar_init(bar_q_full, 1);
    mbar_init(bar_drain, 1);
    mbar_init(bar_drain + 8, 1);
    mbar_init(bar_setup, 1);
    mbar_init(bar_recv(0), 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  // half of a cluster barrier: its other half, before the first store into
  // another CTA, makes that CTA's barriers initialised
  cluster_arrive();
  if (tid == 0) SMQ_MARK(0);
  // Until the previous kernel of the stream has finished, nothing it may have
  // written is read: the row's inputs are only prefetched into L2 (address
  // translations included), so that the loads after the wait hit there.
  if (warp == 0) {
    if (lane * 32 < p.ncb) prefetch_l2(p.candidate_blocks + static_cast<int64_t>(r) * p.ncb + lane * 32);
    if (lane == 0) prefetch_l2(p.row_ke + r);
    if (lane == 1 && p.row_indices) prefetch_l2(p.row_indices + r);
    if (lane == 2) prefetch_l2(p.q_scale + r);
    if (lane == 3 && !p.fused) prefetch_l2(p.end + r);
    if (lane == 4) prefetch_l2(p.weights + static_cast<int64_t>(r) * H);
    if (!p.fused)
      for (int i = lane * 32; i < p.nsb; i += 32 * 32) prefetch_l2(p.sparse_indices + static_cast<int64_t>(r) * p.nsb + i);
  } else if (warp == kQueryWarp && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tma_2d(&tm_q, 0, r * H);
  } else if (warp == 2 && rank == 0) {
    // the rows this cluster writes: their first lines (and address translations)
    if (lane == 0) prefetch_l2(p.topk_out + static_cast<int64_t>(r) * p.topk_ld);
    if (lane == 1 && p.col_indices) prefetch_l2(p.col_indices + static_cast<int64_t>(r) * p.topk);
    if (lane == 2 && p.fused) prefetch_l2(p.sparse_indices_out + static_cast<int64_t>(r) * p.nsb);
    if (lane == 3 && p.fused) prefetch_l2(p.end_out + r);
    if (lane == 4 && p.logits_out) prefetch_l2(p.logits_out + static_cast<int64_t>(r) * S);
  } else if (warp >= 6 && warp < 10) {
    // the block-table row of request r (the row's request when row_indices is the identity)
    const int32_t* bt = p.block_table + static_cast<int64_t>(r < p.bt_rows ? r : 0) * p.bt_stride;
    for (int i = (tid - 6 * 32) * 32; i < p.bt_stride; i += kLoaderThreads * 32) prefetch_l2(bt + i);
  }
  griddep_launch_dependents();
  griddep_wait();
  if (tid == 0) SMQ_MARK(1);

  // this CTA's tiles of the row
  int bound = p.fused ? p.row_ke[r] : p.end[r];
  bound = bound < 0 ? 0 : (bound > S ? S : bound);
  const int T = (bound + kTileM - 1) / kTileM;
  const int t0 = static_cast<int>(static_cast<int64_t>(T) * rank / C);
  const int n = static_cast<int>(static_cast<int64_t>(T) * (rank + 1) / C) - t0;
  const int c0 = t0 * kTileM;  // the first sparse column of this CTA
  if (tid == 0) SMQ_MARK(2);
  // the scheduler's loads go out before the set-up below
  int s_ke = 0, s_brow = 0, s_c0 = -1, s_c1 = -1;
  if (warp == 0) {
    s_ke = p.row_ke[r];
    s_brow = p.row_indices ? p.row_indices[r] : r;
    if (p.fused) {
      const int32_t* cb = p.candidate_blocks + static_cast<int64_t>(r) * p.ncb;
      s_c0 = lane < p.ncb ? cb[lane] : -1;
      s_c1 = lane + 32 < p.ncb ? cb[lane + 32] : -1;
    }
  }

  uint32_t tmem = 0;
  if (n > 0) {
    if (warp == 1) tmem_alloc(smem_addr(tmem_slot), p.tmem_cols);
    uint32_t* sf_one = reinterpret_cast<uint32_t*>(smem + lay.sf + kScoreStages * kHalves * 512);
    if (tid < 128) sf_one[tid] = 0x7F7F7F7Fu;
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    tmem = *tmem_slot;
    if (tid == 32) {
      tmem_cp_32x128b_x4(tmem + NA * kHalves * kN + 4 * kHalves * NS, rows16_desc(smem_addr(sf_one)));
      mma_commit(bar_setup);
      if (!mbar_wait(bar_setup, 0, abort_flag, static_cast<uint64_t>(p.wait_ns))) {
        set_status(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tm_sfa = tmem + NA * kHalves * kN;
  const uint32_t tm_sfb = tm_sfa + 4 * kHalves * NS;
  if (tid == 0) SMQ_MARK(3);

  if (warp == 0) {
    // ======================= scheduler =======================
    // The row's expansion into shared memory (expanded here, or the one passed
    // in), then the source addresses of this CTA's sub-blocks, tile by tile.
    const int64_t L = s_ke > 0 ? s_ke : 0;
    const int brow = s_brow;
    const int spb = p.cbs / sbkv;
#ifdef SMQ_TRACE
    if (__shfl_sync(kFullMask, s_c0 ^ s_c1 ^ s_ke ^ s_brow, 0) != 0x5a5a5a5a && lane == 0) SMQ_MARK(17);
#endif
    // Sub-blocks per candidate block and per cache page: shifts where they are
    // powers of two (the usual case), divisions otherwise.
    const int spp = p.page_size / sbkv;
    const int spb_sh = (spb & (spb - 1)) == 0 ? __ffs(spb) - 1 : -1;
    const int spp_sh = (spp & (spp - 1)) == 0 ? __ffs(spp) - 1 : -1;
    auto div_spb = [&](int x) { return spb_sh >= 0 ? x >> spb_sh : x / spb; };
    auto div_spp = [&](int x) { return spp_sh >= 0 ? x >> spp_sh : x / spp; };
    int e = 0, nkept = 0;
    if (p.fused) {
      const int cols = expand_row_in_warp(p.ncb, p.cbs, L, s_c0, s_c1, sorted, &nkept, lane);
      if (lane == 0) SMQ_MARK(18);
      e = cols < 0 ? 0 : (cols > S ? S : cols);
    } else {
      e = p.end[r];
      e = e < 0 ? 0 : (e > S ? S : e);
      for (int slot = lane; slot < p.nsb; slot += 32) sidx[slot] = p.sparse_indices[static_cast<int64_t>(r) * p.nsb + slot];
    }
    // the row's sparse sub-block list from the sorted blocks (fused): after
    // the first block-table loads, off the path to the first tile
    auto fill_sidx = [&]() {
      for (int slot = lane; slot < p.nsb; slot += 32) {
        const int k = div_spb(slot);
        int v = -1;
        if (k < nkept) {
          const int sub = sorted[k] * spb + (slot - k * spb);
          if (static_cast<int64_t>(sub) * sbkv < L) v = sub;
        }
        sidx[slot] = v;
      }
    };
    if (lane == 0) st_volatile_s32(end_sm, e);
    if (lane == 0) SMQ_MARK(4);
    __syncwarp();  // sidx (passed-in expansion) or sorted (fused) is read by every lane below
    bool sidx_ready = !p.fused;
    bool owner = p.fused && rank == 0;  // writes the row's expansion once its first tiles are published
    bool ok = true;
    int it = 0;
    const int tiles_per_batch = 32 / spt;
    for (int tb = 0; tb < n && ok; tb += tiles_per_batch) {
      const int tl = tb + lane / spt;  // local tile
      const int sub = lane % spt;
      const int col_sub = (t0 + tl) * spt + sub;
      const bool want = tl < n && col_sub * sbkv < e;
      int pg = -1, tok = 0;
      if (want) {
        // columns below end lie in the leading sub-blocks of the kept blocks, all valid
        int sb;
        if (p.fused) {
          const int k = div_spb(col_sub);
          sb = sorted[k] * spb + (col_sub - k * spb);
        } else {
          sb = sidx[col_sub];
        }
        const int slot = div_spp(sb);
        tok = (sb - slot * spp) * sbkv;
        if (sb >= 0 && brow >= 0 && brow < p.bt_rows && slot < p.bt_stride)
          pg = p.block_table[static_cast<int64_t>(brow) * p.bt_stride + slot];
      }
      int ntok = 0, trow = 0, tpage = 0;
      const uint8_t* vsrc = nullptr;
      const uint8_t* ssrc = nullptr;
      if (want) {
        if (pg >= 0 && pg < p.num_pages) {
          const uint8_t* base = p.k_cache + static_cast<int64_t>(pg) * p.page_bytes;
          vsrc = base + tok * (kHeadDim / 2);
          ssrc = base + p.page_size * (kHeadDim / 2) + tok * kScaleWordBytes;
          trow = tok;
          tpage = pg;
          ntok = sbkv;
        } else {
          set_status(p.status, kStatusBounds);
        }
      }
      for (int k = 0; k < tiles_per_batch; ++k) {
        if (tb + k >= n) break;
        const int base = k * spt;
        const int dslot = it % kDescRing;
        bool e_ok = true;
        if (lane == 0) e_ok = mbar_wait(bar_desc_empty(dslot), ((it / kDescRing) & 1) ^ 1, abort_flag, static_cast<uint64_t>(p.wait_ns));
        ok = __shfl_sync(kFullMask, e_ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        if (lane >= base && lane < base + spt)
          put_src(&desc[dslot * kMaxSubsPerTile + (lane - base)], vsrc, ssrc, trow, tpage, ntok);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_desc_full(dslot));
        if (lane == 0 && it == 0) SMQ_MARK(5);
        if (lane == 0 && it == n - 1) SMQ_MARK(6);
        ++it;
      }
      if (!sidx_ready) {
        fill_sidx();
        sidx_ready = true;
        __syncwarp();
      }
      if (owner) {
        for (int slot = lane; slot < p.nsb; slot += 32)
          p.sparse_indices_out[static_cast<int64_t>(r) * p.nsb + slot] = sidx[slot];
        if (lane == 0) p.end_out[r] = e;
        owner = false;
      }
    }
    if (!sidx_ready) {  // a CTA without a tile (or one that gave up) still holds the row's list for the top-k
      fill_sidx();
      __syncwarp();
    }
    if (owner) {  // a row with no tile in this CTA
      for (int slot = lane; slot < p.nsb; slot += 32)
        p.sparse_indices_out[static_cast<int64_t>(r) * p.nsb + slot] = sidx[slot];
      if (lane == 0) p.end_out[r] = e;
    }
    if (!ok) {
      set_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    __syncwarp();
  } else if (warp == kQueryWarp) {
    // ======================= query loader =======================
    if (lane == 0 && n > 0) {
      *qscale_sm = p.q_scale[r];
      mbar_arrive_expect_tx(bar_q_full, kN * kRowBytes + H * 2);
      tma_load_2d(smem_addr(smem + lay.q), &tm_q, 0, r * H, bar_q_full);
      bulk_load(smem_addr(smem + lay.w), p.weights + static_cast<int64_t>(r) * H, H * 2, bar_q_full);
      const volatile int never = 0;
      mbar_wait(bar_q_full, 0, &never, static_cast<uint64_t>(p.wait_ns));  // the copies land before the CTA can exit
    }
    __syncwarp();
  } else if (warp == 1 || warp == kMmaWarp1) {
    // ======================= MMA issuers (alternate tiles) =======================
    const int par = warp == 1 ? 0 : 1;
    if (lane == 0 && n > 0) {
      uint32_t idesc[4];
      for (int g = 0; g < 4; ++g) idesc[g] = mxf8f6f4_idesc(kE2M1, kE4M3, kMmaM, kN, g, g);
      bool ok = mbar_wait(bar_q_full, 0, abort_flag, static_cast<uint64_t>(p.wait_ns));
      if (warp == 1) SMQ_MARK(20);
      const uint64_t bdesc = sw128_desc(smem_addr(smem + lay.q));
      for (int it = 0; it < n && ok; ++it) {
        if (NA > 1 ? ((it & 1) != par) : (par != 0)) continue;
        const int s = it % NS;
        const int a = it % NA;
        ok = mbar_wait(bar_full(s), (it / NS) & 1, abort_flag, static_cast<uint64_t>(p.wait_ns)) &&
             mbar_wait(bar_acc_empty(a), ((it / NA) & 1) ^ 1, abort_flag, static_cast<uint64_t>(p.wait_ns));
        if (!ok) break;
        tc_fence_after();
        const uint32_t stage_addr = smem_addr(smem + lay.kv + s * (kTileM * kRowBytes));
        for (int h = 0; h < kHalves; ++h) {
          const uint32_t sfa = tm_sfa + 4 * (s * kHalves + h);
          tmem_cp_32x128b_x4(sfa, rows16_desc(smem_addr(smem + lay.sf + (s * kHalves + h) * 512)));
          const uint64_t adesc = sw128_desc(stage_addr + h * (kMmaM * kRowBytes));
          for (int g = 0; g < 4; ++g)
            mma_mxf8f6f4(tmem + (a * kHalves + h) * kN, adesc + 2 * g, bdesc + 2 * g, idesc[g], sfa, tm_sfb, g > 0);
        }
        mma_commit(bar_acc_full(a));
        if (it == 0) SMQ_MARK(9);
        if (it == n - 1) SMQ_MARK(10);
      }
      if (!ok) {
        set_status(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      const uint32_t drain = bar_drain + 8 * par;
      mma_commit(drain);
      const volatile int never = 0;
      mbar_wait(drain, 0, &never, static_cast<uint64_t>(p.wait_ns));
    }
    __syncwarp();
  } else if (warp < 6) {
    // ======================= epilogue (warps 2..5) =======================
    // One TMEM lane (one key position of each half) per thread. The logit goes
    // to shared memory (and the caller's logits_out), and its top 12 bits are
    // counted for the top-k.
    const int q4 = warp & 3;
    const int m = 32 * q4 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
    bool ok = n > 0 ? warp_wait(bar_q_full, 0, abort_flag, static_cast<uint64_t>(p.wait_ns)) : true;
    // head weights: packed pairs (2j, 2j + 1) for the packed FMA at 64 heads;
    // scalars at 128 heads (pairs would not fit the registers)
    constexpr bool kPacked = kN == 64;
    uint64_t w2[kPacked ? kN / 2 : 1];
    float w[kPacked ? 1 : kN];
    const uint16_t* wsm = reinterpret_cast<const uint16_t*>(smem + lay.w);
    if constexpr (kPacked) {
#pragma unroll
      for (int j = 0; j < kN / 2; ++j)
        w2[j] = pack2(2 * j < H ? bf16_to_f32(wsm[2 * j]) : 0.f, 2 * j + 1 < H ? bf16_to_f32(wsm[2 * j + 1]) : 0.f);
    } else {
#pragma unroll
      for (int h = 0; h < kN; ++h) w[h] = h < H ? bf16_to_f32(wsm[h]) : 0.f;
    }
    const float qs = n > 0 ? *qscale_sm : 0.f;
    float* lout = p.logits_out ? p.logits_out + static_cast<int64_t>(r) * S : nullptr;
    uint16_t* lout16 = p.logits_bf16 ? p.logits_bf16 + static_cast<int64_t>(r) * S : nullptr;
    int e = 0;
    for (int ie = 0; ie < n && ok; ++ie) {
      const int a = ie % NA;
      ok = warp_wait(bar_acc_full(a), (ie / NA) & 1, abort_flag, static_cast<uint64_t>(p.wait_ns));
      if (!ok) break;
      if (ie == 0) e = ld_volatile_s32(end_sm);  // written before the first tile was published
      if (warp == 2 && lane == 0) mbar_arrive(bar_empty(ie % NS));
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < kHalves; ++h) {
        uint64_t lo = 0, hi = 0;  // heads h mod 4: two packed pairs of partial sums (64 heads)
        float acc4[4] = {0.f, 0.f, 0.f, 0.f};  // or four scalars (128 heads)
        const uint32_t tacc = tmem + (a * kHalves + h) * kN + lane_base;
#pragma unroll
        for (int c = 0; c < kN; c += 32) {
          uint32_t v0[16], v1[16];
          tmem_ld16(tacc + c, v0);
          tmem_ld16(tacc + c + 16, v1);
          tmem_wait_ld();
          if (h == kHalves - 1 && c + 32 >= kN) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_acc_empty(a));
          }
          if constexpr (kPacked) {
#pragma unroll
            for (int hh = 0; hh < 16; hh += 4) {
              relu2_fma2(lo, w2[(c + hh) / 2], __uint_as_float(v0[hh]), __uint_as_float(v0[hh + 1]));
              relu2_fma2(hi, w2[(c + hh) / 2 + 1], __uint_as_float(v0[hh + 2]), __uint_as_float(v0[hh + 3]));
            }
#pragma unroll
            for (int hh = 0; hh < 16; hh += 4) {
              relu2_fma2(lo, w2[(c + 16 + hh) / 2], __uint_as_float(v1[hh]), __uint_as_float(v1[hh + 1]));
              relu2_fma2(hi, w2[(c + 16 + hh) / 2 + 1], __uint_as_float(v1[hh + 2]), __uint_as_float(v1[hh + 3]));
            }
          } else {
#pragma unroll
            for (int hh = 0; hh < 16; ++hh)
              acc4[hh & 3] = fmaf(w[c + hh], fmaxf(__uint_as_float(v0[hh]), 0.f), acc4[hh & 3]);
#pragma unroll
            for (int hh = 0; hh < 16; ++hh)
              acc4[hh & 3] = fmaf(w[c + 16 + hh], fmaxf(__uint_as_float(v1[hh]), 0.f), acc4[hh & 3]);
          }
        }
        // the head sums (twice them, exactly, from the packed form)
        const float2 l2 = kPacked ? unpack2(lo) : make_float2(acc4[0], acc4[1]);
        const float2 h2 = kPacked ? unpack2(hi) : make_float2(acc4[2], acc4[3]);
        const float qscale = kPacked ? 0.5f * qs : qs;
        const float logit = ((l2.x + l2.y) + (h2.x + h2.y)) * qscale;
        const int lc = ie * kTileM + h * kMmaM + m;  // local column
        const int col = c0 + lc;
        if (col < e) lg[col] = logit;
        if (lout && col < S) lout[col] = col < e ? logit : -INFINITY;
        if (lout16 && col < S) lout16[col] = col < e ? to_bf16(logit) : kBf16NegInf;
      }
      if (warp == 2 && lane == 0 && ie == 0) SMQ_MARK(11);
      if (warp == 2 && lane == 0 && ie == n - 1) SMQ_MARK(12);
    }
    if (!ok) {
      set_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
  } else if (warp >= 6 && warp < 10) {
    // ======================= loaders (warps 6..9) =======================
    // Coalesced 16-byte loads two tiles ahead into registers, then stores into
    // the MMA's padded containers (as in the persistent kernel).
    constexpr int kChunks = kTileM / 32;
    const int q4 = warp & 3;
    const int m = 32 * q4 + lane;
    const uint32_t sf_base = smem_addr(smem + lay.sf);
    const uint32_t kv_base = smem_addr(smem + lay.kv);
    const int vch = m & 3;
    int vu[kChunks], vtk[kChunks];
#pragma unroll
    for (int k8 = 0; k8 < kChunks; ++k8) {
      const int pos = (m >> 2) + 32 * k8;
      vu[k8] = pos / sbkv;
      vtk[k8] = pos % sbkv;
    }
    int su[kHalves], stk[kHalves];
#pragma unroll
    for (int h = 0; h < kHalves; ++h) {
      su[h] = (m + h * kMmaM) / sbkv;
      stk[h] = (m + h * kMmaM) % sbkv;
    }
    uint4 v[2][kChunks];
    uint32_t sw[2][kHalves];
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
      for (int k8 = 0; k8 < kChunks; ++k8) v[k][k8] = make_uint4(0u, 0u, 0u, 0u);
    auto store_tile = [&](const uint4 (&vv)[kChunks], const uint32_t (&ss)[kHalves], int j) {
      const int s = j % NS;
      const uint32_t stage = kv_base + s * (kTileM * kRowBytes);
#pragma unroll
      for (int k8 = 0; k8 < kChunks; ++k8) {
        const int pos = (m >> 2) + 32 * k8;
        const uint32_t dst = stage + static_cast<uint32_t>(pos) * kRowBytes;
        const uint32_t swz = static_cast<uint32_t>(pos & 7);
        sts_v2(dst + (((2 * vch) ^ swz) << 4), vv[k8].x, vv[k8].y);
        sts_v2(dst + (((2 * vch + 1) ^ swz) << 4), vv[k8].z, vv[k8].w);
      }
#pragma unroll
      for (int h = 0; h < kHalves; ++h) sts_u32(sf_base + (s * kHalves + h) * 512 + 16 * lane + 4 * q4, ss[h]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && !(j == p.stall_tile && blockIdx.x == 0)) mbar_arrive(bar_full(s));
      if (warp == 6 && lane == 0 && j == 0) SMQ_MARK(7);
      if (warp == 6 && lane == 0 && j == n - 1) SMQ_MARK(8);
    };
    auto load_tile = [&](uint4 (&vv)[kChunks], uint32_t (&ss)[kHalves], int i) {
      const SubBlockSrc* dring = desc + (i % kDescRing) * kMaxSubsPerTile;
#pragma unroll
      for (int k8 = 0; k8 < kChunks; ++k8) {
        const SubBlockSrc d = get_src(dring + vu[k8]);
        ldg_stream_v4_if(vv[k8], d.values + static_cast<int64_t>(vtk[k8]) * (kHeadDim / 2) + 16 * vch,
                         d.values != nullptr && vtk[k8] < d.positions);
      }
#pragma unroll
      for (int h = 0; h < kHalves; ++h) {
        const SubBlockSrc ds = get_src(dring + su[h]);
        ss[h] = 0x7F7F7F7Fu;
        ldg_stream_u32_if(ss[h], ds.scales + static_cast<int64_t>(stk[h]) * kScaleWordBytes,
                          ds.values != nullptr && stk[h] < ds.positions);
      }
    };
    bool ok = true;
    // Two register slots: each slot's tile is stored, then the slot takes its
    // next tile at once, so that the next load is out before the other slot's
    // stores.
    for (int i0 = 0; i0 < n + 2 && ok; i0 += 2) {
      const int j0 = i0 - 2;
      if (j0 >= 0 && j0 < n) {
        const int jl = j0 + 1 < n ? j0 + 1 : j0;
        ok = warp_wait(bar_empty(jl % NS), ((jl / NS) & 1) ^ 1, abort_flag, static_cast<uint64_t>(p.wait_ns));
        if (!ok) break;
        store_tile(v[0], sw[0], j0);
      }
      if (i0 < n) {
        ok = warp_wait(bar_desc_full(i0 % kDescRing), (i0 / kDescRing) & 1, abort_flag, static_cast<uint64_t>(p.wait_ns));
        if (!ok) break;
        if (warp == 6 && lane == 0 && i0 == 0) SMQ_MARK(19);
        load_tile(v[0], sw[0], i0);
      }
      if (j0 >= 0 && j0 + 1 < n) store_tile(v[1], sw[1], j0 + 1);
      if (i0 + 1 < n) {
        ok = warp_wait(bar_desc_full((i0 + 1) % kDescRing), ((i0 + 1) / kDescRing) & 1, abort_flag,
                       static_cast<uint64_t>(p.wait_ns));
        if (!ok) break;
        load_tile(v[1], sw[1], i0 + 1);
      }
      if (i0 < n) {
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar_desc_empty(i0 % kDescRing));
          if (i0 + 1 < n) mbar_arrive(bar_desc_empty((i0 + 1) % kDescRing));
        }
      }
    }
    if (!ok) {
      set_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
  }

  // ---- teardown ----
  tc_fence_before();
  __syncthreads();
  if (tid == 0) SMQ_MARK(13);
  if (n > 0 && warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }

  // ---- top-k: the other CTAs' logits into CTA 0, which selects ----
  // Each other CTA stores its valid logits into CTA 0's row of logits
  // (asynchronous stores completing on CTA 0's barrier) and leaves. CTA 0
  // then selects on shared memory alone. Every CTA computes the same `end`, so
  // all take the same branch.
  const int e = ld_volatile_s32(end_sm);
  const int k = p.topk;
  int32_t* out = p.topk_out + static_cast<int64_t>(r) * p.topk_ld;
  int32_t* colo = p.col_indices ? p.col_indices + static_cast<int64_t>(r) * p.topk : nullptr;
  if (rank == C - 1 && p.logits_out)  // columns past the last tile
    for (int c = T * kTileM + tid; c < S; c += kScoreThreads) p.logits_out[static_cast<int64_t>(r) * S + c] = -INFINITY;
  if (rank == C - 1 && p.logits_bf16)
    for (int c = T * kTileM + tid; c < S; c += kScoreThreads) p.logits_bf16[static_cast<int64_t>(r) * S + c] = kBf16NegInf;
  auto valid_cols = [&](int cr) {  // valid columns of CTA cr: [T cr / C * 256, ...) below e
    const int a = static_cast<int>(static_cast<int64_t>(T) * cr / C) * kTileM;
    const int b = static_cast<int>(static_cast<int64_t>(T) * (cr + 1) / C) * kTileM;
    const int hi = b < e ? b : e;
    return hi > a ? hi - a : 0;
  };
  const bool select = e > k;
  cluster_wait();  // every CTA of the cluster has initialised its barriers
  if (tid == 0) SMQ_MARK(21);
  if (rank != 0) {
    if (select) {
      const int nv = valid_cols(rank);
      const uint32_t src = smem_addr(lg + c0), bar = bar_recv(0);
      for (int i = tid; 4 * i + 3 < nv; i += kScoreThreads)
        st_async_v4(src + 16u * i, 0, *reinterpret_cast<const uint4*>(lg + c0 + 4 * i), bar);
      for (int c = (nv & ~3) + tid; c < nv; c += kScoreThreads)
        st_async_u32(src + 4u * c, 0, __float_as_uint(lg[c0 + c]), bar);
    }
    return;
  }
  if (!select) {  // every valid column is selected, in column order
    const int sb_shift = 31 - __clz(sbkv);
    for (int c = tid; c < k; c += kScoreThreads) {
      out[c] = c < e ? (sidx[c >> sb_shift] << sb_shift) | (c & (sbkv - 1)) : -1;
      if (colo) colo[c] = c < e ? c : -1;
    }
    if (tid == 0) SMQ_MARK(16);
    return;
  }
  int incoming = 0;
  for (int cr = 1; cr < C; ++cr) incoming += valid_cols(cr);
  if (tid == 0) mbar_arrive_expect_tx(bar_recv(0), static_cast<uint32_t>(incoming) * 4u);
  fence_proxy_async_smem();  // the key stages (written for the tensor core) become plain scratch
  uint8_t* scr = smem + lay.kv;
  TopkScratch sm;
  sm.hist = reinterpret_cast<uint32_t*>(scr);
  sm.bsum = nullptr;
  sm.wsum = reinterpret_cast<int*>(scr + kTopkBins * 4);
  sm.chunk = reinterpret_cast<uint32_t*>(sm.wsum + 32);
  sm.sel = reinterpret_cast<int*>(sm.chunk + 32 * 32);
  sm.sidx = sidx;
  if (!warp_wait(bar_recv(0), 0, abort_flag, static_cast<uint64_t>(p.wait_ns))) set_status(p.status, kStatusTimeout);
  if (tid == 0) SMQ_MARK(14);
  select_topk<kScoreThreads, kJ, true, true>(lg, S, end_sm, k, nullptr, p.nsb, sbkv, out, colo, nullptr, nullptr, sm);
  if (tid == 0) SMQ_MARK(16);
}

// ===========================================================================
// Candidate source: dense layout, then block maxima and the best blocks.
// ===========================================================================
// One warp per row: sub-block j of the row's context is sparse sub-block j
// (every position a column, in order); end = the context length.
__global__ void __launch_bounds__(256) source_layout_kernel(const __grid_constant__ SourceParams p) {
  griddep_launch_dependents();
  griddep_wait();
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= p.rows) return;
  int L = p.row_ke[r];
  if (L > p.num_cols) {
    if (lane == 0) set_status(p.status, kStatusBounds);  // a context longer than the call's bound
    L = p.num_cols;
  }
  L = L < 0 ? 0 : L;
  int32_t* si = p.sparse_indices + static_cast<int64_t>(r) * p.nsb;
  for (int j = lane; j < p.nsb; j += 32) si[j] = j * p.sbkv < L ? j : -1;
  if (lane == 0) p.end[r] = L;
}

// One CTA per row: block b's score is the largest logit of its positions
// below the row's end; the ncb best blocks (ties to the lower id) come out in
// that order, then -1. Keys (score order, then the complement of the block
// id) are sorted in shared memory, descending, by a bitonic network.
__global__ void __launch_bounds__(512) source_select_kernel(const __grid_constant__ SourceParams p) {
  extern __shared__ uint64_t src_keys[];
  griddep_launch_dependents();
  griddep_wait();
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int L = p.end[r];
  L = L < 0 ? 0 : (L > p.num_cols ? p.num_cols : L);
  const int nb = (L + p.cbs - 1) / p.cbs;
  int n2 = 1;
  while (n2 < nb) n2 <<= 1;
  const float* lg = p.logits + static_cast<int64_t>(r) * p.num_cols;
  for (int b = warp; b < nb; b += 16) {  // a warp per block
    float m = -INFINITY;
    const int lo = b * p.cbs, hi = min(L, lo + p.cbs);
    for (int c = lo + lane; c < hi; c += 32) m = fmaxf(m, __ldcg(lg + c));
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, o));
    if (lane == 0) {
      src_keys[b] = (static_cast<uint64_t>(ordered_key(m)) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(b));
      if (p.block_scores) p.block_scores[static_cast<int64_t>(r) * p.max_blocks + b] = m;
    }
  }
  for (int b = nb + tid; b < n2; b += 512) src_keys[b] = 0;  // below every block
  if (p.block_scores)
    for (int b = nb + tid; b < p.max_blocks; b += 512) p.block_scores[static_cast<int64_t>(r) * p.max_blocks + b] = -INFINITY;
  __syncthreads();
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < n2; i += 512) {
        const int x = i ^ j;
        if (x > i) {
          const uint64_t a = src_keys[i], b = src_keys[x];
          const bool desc = (i & k) == 0;  // descending runs where bit k of i is clear
          if ((a < b) == desc) {
            src_keys[i] = b;
            src_keys[x] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  int32_t* out = p.candidate_blocks + static_cast<int64_t>(r) * p.ncb;
  for (int i = tid; i < p.ncb; i += 512)
    out[i] = i < nb ? static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(src_keys[i] & 0xFFFFFFFFu)) : -1;
}

// ===========================================================================
// Launchers
// ===========================================================================
cudaError_t prepare_kernels(int n_mma) {
  const int max_smem = 232448;  // 227 KB opt-in per block
  cudaError_t err;
  // one shared-memory carveout for every kernel of a step, so that consecutive
  // kernels never wait for the SM to re-split L1 and shared memory
  const void* all[] = {reinterpret_cast<const void*>(&score_kernel<true, 64, true>),
                       reinterpret_cast<const void*>(&score_kernel<true, 64, false>),
                       reinterpret_cast<const void*>(&score_kernel<false, 64, false>),
                       reinterpret_cast<const void*>(&score_kernel<true, 128, true>),
                       reinterpret_cast<const void*>(&score_kernel<true, 128, false>),
                       reinterpret_cast<const void*>(&score_kernel<false, 128, false>),
                       reinterpret_cast<const void*>(&score_kernel<true, 64, true, true>),
                       reinterpret_cast<const void*>(&topk_kernel<256, 8>),
                       reinterpret_cast<const void*>(&topk_kernel<256, 16>),
                       reinterpret_cast<const void*>(&topk_kernel<512, 16>),
                       reinterpret_cast<const void*>(&topk_kernel<512, 32>),
                       reinterpret_cast<const void*>(&topk_warp_kernel),
                       reinterpret_cast<const void*>(&expand_kernel),
                       reinterpret_cast<const void*>(&gather_kernel),
                       reinterpret_cast<const void*>(&source_layout_kernel),
                       reinterpret_cast<const void*>(&source_select_kernel)};
  for (const void* f : all) {
    err = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (err != cudaSuccess) return err;
  }
  const void* score[] = {reinterpret_cast<const void*>(&score_kernel<true, 64, true>),
                         reinterpret_cast<const void*>(&score_kernel<true, 64, false>),
                         reinterpret_cast<const void*>(&score_kernel<false, 64, false>),
                         reinterpret_cast<const void*>(&score_kernel<true, 64, true, true>),
                         reinterpret_cast<const void*>(&score_kernel<true, 128, true>),
                         reinterpret_cast<const void*>(&score_kernel<true, 128, false>),
                         reinterpret_cast<const void*>(&score_kernel<false, 128, false>)};
  for (int i = 0; i < 7; ++i) {
    if ((i < 4) != (n_mma == 64)) continue;
    err = cudaFuncSetAttribute(score[i], cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (err != cudaSuccess) return err;
  }
  const void* rc[] = {reinterpret_cast<const void*>(&row_cluster_kernel<64, 11>),
                      reinterpret_cast<const void*>(&row_cluster_kernel<64, 22>),
                      reinterpret_cast<const void*>(&row_cluster_kernel<128, 11>),
                      reinterpret_cast<const void*>(&row_cluster_kernel<128, 22>)};
  for (int i = 0; i < 4; ++i) {
    if ((i < 2) != (n_mma == 64)) continue;
    err = cudaFuncSetAttribute(rc[i], cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(rc[i], cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (err != cudaSuccess) return err;
  }
  if (err != cudaSuccess) return err;

  err = cudaFuncSetAttribute(source_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSourceMaxBlocks * 8);
  if (err != cudaSuccess) return err;
  // the widest rows of the warp top-k: kTopkWarpMaxCols columns in sub-blocks of 16
  err = cudaFuncSetAttribute(topk_warp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(topk_warp_smem(kTopkWarpMaxCols / 16)));
  if (err != cudaSuccess) return err;
  return cudaFuncSetAttribute(expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kExpandWarps * 2 * 512 * 4);
}

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel of the stream finishes; it waits (griddepcontrol.wait)
// before touching anything an earlier kernel wrote.
template <typename P>
cudaError_t launch_pdl(void (*kernel)(P), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                       const P& params) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, params);
}

template <typename... A>
cudaError_t launch_pdl_n(void (*kernel)(A...), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                         const A&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_expand(const ExpandParams& p, cudaStream_t stream) {
  const int grid = (p.rows + kExpandWarps - 1) / kExpandWarps;
  const size_t smem = static_cast<size_t>(kExpandWarps) * 2 * p.ncb * sizeof(int32_t);
  return launch_pdl(expand_kernel, grid, kExpandWarps * 32, smem, stream, p);
}

cudaError_t launch_score(const ScoreParams& p, bool paged, bool copy, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                         int grid, size_t smem, cudaStream_t stream) {
  const bool stat = paged && p.fused;
  if (p.n_mma == 64) {
    if (stat && copy)
      return launch_pdl_n(score_kernel<true, 64, true, true>, grid, kScoreThreads, smem, stream, p, tm_q, tm_k);
    if (stat) return launch_pdl_n(score_kernel<true, 64, true>, grid, kScoreThreads, smem, stream, p, tm_q, tm_k);
    if (paged) return launch_pdl_n(score_kernel<true, 64, false>, grid, kScoreThreads, smem, stream, p, tm_q, tm_k);
    return launch_pdl_n(score_kernel<false, 64, false>, grid, kScoreThreads, smem, stream, p, tm_q, tm_k);
  }
  if (stat) return launch_pdl_n(score_kernel<true, 128, true>, grid, kScoreThreads, smem, stream, p, tm_q, tm_k);
  if (paged) return launch_pdl_n(score_kernel<true, 128, false>, grid, kScoreThreads, smem, stream, p, tm_q, tm_k);
  return launch_pdl_n(score_kernel<false, 128, false>, grid, kScoreThreads, smem, stream, p, tm_q, tm_k);
}

template <int kN, int kJ>
cudaError_t launch_rc(const ScoreParams& p, const CUtensorMap& tm_q, size_t smem, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.rows) * static_cast<unsigned>(p.cluster));
  cfg.blockDim = dim3(kScoreThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(p.cluster);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, row_cluster_kernel<kN, kJ>, p, tm_q);
}

cudaError_t launch_row_cluster(const ScoreParams& p, const CUtensorMap& tm_q, size_t smem, cudaStream_t stream) {
  const bool narrow = p.num_cols <= kScoreThreads * 11;  // keys per thread of the selection
  static_assert(kScoreThreads * 22 >= kRowClusterMaxCols, "the widest row's keys fit the selection");
  if (p.n_mma == 64) return narrow ? launch_rc<64, 11>(p, tm_q, smem, stream) : launch_rc<64, 22>(p, tm_q, smem, stream);
  return narrow ? launch_rc<128, 11>(p, tm_q, smem, stream) : launch_rc<128, 22>(p, tm_q, smem, stream);
}

cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(p.nsb) * 4;
  // narrow rows: a warp per row (float4 reads of the logits)
  if (p.num_cols <= kTopkWarpMaxCols && (reinterpret_cast<uintptr_t>(p.logits) & 15u) == 0 && p.num_cols % 4 == 0) {
    const int grid = p.rows < p.num_sms ? p.rows : p.num_sms;
    return launch_pdl(topk_warp_kernel, static_cast<unsigned>(grid), 32 * kTopkWarps, topk_warp_smem(p.nsb), stream, p);
  }
  if (p.num_cols <= 8 * 256) return launch_pdl(topk_kernel<256, 8>, p.rows, 256, smem, stream, p);
  if (p.num_cols <= 16 * 256) return launch_pdl(topk_kernel<256, 16>, p.rows, 256, smem, stream, p);
  if (p.num_cols <= 16 * 512) return launch_pdl(topk_kernel<512, 16>, p.rows, 512, smem, stream, p);
  static_assert(32 * 512 >= kMaxSparseCols, "the widest top-k kernel covers every row");
  return launch_pdl(topk_kernel<512, 32>, p.rows, 512, smem, stream, p);
}

cudaError_t launch_source_layout(const SourceParams& p, cudaStream_t stream) {
  return launch_pdl(source_layout_kernel, static_cast<unsigned>((p.rows + 7) / 8), 256, 0, stream, p);
}

cudaError_t launch_source_select(const SourceParams& p, cudaStream_t stream) {
  int n2 = 1;
  while (n2 < p.max_blocks) n2 <<= 1;
  return launch_pdl(source_select_kernel, static_cast<unsigned>(p.rows), 512, static_cast<size_t>(n2) * 8, stream, p);
}

cudaError_t launch_gather(const GatherParams& p, cudaStream_t stream) {
  const int64_t blocks = (p.total_len + 255) / 256;
  return launch_pdl(gather_kernel, static_cast<unsigned>(blocks), 256, 0, stream, p);
}

}  // namespace smq
