// Window-major prefill scoring for sm_103a.
//
// The rows of a prefill chunk draw their candidate blocks from the same
// sequences, so each 128-key window of the gathered workspace is selected by
// many rows. Here the score runs per window: the window's keys (E2M1 values
// unpacked into the MMA's 16-byte containers, UE8M0 scale words) are loaded
// into shared memory once and stay there, and the E4M3 query tiles of the rows
// that selected it stream past, two rows per block-scaled MMA (N = 128, the
// full rate of tcgen05.mma kind::mxf8f6f4). The logits are the same as the
// row-major score kernel's, bit for bit: q_scale * sum_h w_h * max(q_h . k, 0)
// with the same accumulation order, written to the row's sparse column.
//
//   bm_records_kernel  one warp per row: the row's (row, window) records, the
//                      per-window record counts, the row's float weights
//   bm_tilesum_kernel  groups of two records per window, summed per tile of
//   bm_plan_kernel     positions; then numbered window by window (each tile
//                      offset by the tiles before it, scanned within)
//   bm_fill_kernel     one warp per row: each record to its group slot
//   bm_score_kernel    persistent, one CTA per SM over a contiguous range of
//                      groups: a window loader, 3 MMA issuers (which also load
//                      the query tiles) and 24 epilogue warps (which fetch
//                      their rows' params)
//
// The formula is the indexer's score ("sparse_mqa_indexer" docs, the
// SparseMQAIndexer forward's MQA-logits call); the record and group layout is
// in smq_kernels.cuh.
#include "smq_kernels.cuh"
#include "smq_ptx.cuh"

#include <cuda_bf16.h>

namespace smq {

namespace {

constexpr uint32_t kAll = 0xffffffffu;
constexpr uint32_t kTypeE2M1 = 5, kTypeE4M3 = 0;
constexpr int kBmAcc = 3;                                   // TMEM accumulators of kBmN columns
constexpr int kBmN = 128;                                   // MMA N: two rows of 64 heads
constexpr int kBmHeads = 64;
constexpr int kQRowBytes = kBmHeads * 128;                  // one row's query tile
constexpr int kRowParamBytes = kBmRowParams * 4;            // 272
constexpr int kWindowBytes = 128 * 128;                     // 128 keys in 16-byte containers
constexpr int kQPer = kBmStages / kBmAcc;                    // query stages of each MMA issuer
constexpr int kPrmPer = 3;                                  // params slots of each epilogue warp
constexpr int kEpiWarps = 8 * kBmAcc;                        // two warpgroups per accumulator, one per row
constexpr int kSlotBytes = 32 + kRowParamBytes;              // a group's descriptor and one row's params
constexpr int kBmEpiWarp0 = 1 + kBmAcc;                     // first epilogue warp; warp 0 is the stager
constexpr int kRecordWarps = 8;
static_assert(kBmStages % kBmAcc == 0 && kQPer >= 2, "each issuer owns at least two query stages");

struct BmLayout {  // offsets from the 1024-byte aligned base of dynamic shared memory
  static constexpr uint32_t window = 0;                                   // 2 x 16 KB
  static constexpr uint32_t q = 2 * kWindowBytes;                         // kBmStages x 16 KB
  static constexpr uint32_t window_sf = q + kBmStages * 2 * kQRowBytes;   // 2 x 512 B
  static constexpr uint32_t sf_one = window_sf + 2 * 512;                 // 512 B of 0x7F
  static constexpr uint32_t prm = sf_one + 512;                           // kEpiWarps x kPrmPer x kSlotBytes
  static constexpr uint32_t bars = prm + kEpiWarps * kPrmPer * kSlotBytes;
  static constexpr int nbars = 4 + 2 * kBmStages + 3 * kBmAcc;
  static constexpr uint32_t misc = bars + nbars * 8;                      // TMEM address, abort flag
  static constexpr uint32_t bytes = misc + 16;
};
static_assert(BmLayout::prm % 16 == 0 && kSlotBytes % 16 == 0 && kRowParamBytes % 16 == 0,
              "16-byte aligned params");
static_assert(BmLayout::bars % 8 == 0, "mbarriers are 8-byte aligned");
static_assert(kBmAcc * kBmN + 12 * kBmAcc <= 512, "accumulators, each issuer's window and query scales fit in TMEM");

__device__ __forceinline__ void status_or(int32_t* s, int code) { atomicOr(s, code); }
__device__ __forceinline__ float bf16_bits(uint32_t b) { return __uint_as_float(b << 16); }
__device__ __forceinline__ uint16_t round_bf16(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

// Entry j of a row's sparse list: whether it names a sub-block inside the
// workspace, its window u (relative to the row's ks) and its slot there.
struct Entry {
  bool ok;
  int u;
  int slot;
};

__device__ __forceinline__ Entry decode_entry(const int32_t* si, int j, int64_t ks, const BmIndexParams& p, int shift) {
  Entry e;
  const int sb = si[j];
  const int64_t rel = static_cast<int64_t>(sb) << shift;
  const int64_t pos = ks + rel;
  e.ok = sb >= 0 && ks >= 0 && pos < p.total_len;
  e.u = static_cast<int>(rel >> 7);
  e.slot = static_cast<int>((rel & 127) >> shift);
  return e;
}

}  // namespace

// ---------------------------------------------------------------------------
// Index
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kRecordWarps * 32) bm_records_kernel(const __grid_constant__ BmIndexParams p) {
  griddep_launch_dependents();
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kRecordWarps + warp;
  if (r >= p.rows) return;
  // the row's epilogue parameters: its 64 head weights as float, then q_scale
  float* rp = p.rowparams + static_cast<int64_t>(r) * kBmRowParams;
  const uint32_t w2 = reinterpret_cast<const uint32_t*>(p.weights + static_cast<int64_t>(r) * kBmHeads)[lane];
  reinterpret_cast<float2*>(rp)[lane] = make_float2(bf16_bits(w2 & 0xffffu), bf16_bits(w2 >> 16));
  if (lane < 4) rp[kBmHeads + lane] = lane == 0 ? p.q_scale[r] : 0.f;

  int e = p.end[r];
  e = e < 0 ? 0 : (e > p.num_cols ? p.num_cols : e);
  const int shift = 31 - __clz(p.sbkv);  // the sub-block size is a power of two
  const int nent = (e + p.sbkv - 1) >> shift;  // entries holding at least one valid column
  const int64_t ks = p.row_ks[r];
  const int32_t* si = p.sparse_indices + static_cast<int64_t>(r) * p.nsb;
  int nrec = 0;
  Entry prev{false, 0, 0};  // the entry before this chunk
  for (int base = 0; base < nent; base += 32) {
    const int j = base + lane;
    Entry cur{false, 0, 0};
    if (j < nent) {
      cur = decode_entry(si, j, ks, p, shift);
      if (!cur.ok) status_or(p.status, kStatusBounds);
    }
    Entry before;
    before.ok = __shfl_up_sync(kAll, cur.ok ? 1 : 0, 1) != 0;
    before.u = __shfl_up_sync(kAll, cur.u, 1);
    before.slot = __shfl_up_sync(kAll, cur.slot, 1);
    if (lane == 0) before = prev;
    // a record starts at every valid entry that does not continue its
    // predecessor's run (same window, higher slot)
    const bool head = cur.ok && !(before.ok && before.u == cur.u && before.slot < cur.slot);
    const uint32_t heads = __ballot_sync(kAll, head);
    if (head) {
      uint32_t mask = 1u << cur.slot;
      int last = cur.slot;
      for (int t = j + 1; t < nent; ++t) {  // at most 128 / sbkv - 1 steps: the slots rise
        const Entry nx = decode_entry(si, t, ks, p, shift);
        if (!nx.ok || nx.u != cur.u || nx.slot <= last) break;
        mask |= 1u << nx.slot;
        last = nx.slot;
      }
      const int k = nrec + __popc(heads & ((1u << lane) - 1u));
      const int P = static_cast<int>(ks + (static_cast<int64_t>(cur.u) << 7));
      p.rec[static_cast<int64_t>(r) * p.nsb + k] = make_int2(P, static_cast<int>((static_cast<uint32_t>(j) << shift) | (mask << 24)));
      atomicAdd(p.cnt + P, 1);
    }
    nrec += __popc(heads);
    prev.ok = __shfl_sync(kAll, cur.ok ? 1 : 0, 31) != 0;
    prev.u = __shfl_sync(kAll, cur.u, 31);
    prev.slot = __shfl_sync(kAll, cur.slot, 31);
  }
  if (lane == 0) p.nrec[r] = nrec;
}

// Groups of two records per window, windows in position order: cursor[P]
// becomes the first record slot of window P (2 x its first group), and
// cnt[P] the window's ordinal. Positions go in tiles of kScanTile: one kernel
// sums each tile's groups and windows, the next gives each tile its offsets
// (the sums of the tiles before it) and scans the tile.
// Thread t of a tile takes its positions 8 t .. 8 t + 7 (two 16-byte loads).
constexpr int kScanThreads = 256;
constexpr int kScanTile = 8 * kScanThreads;

__device__ __forceinline__ void load_tile_counts(const int32_t* cnt, int64_t total, int64_t i0, int (&c)[8]) {
  if (i0 + 8 <= total) {
    const int4 a = *reinterpret_cast<const int4*>(cnt + i0);
    const int4 b = *reinterpret_cast<const int4*>(cnt + i0 + 4);
    c[0] = a.x; c[1] = a.y; c[2] = a.z; c[3] = a.w;
    c[4] = b.x; c[5] = b.y; c[6] = b.z; c[7] = b.w;
  } else {
#pragma unroll
    for (int x = 0; x < 8; ++x) c[x] = i0 + x < total ? cnt[i0 + x] : 0;
  }
}

// Block-wide exclusive scan of one value per thread; *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kAll, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < kScanThreads / 32 ? wsum[lane] : 0;
    int x = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kAll, x, o);
      if (lane >= o) x += y;
    }
    if (lane < kScanThreads / 32) wsum[lane] = x - w;
    if (lane == kScanThreads / 32 - 1) wsum[32] = x;
  }
  __syncthreads();
  *total = wsum[32];
  return wsum[warp] + incl - v;
}

__global__ void __launch_bounds__(kScanThreads) bm_tilesum_kernel(const __grid_constant__ BmIndexParams p) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ int wsum[33];
  int c[8];
  load_tile_counts(p.cnt, p.total_len, static_cast<int64_t>(blockIdx.x) * kScanTile + 8 * threadIdx.x, c);
  int groups = 0, windows = 0;
#pragma unroll
  for (int x = 0; x < 8; ++x) {
    groups += (c[x] + 1) >> 1;
    windows += c[x] > 0 ? 1 : 0;
  }
  int total_g, total_w;
  block_exclusive_scan(groups, wsum, &total_g);
  __syncthreads();
  block_exclusive_scan(windows, wsum, &total_w);
  if (threadIdx.x == 0) {
    p.tile_groups[blockIdx.x] = total_g;
    p.tile_windows[blockIdx.x] = total_w;
  }
}

__global__ void __launch_bounds__(kScanThreads) bm_plan_kernel(const __grid_constant__ BmIndexParams p) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ int wsum[33];
  __shared__ int red[2][kScanThreads / 32];
  const int b = blockIdx.x;
  // this tile's offsets: the groups and the windows of the tiles before it
  int before_g = 0, before_w = 0;
  for (int i = threadIdx.x; i < b; i += kScanThreads) {
    before_g += p.tile_groups[i];
    before_w += p.tile_windows[i];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before_g += __shfl_xor_sync(kAll, before_g, o);
    before_w += __shfl_xor_sync(kAll, before_w, o);
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = before_g;
    red[1][threadIdx.x >> 5] = before_w;
  }
  int c[8];
  const int64_t i0 = static_cast<int64_t>(b) * kScanTile + 8 * threadIdx.x;
  load_tile_counts(p.cnt, p.total_len, i0, c);
  int groups = 0, windows = 0;
#pragma unroll
  for (int x = 0; x < 8; ++x) {
    groups += (c[x] + 1) >> 1;
    windows += c[x] > 0 ? 1 : 0;
  }
  int total_g, total_w;
  int g = block_exclusive_scan(groups, wsum, &total_g);  // its __syncthreads also publish red[]
  __syncthreads();
  int w = block_exclusive_scan(windows, wsum, &total_w);
  int offset_g = 0, offset_w = 0;
#pragma unroll
  for (int x = 0; x < kScanThreads / 32; ++x) {
    offset_g += red[0][x];
    offset_w += red[1][x];
  }
  g += offset_g;
  w += offset_w;
#pragma unroll
  for (int x = 0; x < 8; ++x) {
    if (c[x] == 0) continue;
    p.cursor[i0 + x] = 2 * g;
    p.cnt[i0 + x] = w++;  // the count is read; the position now keeps its window's ordinal
    if (c[x] & 1) p.groups[g + (c[x] >> 1)].row[1] = -1;  // the window's last group holds one record
    g += (c[x] + 1) >> 1;
  }
  if (b == gridDim.x - 1 && threadIdx.x == 0) *p.ngroups = offset_g + total_g;
}

__global__ void __launch_bounds__(kRecordWarps * 32) bm_fill_kernel(const __grid_constant__ BmIndexParams p) {
  griddep_launch_dependents();
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kRecordWarps + warp;
  if (r >= p.rows) return;
  int e = p.end[r];
  e = e < 0 ? 0 : (e > p.num_cols ? p.num_cols : e);
  const int n = p.nrec[r];
  for (int k = lane; k < n; k += 32) {
    const int2 rc = p.rec[static_cast<int64_t>(r) * p.nsb + k];
    const int at = atomicAdd(p.cursor + rc.x, 1);
    BmGroup* g = p.groups + (at >> 1);
    const int s = at & 1;
    if (s == 0) {
      g->P = rc.x;
      g->wo = p.cnt[rc.x];  // the plan kernel left the window's ordinal there
    }
    g->row[s] = r;
    g->c0m[s] = rc.y;
    g->end[s] = e;
  }
}

// ---------------------------------------------------------------------------
// Score
// ---------------------------------------------------------------------------

// Warps: 0 window loader, 1..3 MMA issuers, 4..27 epilogue (six warpgroups).
// Issuer t and epilogue warpgroups 2t (row 0 of each group) and 2t + 1 (row
// 1) own accumulator t and take the groups it = t, t + 3, ...; issuer t also
// loads the query tiles of its groups into its own kQPer stages, and every
// epilogue warp fetches its row's params into a ring of its own. So every
// barrier has one waiter set that sees its phases in order (a parity wait
// cannot match a phase two back), except the windows', which every issuer
// waits for in order.
__global__ void __launch_bounds__(kBmThreads, 1)
    bm_score_kernel(const __grid_constant__ BmScoreParams p, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_kw) {
  using L = BmLayout;
  extern __shared__ uint8_t bm_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(bm_smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int NS = kBmStages;
  constexpr int NA = kBmAcc;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
  auto win_full = [&](int i) { return smem_addr(&bars[i]); };
  auto win_empty = [&](int i) { return smem_addr(&bars[2 + i]); };
  auto q_full = [&](int s) { return smem_addr(&bars[4 + s]); };
  auto q_empty = [&](int s) { return smem_addr(&bars[4 + NS + s]); };
  auto acc_full = [&](int a) { return smem_addr(&bars[4 + 2 * NS + a]); };
  auto acc_empty = [&](int a) { return smem_addr(&bars[4 + 2 * NS + NA + a]); };
  auto bar_drain = [&](int a) { return smem_addr(&bars[4 + 2 * NS + 2 * NA + a]); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc + 4);
  const volatile int never = 0;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(win_full(i), 1);    // the stager's arrival plus the value copy's bytes
      mbar_init(win_empty(i), NA);  // a commit of each MMA issuer
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(q_full(s), 1);   // the issuer's expect plus its copies' bytes
      mbar_init(q_empty(s), 1);  // the issuer's MMA commit
    }
    for (int a = 0; a < NA; ++a) {
      mbar_init(acc_full(a), 1);
      mbar_init(acc_empty(a), 8);  // the two warpgroups of accumulator a
      mbar_init(bar_drain(a), 1);
    }
    *abort_flag = 0;
    mbar_init_fence();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_kw);
  }
  // query scales are all 2^0: one 512-byte block of 0x7F for the SF-B columns
  uint32_t* sf_one = reinterpret_cast<uint32_t*>(smem + L::sf_one);
  if (tid < 128) sf_one[tid] = 0x7F7F7F7Fu;
  fence_proxy_async_smem();
  if (warp == 1) tmem_alloc(smem_addr(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tm_sfa = tmem + NA * kBmN;  // per MMA issuer t: 4 columns per window slot at 8 t
  const uint32_t tm_sfb = tm_sfa + 8 * NA;   // per MMA issuer t: 4 columns at 4 t

  // everything below reads what the index kernels wrote
  griddep_launch_dependents();
  griddep_wait();
  const int G = *p.ngroups;
  const int g_begin = static_cast<int>(static_cast<int64_t>(G) * blockIdx.x / gridDim.x);
  const int g_end = static_cast<int>(static_cast<int64_t>(G) * (blockIdx.x + 1) / gridDim.x);
  const int n = g_end - g_begin;
  const BmGroup* groups = p.groups + g_begin;

  if (warp == 0) {
    // ======================= window loader =======================
    // Walks the groups' window ids in order (batches of 32, one batch ahead).
    // A new window: its 128 rows of values by one tensor copy that unpacks
    // E2M1 into the MMA's containers (positions past the workspace read as
    // zero), its scale words through registers into the layout tcgen05.cp
    // places at lane m, column m / 32: word 4 (m % 32) + m / 32.
    bool ok = true;
    int nw = 0, cur = -1;
    const uint32_t* scales = reinterpret_cast<const uint32_t*>(p.k_scales);
    auto load_P = [&](int b) { return b + lane < n ? groups[b + lane].P : -1; };
    auto walk = [&](int base, int myP) {
      for (int k = 0; k < 32 && base + k < n && ok; ++k) {
        const int P = __shfl_sync(kAll, myP, k);
        if (P == cur) continue;
        cur = P;
        const int slot = nw & 1;
        ok = warp_wait(win_empty(slot), ((nw >> 1) & 1) ^ 1, abort_flag, p.wait_ns);
        if (!ok) break;
        if (lane == 0) {
          mbar_expect_tx(win_full(slot), 128 * (kHeadDim / 2));  // the packed source bytes
          tma_load_3d(smem_addr(smem + L::window + slot * kWindowBytes), &tm_kw, 0, P, 0, win_full(slot));
        }
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int64_t pos = static_cast<int64_t>(P) + 32 * q + lane;
          w[q] = pos < p.total_len ? __ldg(scales + pos) : 0x7F7F7F7Fu;
        }
        const uint32_t sdst = smem_addr(smem + L::window_sf + slot * 512 + 16 * lane);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sdst), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                     : "memory");
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(win_full(slot));
        ++nw;
      }
    };
    int pa = load_P(0);
    for (int base = 0; base < n && ok; base += 64) {
      const int pb = load_P(base + 32);
      walk(base, pa);
      pa = load_P(base + 64);
      walk(base + 32, pb);
    }
    if (!ok) {
      if (lane == 0) status_or(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    // the last windows' copies may still be in flight when another warp gave up
    if (lane == 0)
      for (int t = nw > 2 ? nw - 2 : 0; t < nw; ++t) mbar_wait(win_full(t & 1), (t >> 1) & 1, &never, p.wait_ns);
    __syncwarp();
  } else if (warp <= NA) {
    // ======================= MMA issuers =======================
    // Issuing tcgen05 instructions costs a thread about as much as they take
    // to run, so three threads share it; each shares its scheduler with six
    // epilogue warps, so its work per group is kept to a few instructions.
    // Issuer t takes the groups it = t, t + 3, ... (its own groups k = 0, 1,
    // ...); lane l holds the descriptor head (P, row0, row1, window ordinal)
    // of own group base + l, for two alternating batches of 32, each loaded
    // a batch ahead. Each issuer keeps its own scale columns; a window's slot
    // is free once every issuer committed past it. A window an issuer has no
    // group in is committed after it has loaded (so that a commit for the
    // slot's next window cannot pass it). After the MMAs of own group k it
    // loads the query tiles of own group k + kQPer - 1 into stage
    // (k + kQPer - 1) % kQPer of its own. Lane 0 issues.
    const int t = warp - 1;
    const uint32_t sfa = tm_sfa + 8 * t, sfb = tm_sfb + 4 * t;
    uint32_t idesc[4];
    for (int g = 0; g < 4; ++g) idesc[g] = mxf8f6f4_idesc(kTypeE2M1, kTypeE4M3, 128, kBmN, g, g);
    if (lane == 0) tmem_cp_32x128b_x4(sfb, rows16_desc(smem_addr(sf_one)));
    const int own = n > t ? (n - t + NA - 1) / NA : 0;
    const int wo0 = n > 0 ? groups[0].wo : 0;               // the range's first window ordinal
    const int nwin = n > 0 ? groups[n - 1].wo - wo0 + 1 : 0;  // windows of the range
    bool ok = true;
    int mine = -1;    // the window this issuer is in
    int issued = 0;   // own groups whose query tiles are out
    auto head = [&](int k) {  // descriptor head of own group k
      return k < own ? *reinterpret_cast<const int4*>(groups + t + NA * k) : make_int4(0, -1, -1, 0);
    };
    int4 hcur = head(lane), hnxt = head(32 + lane);
    int base = 0;  // own group of hcur's lane 0
    auto get = [&](int k) {  // own group k's head, base <= k < base + 64 (k uniform)
      const int d = k - base;
      const int4 h = d < 32 ? hcur : hnxt;
      int4 r;
      r.x = __shfl_sync(kAll, h.x, d & 31);
      r.y = __shfl_sync(kAll, h.y, d & 31);
      r.z = __shfl_sync(kAll, h.z, d & 31);
      r.w = __shfl_sync(kAll, h.w, d & 31);
      return r;
    };
    auto pass_windows = [&](int upto) {  // lane 0: commit windows [max(mine, 0), upto) this issuer leaves
      for (int w = mine < 0 ? 0 : mine; w < upto && ok; ++w) {
        if (w != mine) ok = mbar_wait(win_full(w & 1), (w >> 1) & 1, abort_flag, p.wait_ns);
        mma_commit(win_empty(w & 1));
      }
    };
    auto load_q = [&](int k, int r0, int r1) {  // lane 0: query tiles of own group k
      const int g = t + NA * k;
      const int s = t * kQPer + k % kQPer;
      ok = ok && mbar_wait(q_empty(s), ((k / kQPer) & 1) ^ 1, abort_flag, p.wait_ns);
      if (ok && !(g == p.stall_group && blockIdx.x == 0)) {
        const uint32_t qdst = smem_addr(smem + L::q + s * 2 * kQRowBytes);
        mbar_arrive_expect_tx(q_full(s), (r1 >= 0 ? 2 : 1) * kQRowBytes);
        tma_load_2d(qdst, &tm_q, 0, r0 * kBmHeads, q_full(s));
        if (r1 >= 0) tma_load_2d(qdst + kQRowBytes, &tm_q, 0, r1 * kBmHeads, q_full(s));
      }
      issued = k + 1;
    };
    for (int k = 0; k < kQPer - 1 && k < own; ++k) {
      const int4 h = get(k);
      if (lane == 0) load_q(k, h.y, h.z);
    }
    for (int k = 0; k < own; ++k) {
      if (k >= base + 32) {  // slide the batches: the next one was loaded a batch ago
        base += 32;
        hcur = hnxt;
        hnxt = head(base + 32 + lane);
      }
      const int4 h = get(k);
      const int4 hq = get(k + kQPer - 1 < own ? k + kQPer - 1 : k);
      if (lane == 0 && ok) {
        const int wi = h.w - wo0;
        if (wi != mine) {
          pass_windows(wi);
          ok = ok && mbar_wait(win_full(wi & 1), (wi >> 1) & 1, abort_flag, p.wait_ns);
          if (ok) {
            tc_fence_after();
            tmem_cp_32x128b_x4(sfa + 4 * (wi & 1), rows16_desc(smem_addr(smem + L::window_sf + (wi & 1) * 512)));
            mine = wi;
          }
        }
        const int s = t * kQPer + k % kQPer;
        ok = ok && mbar_wait(q_full(s), (k / kQPer) & 1, abort_flag, p.wait_ns) &&
             mbar_wait(acc_empty(t), (k & 1) ^ 1, abort_flag, p.wait_ns);
        if (ok) {
          tc_fence_after();
          const int slot = wi & 1;
          const uint64_t adesc = sw128_desc(smem_addr(smem + L::window + slot * kWindowBytes));
          const uint64_t bdesc = sw128_desc(smem_addr(smem + L::q + s * 2 * kQRowBytes));
#pragma unroll
          for (int g = 0; g < 4; ++g)  // K = 32 per MMA: 32 bytes along the swizzled rows
            mma_mxf8f6f4(tmem + t * kBmN, adesc + 2 * g, bdesc + 2 * g, idesc[g], sfa + 4 * slot, sfb, g > 0);
          mma_commit(acc_full(t));
          mma_commit(q_empty(s));
          // the query tiles of own group k + kQPer - 1, into the stage of
          // group k - 1: after this group's MMAs are out, so that waiting for
          // the previous group's MMAs to finish overlaps this group's
          if (k + kQPer - 1 < own) load_q(k + kQPer - 1, hq.y, hq.z);
        }
      }
      if (__shfl_sync(kAll, ok ? 1 : 0, 0) == 0) break;
    }
    if (lane == 0) {
      if (ok) pass_windows(nwin);  // the windows left: this issuer's last and those with none of its groups
      if (!ok) {
        status_or(p.status, kStatusTimeout);
        *abort_flag = 1;
        // query tiles issued but not consumed may still be in flight: let them land
        for (int k = issued > kQPer ? issued - kQPer : 0; k < issued; ++k)
          mbar_wait(q_full(t * kQPer + k % kQPer), (k / kQPer) & 1, &never, p.wait_ns);
      }
      mma_commit(bar_drain(t));  // every tcgen05 operation of this thread has finished once this arrives
      mbar_wait(bar_drain(t), 0, &never, p.wait_ns);
    }
    __syncwarp();
  } else {
    // ======================= epilogue (warps 4..27) =======================
    // Warpgroups 2t and 2t + 1 take the groups it = t, t + 3, ..., one row
    // each: so an accumulator goes back after one round of loads and half a
    // row's arithmetic. Each warp fetches each group's descriptor and its
    // row's params itself, one group ahead, by 16-byte asynchronous copies
    // into a ring of kPrmPer slots of its own (no barrier across warps); the
    // rows of the group after that come from a load two groups ahead.
    const int ew = warp - kBmEpiWarp0;  // epilogue warp: its ring
    const int a = ew >> 3;              // accumulator (and issuer) of its groups
    const int e = (ew >> 2) & 1;        // its row of each group
    const int q4 = warp & 3;            // TMEM lane quarter
    const int m = 32 * q4 + lane;       // key of the window
    const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
    const int shift = 31 - __clz(p.sbkv);
    const int sl = m >> shift;
    const uint32_t below = (1u << sl) - 1u;
    const int moff = m & (p.sbkv - 1);
    const int own = n > a ? (n - a + NA - 1) / NA : 0;
    constexpr int kChunks = kSlotBytes / 16;  // 19: descriptor, then the row's params
    static_assert(kChunks <= 32, "one chunk per lane");
    auto fetch = [&](int k, int r) {  // group k's descriptor and row params into slot k % kPrmPer
      if (k < own && lane < kChunks) {
        const uint32_t dst = smem_addr(smem + L::prm + (ew * kPrmPer + k % kPrmPer) * kSlotBytes) + 16 * lane;
        const uint8_t* src =
            lane < 2 ? reinterpret_cast<const uint8_t*>(groups + a + NA * k) + 16 * lane
                     : reinterpret_cast<const uint8_t*>(p.rowparams + static_cast<int64_t>(r < 0 ? 0 : r) * kBmRowParams) +
                           16 * (lane - 2);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    auto row_of = [&](int k) {  // this warp's row of group k, or -1
      if (k >= own) return -1;
      const int4 d = *reinterpret_cast<const int4*>(groups + a + NA * k);  // (P, row0, row1, c0m0)
      return e == 0 ? d.y : d.z;
    };
    int r1n = row_of(1);  // the next group's row
    fetch(0, row_of(0));
    bool ok = true;
    for (int k = 0; k < own && ok; ++k) {
      const int r2n = row_of(k + 2);  // used next step
      fetch(k + 1, r1n);
      asm volatile("cp.async.wait_group 1;" ::: "memory");  // this lane's copies of group k
      ok = warp_wait(acc_full(a), k & 1, abort_flag, p.wait_ns);  // its __syncwarp also publishes the lanes' copies
      if (!ok) break;
      tc_fence_after();
      const uint8_t* prm = smem + L::prm + (ew * kPrmPer + k % kPrmPer) * kSlotBytes;
      const BmGroup* gd = reinterpret_cast<const BmGroup*>(prm);
      const int row = gd->row[e];
      // Two halves of 32 heads: the second half's loads are this warp's last
      // reads of the accumulator. Heads h = 0, 1 (mod 4) accumulate in lo and
      // h = 2, 3 (mod 4) in hi, each in head order.
      uint64_t lo = 0, hi = 0;  // (+0, +0) as packed pairs
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t v[32];
        const uint32_t tacc = tmem + a * kBmN + e * kBmHeads + 32 * half + lane_base;
        tmem_ld16(tacc, *reinterpret_cast<uint32_t(*)[16]>(v));
        tmem_ld16(tacc + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
        tmem_wait_ld();
        if (half == 1) {  // this warp's columns are in registers: its share of the hand-back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty(a));
        }
        if (row < 0) continue;
        const ulonglong2* w4 = reinterpret_cast<const ulonglong2*>(prm + 32) + 8 * half;
#pragma unroll
        for (int h4 = 0; h4 < 8; ++h4) {
          const ulonglong2 w = w4[h4];  // weights of heads 4 h4 .. 4 h4 + 3 as two pairs
          const uint32_t* x = v + 4 * h4;
          relu2_fma2(lo, w.x, __uint_as_float(x[0]), __uint_as_float(x[1]));
          relu2_fma2(hi, w.y, __uint_as_float(x[2]), __uint_as_float(x[3]));
        }
      }
      if (row >= 0) {
        const float qs = reinterpret_cast<const float*>(prm + 32)[kBmHeads];
        const float2 l = unpack2(lo), h = unpack2(hi);  // twice the head sums, exactly
        const float logit = ((l.x + l.y) + (h.x + h.y)) * (0.5f * qs);
        const uint32_t c0m = static_cast<uint32_t>(gd->c0m[e]);
        const uint32_t mask = c0m >> 24;
        if ((mask >> sl) & 1u) {
          const int col = static_cast<int>(c0m & 0xFFFFFFu) + (__popc(mask & below) << shift) + moff;
          if (col < gd->end[e]) {
            const int64_t at = static_cast<int64_t>(row) * p.num_cols + col;
            p.logits[at] = logit;
            if (p.logits_bf16) p.logits_bf16[at] = round_bf16(logit);
          }
        }
      }
      r1n = r2n;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // no copy into shared memory outlives the CTA
    if (!ok) {
      if (lane == 0) status_or(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------

namespace {

template <typename... A>
cudaError_t launch_pdl_bm(void (*kernel)(A...), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
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

}  // namespace

size_t bm_score_smem_bytes() { return BmLayout::bytes + 1024; }

cudaError_t prepare_bm_kernels() {
  cudaError_t err = cudaFuncSetAttribute(bm_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bm_score_smem_bytes()));
  if (err != cudaSuccess) return err;
  const void* all[] = {reinterpret_cast<const void*>(&bm_score_kernel),
                       reinterpret_cast<const void*>(&bm_records_kernel),
                       reinterpret_cast<const void*>(&bm_tilesum_kernel), reinterpret_cast<const void*>(&bm_plan_kernel),
                       reinterpret_cast<const void*>(&bm_fill_kernel)};
  for (const void* f : all) {
    err = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

cudaError_t launch_bm_index(const BmIndexParams& p, cudaStream_t stream) {
  cudaError_t err = cudaMemsetAsync(p.cnt, 0, static_cast<size_t>(p.total_len) * sizeof(int32_t), stream);
  if (err != cudaSuccess) return err;
  const unsigned row_grid = static_cast<unsigned>((p.rows + kRecordWarps - 1) / kRecordWarps);
  err = launch_pdl_bm(bm_records_kernel, row_grid, kRecordWarps * 32, 0, stream, p);
  if (err != cudaSuccess) return err;
  const unsigned tiles = static_cast<unsigned>((p.total_len + kScanTile - 1) / kScanTile);
  err = launch_pdl_bm(bm_tilesum_kernel, tiles, kScanThreads, 0, stream, p);
  if (err != cudaSuccess) return err;
  err = launch_pdl_bm(bm_plan_kernel, tiles, kScanThreads, 0, stream, p);
  if (err != cudaSuccess) return err;
  return launch_pdl_bm(bm_fill_kernel, row_grid, kRecordWarps * 32, 0, stream, p);
}

cudaError_t launch_bm_score(const BmScoreParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kw, int grid,
                            cudaStream_t stream) {
  return launch_pdl_bm(bm_score_kernel, static_cast<unsigned>(grid), kBmThreads, bm_score_smem_bytes(), stream, p, tm_q,
                       tm_kw);
}

}  // namespace smq
