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
// per SM:
//  - warp 0 (producer): for each 128-position tile it TMA-loads the FP4 key
//    values of the tile's sub-blocks. A 16U4_ALIGN16B tensor map unpacks
//    them into the padded layout the MMA reads, and per-position UE8M0 scales
//    come in by bulk copy. When the row changes it also loads the row's Q tile
//    (E4M3, 128-byte swizzle) and bf16 head weights.
//  - warp 1 (MMA): one thread issues 4 x tcgen05.mma kind::mxf8f6f4 with
//    UE8M0 block scales, M = 128 positions, N = heads, K = 32 each. The
//    accumulator (fp32) goes to TMEM, double-buffered.
//  - warps 2..5 (epilogue): they write each tile's key scales into TMEM,
//    where row m of A reads lane m, column base + m/32, byte = scale id.
//    Then they read the accumulator, one TMEM lane (= one position) per
//    thread, and reduce over heads with ReLU and the weights.
// Every wait is bounded. A wait that gives up sets SMQ_ERR_TIMEOUT in the
// status word and the CTA winds down. Out-of-range page / row / block ids set
// SMQ_ERR_BOUNDS, and the load is skipped.
#include "smq_kernels.cuh"
#include "smq_ptx.cuh"

#include <cfloat>

namespace smq {

namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr uint32_t kFullMask = 0xffffffffu;
constexpr uint32_t kE2M1 = 5, kE4M3 = 0;

__host__ __device__ constexpr uint32_t round_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Byte offsets inside the score kernel's dynamic shared memory (base aligned to 1024).
struct ScoreLayout {
  uint32_t kv, q, sf, sf_region, sf_stage, w, w_stride, meta, rem, bars, misc, scan, prefix, total;
  __host__ __device__ ScoreLayout(int n_mma, int heads, int sbkv, int stages, int rows) {
    uint32_t o = 0;
    kv = o;  // [stages][128 rows][128 B] padded FP4 keys, 128-byte swizzle
    o += static_cast<uint32_t>(stages) * kTileM * kRowBytes;
    q = o;  // [2][n_mma rows][128 B] E4M3 queries, 128-byte swizzle
    o += 2u * static_cast<uint32_t>(n_mma) * kRowBytes;
    // one region per sub-block: sbkv + 4 scale words, 128-byte aligned (tensor-copy destination)
    sf_region = round_up(static_cast<uint32_t>(sbkv + 4) * 4u, 128);
    sf_stage = static_cast<uint32_t>(kTileM / sbkv) * sf_region;
    sf = o;  // [stages][sub-blocks][sf_region bytes]
    o += static_cast<uint32_t>(stages) * sf_stage;
    w_stride = round_up(static_cast<uint32_t>(heads) * 2u, 16);
    w = o;  // [2][heads] bf16 weights
    o += 2u * w_stride;
    meta = o;  // [2] {row, end, q_scale bits, unused}
    o += 2u * 16u;
    rem = o;  // [stages] int: word offset of the first scale in the stage
    o += round_up(static_cast<uint32_t>(stages) * 4u, 16);
    bars = o;  // full, empty, sf_full [stages]; acc_full, acc_empty, q_full, q_empty [2]; drain
    o += round_up((3u * static_cast<uint32_t>(stages) + 9u) * 8u, 16);
    misc = o;  // tmem base, abort flag
    o += 16u;
    scan = o;  // per-warp partial sums of the prologue scan
    o += 32u;
    prefix = o;  // [rows + 1] exclusive prefix of tiles per row
    o += round_up((static_cast<uint32_t>(rows) + 1u) * 4u, 16);
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

}  // namespace

size_t score_smem_bytes(int n_mma, int heads, int sbkv, int stages, int rows) {
  return ScoreLayout(n_mma, heads, sbkv, stages, rows).total + 1024;
}

// ===========================================================================
// Candidate expansion: one warp per row.
// ===========================================================================
__global__ void __launch_bounds__(kExpandWarps * 32) expand_kernel(const __grid_constant__ ExpandParams p) {
  extern __shared__ int32_t expand_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kExpandWarps + warp;
  if (r >= p.rows) return;
  int32_t* cand = expand_smem + warp * 2 * p.ncb;
  int32_t* kept = cand + p.ncb;
  const int64_t ks = p.row_ks ? p.row_ks[r] : 0;
  int64_t L = static_cast<int64_t>(p.row_ke[r]) - ks;
  if (L < 0) L = 0;
  for (int i = lane; i < p.ncb; i += 32) cand[i] = p.candidate_blocks[static_cast<int64_t>(r) * p.ncb + i];
  __syncwarp();
  // keep a block if it is in range and its first occurrence; others -> INT_MAX
  for (int i = lane; i < p.ncb; i += 32) {
    const int32_t b = cand[i];
    bool keep = b >= 0 && static_cast<int64_t>(b) * p.cbs < L;
    for (int j = 0; keep && j < i; ++j) keep = cand[j] != b;
    kept[i] = keep ? b : INT_MAX;
  }
  __syncwarp();
  const int spb = p.cbs / p.sbkv;
  int32_t* si = p.sparse_indices + static_cast<int64_t>(r) * p.nsb;
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
template <bool kPaged, int kN>
__global__ void __launch_bounds__(kScoreThreads, 1)
    score_kernel(const __grid_constant__ ScoreParams p, const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_ks) {
  extern __shared__ uint8_t score_smem_raw[];
  uint8_t* smem = align1024(score_smem_raw);
  const ScoreLayout lay(kN, p.heads, p.sbkv, p.stages, p.rows);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NS = p.stages;
  const int S = p.num_cols;
  const int R = p.rows;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
  auto bar_full = [&](int s) { return smem_addr(&bars[s]); };
  auto bar_empty = [&](int s) { return smem_addr(&bars[NS + s]); };
  auto bar_sf = [&](int s) { return smem_addr(&bars[2 * NS + s]); };
  auto bar_acc_full = [&](int a) { return smem_addr(&bars[3 * NS + a]); };
  auto bar_acc_empty = [&](int a) { return smem_addr(&bars[3 * NS + 2 + a]); };
  auto bar_q_full = [&](int b) { return smem_addr(&bars[3 * NS + 4 + b]); };
  auto bar_q_empty = [&](int b) { return smem_addr(&bars[3 * NS + 6 + b]); };
  const uint32_t bar_drain = smem_addr(&bars[3 * NS + 8]);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + lay.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + lay.misc + 4);
  int32_t* scan = reinterpret_cast<int32_t*>(smem + lay.scan);
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + lay.prefix);
  RowMeta* meta = reinterpret_cast<RowMeta*>(smem + lay.meta);
  int32_t* stage_rem = reinterpret_cast<int32_t*>(smem + lay.rem);

  // ---- prologue: barriers, per-row tile counts and their prefix ---------
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
      mbar_init(bar_sf(s), 128);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_acc_full(a), 1);
      mbar_init(bar_acc_empty(a), 128);
      mbar_init(bar_q_full(a), 1);
      mbar_init(bar_q_empty(a), 1 + 4);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (tid == 32) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    if constexpr (!kPaged) prefetch_tmap(&tm_ks);
  }
  const int per = (R + kScoreThreads - 1) / kScoreThreads;
  const int r0 = min(R, tid * per), r1 = min(R, r0 + per);
  auto tiles_of = [&](int r) {
    int e = p.end[r];
    e = e < 0 ? 0 : (e > S ? S : e);
    return (e + kTileM - 1) / kTileM;
  };
  int mine = 0;
  for (int r = r0; r < r1; ++r) mine += tiles_of(r);
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
  if (n <= 0) return;

  // ---- TMEM: [acc 0 | acc 1 | SF-A per stage (4 cols) | SF-B (4 cols)] ----
  if (warp == 1) tmem_alloc(smem_addr(tmem_slot), p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tm_sfa = tmem + 2 * kN;
  const uint32_t tm_sfb = tm_sfa + 4 * NS;
  if (warp >= 2) {  // B (query) scales are all 2^0
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    tmem_st4(tm_sfb + lane_base, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int spt = p.subs_per_tile;
  const int sbkv = p.sbkv;
  const int H = p.heads;

  if (warp == 0) {
    // ======================= producer =======================
    const int tiles_per_batch = 32 / spt;
    int cur_row = -1;
    uint32_t quse = 0;
    int it = 0;
    bool ok = true;
    for (int64_t tb = t_begin; tb < t_end && ok; tb += tiles_per_batch) {
      // each lane resolves one sub-block of the batch
      const int64_t t = tb + lane / spt;
      const int sub = lane % spt;
      int r = 0, e = 0, valid = 0, page = 0, tok = 0;
      int64_t pos = 0;
      float qs = 0.f;
      if (t < t_end) {
        r = find_row(prefix, R, t);
        const int j = static_cast<int>(t - prefix[r]);
        e = p.end[r];
        e = e < 0 ? 0 : (e > S ? S : e);
        qs = p.q_scale[r];
        const int col_sub = j * spt + sub;
        if (col_sub * sbkv < e) {
          const int sb = p.sparse_indices[static_cast<int64_t>(r) * p.nsb + col_sub];
          if (sb >= 0) {
            if constexpr (kPaged) {
              const int64_t tpos = static_cast<int64_t>(sb) * sbkv;
              const int64_t slot = tpos / p.page_size;
              const int brow = p.row_indices ? p.row_indices[r] : r;
              if (brow >= 0 && brow < p.bt_rows && slot < p.bt_stride) {
                const int pg = p.block_table[static_cast<int64_t>(brow) * p.bt_stride + slot];
                if (pg >= 0 && pg < p.num_pages) {
                  page = pg;
                  tok = static_cast<int>(tpos % p.page_size);
                  valid = 1;
                }
              }
            } else {
              pos = static_cast<int64_t>(p.row_ks[r]) + static_cast<int64_t>(sb) * sbkv;
              valid = (pos >= 0 && pos < p.total_len) ? 1 : 0;
            }
          }
          if (!valid) set_status(p.status, kStatusBounds);
        }
      }
      for (int k = 0; k < tiles_per_batch; ++k) {
        if (tb + k >= t_end) break;
        const int base = k * spt;
        const int rk = __shfl_sync(kFullMask, r, base);
        const int ek = __shfl_sync(kFullMask, e, base);
        const float qsk = __shfl_sync(kFullMask, qs, base);
        if (rk != cur_row) {
          const int qb = quse & 1;
          bool w_ok = true;
          if (lane == 0) w_ok = mbar_wait(bar_q_empty(qb), ((quse >> 1) & 1) ^ 1, abort_flag, kWaitLimitNs);
          ok = __shfl_sync(kFullMask, w_ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          if (lane == 0) {
            meta[qb].row = rk;
            meta[qb].end = ek;
            meta[qb].q_scale = qsk;
            const uint32_t q_dst = smem_addr(smem + lay.q + qb * kN * kRowBytes);
            const uint32_t w_dst = smem_addr(smem + lay.w + qb * lay.w_stride);
            mbar_arrive_expect_tx(bar_q_full(qb), kN * kRowBytes + H * 2);
            tma_load_2d(q_dst, &tm_q, 0, rk * H, bar_q_full(qb));
            bulk_load(w_dst, p.weights + static_cast<int64_t>(rk) * H, H * 2, bar_q_full(qb));
          }
          cur_row = rk;
          ++quse;
        }
        const int s = it % NS;
        bool e_ok = true;
        if (lane == 0) e_ok = mbar_wait(bar_empty(s), ((it / NS) & 1) ^ 1, abort_flag, kWaitLimitNs);
        ok = __shfl_sync(kFullMask, e_ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        // bytes this stage will receive
        const uint32_t kv_stage = smem_addr(smem + lay.kv + s * (kTileM * kRowBytes));
        const uint32_t sf_stage = smem_addr(smem + lay.sf + s * lay.sf_stage);
        // tensor copies land on 128-byte boundaries (1024 for the swizzled keys); a
        // destination that is not is reported and skipped instead of issued
        auto dst_ok = [&](int u) {
          return ((kv_stage + u * sbkv * kRowBytes) & 1023u) == 0 && ((sf_stage + u * lay.sf_region) & 127u) == 0;
        };
        uint32_t bytes = 0;
        int rem = 0;
        for (int u = 0; u < spt; ++u) {
          const int v = __shfl_sync(kFullMask, valid, base + u);
          const int64_t pu = __shfl_sync(kFullMask, pos, base + u);
          if (v && !dst_ok(u)) {
            if (lane == 0) set_status(p.status, kStatusBounds);
          } else if (v) {
            bytes += static_cast<uint32_t>(sbkv) * (kHeadDim / 2);  // packed FP4 bytes
            if constexpr (kPaged) {
              bytes += static_cast<uint32_t>(sbkv) * kScaleWordBytes;
            } else {
              bytes += static_cast<uint32_t>(sbkv + 4) * kScaleWordBytes;
              rem = static_cast<int>(pu & 3);
            }
          }
        }
        if (lane == 0) {
          stage_rem[s] = rem;
          mbar_arrive_expect_tx(bar_full(s), bytes);
        }
        for (int u = 0; u < spt; ++u) {
          const int v = __shfl_sync(kFullMask, valid, base + u);
          const int pg = __shfl_sync(kFullMask, page, base + u);
          const int tk = __shfl_sync(kFullMask, tok, base + u);
          const int64_t pu = __shfl_sync(kFullMask, pos, base + u);
          if (lane == 0 && v && dst_ok(u)) {
            const uint32_t kv_dst = kv_stage + u * sbkv * kRowBytes;
            const uint32_t sf_dst = sf_stage + u * lay.sf_region;
            if constexpr (kPaged) {
              tma_load_3d(kv_dst, &tm_k, 0, tk, pg, bar_full(s));
              const uint8_t* src = p.k_cache + static_cast<int64_t>(pg) * p.page_bytes +
                                   static_cast<int64_t>(p.page_size) * (kHeadDim / 2) +
                                   static_cast<int64_t>(tk) * kScaleWordBytes;
              bulk_load(sf_dst, src, sbkv * kScaleWordBytes, bar_full(s));
            } else {
              tma_load_2d(kv_dst, &tm_k, 0, static_cast<int32_t>(pu), bar_full(s));
              tma_load_1d(sf_dst, &tm_ks, static_cast<int32_t>(pu & ~int64_t(3)), bar_full(s));
            }
          }
        }
        ++it;
      }
    }
    if (!ok) {
      set_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    // let every load this warp issued land before the CTA exits
    if (lane == 0) {
      const volatile int never = 0;
      for (int i = (it > NS ? it - NS : 0); i < it; ++i)
        mbar_wait(bar_full(i % NS), (i / NS) & 1, &never, kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      uint32_t idesc[4];
      for (int g = 0; g < 4; ++g) idesc[g] = mxf8f6f4_idesc(kE2M1, kE4M3, kTileM, kN, g, g);
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
          ok = mbar_wait(bar_q_full(qb), (quse >> 1) & 1, abort_flag, kWaitLimitNs);
          ++quse;
          if (!ok) break;
        }
        const bool last_of_row = (t + 1 >= t_end) || (t + 1 >= prefix[r + 1]);
        const int s = it % NS;
        const uint32_t ph = (it / NS) & 1;
        const int a = it & 1;
        ok = mbar_wait(bar_full(s), ph, abort_flag, kWaitLimitNs) &&
             mbar_wait(bar_sf(s), ph, abort_flag, kWaitLimitNs) &&
             mbar_wait(bar_acc_empty(a), ((it >> 1) & 1) ^ 1, abort_flag, kWaitLimitNs);
        if (!ok) break;
        tc_fence_after();
        const uint64_t adesc = sw128_desc(smem_addr(smem + lay.kv + s * (kTileM * kRowBytes)));
        const uint64_t bdesc = sw128_desc(smem_addr(smem + lay.q + qb * kN * kRowBytes));
        for (int g = 0; g < 4; ++g)  // K = 32 per MMA; advance 32 bytes along the swizzled rows
          mma_mxf8f6f4(tmem + a * kN, adesc + 2 * g, bdesc + 2 * g, idesc[g], tm_sfa + 4 * s, tm_sfb, g > 0);
        mma_commit(bar_empty(s));
        mma_commit(bar_acc_full(a));
        if (last_of_row) mma_commit(bar_q_empty(qb));
      }
      if (!ok) {
        set_status(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      mma_commit(bar_drain);  // every MMA issued above has finished once this arrives
      const volatile int never = 0;
      mbar_wait(bar_drain, 0, &never, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // ======================= epilogue (warps 2..5) =======================
    const int q4 = warp & 3;  // TMEM lane quarter this warp may access
    const int m = 32 * q4 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
    const int sub_of_m = m / sbkv, tok_of_m = m % sbkv;
    int r = find_row(prefix, R, t_begin);
    int cur = -1, qb = 0, row = 0, e = 0;
    uint32_t quse = 0;
    float qs = 0.f;
    float w[kN];
    bool ok = true;
    for (int it = 0; it <= n && ok; ++it) {
      if (it < n) {
        // key scales of tile `it` into TMEM (row m reads lane m, column m / 32)
        const int s = it % NS;
        ok = mbar_wait(bar_full(s), (it / NS) & 1, abort_flag, kWaitLimitNs);
        if (!ok) break;
        const uint32_t* words = reinterpret_cast<const uint32_t*>(smem + lay.sf + s * lay.sf_stage);
        const uint32_t word = words[sub_of_m * (lay.sf_region / 4) + stage_rem[s] + tok_of_m];
        tmem_st1(tm_sfa + 4 * s + lane_base + q4, word);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_sf(s));
      }
      if (it > 0) {
        const int ie = it - 1;
        const int64_t t = t_begin + ie;
        while (prefix[r + 1] <= t) ++r;
        if (r != cur) {
          cur = r;
          qb = quse & 1;
          ok = mbar_wait(bar_q_full(qb), (quse >> 1) & 1, abort_flag, kWaitLimitNs);
          ++quse;
          if (!ok) break;
          row = meta[qb].row;
          e = meta[qb].end;
          qs = meta[qb].q_scale;
          const uint16_t* wsm = reinterpret_cast<const uint16_t*>(smem + lay.w + qb * lay.w_stride);
#pragma unroll
          for (int h = 0; h < kN; ++h) w[h] = h < H ? bf16_to_f32(wsm[h]) : 0.f;
        }
        const bool last_of_row = (t + 1 >= t_end) || (t + 1 >= prefix[r + 1]);
        const int a = ie & 1;
        ok = mbar_wait(bar_acc_full(a), (ie >> 1) & 1, abort_flag, kWaitLimitNs);
        if (!ok) break;
        tc_fence_after();
        float acc = 0.f;
        const uint32_t tacc = tmem + a * kN + lane_base;
#pragma unroll
        for (int c = 0; c < kN; c += 32) {
          uint32_t v0[16], v1[16];
          tmem_ld16(tacc + c, v0);
          tmem_ld16(tacc + c + 16, v1);
          tmem_wait_ld();
          if (c + 32 >= kN) {  // every column read: hand the accumulator back
            tc_fence_before();
            mbar_arrive(bar_acc_empty(a));
          }
#pragma unroll
          for (int h = 0; h < 16; ++h) acc = fmaf(w[c + h], fmaxf(__uint_as_float(v0[h]), 0.f), acc);
#pragma unroll
          for (int h = 0; h < 16; ++h) acc = fmaf(w[c + 16 + h], fmaxf(__uint_as_float(v1[h]), 0.f), acc);
        }
        const int col = static_cast<int>(t - prefix[r]) * kTileM + m;
        if (col < e) p.logits[static_cast<int64_t>(row) * S + col] = acc * qs;
        if (last_of_row) {
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_q_empty(qb));
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
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

// ===========================================================================
// Top-k: radix select over order-preserving keys, one CTA per row.
// ===========================================================================
__device__ __forceinline__ uint32_t ordered_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const __grid_constant__ TopkParams p) {
  extern __shared__ uint32_t topk_smem[];
  constexpr int kWarps = kTopkThreads / 32;
  __shared__ int hist[256];
  __shared__ int warp_a[kWarps], warp_b[kWarps];
  __shared__ int sel_bin, sel_need;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.x;
  const int S = p.num_cols;
  const int k = p.topk;
  uint32_t* keys = topk_smem;
  int32_t* sidx = reinterpret_cast<int32_t*>(topk_smem + S);
  int e = p.end[r];
  e = e < 0 ? 0 : (e > S ? S : e);
  for (int i = tid; i < p.nsb; i += kTopkThreads) sidx[i] = p.sparse_indices[static_cast<int64_t>(r) * p.nsb + i];
  if (p.logits_fill)
    for (int c = e + tid; c < S; c += kTopkThreads) p.logits_fill[static_cast<int64_t>(r) * S + c] = -INFINITY;
  int32_t* out = p.topk_out + static_cast<int64_t>(r) * p.topk_ld;
  int32_t* colo = p.col_indices ? p.col_indices + static_cast<int64_t>(r) * k : nullptr;
  const int sbkv = p.sbkv;
  __syncthreads();
  auto token = [&](int c) { return sidx[c / sbkv] * sbkv + c % sbkv; };
  if (e <= k) {
    for (int c = tid; c < k; c += kTopkThreads) {
      out[c] = c < e ? token(c) : -1;
      if (colo) colo[c] = c < e ? c : -1;
    }
    return;
  }
  const float* L = p.logits + static_cast<int64_t>(r) * S;
  for (int c = tid; c < e; c += kTopkThreads) keys[c] = ordered_key(L[c]);
  uint32_t prefix = 0;
  int need = k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int c0 = 0; c0 < e; c0 += kTopkThreads) {
      const int c = c0 + tid;
      int bin = -1;
      if (c < e) {
        const uint32_t key = keys[c];
        const bool match = pass == 0 || ((key ^ prefix) >> (shift + 8)) == 0;
        if (match) bin = static_cast<int>((key >> shift) & 255u);
      }
      const uint32_t peers = __match_any_sync(kFullMask, bin);
      if (bin >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
    }
    __syncthreads();
    // inclusive scan over bins in descending order: thread i holds bin 255 - i
    int cnt = tid < 256 ? hist[255 - tid] : 0;
    int incl = cnt;
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_a[warp] = incl;
    __syncthreads();
    for (int w2 = 0; w2 < warp; ++w2) incl += warp_a[w2];
    const int excl = incl - cnt;
    if (tid < 256 && excl < need && need <= incl) {
      sel_bin = 255 - tid;
      sel_need = need - excl;
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(sel_bin) << shift;
    need = sel_need;
    __syncthreads();
  }
  const uint32_t thr = prefix;  // key of the k-th largest logit
  const int need_eq = need;     // how many keys equal to thr are selected
  int base_gt = 0, base_eq = 0;
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int c0 = 0; c0 < e; c0 += kTopkThreads) {
    const int c = c0 + tid;
    const uint32_t key = c < e ? keys[c] : 0u;
    const bool gt = c < e && key > thr;
    const bool eq = c < e && key == thr;
    const uint32_t bg = __ballot_sync(kFullMask, gt), be = __ballot_sync(kFullMask, eq);
    if (lane == 0) {
      warp_a[warp] = __popc(bg);
      warp_b[warp] = __popc(be);
    }
    __syncthreads();
    int off_gt = base_gt, off_eq = base_eq, tot_gt = 0, tot_eq = 0;
    for (int w2 = 0; w2 < kWarps; ++w2) {
      if (w2 < warp) {
        off_gt += warp_a[w2];
        off_eq += warp_b[w2];
      }
      tot_gt += warp_a[w2];
      tot_eq += warp_b[w2];
    }
    const int pg = off_gt + __popc(bg & lt_mask);
    const int pe = off_eq + __popc(be & lt_mask);
    int slot = -1;
    if (gt) slot = pg + min(pe, need_eq);
    else if (eq && pe < need_eq) slot = pg + pe;
    if (slot >= 0 && slot < k) {
      out[slot] = token(c);
      if (colo) colo[slot] = c;
    }
    base_gt += tot_gt;
    base_eq += tot_eq;
    __syncthreads();
  }
}

// ===========================================================================
// Paged -> contiguous K gather: one thread per workspace row.
// ===========================================================================
__global__ void __launch_bounds__(256) gather_kernel(const __grid_constant__ GatherParams p) {
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
  const int64_t pos = wrow - start;
  const int64_t slot = pos / p.page_size;
  if (slot >= p.bt_stride) {
    set_status(p.status, kStatusBounds);
    return;
  }
  const int page = p.block_table[static_cast<int64_t>(lo) * p.bt_stride + slot];
  if (page < 0 || page >= p.num_pages) {
    set_status(p.status, kStatusBounds);
    return;
  }
  const int64_t tok = pos % p.page_size;
  const uint8_t* base = p.k_cache + static_cast<int64_t>(page) * p.page_bytes;
  const uint4* src = reinterpret_cast<const uint4*>(base + tok * (kHeadDim / 2));
  uint4* dst = reinterpret_cast<uint4*>(p.k_values + wrow * (kHeadDim / 2));
#pragma unroll
  for (int i = 0; i < kHeadDim / 32; ++i) dst[i] = src[i];
  const uint32_t* ssrc = reinterpret_cast<const uint32_t*>(base + static_cast<int64_t>(p.page_size) * (kHeadDim / 2) +
                                                           tok * kScaleWordBytes);
  reinterpret_cast<uint32_t*>(p.k_scales)[wrow] = *ssrc;
}

// ===========================================================================
// Launchers
// ===========================================================================
cudaError_t prepare_kernels(int n_mma) {
  const int max_smem = 232448;  // 227 KB opt-in per block
  cudaError_t err;
  if (n_mma == 64) {
    err = cudaFuncSetAttribute(score_kernel<true, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(score_kernel<false, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  } else {
    err = cudaFuncSetAttribute(score_kernel<true, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(score_kernel<false, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  }
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (kMaxSparseCols + kMaxSparseCols / 16) * 4);
  if (err != cudaSuccess) return err;
  return cudaFuncSetAttribute(expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kExpandWarps * 2 * 512 * 4);
}

cudaError_t launch_expand(const ExpandParams& p, cudaStream_t stream) {
  const int grid = (p.rows + kExpandWarps - 1) / kExpandWarps;
  const size_t smem = static_cast<size_t>(kExpandWarps) * 2 * p.ncb * sizeof(int32_t);
  expand_kernel<<<grid, kExpandWarps * 32, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_score_paged(const ScoreParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k, int grid,
                               size_t smem, cudaStream_t stream) {
  if (p.n_mma == 64)
    score_kernel<true, 64><<<grid, kScoreThreads, smem, stream>>>(p, tm_q, tm_k, tm_k);
  else
    score_kernel<true, 128><<<grid, kScoreThreads, smem, stream>>>(p, tm_q, tm_k, tm_k);
  return cudaGetLastError();
}

cudaError_t launch_score_contig(const ScoreParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_ks, int grid, size_t smem, cudaStream_t stream) {
  if (p.n_mma == 64)
    score_kernel<false, 64><<<grid, kScoreThreads, smem, stream>>>(p, tm_q, tm_k, tm_ks);
  else
    score_kernel<false, 128><<<grid, kScoreThreads, smem, stream>>>(p, tm_q, tm_k, tm_ks);
  return cudaGetLastError();
}

cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(p.num_cols + p.nsb) * 4;
  topk_kernel<<<p.rows, kTopkThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_gather(const GatherParams& p, cudaStream_t stream) {
  const int64_t blocks = (p.total_len + 255) / 256;
  gather_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace smq
