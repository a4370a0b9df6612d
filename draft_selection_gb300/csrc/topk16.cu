// Top-16 per row of the drafter logits ("DFlash 2: Keep Drafting Parallel",
// 方法细节 > 轻量级路径选择器: keep the 16 highest-logit candidates at every
// draft position), ordered by value descending, then index ascending.
//
// Design (HBM-bound, one pass over the logits):
//   * Persistent grid: the rows*tiles_per_row 8 KB tiles are cut into equal
//     contiguous shares, one per CTA, so every SM streams the same number of
//     bytes whatever B*L is (16 rows at batch 1, 4096 at batch 256).
//   * One producer thread stages tiles into a 7-deep shared-memory ring with
//     bulk async copies (cp.async.bulk, completion on mbarriers); eight
//     consumer warps read the tiles from shared memory, two 16-byte vectors
//     per lane per tile (each warp: two blocks of 32 vectors).
//   * Bound: the first tiles of each row segment are held while every warp
//     reduces its block maxima; the 16th largest of those maxima (16 distinct
//     elements, so no larger than the row's 16th value) becomes the bound T.
//   * Candidates: every element >= T is appended, as a 64-bit key
//     (ordered value << 32 | ~index, unique, larger = better), to a shared
//     candidate buffer with one warp-aggregated atomic; a tile with no such
//     element costs two packed maxima and one vote per lane.  Past the
//     buffer's capacity a warp keeps its overflow in an exact per-warp list.
//   * Selection by rank: each thread counts the keys that beat its key (one
//     pass over shared memory, stopping at 16) and a key of rank r < 16 writes
//     itself to slot r.  Keys are unique, so this is the exact top 16 with no
//     sorting network.  Rows split across CTAs publish partial lists and the
//     last CTA to arrive (atomicInc ticket, which also resets itself) ranks
//     them.  No CTA ever waits for another.
#include <algorithm>

#include "dfl2_internal.cuh"

namespace dfl2 {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kTileBytes = 8192;
constexpr int kStages = 7;
constexpr int kMaxGrid = 2048;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kBlocksPerTile = 2 * kConsumerWarps;  // blocks of 32 vectors (512 bytes)
// Tiles at the start of each row segment that feed the block-maximum bound;
// later tiles skip the reduction and the CTA barrier.
constexpr int kBoundTiles = 3;
constexpr int kCandCap = 1024;   // candidate keys buffered per row segment
constexpr int kMinTilesPerCta = 4;
static_assert(kBoundTiles < kStages, "held bound tiles must leave the ring room to stream");
constexpr int kConsumers = kConsumerWarps * 32;
// [stages][full][empty][cand][extra: per-warp overflow lists][res][block maxima][flags]
constexpr size_t kSmemBytes = size_t(kStages) * kTileBytes + 2 * kStages * sizeof(uint64_t) +
                              size_t(kCandCap) * sizeof(uint64_t) +
                              size_t(kConsumerWarps) * kCand * sizeof(uint64_t) +
                              kCand * sizeof(uint64_t) +
                              size_t(kBoundTiles) * kBlocksPerTile * sizeof(float) + 32;
static_assert(kTileBytes == kBlocksPerTile * 32 * 16, "a tile is one iteration of all warps");

struct TopkArgs {
  const uint8_t* logits;
  int V;
  int tiles_per_row;
  long long total_tiles;
  int max_contrib;
  uint64_t* partial;
  uint32_t* tickets;
  int32_t* out_idx;
  float* out_val;
  uint32_t* err;
};

__device__ __forceinline__ uint64_t shfl64(uint64_t v, int src) {
  uint32_t lo = __shfl_sync(kFull, static_cast<uint32_t>(v), src);
  uint32_t hi = __shfl_sync(kFull, static_cast<uint32_t>(v >> 32), src);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl_xor64(uint64_t v, int m) {
  uint32_t lo = __shfl_xor_sync(kFull, static_cast<uint32_t>(v), m);
  uint32_t hi = __shfl_xor_sync(kFull, static_cast<uint32_t>(v >> 32), m);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Bitonic sort of one key per lane, descending across lanes 0..31.
__device__ __forceinline__ uint64_t warp_sort32_desc(uint64_t x, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t y = shfl_xor64(x, j);
      const bool keep_max = (((lane & j) == 0) == ((lane & k) == 0));
      x = keep_max ? (x > y ? x : y) : (x < y ? x : y);
    }
  }
  return x;
}

// Lanes 0..15 descending and lanes 16..31 ascending (a bitonic sequence) ->
// all 32 descending; the merged top 16 ends up in lanes 0..15.
__device__ __forceinline__ uint64_t warp_merge32_desc(uint64_t x, int lane) {
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const uint64_t y = shfl_xor64(x, j);
    x = ((lane & j) == 0) ? (x > y ? x : y) : (x < y ? x : y);
  }
  return x;
}

__device__ __forceinline__ uint64_t shfl_up64(uint64_t v, int d) {
  uint32_t lo = __shfl_up_sync(kFull, static_cast<uint32_t>(v), d);
  uint32_t hi = __shfl_up_sync(kFull, static_cast<uint32_t>(v >> 32), d);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Insert one key (the same in every lane) into the descending list in lanes 0..15.
__device__ __forceinline__ uint64_t insert_one(uint64_t list, uint64_t key, int lane) {
  const int pos = __popc(__ballot_sync(kFull, lane < 16 && list > key));
  const uint64_t up = shfl_up64(list, 1);
  if (lane >= 16) return 0ull;
  return lane < pos ? list : (lane == pos ? key : up);
}

// Merge 16 descending keys held in lanes 0..15 of `cand` into `list`.
__device__ __forceinline__ uint64_t merge_sorted16(uint64_t list, uint64_t cand, int lane) {
  const uint64_t rev = shfl64(cand, 31 - lane);
  return warp_merge32_desc(lane < 16 ? list : rev, lane);
}

__device__ __forceinline__ int owner_cta(long long g, long long T, int G) {
  return static_cast<int>(((g + 1) * G - 1) / T);
}

template <int EPV>  // elements per 16-byte vector: 4 (float32) or 8 (bf16)
__device__ __forceinline__ void unpack(const uint4& q, float (&f)[EPV]) {
  if constexpr (EPV == 4) {
    f[0] = __uint_as_float(q.x);
    f[1] = __uint_as_float(q.y);
    f[2] = __uint_as_float(q.z);
    f[3] = __uint_as_float(q.w);
  } else {
    const uint32_t r[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(r[i] << 16);
      f[2 * i + 1] = __uint_as_float(r[i] & 0xFFFF0000u);
    }
  }
}

__device__ __forceinline__ float warp_max_f(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, off));
  return x;
}

// Maximum of one 16-byte vector, as float.
template <int EPV>
__device__ __forceinline__ float vec_max(const uint4& q) {
  if constexpr (EPV == 4) {
    return fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)),
                 fmaxf(__uint_as_float(q.z), __uint_as_float(q.w)));
  } else {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&q.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&q.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&q.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&q.w);
    const __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
    return fmaxf(__low2float(m), __high2float(m));
  }
}

struct WarpTop {
  uint64_t list;  // lanes 0..15: this warp's overflow keys by rank, 0 = empty
  float bound;    // the segment's bound T
};

// Exact insertion of one key per lane (0 = none) into the warp's list.
__device__ __forceinline__ void insert_lane_keys(WarpTop& w, uint64_t cand, int lane) {
  const unsigned who = __ballot_sync(kFull, cand != 0);
  if (!who) return;
  if (__popc(who) <= 2) {
    unsigned rest = who;
    while (rest) {
      const int src = __ffs(rest) - 1;
      rest &= rest - 1;
      const uint64_t k = shfl64(cand, src);
      if (k > shfl64(w.list, 15)) w.list = insert_one(w.list, k, lane);
    }
  } else {
    w.list = merge_sorted16(w.list, warp_sort32_desc(cand, lane), lane);
  }
}

// The lane's elements at or above the bound go to the CTA candidate buffer
// (or, past its capacity, into the warp's own exact list).
template <int EPV>
__device__ __forceinline__ void collect_hits(WarpTop& w, const uint4& qa, const uint4& qb, bool va,
                                             bool vb, uint32_t idxA, uint32_t idxB, int lane,
                                             uint64_t* cand, uint32_t* cand_count) {
  float f[2 * EPV];
  {
    float fa[EPV], fb[EPV];
    unpack<EPV>(qa, fa);
    unpack<EPV>(qb, fb);
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      f[e] = fa[e];
      f[EPV + e] = fb[e];
    }
  }
  uint32_t mask = 0;
#pragma unroll
  for (int e = 0; e < 2 * EPV; ++e)
    if ((e < EPV ? va : vb) && f[e] >= w.bound) mask |= 1u << e;
  const int n = __popc(mask);
  int pre = n;  // inclusive warp scan of the counts
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(kFull, pre, off);
    if (lane >= off) pre += o;
  }
  const int total = __shfl_sync(kFull, pre, 31);
  uint32_t base = 0;
  if (lane == 0) base = atomicAdd(cand_count, static_cast<uint32_t>(total));
  base = __shfl_sync(kFull, base, 0);
  uint32_t pos = base + static_cast<uint32_t>(pre - n);
  uint32_t over = 0;  // elements that did not fit
#pragma unroll
  for (int e = 0; e < 2 * EPV; ++e) {
    if ((mask >> e) & 1u) {
      const uint64_t k = make_key(f[e], e < EPV ? idxA + e : idxB + (e - EPV));
      if (pos < kCandCap) cand[pos] = k;
      else over |= 1u << e;
      ++pos;
    }
  }
  while (__any_sync(kFull, over != 0)) {  // only once the buffer is full: exact per-warp list
    uint64_t k = 0;
    if (over) {
      const int e = __ffs(over) - 1;
      over &= over - 1;
      float v = f[0];
#pragma unroll
      for (int e2 = 1; e2 < 2 * EPV; ++e2) v = (e2 == e) ? f[e2] : v;
      k = make_key(v, e < EPV ? idxA + e : idxB + (e - EPV));
    }
    insert_lane_keys(w, k, lane);
  }
}

__device__ __forceinline__ void write_row(const TopkArgs& a, long long row, uint64_t key, int lane) {
  if (lane < kCand) {
    a.out_idx[row * kCand + lane] = static_cast<int32_t>(~static_cast<uint32_t>(key));
    a.out_val[row * kCand + lane] = unord_f32(static_cast<uint32_t>(key >> 32));
  }
}

// res[r] = the key of rank r (0-based, by descending key) among keys[0..n),
// for r < 16.  Keys are unique (0 = empty, skipped); res must hold zeros for
// ranks that no key takes.  All consumer threads call it; no barrier inside.
__device__ __forceinline__ void rank_select16(const uint64_t* keys, int n, uint64_t* res,
                                              int tid) {
  for (int i = tid; i < n; i += kConsumers) {
    const uint64_t k = keys[i];
    if (k == 0) continue;
    int r = 0;
    int j = 0;
    for (; j + 8 <= n && r < kCand; j += 8) {
#pragma unroll
      for (int u = 0; u < 8; ++u) r += keys[j + u] > k;
    }
    for (; j < n && r < kCand; ++j) r += keys[j] > k;
    if (r < kCand) res[r] = k;
  }
}

// The 16th largest of n block maxima (ties ranked by position); -inf if n < 16.
__device__ __forceinline__ void rank_bound(const float* bm, int n, float* out, int tid) {
  for (int i = tid; i < n; i += kConsumers) {
    const float v = bm[i];
    int r = 0;
    for (int j = 0; j < n; ++j) r += (bm[j] > v) || (bm[j] == v && j < i);
    if (r == kCand - 1) *out = v;
  }
}

template <int EPV>
__global__ void __launch_bounds__(kThreads, 3) topk16_kernel(TopkArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + size_t(kStages) * kTileBytes);
  uint64_t* empty_bar = full_bar + kStages;
  uint64_t* cand = empty_bar + kStages;                          // [kCandCap]
  uint64_t* extra = cand + kCandCap;                              // [kConsumerWarps][16]
  uint64_t* res = extra + kConsumerWarps * kCand;                 // [16]
  float* bmax = reinterpret_cast<float*>(res + kCand);            // [kBoundTiles][16]
  uint32_t* last_flag = reinterpret_cast<uint32_t*>(bmax + kBoundTiles * kBlocksPerTile);
  uint32_t* cand_count = last_flag + 1;
  float* bound_s = reinterpret_cast<float*>(cand_count + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long T = a.total_tiles;
  const int G = gridDim.x, c = blockIdx.x;
  const long long g0 = (long long)c * T / G, g1 = (long long)(c + 1) * T / G;
  const int tpr = a.tiles_per_row;
  const size_t row_bytes = size_t(a.V) * (16 / EPV);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConsumerWarps);
    }
    fence_mbar_init();
    *cand_count = 0u;
    for (int k = 0; k < kCand; ++k) res[k] = 0ull;
  }
  __syncthreads();
  pdl_wait();  // the logits may come from the previous kernel on the stream

  if (warp == kConsumerWarps) {  // producer
    if (lane == 0) {
      for (long long g = g0; g < g1; ++g) {
        const int i = static_cast<int>(g - g0), s = i % kStages;
        if (i >= kStages && !mbar_wait(&empty_bar[s], ((i / kStages) - 1) & 1))
          record_error(a.err, kDevErrTopkEmpty);
        const long long row = g / tpr;
        const size_t off = size_t(g % tpr) * kTileBytes;
        const uint32_t bytes = static_cast<uint32_t>(min(size_t(kTileBytes), row_bytes - off));
        mbar_arrive_expect_tx(&full_bar[s], bytes);
        bulk_g2s(stages + size_t(s) * kTileBytes, a.logits + size_t(row) * row_bytes + off, bytes,
                 &full_bar[s]);
      }
    }
    return;
  }

  long long g = g0;
  int i = 0, seg = 0;
  while (g < g1) {
    const long long row = g / tpr;
    const long long seg_end = min(g1, (row + 1) * tpr);
    WarpTop w{0ull, -INFINITY};
    const int nbound = static_cast<int>((seg_end - g < kBoundTiles ? seg_end - g : kBoundTiles));
    // ---- bound: hold the first nbound tiles, rank their block maxima ----
    uint4 hqa[kBoundTiles], hqb[kBoundTiles];
    bool hva[kBoundTiles], hvb[kBoundTiles];
    float hma[kBoundTiles], hmb[kBoundTiles];
    uint32_t hia[kBoundTiles], hib[kBoundTiles];
#pragma unroll
    for (int k = 0; k < kBoundTiles; ++k) {
      hva[k] = hvb[k] = false;
      hma[k] = hmb[k] = -INFINITY;
      hqa[k] = hqb[k] = make_uint4(0u, 0u, 0u, 0u);
      hia[k] = hib[k] = 0u;
      if (k < nbound) {
        const int s = (i + k) % kStages;
        if (!mbar_wait(&full_bar[s], ((i + k) / kStages) & 1)) record_error(a.err, kDevErrTopkFull);
        const int t = static_cast<int>((g + k) % tpr);
        const int nvec = static_cast<int>(min(size_t(kTileBytes), row_bytes - size_t(t) * kTileBytes) / 16);
        const uint32_t elem_base = static_cast<uint32_t>(t) * (kTileBytes / (16 / EPV));
        const uint4* tile = reinterpret_cast<const uint4*>(stages + size_t(s) * kTileBytes);
        const int v_a = warp * 64 + lane, v_b = v_a + 32;
        hva[k] = v_a < nvec;
        hvb[k] = v_b < nvec;
        if (hva[k]) hqa[k] = tile[v_a];
        if (hvb[k]) hqb[k] = tile[v_b];
        hma[k] = hva[k] ? vec_max<EPV>(hqa[k]) : -INFINITY;
        hmb[k] = hvb[k] ? vec_max<EPV>(hqb[k]) : -INFINITY;
        hia[k] = elem_base + static_cast<uint32_t>(v_a) * EPV;
        hib[k] = elem_base + static_cast<uint32_t>(v_b) * EPV;
        const float bma = warp_max_f(hma[k]), bmb = warp_max_f(hmb[k]);
        if (lane == 0) {
          bmax[k * kBlocksPerTile + 2 * warp] = bma;
          bmax[k * kBlocksPerTile + 2 * warp + 1] = bmb;
        }
      }
    }
    if (threadIdx.x == 0) *bound_s = -INFINITY;  // read last at the previous segment's start
    named_sync(1, kConsumers);
    rank_bound(bmax, nbound * kBlocksPerTile, bound_s, threadIdx.x);
    named_sync(1, kConsumers);
    w.bound = *bound_s;
#pragma unroll
    for (int k = 0; k < kBoundTiles; ++k) {
      if (k < nbound) {
        if (__any_sync(kFull, (hva[k] && hma[k] >= w.bound) || (hvb[k] && hmb[k] >= w.bound)))
          collect_hits<EPV>(w, hqa[k], hqb[k], hva[k], hvb[k], hia[k], hib[k], lane, cand,
                            cand_count);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[(i + k) % kStages]);
      }
    }
    g += nbound;
    i += nbound;
    // ---- stream the rest of the segment against the bound ----
    for (; g < seg_end; ++g, ++i) {
      const int s = i % kStages;
      if (!mbar_wait(&full_bar[s], (i / kStages) & 1)) record_error(a.err, kDevErrTopkFull);
      const int t = static_cast<int>(g % tpr);
      const size_t off = size_t(t) * kTileBytes;
      const int nvec = static_cast<int>(min(size_t(kTileBytes), row_bytes - off) / 16);
      const uint32_t elem_base = static_cast<uint32_t>(t) * (kTileBytes / (16 / EPV));
      const uint4* tile = reinterpret_cast<const uint4*>(stages + size_t(s) * kTileBytes);
      const int v_a = warp * 64 + lane, v_b = v_a + 32;
      const bool ok_a = v_a < nvec, ok_b = v_b < nvec;
      const uint4 qa = ok_a ? tile[v_a] : make_uint4(0u, 0u, 0u, 0u);
      const uint4 qb = ok_b ? tile[v_b] : make_uint4(0u, 0u, 0u, 0u);
      const float ma = ok_a ? vec_max<EPV>(qa) : -INFINITY;
      const float mb = ok_b ? vec_max<EPV>(qb) : -INFINITY;
      if (__any_sync(kFull, (ok_a && ma >= w.bound) || (ok_b && mb >= w.bound)))
        collect_hits<EPV>(w, qa, qb, ok_a, ok_b, elem_base + static_cast<uint32_t>(v_a) * EPV,
                          elem_base + static_cast<uint32_t>(v_b) * EPV, lane, cand, cand_count);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }

    // ---- the segment's top 16 by rank over the candidates (+ overflow lists) ----
    if (lane < kCand) extra[warp * kCand + lane] = w.list;
    named_sync(1, kConsumers);
    const uint32_t cnt = *reinterpret_cast<volatile uint32_t*>(cand_count);
    const int ncand = static_cast<int>(min(cnt, static_cast<uint32_t>(kCandCap)));
    // The overflow lists sit right after the buffer, so one ranking covers both.
    if (cnt > static_cast<uint32_t>(kCandCap)) {
      rank_select16(cand, kCandCap + kConsumerWarps * kCand, res, threadIdx.x);
    } else {
      rank_select16(cand, ncand, res, threadIdx.x);
    }
    const int c_first = owner_cta(row * tpr, T, G);
    const int c_last = owner_cta(row * tpr + tpr - 1, T, G);
    const int ncontrib = c_last - c_first + 1;
    uint64_t* part = a.partial + size_t(row) * a.max_contrib * kCand;
    named_sync(1, kConsumers);
    if (warp == 0) {
      const uint64_t x = lane < kCand ? res[lane] : 0ull;
      uint32_t last = 0;
      if (ncontrib == 1) {
        write_row(a, row, x, lane);
      } else {
        if (lane < kCand) part[(c - c_first) * kCand + lane] = x;
        __threadfence();
        __syncwarp();
        uint32_t ticket = 0;
        if (lane == 0) ticket = atomicInc(&a.tickets[row], static_cast<unsigned>(ncontrib - 1));
        last = __shfl_sync(kFull, ticket, 0) == static_cast<uint32_t>(ncontrib - 1);
      }
      if (lane < kCand) res[lane] = 0ull;
      if (lane == 0) {
        *last_flag = last;
        *cand_count = 0u;  // every warp has read it before the barrier above
      }
    }
    named_sync(1, kConsumers);
    if (*last_flag) {
      // Last CTA of a split row: rank the partial lists, kCandCap - 16 keys at a
      // time, carrying the running top 16 in front of each batch.
      __threadfence();
      const unsigned long long* pp = reinterpret_cast<const unsigned long long*>(part);
      const int total = ncontrib * kCand;
      constexpr int kBatchKeys = kCandCap - kCand;
      for (int b0 = 0; b0 < total; b0 += kBatchKeys) {
        const int nb = min(kBatchKeys, total - b0);
        for (int e = threadIdx.x; e < nb; e += kConsumers) cand[kCand + e] = __ldcg(pp + b0 + e);
        if (threadIdx.x < kCand) cand[threadIdx.x] = res[threadIdx.x];
        named_sync(1, kConsumers);
        if (threadIdx.x < kCand) res[threadIdx.x] = 0ull;
        named_sync(1, kConsumers);
        rank_select16(cand, kCand + nb, res, threadIdx.x);
        named_sync(1, kConsumers);
      }
      if (warp == 0) {
        write_row(a, row, lane < kCand ? res[lane] : 0ull, lane);
        if (lane < kCand) res[lane] = 0ull;
      }
      named_sync(1, kConsumers);
    }
    ++seg;
  }
  pdl_launch_dependents();
}

struct KernelSetup {
  bool done = false;
  int occ4 = 1, occ2 = 1;
};
KernelSetup g_setup[64];

cudaError_t ensure_setup(int dev, KernelSetup*& out) {
  KernelSetup& k = g_setup[dev & 63];
  if (!k.done) {
    cudaError_t e;
    e = cudaFuncSetAttribute(topk16_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(topk16_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k.occ4, topk16_kernel<4>, kThreads,
                                                      kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k.occ2, topk16_kernel<8>, kThreads,
                                                      kSmemBytes);
    if (e != cudaSuccess) return e;
    k.done = true;
  }
  out = &k;
  return cudaSuccess;
}

}  // namespace

TopkPlan topk_plan(int rows, int V, int elem_bytes) {
  TopkPlan p{};
  p.rows = rows;
  p.V = V;
  p.elem_bytes = elem_bytes;
  p.tiles_per_row = static_cast<int>((size_t(V) * elem_bytes + kTileBytes - 1) / kTileBytes);
  // Workspace stride: contributors per row are at most the row's tiles and at
  // most ceil(grid / rows) + 1; sized for float32 rows and the largest grid so
  // the size does not depend on the device or the dtype.
  const long long tiles_f32 = (size_t(V) * 4 + kTileBytes - 1) / kTileBytes;
  p.max_contrib = static_cast<int>(std::min<long long>(tiles_f32, (kMaxGrid + rows - 1) / rows + 1));
  p.partial_off = 256;
  p.ticket_off = align_up(p.partial_off + size_t(rows) * p.max_contrib * kCand * 8, 256);
  p.ws_bytes = align_up(p.ticket_off + size_t(rows) * 4, 256);
  p.grid = 0;  // filled by launch_topk from the device's SM count
  return p;
}

cudaError_t launch_topk(const TopkPlan& plan, const void* logits, int32_t* idx, float* val,
                        void* ws, cudaStream_t s, bool pdl) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  KernelSetup* k = nullptr;
  e = ensure_setup(dev, k);
  if (e != cudaSuccess) return e;
  const DeviceInfo info = device_info();
  const int occ = plan.elem_bytes == 4 ? k->occ4 : k->occ2;
  const long long T = (long long)plan.rows * plan.tiles_per_row;
  // One wave of resident CTAs, but no fewer than kMinTilesPerCta tiles per CTA
  // while that still puts one CTA on every SM (fewer partial lists per row).
  long long grid_l = std::min<long long>(kMaxGrid, (long long)info.sms * std::max(occ, 1));
  grid_l = std::min(grid_l, std::max<long long>(info.sms, (T + kMinTilesPerCta - 1) / kMinTilesPerCta));
  const int grid = static_cast<int>(std::min<long long>(T, grid_l));
  TopkArgs a;
  a.logits = static_cast<const uint8_t*>(logits);
  a.V = plan.V;
  a.tiles_per_row = plan.tiles_per_row;
  a.total_tiles = T;
  a.max_contrib = plan.max_contrib;
  a.partial = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(ws) + plan.partial_off);
  a.tickets = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + plan.ticket_off);
  a.out_idx = idx;
  a.out_val = val;
  a.err = device_error_word();
  if (plan.elem_bytes == 4)
    return launch_k(topk16_kernel<4>, dim3(grid), dim3(kThreads), kSmemBytes, s, pdl, a);
  return launch_k(topk16_kernel<8>, dim3(grid), dim3(kThreads), kSmemBytes, s, pdl, a);
}

}  // namespace dfl2
