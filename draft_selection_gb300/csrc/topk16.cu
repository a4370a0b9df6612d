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
//   * Bound: the first tiles of each row segment are held while every lane
//     takes the maximum of its own elements in them; the 16th largest of those
//     lane maxima (maxima of 16 disjoint element sets, so no larger than the
//     segment's 16th value) becomes the bound T.  Each warp sorts its 32 lane
//     maxima and the 16th largest of the union is found by rank with binary
//     searches over the other warps' sorted lists.
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
constexpr int kVecPerLane = kTileBytes / 16 / 32;  // 16-byte vectors per lane per tile
constexpr int kStages = 8;
constexpr int kMaxGrid = 2048;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kCandCap = 1024;   // candidate keys buffered per row segment
constexpr int kRaise = 64;       // candidates per bound-raising window (2 per lane)
constexpr int kMinTilesPerCta = 4;
constexpr int kConsumers = kConsumerWarps * 32;
// [stages][full][empty][cand][extra: per-warp overflow lists][res][lane maxima][flags]
constexpr size_t kSmemBytes = size_t(kStages) * kTileBytes + 2 * kStages * sizeof(uint64_t) +
                              size_t(kCandCap) * sizeof(uint64_t) +
                              size_t(kConsumerWarps) * kCand * sizeof(uint64_t) +
                              kCand * sizeof(uint64_t) +
                              size_t(kConsumerWarps) * kCand * sizeof(float) + 32;  // flags: 5 words
static_assert(kVecPerLane <= 32, "hit masks are 32 bits");
static_assert((size_t(kStages) * kTileBytes + 2 * kStages * 8 + size_t(kCandCap) * 8 +
               size_t(kConsumerWarps) * kCand * 8 + kCand * 8) % 16 == 0,
              "the lane-maximum lists are read 16 bytes at a time");
static_assert(kStages >= kConsumerWarps, "the held bound tiles must fit in the ring");

struct TopkArgs {
  const uint8_t* logits;
  int V, rows;
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

// Bitonic sort of one float per lane, descending across lanes 0..31.
__device__ __forceinline__ float warp_sort32_desc_f(float x, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float y = __shfl_xor_sync(kFull, x, j);
      const bool keep_max = (((lane & j) == 0) == ((lane & k) == 0));
      x = keep_max ? fmaxf(x, y) : fminf(x, y);
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

// The lane's elements of one 16-byte vector at or above the bound go to the
// CTA candidate buffer with one warp-aggregated atomic (or, past its
// capacity, into the warp's own exact list).
template <int EPV>
__device__ __forceinline__ void collect_vec(WarpTop& w, const uint4& q, bool valid, uint32_t idx0,
                                            int lane, uint64_t* cand, uint32_t* cand_count,
                                            uint32_t* raise_s) {
  float f[EPV];
  unpack<EPV>(q, f);
  uint32_t mask = 0;
#pragma unroll
  for (int e = 0; e < EPV; ++e)
    if (valid && f[e] >= w.bound) mask |= 1u << e;
  const int n = __popc(mask);
  const unsigned who = __ballot_sync(kFull, n != 0);
  if (!who) return;
  int pre, total;
  uint32_t base;
  if ((who & (who - 1)) == 0) {  // one lane hits (the common case): no scan
    const int src = __ffs(who) - 1;
    total = __shfl_sync(kFull, n, src);
    pre = n;
    uint32_t b0 = 0;
    if (lane == src) b0 = atomicAdd(cand_count, static_cast<uint32_t>(n));
    base = __shfl_sync(kFull, b0, src);
  } else {
    pre = n;  // inclusive warp scan of the counts
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(kFull, pre, off);
      if (lane >= off) pre += o;
    }
    total = __shfl_sync(kFull, pre, 31);
    uint32_t b0 = 0;
    if (lane == 0) b0 = atomicAdd(cand_count, static_cast<uint32_t>(total));
    base = __shfl_sync(kFull, b0, 0);
  }
  uint32_t pos = base + static_cast<uint32_t>(pre - n);
  uint32_t over = 0;  // elements that did not fit
#pragma unroll
  for (int e = 0; e < EPV; ++e) {
    if ((mask >> e) & 1u) {
      if (pos < kCandCap) cand[pos] = make_key(f[e], idx0 + e);
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
      for (int e2 = 1; e2 < EPV; ++e2) v = (e2 == e) ? f[e2] : v;
      k = make_key(v, idx0 + e);
    }
    insert_lane_keys(w, k, lane);
  }
  // Raising the bound: the warp whose keys complete a window of kRaise buffer
  // slots ranks that window (two slots per lane, the lane's larger one).  The
  // 16th largest of those 32 maxima stands for 16 distinct elements of the
  // segment, so it is still a lower bound on the segment's 16th value.  Slots
  // other warps have reserved but not yet written read as empty (the buffer is
  // cleared at every segment's end), which only lowers the result.
  const uint32_t end = base + static_cast<uint32_t>(total);
  if (end / kRaise != base / kRaise && end <= static_cast<uint32_t>(kCandCap)) {
    __syncwarp();
    const uint32_t m0 = (end / kRaise - 1) * kRaise;
    const volatile uint64_t* wnd = cand + m0;
    const uint64_t k0 = wnd[2 * lane], k1 = wnd[2 * lane + 1];
    float v = -INFINITY;
    if (k0 != 0ull) v = unord_f32(static_cast<uint32_t>(k0 >> 32));
    if (k1 != 0ull) v = fmaxf(v, unord_f32(static_cast<uint32_t>(k1 >> 32)));
    v = warp_sort32_desc_f(v, lane);
    const float nb = __shfl_sync(kFull, v, kCand - 1);
    if (nb > w.bound) {
      w.bound = nb;
      if (lane == 0) atomicMax(raise_s, ord_f32(nb));
    }
  }
}

// One warp's pass over one staged tile: the lane reads vectors lane + 32*j,
// j < 16; vectors whose maximum reaches the bound are re-read and collected.
template <int EPV>
__device__ __forceinline__ void scan_tile(WarpTop& w, const uint4* tile, int nvec, uint32_t elem_base,
                                          int lane, uint64_t* cand, uint32_t* cand_count,
                                          uint32_t* raise_s) {
  uint32_t hit = 0;
#pragma unroll
  for (int j = 0; j < kVecPerLane; ++j) {
    const int v = lane + 32 * j;
    if (v < nvec && vec_max<EPV>(tile[v]) >= w.bound) hit |= 1u << j;
  }
  uint32_t any = __reduce_or_sync(kFull, hit);
  while (any) {
    const int j = __ffs(any) - 1;
    any &= any - 1;
    const int v = lane + 32 * j;
    const bool ok = v < nvec;
    const uint4 q = ok ? tile[v] : make_uint4(0u, 0u, 0u, 0u);
    collect_vec<EPV>(w, q, ok, elem_base + static_cast<uint32_t>(v) * EPV, lane, cand, cand_count,
                     raise_s);
  }
}

// The lane's maximum over its vectors of a staged tile.
template <int EPV>
__device__ __forceinline__ float lane_max_tile(const uint4* tile, int nvec, int lane) {
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < kVecPerLane; ++j) {
    const int v = lane + 32 * j;
    if (v < nvec) m = fmaxf(m, vec_max<EPV>(tile[v]));
  }
  return m;
}


// A logits row as streamed: the 16-byte-aligned window [lo, hi) of the flat
// logits buffer around the row's bytes [s, e).  Rows need not start on 16
// bytes (V * element size may be any even number); the buffer's bytes past its
// last whole 16 bytes (floor16) cannot be bulk-copied and are read by plain
// loads (finish_tile).
struct RowWin {
  size_t s, e, lo, hi;
};
__device__ __forceinline__ RowWin row_window(long long row, size_t rb, size_t floor16) {
  RowWin w;
  w.s = size_t(row) * rb;
  w.e = w.s + rb;
  w.lo = w.s & ~size_t(15);
  w.hi = min((w.e + 15) & ~size_t(15), floor16);
  return w;
}
// Bytes the bulk copy moves for tile t of a window (0 past its end).
__device__ __forceinline__ uint32_t tile_bytes(const RowWin& w, int t) {
  const size_t a = w.lo + size_t(t) * kTileBytes;
  return a < w.hi ? static_cast<uint32_t>(min(size_t(kTileBytes), w.hi - a)) : 0u;
}
// Row index of tile t's first element, as a 32-bit value that wraps below 0
// (the window may start up to 7 elements before the row).
template <int EPV>
__device__ __forceinline__ uint32_t tile_ebase(const RowWin& w, int t) {
  constexpr int es = 16 / EPV;
  return static_cast<uint32_t>(static_cast<long long>(t) * (kTileBytes / es) -
                               static_cast<long long>((w.s - w.lo) / es));
}
// Completes a staged tile before the one warp that scans it does so.  The
// window's elements outside the row (before its start, after its end) become
// -inf: their keys carry indices outside [0, V), which rank below every
// element of the row, so with V >= 16 none is ever selected.  The row's
// elements past the buffer's last whole 16 bytes (its last row only) are read
// with plain loads into the vector after the copied bytes.  Every lane calls
// it; returns the tile's vector count.
template <int EPV>
__device__ __forceinline__ int finish_tile(uint8_t* tile, int t, const RowWin& w, size_t floor16,
                                           const uint8_t* logits, int lane) {
  constexpr int es = 16 / EPV;
  const size_t a = w.lo + size_t(t) * kTileBytes;  // flat byte of the tile's start
  int nbytes = static_cast<int>(tile_bytes(w, t));
  if (lane == 0 && ((w.s | w.e) & 15)) {
    auto neg_inf = [&](size_t g) {  // element at flat byte g of this tile
      if constexpr (es == 2)
        *reinterpret_cast<uint16_t*>(tile + (g - a)) = 0xFF80u;
      else
        *reinterpret_cast<uint32_t*>(tile + (g - a)) = 0xFF800000u;
    };
    bool wrote = false;
    if (w.e > floor16 && floor16 >= a && floor16 < a + kTileBytes) {
      for (size_t g = floor16; g < floor16 + 16; g += es) {
        if (g < w.e) {
          if constexpr (es == 2)
            *reinterpret_cast<uint16_t*>(tile + (g - a)) = *reinterpret_cast<const uint16_t*>(logits + g);
          else
            *reinterpret_cast<uint32_t*>(tile + (g - a)) = *reinterpret_cast<const uint32_t*>(logits + g);
        } else {
          neg_inf(g);
        }
      }
      nbytes = static_cast<int>(floor16 - a) + 16;
      wrote = true;
    }
    if (t == 0 && w.s > w.lo) {
      for (size_t g = w.lo; g < w.s; g += es) neg_inf(g);
      wrote = true;
    }
    if ((w.e & 15) && w.e <= floor16 && w.e >= a && w.e < a + size_t(nbytes)) {
      for (size_t g = w.e; g < ((w.e + 15) & ~size_t(15)); g += es) neg_inf(g);
      wrote = true;
    }
    // these generic writes come before the next bulk copy into the stage
    if (wrote) fence_proxy_async_smem();
  }
  nbytes = __shfl_sync(kFull, nbytes, 0);
  __syncwarp();
  return nbytes / 16;
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

// lm holds kConsumerWarps descending lists of 16 lane maxima.  Entry (w, i)
// ranks as i plus, in every other list w2, the entries above it (ties go to
// the lower list), counted with independent 16-byte loads; the entry of rank
// 15 is the 16th largest of the union.
__device__ __forceinline__ void rank_bound(const float* lm, float* out, int tid) {
  if (tid >= kConsumerWarps * kCand) return;
  const int w = tid / kCand;
  const float v = lm[tid];
  int r = tid % kCand;
#pragma unroll
  for (int w2 = 0; w2 < kConsumerWarps; ++w2) {
    if (w2 == w) continue;
    const float4* L2 = reinterpret_cast<const float4*>(lm + w2 * kCand);
    const bool lower = w2 < w;
#pragma unroll
    for (int q = 0; q < kCand / 4; ++q) {
      const float4 e = L2[q];
      r += (e.x > v || (lower && e.x == v)) + (e.y > v || (lower && e.y == v)) +
           (e.z > v || (lower && e.z == v)) + (e.w > v || (lower && e.w == v));
    }
  }
  if (r == kCand - 1) *out = v;
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
  float* lmax = reinterpret_cast<float*>(res + kCand);            // [kConsumerWarps][16]
  uint32_t* last_flag = reinterpret_cast<uint32_t*>(lmax + kConsumerWarps * kCand);
  uint32_t* cand_count = last_flag + 1;
  float* bound_s = reinterpret_cast<float*>(cand_count + 1);
  uint32_t* raise_s = reinterpret_cast<uint32_t*>(bound_s + 1);  // raised bound, ordered bits
  uint32_t* issued = raise_s + 1;  // tiles the producer has issued so far

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long T = a.total_tiles;
  const int G = gridDim.x, c = blockIdx.x;
  const long long g0 = (long long)c * T / G, g1 = (long long)(c + 1) * T / G;
  const int tpr = a.tiles_per_row;
  const size_t row_bytes = size_t(a.V) * (16 / EPV);
  const size_t floor16 = (size_t(a.rows) * row_bytes) & ~size_t(15);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);  // the one warp that scans the tile
    }
    fence_mbar_init();
    *cand_count = 0u;
    *issued = 0u;
    for (int k = 0; k < kCand; ++k) res[k] = 0ull;
  }
  for (int e = threadIdx.x; e < kCandCap; e += kThreads) cand[e] = 0ull;
  __syncthreads();
  pdl_wait();  // the logits may come from the previous kernel on the stream

  if (warp == kConsumerWarps) {  // producer
    if (lane == 0) {
      long long row = g0 / tpr;
      int t = static_cast<int>(g0 - row * tpr);
      const int n = static_cast<int>(g1 - g0);
      for (int i = 0, s = 0, ph = 0; i < n; ++i) {
        if (i >= kStages && !mbar_wait(&empty_bar[s], ph ^ 1, a.err)) record_error(a.err, kDevErrTopkEmpty);
        const RowWin win = row_window(row, row_bytes, floor16);
        const uint32_t bytes = tile_bytes(win, t);
        mbar_arrive_expect_tx(&full_bar[s], bytes);
        if (bytes)
          bulk_g2s(stages + size_t(s) * kTileBytes, a.logits + win.lo + size_t(t) * kTileBytes,
                   bytes, &full_bar[s]);
        st_release_cta(issued, static_cast<uint32_t>(i + 1));
        if (++t == tpr) {
          t = 0;
          ++row;
        }
        if (++s == kStages) {
          s = 0;
          ph ^= 1;
        }
      }
    }
    return;
  }

  // Tile i of this CTA (0-based over its share) sits in stage i % kStages and
  // is scanned by warp i % kConsumerWarps.  Warps do not move in step, so a
  // warp may reach tile i while the producer still waits to reuse the stage
  // for tile i - kStages: the stage's full barrier is then two phases behind
  // and its parity alone cannot tell.  A warp therefore first waits until the
  // producer has issued tile i (which it does only after tile i - kStages was
  // released), and only then on the barrier's parity.
  long long g = g0;
  long long row = g0 / tpr;
  int t0 = static_cast<int>(g0 - row * tpr);  // tile of the row where the segment starts
  int i0 = 0;                                  // CTA tile index where the segment starts
  while (g < g1) {
    const long long seg_end = min(g1, (row + 1) * tpr);
    const int nseg = static_cast<int>(seg_end - g);
    const int nbound = nseg < kConsumerWarps ? nseg : kConsumerWarps;
    WarpTop w{0ull, -INFINITY};
    // this warp's first tile of the segment (segment-relative)
    const int jw = ((warp - i0) % kConsumerWarps + kConsumerWarps) % kConsumerWarps;
    auto tile_of = [&](int j, const uint4*& tile, int& nvec, uint32_t& elem_base) {
      const int i = i0 + j, st = i % kStages;
      if (!wait_count_above(issued, static_cast<uint32_t>(i), a.err) ||
          !mbar_wait(&full_bar[st], (i / kStages) & 1, a.err))
        record_error(a.err, kDevErrTopkFull);
      const int t = t0 + j;
      const RowWin win = row_window(row, row_bytes, floor16);
      nvec = finish_tile<EPV>(stages + size_t(st) * kTileBytes, t, win, floor16, a.logits, lane);
      elem_base = tile_ebase<EPV>(win, t);
      tile = reinterpret_cast<const uint4*>(stages + size_t(st) * kTileBytes);
    };
    auto release = [&](int j) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[(i0 + j) % kStages]);
    };
    // ---- bound: the first nbound tiles (one per warp) stay staged while every
    // lane takes its maximum over them; the 16th largest lane maximum is T ----
    {
      float lm = -INFINITY;
      if (jw < nbound) {
        const uint4* tile;
        int nvec;
        uint32_t eb;
        tile_of(jw, tile, nvec, eb);
        lm = lane_max_tile<EPV>(tile, nvec, lane);
      }
      // the lane's rank in its warp from 32 independent shuffles (ties by lane):
      // the warp's best 16 land in lmax in descending order
      int r = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float o = __shfl_sync(kFull, lm, j);
        r += (o > lm) || (o == lm && j < lane);
      }
      if (r < kCand) lmax[warp * kCand + r] = lm;
    }
    if (threadIdx.x == 0) {  // both read last at the previous segment's start
      *bound_s = -INFINITY;
      *raise_s = ord_f32(-INFINITY);
    }
    named_sync(1, kConsumers);
    rank_bound(lmax, bound_s, threadIdx.x);
    named_sync(1, kConsumers);
    w.bound = *bound_s;
    // ---- every tile of the segment against the bound (the held one first) ----
    for (int j = jw; j < nseg; j += kConsumerWarps) {
      const uint4* tile;
      int nvec;
      uint32_t eb;
      tile_of(j, tile, nvec, eb);
      w.bound = fmaxf(w.bound, unord_f32(*reinterpret_cast<volatile uint32_t*>(raise_s)));
      scan_tile<EPV>(w, tile, nvec, eb, lane, cand, cand_count, raise_s);
      release(j);
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
    const bool was_last = *last_flag != 0u;
    if (was_last) {
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
    // Clear the slots this segment used: the next segment's bound raises read
    // slots that are reserved but not yet written as empty.
    {
      const int used = was_last ? kCandCap : ncand;
      for (int e = threadIdx.x; e < used; e += kConsumers) cand[e] = 0ull;
    }
    g = seg_end;
    i0 += nseg;
    ++row;
    t0 = 0;
  }
  pdl_launch_dependents();
}

// ============================================================================
// Few rows (batch 1 and small batches): one thread-block cluster per row.
//
// The persistent kernel above balances any number of rows, but at batch 1 its
// per-segment bound, ranking and the global ticket merge of about ten partial
// lists per row form a long dependent chain.  Here the C CTAs of a cluster
// share one row (C <= 8), each streaming at most kRMaxTilesPerCta tiles, and
// the chain is kept short: warp-collective sorting networks (tens of
// dependent shuffles each) are replaced by counting that runs in parallel.
//   * Each lane takes its maximum key (value, then lowest index) over its
//     vectors of the warp's first tile; a lane learns its rank among the
//     warp's 32 maxima from 32 independent shuffles, which lays out each
//     warp's best 16 in order, and binary searches in the other warps' lists
//     rank those 128.  The 16th largest, T, bounds the CTA's share of the row
//     (16 distinct elements reach it).
//   * Every element whose key reaches T is appended to a shared buffer (a few
//     dozen; a key bound also caps all-tied rows); the CTA's top 16 follow by
//     counting, for each candidate, the candidates above it.
//   * The CTAs hand their 16 keys to the cluster's first CTA through
//     distributed shared memory and arrive on its mbarrier; it ranks the C
//     lists by binary search in each.  No global atomics or fences.
// ============================================================================
constexpr int kRStages = 8;       // clusters of C > 1 CTAs per row (few tiles per CTA)
constexpr int kRStagesRow = 12;   // one CTA per row (a whole row streams through the ring)
constexpr int kRowLoopCtasPerSm = 2;  // resident CTAs of the row-looping kernel per SM
constexpr int kRMaxCluster = 8;
constexpr int kRMaxTilesPerCta = 16;
constexpr int kRCandCap = 1024;
// Shared memory: [stages][full][empty][list barrier, pad][cand][extra][res]
// [cluster lists][lane maxima][their top 16][flags]; every region after the
// barriers starts on a 16-byte boundary (the lists are read 16 bytes at a time).
template <int NST>
struct RowsLayout {
  static constexpr size_t bars = size_t(NST) * kTileBytes;
  static constexpr size_t cand = bars + (2 * NST + 2) * sizeof(uint64_t);
  static constexpr size_t extra = cand + size_t(kRCandCap) * sizeof(uint64_t);
  static constexpr size_t res = extra + size_t(kConsumerWarps) * kCand * sizeof(uint64_t);
  static constexpr size_t clists = res + kCand * sizeof(uint64_t);
  static constexpr size_t wsorted = clists + size_t(kRMaxCluster) * kCand * sizeof(uint64_t);
  static constexpr size_t tres = wsorted + size_t(kConsumerWarps) * kCand * sizeof(uint64_t);
  static constexpr size_t flags = tres + kCand * sizeof(uint64_t);
  static constexpr size_t bytes = flags + 16;
  static_assert(cand % 16 == 0 && extra % 16 == 0 && res % 16 == 0 && clists % 16 == 0 &&
                    wsorted % 16 == 0 && tres % 16 == 0,
                "16-byte aligned regions");
};
static_assert(kConsumerWarps <= kRMaxCluster, "lists ranked by rank_sorted_lists16");

struct RowsArgs {
  const uint8_t* logits;
  int V, rows, tiles_per_row, C;
  int32_t* out_idx;
  float* out_val;
  uint32_t* err;
};

__device__ __forceinline__ void st_cluster_u64(uint32_t addr, uint64_t v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

// The lane's largest key over its vectors of a staged tile (0 if it has none);
// vm receives the vectors' maximum values.
template <int EPV>
__device__ __forceinline__ uint64_t lane_max_key(const uint4* tile, int nvec, uint32_t elem_base,
                                                 int lane, float (&vm)[kVecPerLane]) {
  float lm = -INFINITY;
#pragma unroll
  for (int j = 0; j < kVecPerLane; ++j) {
    const int v = lane + 32 * j;
    vm[j] = v < nvec ? vec_max<EPV>(tile[v]) : -INFINITY;
    lm = fmaxf(lm, vm[j]);
  }
  uint32_t at = 0;  // vectors holding the maximum
#pragma unroll
  for (int j = 0; j < kVecPerLane; ++j)
    if (lane + 32 * j < nvec && vm[j] == lm) at |= 1u << j;
  if (at == 0u) return 0ull;
  const int v = lane + 32 * (__ffs(at) - 1);
  float f[EPV];
  unpack<EPV>(tile[v], f);
  uint32_t em = 0;
#pragma unroll
  for (int e = 0; e < EPV; ++e)
    if (f[e] == lm) em |= 1u << e;  // -0.0 == +0.0, as the keys treat them
  return make_key(lm, elem_base + static_cast<uint32_t>(v) * EPV + (__ffs(em) - 1));
}

// The lane's keys >= T (other than `skip`) over the vectors in `hit`, in a
// fixed order; calls f(key) for each.
template <int EPV, typename F>
__device__ __forceinline__ void for_keys_at_least(const uint4* tile, uint32_t hit, uint32_t elem_base,
                                                  int lane, uint64_t T, float bval, uint64_t skip,
                                                  F&& f) {
  for (uint32_t h = hit; h; h &= h - 1) {
    const int j = __ffs(h) - 1;
    const int v = lane + 32 * j;
    float x[EPV];
    unpack<EPV>(tile[v], x);
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      if (x[e] < bval) continue;
      const uint64_t k = make_key(x[e], elem_base + static_cast<uint32_t>(v) * EPV + e);
      if (k >= T && k != skip) f(k);
    }
  }
}

// Appends the lane's keys >= T (other than `skip`) to `cand` (capacity
// kRCandCap - 16) with one atomic per lane; keys past the capacity go, one per
// lane per round, into the warp's exact list.
template <int EPV>
__device__ __forceinline__ void append_tile_keys(WarpTop& w, const uint4* tile, int nvec,
                                                 uint32_t elem_base, const float (&vm)[kVecPerLane],
                                                 uint64_t T, float bval, uint64_t skip, int lane,
                                                 uint64_t* cand, uint32_t* cand_count) {
  constexpr uint32_t kCap = kRCandCap - kCand;
  uint32_t hit = 0;
#pragma unroll
  for (int j = 0; j < kVecPerLane; ++j)
    if (lane + 32 * j < nvec && vm[j] >= bval) hit |= 1u << j;
  uint32_t c = 0;
  uint64_t k1 = 0ull, k2 = 0ull;  // the first two, kept to spare a second pass
  for_keys_at_least<EPV>(tile, hit, elem_base, lane, T, bval, skip, [&](uint64_t k) {
    if (c == 0) k1 = k;
    else if (c == 1) k2 = k;
    ++c;
  });
  const uint32_t pos = c ? atomicAdd(cand_count, c) : 0u;
  const uint32_t first_spill = pos + c > kCap ? (pos >= kCap ? 0u : kCap - pos) : c;
  if (c <= 2) {
    if (c > 0 && first_spill > 0) cand[pos] = k1;
    if (c > 1 && first_spill > 1) cand[pos + 1] = k2;
  } else {
    uint32_t o = 0;
    for_keys_at_least<EPV>(tile, hit, elem_base, lane, T, bval, skip, [&](uint64_t k) {
      if (o < first_spill) cand[pos + o] = k;
      ++o;
    });
  }
  // Rare: the buffer is full.  Each lane offers its spilled keys, largest
  // first, one per round.
  bool spill = first_spill < c;
  uint64_t last = ~0ull;
  while (__any_sync(kFull, spill)) {
    uint64_t best = 0ull;
    if (spill) {
      uint32_t o = 0;
      for_keys_at_least<EPV>(tile, hit, elem_base, lane, T, bval, skip, [&](uint64_t k) {
        if (o >= first_spill && k < last && k > best) best = k;
        ++o;
      });
      if (best == 0ull) spill = false;
    }
    insert_lane_keys(w, best, lane);
    last = best;
  }
}

// res[r] for r < 16: the key of rank r among n lists of 16 keys (0 = empty,
// skipped; keys unique); thread t < 16n places key t of list t/16, given its
// rank inside its own list (lists are descending), by counting the keys above
// it in the other lists: independent loads, no dependent search.
__device__ __forceinline__ void rank_lists16(const uint64_t* lists, int n, uint64_t* res, int tid) {
  if (tid >= n * kCand) return;
  const uint64_t v = lists[tid];
  if (v == 0ull) return;
  const int own = tid / kCand;
  int r = tid % kCand;
  for (int l = 0; l < n; ++l) {
    if (l == own) continue;
    const ulonglong2* L = reinterpret_cast<const ulonglong2*>(lists + l * kCand);
#pragma unroll
    for (int q = 0; q < kCand / 2; ++q) {
      const ulonglong2 p = L[q];
      r += (p.x > v) + (p.y > v);
    }
  }
  if (r < kCand) res[r] = v;
}

template <int EPV, int NST>
__global__ void __launch_bounds__(kThreads, 2) topk16_rows_kernel(RowsArgs a) {
  using Lay = RowsLayout<NST>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + Lay::bars);
  uint64_t* empty_bar = full_bar + NST;
  uint64_t* list_bar = empty_bar + NST;  // first CTA: the others' lists arrived
  uint64_t* cand = reinterpret_cast<uint64_t*>(smem + Lay::cand);       // [kRCandCap]
  uint64_t* extra = reinterpret_cast<uint64_t*>(smem + Lay::extra);     // [kConsumerWarps][16]
  uint64_t* res = reinterpret_cast<uint64_t*>(smem + Lay::res);         // [16]
  uint64_t* clists = reinterpret_cast<uint64_t*>(smem + Lay::clists);   // [kRMaxCluster][16]
  uint64_t* wsorted = reinterpret_cast<uint64_t*>(smem + Lay::wsorted); // [warps][16] lane maxima
  uint64_t* tres = reinterpret_cast<uint64_t*>(smem + Lay::tres);       // [16] their top 16
  uint32_t* cand_count = reinterpret_cast<uint32_t*>(smem + Lay::flags);
  uint32_t* issued = cand_count + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = a.C, rank = static_cast<int>(blockIdx.x) % C;
  const long long row = blockIdx.x / C;
  const int tpr = a.tiles_per_row;
  const int t_lo = rank * tpr / C, t_hi = (rank + 1) * tpr / C;  // this CTA's tiles of the row
  const int n = t_hi - t_lo;
  const size_t row_bytes = size_t(a.V) * (16 / EPV);
  const size_t floor16 = (size_t(a.rows) * row_bytes) & ~size_t(15);
  const RowWin win = row_window(row, row_bytes, floor16);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(list_bar, C > 1 ? C - 1 : 1);
    fence_mbar_init();
    *issued = 0u;
    *cand_count = 0u;
  }
  if (threadIdx.x < kCand) {
    res[threadIdx.x] = 0ull;
    tres[threadIdx.x] = 0ull;
  }
  if (threadIdx.x < kConsumerWarps * kCand) wsorted[threadIdx.x] = 0ull;
  __syncthreads();
  if (C > 1) cluster_arrive_release();  // the list barrier is initialised (waited before use)
  pdl_wait();  // the logits may come from the previous kernel on the stream

  if (warp == kConsumerWarps) {  // producer
    if (lane == 0) {
      for (int i = 0, s = 0, ph = 0; i < n; ++i) {
        if (i >= NST && !mbar_wait(&empty_bar[s], ph ^ 1, a.err)) record_error(a.err, kDevErrTopkEmpty);
        const uint32_t bytes = tile_bytes(win, t_lo + i);
        mbar_arrive_expect_tx(&full_bar[s], bytes);
        if (bytes)
          bulk_g2s(stages + size_t(s) * kTileBytes,
                   a.logits + win.lo + size_t(t_lo + i) * kTileBytes, bytes, &full_bar[s]);
        st_release_cta(issued, static_cast<uint32_t>(i + 1));
        if (++s == NST) {
          s = 0;
          ph ^= 1;
        }
      }
    }
    if (C > 1) cluster_wait_acquire();
  } else {
    // Warp w scans tiles w, w + 8, ...: each stage serves one warp only.
    auto stage_of = [&](int i, const uint4*& tile, int& nvec, uint32_t& eb) {
      const int st = i % NST;
      if (!wait_count_above(issued, static_cast<uint32_t>(i), a.err) ||
          !mbar_wait(&full_bar[st], (i / NST) & 1, a.err))
        record_error(a.err, kDevErrTopkFull);
      const int t = t_lo + i;
      nvec = finish_tile<EPV>(stages + size_t(st) * kTileBytes, t, win, floor16, a.logits, lane);
      eb = tile_ebase<EPV>(win, t);
      tile = reinterpret_cast<const uint4*>(stages + size_t(st) * kTileBytes);
    };
    WarpTop w{0ull, -INFINITY};
    float vm[kVecPerLane];
    const uint4* tile = nullptr;
    int nvec = 0;
    uint32_t eb = 0;
    // ---- the bound T: the 16th largest lane-maximum key over the CTA's first
    // wave of tiles.  A lane's rank in its warp (32 shuffles) puts the warp's
    // best 16 in order; the 128 are then ranked by binary search. ----
    uint64_t lk = 0ull;
    if (warp < n) {
      stage_of(warp, tile, nvec, eb);
      lk = lane_max_key<EPV>(tile, nvec, eb, lane, vm);
    }
    {
      int r = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) r += shfl64(lk, j) > lk;
      if (r < kCand && lk != 0ull) wsorted[warp * kCand + r] = lk;
    }
    const int nw = n < kConsumerWarps ? n : kConsumerWarps;
    named_sync(1, kConsumers);
    rank_lists16(wsorted, nw, tres, threadIdx.x);
    named_sync(1, kConsumers);
    const uint64_t T = tres[kCand - 1];  // 0 (fewer than 16 keys): accept all
    const float bval = T ? unord_f32(static_cast<uint32_t>(T >> 32)) : -INFINITY;
    // ---- candidates.  With T set, the 16 lane maxima at or above it (tres)
    // are in; a lane that holds one adds its other elements >= T (rare), and
    // later tiles add every element >= T.  Without T every element goes in.
    // Slots 0..15 hold tres, appended keys start at 16. ----
    if (threadIdx.x < kCand) cand[threadIdx.x] = T ? tres[threadIdx.x] : 0ull;
    for (int i = warp; i < n; i += kConsumerWarps) {
      if (i != warp) {
        stage_of(i, tile, nvec, eb);
#pragma unroll
        for (int j = 0; j < kVecPerLane; ++j) {
          const int v = lane + 32 * j;
          vm[j] = v < nvec ? vec_max<EPV>(tile[v]) : -INFINITY;
        }
        append_tile_keys<EPV>(w, tile, nvec, eb, vm, T, bval, 0ull, lane, cand + kCand,
                              cand_count);
      } else if (T == 0ull) {
        append_tile_keys<EPV>(w, tile, nvec, eb, vm, 0ull, -INFINITY, 0ull, lane, cand + kCand,
                              cand_count);
      } else {
        // only a lane whose maximum reaches T can hold more; its maximum is in tres
        const bool holds = lk >= T;
        float vmh[kVecPerLane];
#pragma unroll
        for (int j = 0; j < kVecPerLane; ++j) vmh[j] = holds ? vm[j] : -INFINITY;
        append_tile_keys<EPV>(w, tile, nvec, eb, vmh, T, bval, lk, lane, cand + kCand, cand_count);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[i % NST]);
    }
    if (lane < kCand) extra[warp * kCand + lane] = w.list;
    named_sync(1, kConsumers);
    const uint32_t cnt = *reinterpret_cast<volatile uint32_t*>(cand_count);
    if (cnt == 0u && T != 0ull) {
      if (threadIdx.x < kCand) res[threadIdx.x] = tres[threadIdx.x];  // already in rank order
    } else {
      // The overflow lists sit right after the buffer, so one ranking covers both.
      rank_select16(cand, cnt > static_cast<uint32_t>(kRCandCap - kCand)
                              ? kRCandCap + kConsumerWarps * kCand
                              : kCand + static_cast<int>(cnt),
                    res, threadIdx.x);
    }
    named_sync(1, kConsumers);
    // ---- this CTA's 16 keys (descending: res[r] has rank r) to the first CTA ----
    if (C == 1) {
      if (threadIdx.x < kCand) clists[threadIdx.x] = res[threadIdx.x];
    } else {
      if (warp == 0) cluster_wait_acquire();
      if (rank == 0) {
        if (threadIdx.x < kCand) clists[threadIdx.x] = res[threadIdx.x];
      } else if (threadIdx.x == 0) {
#pragma unroll
        for (int q = 0; q < kCand; ++q)
          st_cluster_u64(dsmem_addr(clists + rank * kCand + q, 0u), res[q]);
        mbar_arrive_remote(list_bar, 0u);  // release: the 16 stores above come first
      }
      if (warp != 0) cluster_wait_acquire();
    }
  }
  if (rank == 0 && warp < kConsumerWarps) {
    if (C > 1 && !mbar_wait_cluster(list_bar, 0, a.err)) record_error(a.err, kDevErrTopkFull);
    named_sync(1, kConsumers);  // the first CTA's own list is in place too
    if (threadIdx.x < kCand) res[threadIdx.x] = 0ull;
    named_sync(1, kConsumers);
    rank_lists16(clists, C, res, threadIdx.x);
    named_sync(1, kConsumers);
    if (threadIdx.x < kCand) {
      const uint64_t key = res[threadIdx.x];
      a.out_idx[row * kCand + threadIdx.x] = static_cast<int32_t>(~static_cast<uint32_t>(key));
      a.out_val[row * kCand + threadIdx.x] = unord_f32(static_cast<uint32_t>(key >> 32));
    }
  }
  pdl_launch_dependents();
}

// One CTA per row, persistent over rows: CTA c takes rows c, c + G, c + 2G, ...
// (G = gridDim.x) and its producer streams their tiles back to back through the
// ring, so the next row's first tiles arrive while the consumers rank the
// current one.  Per row, the same steps as the cluster kernel with C = 1: the
// bound from the first wave of tiles, every element at or above it appended,
// the top 16 by rank.  Tile i of the CTA (counted over its rows) sits in stage
// i % NST; a consumer waits for the producer to have issued it before the
// stage's parity (the producer may be a whole ring ahead).
template <int EPV, int NST>
__global__ void __launch_bounds__(kThreads, 2) topk16_row_loop_kernel(RowsArgs a) {
  using Lay = RowsLayout<NST>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + Lay::bars);
  uint64_t* empty_bar = full_bar + NST;
  uint64_t* cand = reinterpret_cast<uint64_t*>(smem + Lay::cand);       // [kRCandCap]
  uint64_t* extra = reinterpret_cast<uint64_t*>(smem + Lay::extra);     // [kConsumerWarps][16]
  uint64_t* res = reinterpret_cast<uint64_t*>(smem + Lay::res);         // [16]
  uint64_t* wsorted = reinterpret_cast<uint64_t*>(smem + Lay::wsorted); // [warps][16] lane maxima
  uint64_t* tres = reinterpret_cast<uint64_t*>(smem + Lay::tres);       // [16] their top 16
  uint32_t* cand_count = reinterpret_cast<uint32_t*>(smem + Lay::flags);
  uint32_t* issued = cand_count + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long G = gridDim.x;
  const int n = a.tiles_per_row;
  const size_t row_bytes = size_t(a.V) * (16 / EPV);
  const size_t floor16 = (size_t(a.rows) * row_bytes) & ~size_t(15);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    fence_mbar_init();
    *issued = 0u;
    *cand_count = 0u;
  }
  if (threadIdx.x < kCand) {
    res[threadIdx.x] = 0ull;
    tres[threadIdx.x] = 0ull;
  }
  if (threadIdx.x < kConsumerWarps * kCand) wsorted[threadIdx.x] = 0ull;
  __syncthreads();
  pdl_wait();  // the logits may come from the previous kernel on the stream

  if (warp == kConsumerWarps) {  // producer
    if (lane == 0) {
      uint32_t i = 0;
      int s = 0, ph = 0;
      for (long long row = blockIdx.x; row < a.rows; row += G) {
        const RowWin win = row_window(row, row_bytes, floor16);
        for (int t = 0; t < n; ++t, ++i) {
          if (i >= uint32_t(NST) && !mbar_wait(&empty_bar[s], ph ^ 1, a.err))
            record_error(a.err, kDevErrTopkEmpty);
          const uint32_t bytes = tile_bytes(win, t);
          mbar_arrive_expect_tx(&full_bar[s], bytes);
          if (bytes)
            bulk_g2s(stages + size_t(s) * kTileBytes, a.logits + win.lo + size_t(t) * kTileBytes,
                     bytes, &full_bar[s]);
          st_release_cta(issued, i + 1);
          if (++s == NST) {
            s = 0;
            ph ^= 1;
          }
        }
      }
    }
  } else {
    uint32_t base = 0;  // CTA tile index of the row's first tile
    for (long long row = blockIdx.x; row < a.rows; row += G, base += uint32_t(n)) {
      const RowWin win = row_window(row, row_bytes, floor16);
      auto stage_of = [&](int j, const uint4*& tile, int& nvec, uint32_t& eb) {
        const uint32_t i = base + uint32_t(j);
        const int st = int(i % NST);
        if (!wait_count_above(issued, i, a.err) || !mbar_wait(&full_bar[st], (i / NST) & 1, a.err))
          record_error(a.err, kDevErrTopkFull);
        nvec = finish_tile<EPV>(stages + size_t(st) * kTileBytes, j, win, floor16, a.logits, lane);
        eb = tile_ebase<EPV>(win, j);
        tile = reinterpret_cast<const uint4*>(stages + size_t(st) * kTileBytes);
      };
      WarpTop w{0ull, -INFINITY};
      float vm[kVecPerLane];
      const uint4* tile = nullptr;
      int nvec = 0;
      uint32_t eb = 0;
      // ---- the bound T over the row's first wave of tiles (as in the cluster kernel) ----
      uint64_t lk = 0ull;
      if (warp < n) {
        stage_of(warp, tile, nvec, eb);
        lk = lane_max_key<EPV>(tile, nvec, eb, lane, vm);
      }
      {
        int r = 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) r += shfl64(lk, j) > lk;
        if (r < kCand && lk != 0ull) wsorted[warp * kCand + r] = lk;
      }
      const int nw = n < kConsumerWarps ? n : kConsumerWarps;
      named_sync(1, kConsumers);
      rank_lists16(wsorted, nw, tres, threadIdx.x);
      named_sync(1, kConsumers);
      const uint64_t T = tres[kCand - 1];  // 0 (fewer than 16 keys): accept all
      const float bval = T ? unord_f32(static_cast<uint32_t>(T >> 32)) : -INFINITY;
      if (threadIdx.x < kCand) cand[threadIdx.x] = T ? tres[threadIdx.x] : 0ull;
      for (int j = warp; j < n; j += kConsumerWarps) {
        if (j != warp) {
          stage_of(j, tile, nvec, eb);
#pragma unroll
          for (int q = 0; q < kVecPerLane; ++q) {
            const int v = lane + 32 * q;
            vm[q] = v < nvec ? vec_max<EPV>(tile[v]) : -INFINITY;
          }
          append_tile_keys<EPV>(w, tile, nvec, eb, vm, T, bval, 0ull, lane, cand + kCand,
                                cand_count);
        } else if (T == 0ull) {
          append_tile_keys<EPV>(w, tile, nvec, eb, vm, 0ull, -INFINITY, 0ull, lane, cand + kCand,
                                cand_count);
        } else {
          const bool holds = lk >= T;
          float vmh[kVecPerLane];
#pragma unroll
          for (int q = 0; q < kVecPerLane; ++q) vmh[q] = holds ? vm[q] : -INFINITY;
          append_tile_keys<EPV>(w, tile, nvec, eb, vmh, T, bval, lk, lane, cand + kCand,
                                cand_count);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[(base + uint32_t(j)) % NST]);
      }
      if (lane < kCand) extra[warp * kCand + lane] = w.list;
      named_sync(1, kConsumers);
      const uint32_t cnt = *reinterpret_cast<volatile uint32_t*>(cand_count);
      if (cnt == 0u && T != 0ull) {
        if (threadIdx.x < kCand) res[threadIdx.x] = tres[threadIdx.x];  // already in rank order
      } else {
        rank_select16(cand, cnt > static_cast<uint32_t>(kRCandCap - kCand)
                                ? kRCandCap + kConsumerWarps * kCand
                                : kCand + static_cast<int>(cnt),
                      res, threadIdx.x);
      }
      named_sync(1, kConsumers);
      if (threadIdx.x < kCand) {
        const uint64_t key = res[threadIdx.x];
        a.out_idx[row * kCand + threadIdx.x] = static_cast<int32_t>(~static_cast<uint32_t>(key));
        a.out_val[row * kCand + threadIdx.x] = unord_f32(static_cast<uint32_t>(key >> 32));
      }
      named_sync(1, kConsumers);  // every read of this row's lists is done
      // the next row starts from empty lists (the candidate slots it ranks are
      // the ones it writes: below its own count, or all of them on overflow)
      if (threadIdx.x < kCand) {
        res[threadIdx.x] = 0ull;
        tres[threadIdx.x] = 0ull;
      }
      if (threadIdx.x < kConsumerWarps * kCand) wsorted[threadIdx.x] = 0ull;
      if (threadIdx.x == 0) *cand_count = 0u;
      named_sync(1, kConsumers);
    }
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
    e = cudaFuncSetAttribute(topk16_rows_kernel<4, kRStages>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(RowsLayout<kRStages>::bytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(topk16_rows_kernel<8, kRStages>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(RowsLayout<kRStages>::bytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(topk16_rows_kernel<4, kRStagesRow>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(RowsLayout<kRStagesRow>::bytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(topk16_rows_kernel<8, kRStagesRow>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(RowsLayout<kRStagesRow>::bytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(topk16_row_loop_kernel<4, kRStagesRow>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(RowsLayout<kRStagesRow>::bytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(topk16_row_loop_kernel<8, kRStagesRow>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(RowsLayout<kRStagesRow>::bytes));
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
  // tiles of a row's 16-byte-aligned window (up to 30 bytes wider than the row
  // when rows do not start on 16 bytes)
  const size_t rb = size_t(V) * elem_bytes, win = rb % 16 ? rb + 30 : rb;
  p.tiles_per_row = static_cast<int>((win + kTileBytes - 1) / kTileBytes);
  // Workspace stride: contributors per row are at most the row's tiles and at
  // most ceil(grid / rows) + 1; sized for float32 rows and the largest grid so
  // the size does not depend on the device or the dtype.
  const long long tiles_f32 = (size_t(V) * 4 + 30 + kTileBytes - 1) / kTileBytes;
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
  // Few rows: one cluster of C CTAs per row while the clusters fit in about one
  // wave (two CTAs per SM) and each CTA streams at most kRMaxTilesPerCta tiles
  // (ring of kRStages).  Rows enough to give every SM a CTA: one CTA per row,
  // each streaming whole rows through a deeper ring, looping over its share of
  // the rows (1,024 rows of 151,936 bf16: 72 us against 91 for the persistent
  // kernel, whose row segments, bound phases and cross-CTA merges stall its
  // rings).  Otherwise (few rows of many tiles) the persistent kernel spreads
  // the tiles over the whole GPU.
  {
    int C = std::min(kRMaxCluster, plan.tiles_per_row);
    while (C > 1 && (long long)plan.rows * C > 2LL * info.sms) C >>= 1;
    const bool clusters = (long long)plan.rows * C <= 2LL * info.sms &&
                          (plan.tiles_per_row + C - 1) / C <= kRMaxTilesPerCta;
    const bool per_row = !clusters && plan.rows >= info.sms;
    if (clusters || per_row) {
      if (per_row) C = 1;
      RowsArgs r;
      r.logits = static_cast<const uint8_t*>(logits);
      r.V = plan.V;
      r.rows = plan.rows;
      r.tiles_per_row = plan.tiles_per_row;
      r.C = C;
      r.out_idx = idx;
      r.out_val = val;
      r.err = device_error_word();
      const dim3 grid(static_cast<unsigned>(plan.rows * C));
      if (per_row) {
        constexpr size_t smem = RowsLayout<kRStagesRow>::bytes;
        // the fewest rows per CTA that fit the resident CTAs, spread evenly
        // (serving_b64: 4 rows on each of 256 CTAs measured 72.4 us, against
        // 73.4 for 304 CTAs of 3-4 rows and 73.7 for one row per CTA)
        const long long slots = kRowLoopCtasPerSm * (long long)info.sms;
        const long long per = (plan.rows + slots - 1) / slots;
        const dim3 lgrid(static_cast<unsigned>((plan.rows + per - 1) / per));
        if (plan.elem_bytes == 4)
          return launch_k(topk16_row_loop_kernel<4, kRStagesRow>, lgrid, dim3(kThreads), smem, s, pdl, r);
        return launch_k(topk16_row_loop_kernel<8, kRStagesRow>, lgrid, dim3(kThreads), smem, s, pdl, r);
      }
      constexpr size_t smem = RowsLayout<kRStages>::bytes;
      if (plan.elem_bytes == 4)
        return launch_kc(topk16_rows_kernel<4, kRStages>, grid, dim3(kThreads), smem, s, pdl, C, r);
      return launch_kc(topk16_rows_kernel<8, kRStages>, grid, dim3(kThreads), smem, s, pdl, C, r);
    }
  }
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
  a.rows = plan.rows;
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
