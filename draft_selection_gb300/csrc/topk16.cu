// Top-16 per row of the drafter logits ("DFlash 2: Keep Drafting Parallel",
// 方法细节 > 轻量级路径选择器: keep the 16 highest-logit candidates at every
// draft position), ordered by value descending, then index ascending.
//
// Design (HBM-bound, one pass over the logits):
//   * Persistent grid: the rows*tiles_per_row 8 KB tiles are cut into equal
//     contiguous shares, one per CTA, so every SM streams the same number of
//     bytes whatever B*L is (16 rows at batch 1, 4096 at batch 256).
//   * One producer thread stages tiles into an 8-deep shared-memory ring with
//     bulk async copies (cp.async.bulk, completion on mbarriers); eight
//     consumer warps read the tiles from shared memory.
//   * Each consumer warp keeps an exact top-16 of 64-bit keys
//     (ordered value << 32 | ~index) in lanes 0..15.  A block of 256 elements
//     costs one max and one vote when nothing beats the warp's 16th value; the
//     rare hits are merged with a 32-lane bitonic sort + merge network.  The
//     value-only fast filter is exact because a warp meets its elements in
//     increasing index order, so an element equal to the 16th value always
//     loses the index tie-break.
//   * Per CTA the 8 warp lists are merged; rows split across CTAs publish
//     partial lists and the last CTA to arrive (atomicInc ticket, which also
//     resets itself) merges them.  No CTA ever waits for another.
#include <algorithm>

#include "dfl2_internal.cuh"

namespace dfl2 {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kTileBytes = 8192;
constexpr int kStages = 8;
constexpr int kMaxGrid = 2048;
constexpr unsigned kFull = 0xffffffffu;
constexpr size_t kSmemBytes = size_t(kStages) * kTileBytes + 2 * kStages * sizeof(uint64_t) +
                              2 * kConsumerWarps * kCand * sizeof(uint64_t) +
                              (2 + kConsumerWarps) * sizeof(uint32_t);
constexpr int kMergeBatch = 4;  // partial lists each warp loads at once in the final merge

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

struct WarpTop {
  uint64_t list;  // lanes 0..15: keys by rank, 0 = empty
  uint64_t thr;   // the 16th key (0 while fewer than 16 are held)
  float thr_v;    // its value
};

// cta_thr: the best 16th value any warp of this CTA holds for the current row
// (as an order-preserving uint32, 0 = none yet).  Some warp holds 16 elements
// at or above it, so an element strictly below it cannot be in the row's top 16.
template <int EPV>
__device__ __forceinline__ void process_block(WarpTop& w, const float (&f)[EPV], bool valid,
                                              uint32_t idx0, int lane, uint32_t* cta_thr,
                                              uint32_t* warp_v2, int warp) {
  float m = f[0];
#pragma unroll
  for (int e = 1; e < EPV; ++e) m = fmaxf(m, f[e]);
  const uint32_t shared_o = *reinterpret_cast<volatile uint32_t*>(cta_thr);
  const float shared_v = shared_o == 0u ? -INFINITY : unord_f32(shared_o);
  const bool hit = valid && !(m < shared_v) && (w.thr == 0 || m > w.thr_v);
  if (!__any_sync(kFull, hit)) return;
  uint32_t pend = 0;
  if (w.thr == 0) {
    // Empty list: seed it with the 16 best lane maxima in one sort.
    uint64_t lm = 0;
    if (valid) {
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const uint64_t k = make_key(f[e], idx0 + e);
        lm = k > lm ? k : lm;
      }
    }
    const uint64_t srt = warp_sort32_desc(lm, lane);
    w.list = merge_sorted16(w.list, srt, lane);
    w.thr = shfl64(w.list, 15);
    w.thr_v = unord_f32(static_cast<uint32_t>(w.thr >> 32));
    if (valid) {
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const uint64_t k = make_key(f[e], idx0 + e);
        if (k > w.thr && k != lm && !(f[e] < shared_v)) pend |= 1u << e;
      }
    }
  } else if (valid) {
#pragma unroll
    for (int e = 0; e < EPV; ++e)
      if (make_key(f[e], idx0 + e) > w.thr && !(f[e] < shared_v)) pend |= 1u << e;
  }
  while (true) {
    const unsigned who = __ballot_sync(kFull, pend != 0);
    if (!who) break;
    uint64_t cand = 0;
    if (pend) {
      const int e = __ffs(pend) - 1;
      pend &= pend - 1;
      float v = f[0];
#pragma unroll
      for (int e2 = 1; e2 < EPV; ++e2) v = (e2 == e) ? f[e2] : v;
      cand = make_key(v, idx0 + e);
    }
    if (__popc(who) <= 2) {
      // Few candidates (the common case once the list is warm): insert each directly.
      unsigned rest = who;
      while (rest) {
        const int src = __ffs(rest) - 1;
        rest &= rest - 1;
        const uint64_t k = shfl64(cand, src);
        if (k > shfl64(w.list, 15)) w.list = insert_one(w.list, k, lane);
      }
    } else {
      cand = warp_sort32_desc(cand, lane);
      w.list = merge_sorted16(w.list, cand, lane);
    }
    w.thr = shfl64(w.list, 15);
    w.thr_v = unord_f32(static_cast<uint32_t>(w.thr >> 32));
    if (pend) {
#pragma unroll
      for (int e = 0; e < EPV; ++e)
        if (((pend >> e) & 1u) && !(make_key(f[e], idx0 + e) > w.thr)) pend &= ~(1u << e);
    }
  }
  // Publish a tighter CTA bound: besides this warp's 16th value, the smallest of
  // the eight warps' 2nd-best values (8 warps x 2 elements at or above it).
  const uint64_t second = shfl64(w.list, 1);
  if (lane == 0) {
    if (second != 0) warp_v2[warp] = static_cast<uint32_t>(second >> 32);
    uint32_t m2 = 0xFFFFFFFFu;
#pragma unroll
    for (int k = 0; k < 8; ++k) m2 = min(m2, *reinterpret_cast<volatile uint32_t*>(&warp_v2[k]));
    const uint32_t own = w.thr != 0 ? static_cast<uint32_t>(w.thr >> 32) : 0u;
    const uint32_t bound = max(own, m2);
    if (bound != 0u) atomicMax(cta_thr, bound);
  }
}

__device__ __forceinline__ void write_row(const TopkArgs& a, long long row, uint64_t key, int lane) {
  if (lane < kCand) {
    a.out_idx[row * kCand + lane] = static_cast<int32_t>(~static_cast<uint32_t>(key));
    a.out_val[row * kCand + lane] = unord_f32(static_cast<uint32_t>(key >> 32));
  }
}

template <int EPV>
__global__ void __launch_bounds__(kThreads) topk16_kernel(TopkArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + size_t(kStages) * kTileBytes);
  uint64_t* empty_bar = full_bar + kStages;
  uint64_t* merge_buf = empty_bar + kStages;  // [2][kConsumerWarps][16]
  uint32_t* cta_thr = reinterpret_cast<uint32_t*>(merge_buf + 2 * kConsumerWarps * kCand);
  uint32_t* last_flag = cta_thr + 1;
  uint32_t* warp_v2 = cta_thr + 2;  // [kConsumerWarps] each warp's 2nd-best value, ordered

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
    *cta_thr = 0u;
    for (int k = 0; k < kConsumerWarps; ++k) warp_v2[k] = 0u;
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
    WarpTop w{0ull, 0ull, 0.f};
    for (; g < seg_end; ++g, ++i) {
      const int s = i % kStages;
      if (!mbar_wait(&full_bar[s], (i / kStages) & 1)) record_error(a.err, kDevErrTopkFull);
      const int t = static_cast<int>(g % tpr);
      const size_t off = size_t(t) * kTileBytes;
      const int nvec = static_cast<int>(min(size_t(kTileBytes), row_bytes - off) / 16);
      const uint32_t elem_base = static_cast<uint32_t>(t) * (kTileBytes / (16 / EPV));
      const uint4* tile = reinterpret_cast<const uint4*>(stages + size_t(s) * kTileBytes);
      for (int v0 = warp * 32; v0 < nvec; v0 += kConsumerWarps * 32) {
        const int v = v0 + lane;
        const bool valid = v < nvec;
        uint4 q = valid ? tile[v] : make_uint4(0u, 0u, 0u, 0u);
        float f[EPV];
        unpack<EPV>(q, f);
        process_block<EPV>(w, f, valid, elem_base + static_cast<uint32_t>(v) * EPV, lane,
                           cta_thr, warp_v2, warp);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }

    // Merge the warps' lists for this row segment.
    uint64_t* mb = merge_buf + (seg & 1) * kConsumerWarps * kCand;
    if (lane < kCand) mb[warp * kCand + lane] = w.list;
    const int c_first = owner_cta(row * tpr, T, G);
    const int c_last = owner_cta(row * tpr + tpr - 1, T, G);
    const int ncontrib = c_last - c_first + 1;
    uint64_t* part = a.partial + size_t(row) * a.max_contrib * kCand;
    named_sync(1, kConsumerWarps * 32);
    if (warp == 0) {
      uint64_t x = w.list;
      for (int w2 = 1; w2 < kConsumerWarps; ++w2)
        x = warp_merge32_desc(lane < 16 ? x : mb[w2 * kCand + ((31 - lane) & 15)], lane);
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
      if (lane == 0) {
        *last_flag = last;
        *cta_thr = 0u;  // the next segment is another row
        for (int k = 0; k < kConsumerWarps; ++k) warp_v2[k] = 0u;
      }
    }
    named_sync(1, kConsumerWarps * 32);
    if (*last_flag) {
      // Last CTA of a split row: every warp merges a share of the partial lists,
      // loading kMergeBatch lists at a time, then warp 0 merges the warps' results.
      __threadfence();
      const unsigned long long* pp = reinterpret_cast<const unsigned long long*>(part);
      uint64_t acc = 0;
      for (int k0 = warp; k0 < ncontrib; k0 += kConsumerWarps * kMergeBatch) {
        uint64_t y[kMergeBatch];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          const int k = k0 + u * kConsumerWarps;
          y[u] = k < ncontrib ? __ldcg(pp + k * kCand + ((31 - lane) & 15)) : 0ull;
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) acc = warp_merge32_desc(lane < 16 ? acc : y[u], lane);
      }
      uint64_t* mb2 = merge_buf + ((seg + 1) & 1) * kConsumerWarps * kCand;
      if (lane < kCand) mb2[warp * kCand + lane] = acc;
      named_sync(1, kConsumerWarps * 32);
      if (warp == 0) {
        uint64_t x = acc;
        for (int w2 = 1; w2 < kConsumerWarps; ++w2)
          x = warp_merge32_desc(lane < 16 ? x : mb2[w2 * kCand + ((31 - lane) & 15)], lane);
        write_row(a, row, x, lane);
      }
      named_sync(1, kConsumerWarps * 32);
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
  const int grid = static_cast<int>(std::min<long long>(T, std::min(kMaxGrid, info.sms * std::max(occ, 1))));
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
