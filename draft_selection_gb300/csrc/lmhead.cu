// LM head + top-16 in one pass: logits U_t(v) = <h_t, W_lm[v]> for every row t
// of the drafter's last hidden state and every vocabulary entry v, reduced to
// the 16 largest per row (value descending, index ascending) inside the GEMM's
// epilogue, so that the [rows, V] logits never reach HBM.  The top-16 step is
// the selector's first step ("DFlash 2: Keep Drafting Parallel", 方法细节 >
// 轻量级路径选择器, the candidates U_t(.) the pair score reads); the LM head
// that produces U_t(.) is the step before it.
//
// lmhead_topk_kernel: a tcgen05 GEMM.  Rows of h (128 per tile) sit on the TMEM
// lanes, vocabulary entries (256 per tile) on the accumulator columns; both
// operands are K-major bf16, loaded by TMA in the 128-byte swizzle layout; the
// accumulator (fp32) is double-buffered in TMEM (2 x 256 columns) so that the
// epilogue of tile i overlaps the MMAs of tile i+1.  The CTAs of one row tile
// split the vocabulary into contiguous ranges and all run at once, so each
// W_lm tile is fetched from HBM once and served from L2 to the row tiles.
// Eight epilogue warps (two per TMEM lane quarter, one per half of the
// columns) each keep, per thread (= one row), a sorted register list of the 16
// best keys seen so far; a value enters only if it beats the list's 16th and
// is not below the 16th of the row's other half (shared through shared
// memory).  Each thread visits its columns in increasing vocabulary order, so
// a tie with the 16th (equal value, higher index) correctly stays out.  At the
// end the two halves' lists of a row are merged, and each CTA writes one list
// of 16 keys per row.
//
// lmhead_merge_kernel: per row, the top 16 of the vsplits partial lists, one
// warp per 32 lists (lane = list), by sixteen rounds of "take the largest head
// across the warp"; more than 32 lists go through a second round over the
// warps' results.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "dfl2_internal.cuh"

namespace dfl2 {
namespace {

constexpr int kLBM = 128;                  // hidden rows per tile (TMEM lanes)
constexpr int kLBN = 256;                  // vocabulary entries per tile (fp32 columns)
constexpr int kLBK = 64;                   // K per stage: one 128-byte swizzle row of bf16
constexpr int kLMaxStages = 5;
constexpr int kLEpiWarps = 8;              // two per TMEM lane quarter
constexpr int kLThreads = (2 + kLEpiWarps) * 32;
constexpr int kLHalf = kLBN / 2;           // columns per epilogue warp per tile
constexpr int kLAStage = kLBM * kLBK * 2;  // 16 KB
constexpr int kLBStage = kLBN * kLBK * 2;  // 32 KB
constexpr uint32_t kLTmemCols = 2 * kLBN;  // two accumulators
constexpr size_t kLBarBytes = (2 * kLMaxStages + 8) * sizeof(uint64_t);
constexpr size_t kLThrBytes = 2 * kLBM * sizeof(float);           // per half, per row
constexpr size_t kLPairBytes = size_t(kLBM) * kCand * sizeof(uint64_t);  // half 1's lists
constexpr size_t kLFixedBytes = 1024 + kLBarBytes + kLThrBytes + kLPairBytes;
constexpr size_t kLSmemMax = 232448;  // the opt-in shared memory of one CTA
// Stage s holds the h tile (a_rows rows, rounded up to a 1024-byte swizzle
// atom) and then the W_lm tile.  The MMA reads 128 rows of h from the stage's
// start; with fewer rows loaded the rest falls inside the same stage (over the
// W_lm tile) and only feeds accumulator rows past R, which nobody reads.
__host__ __device__ constexpr int lm_a_bytes(int a_rows) { return (a_rows * 128 + 1023) / 1024 * 1024; }
__host__ __device__ constexpr int lm_stage_bytes(int a_rows) { return lm_a_bytes(a_rows) + kLBStage; }
static_assert(lm_stage_bytes(8) >= kLAStage, "the MMA's 128-row read of h stays in its stage");
static_assert(kLFixedBytes + 4 * size_t(lm_stage_bytes(128)) <= kLSmemMax, "four full stages fit");
constexpr int kLMaxSplits = 256;           // CTAs per row tile (workspace bound)
constexpr unsigned kAll = 0xffffffffu;

struct LmArgs {
  int R, V, d;
  int vsplits;      // CTAs sharing one row tile's vocabulary
  int ntiles;       // ceil(V / 256)
  int kblocks;      // ceil(d / 64); K past d reads zeros
  int a_rows;       // rows of the hidden box: R rounded up to 8, at most 128
  int stages;       // pipeline stages: 4 or 5 (more measured slower at B*L = 16)
  uint64_t* lists;  // [R][vsplits][16] descending keys (0 = empty)
  uint32_t* err;
};

__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// Waits for every tcgen05.ld of this thread; names r as its output so that the
// compiler neither reads nor moves r before it.
__device__ __forceinline__ void tmem_ld32_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// Insert (x, ix) into the list (values descending, equal values by ascending
// index), x strictly above the last value.  ix is larger than every index in
// the list, so x goes after the values >= x: its slot is where "x > lv[q]"
// first holds, the entries from there on move down one, and the last falls
// out.  The 16 compares are independent, as are the 16 moves.
__device__ __forceinline__ void list_insert_vi(float (&lv)[kCand], int (&li)[kCand], float x,
                                               int ix) {
  bool gt[kCand];
#pragma unroll
  for (int q = 0; q < kCand; ++q) gt[q] = x > lv[q];
#pragma unroll
  for (int q = kCand - 1; q > 0; --q) {
    lv[q] = gt[q] ? (gt[q - 1] ? lv[q - 1] : x) : lv[q];
    li[q] = gt[q] ? (gt[q - 1] ? li[q - 1] : ix) : li[q];
  }
  lv[0] = gt[0] ? x : lv[0];
  li[0] = gt[0] ? ix : li[0];
}

// One 32-column chunk of a row (the thread's TMEM lane): a bit per column
// that beats the list's 16th value and is not below the other half's, then,
// per set bit in column order, the insertion (re-checked against the risen
// bound).  Columns at or past lim are padding.
__device__ __forceinline__ void scan_chunk(const uint32_t (&r)[32], int c, int lim, int vbase,
                                           float (&lv)[kCand], int (&li)[kCand],
                                           volatile float* my_thr,
                                           volatile const float* other_thr) {
  const float floor_v = *other_thr;
  const float thr = lv[kCand - 1];
  // x passes iff x > thr and x >= floor_v: one strict compare against t
  const float t = floor_v > thr ? nextafterf(floor_v, -INFINITY) : thr;
  uint32_t m = 0;
#pragma unroll
  for (int q = 0; q < 32; ++q) m |= (__uint_as_float(r[q]) > t ? 1u : 0u) << q;
  const int valid = lim - c;
  if (valid < 32) m &= valid <= 0 ? 0u : ((1u << valid) - 1u);
  while (m) {
    const int q = __ffs(m) - 1;
    m &= m - 1;
    // r[q] by a tree of selects on the bits of q (no local memory)
    float s16[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) s16[j] = __uint_as_float((q & 16) ? r[j + 16] : r[j]);
    float s8[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) s8[j] = (q & 8) ? s16[j + 8] : s16[j];
    float s4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) s4[j] = (q & 4) ? s8[j + 4] : s8[j];
    const float s2a = (q & 2) ? s4[2] : s4[0], s2b = (q & 2) ? s4[3] : s4[1];
    const float x = (q & 1) ? s2b : s2a;
    if (x > lv[kCand - 1] && x >= floor_v) {
      list_insert_vi(lv, li, x, vbase + c + q);
      *my_thr = lv[kCand - 1];
    }
  }
}

__global__ void __launch_bounds__(kLThreads, 1)
    lmhead_topk_kernel(const __grid_constant__ LmArgs a, const __grid_constant__ CUtensorMap tmH,
                       const __grid_constant__ CUtensorMap tmW) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int nst = a.stages;
  const int sbytes = lm_stage_bytes(a.a_rows), abytes = lm_a_bytes(a.a_rows);
  uint8_t* stage0 = smem;  // [stages][h rows | 256 W_lm rows][128 B]
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + size_t(nst) * sbytes);
  uint64_t* empty_bar = full_bar + kLMaxStages;
  uint64_t* accf_bar = empty_bar + kLMaxStages;  // [2] accumulator b complete
  uint64_t* acce_bar = accf_bar + 2;          // [2] accumulator b read out
  uint64_t* done_bar = acce_bar + 2;          // the MMA issuer's last commit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  float* thr_s = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full_bar) + kLBarBytes);
  uint64_t* pair = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(thr_s) + kLThrBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int vs = blockIdx.x;
  const int m0 = blockIdx.y * kLBM;
  const int t_lo = static_cast<int>((long long)vs * a.ntiles / a.vsplits);
  const int t_hi = static_cast<int>((long long)(vs + 1) * a.ntiles / a.vsplits);
  const int nt = t_hi - t_lo;  // >= 1: vsplits <= ntiles

  if (tid == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf_bar[b], 1);
      mbar_init(&acce_bar[b], kLEpiWarps);
    }
    mbar_init(done_bar, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmH);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kLTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  // Every CTA of this grid is resident once all have passed this point, so the
  // merge kernel may be scheduled (it waits for this grid's completion itself).
  pdl_launch_dependents();

  // A wait that runs out records the error and ends that role's loop; the
  // producer then waits (bounded) for its copies in flight and the MMA issuer
  // for its MMAs, so the CTA leaves no asynchronous work behind.
  if (warp == 0) {
    if (lane == 0) {  // ---- producer: the h tile and the W_lm tile of each K block ----
      const uint32_t tx = static_cast<uint32_t>(a.a_rows * 128 + kLBStage);
      int s = 0, ph = 0, it = 0;
      bool ok = true;
      for (int i = 0; i < nt && ok; ++i) {
        const int n0 = (t_lo + i) * kLBN;
        for (int kb = 0; kb < a.kblocks; ++kb, ++it) {
          if (it >= nst && !mbar_wait(&empty_bar[s], ph ^ 1, a.err)) {
            record_error(a.err, kDevErrGemm);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_bar[s], tx);
          uint8_t* st = stage0 + size_t(s) * sbytes;
          tma_load_2d(st, &tmH, kb * kLBK, m0, &full_bar[s]);
          tma_load_2d(st + abytes, &tmW, kb * kLBK, n0, &full_bar[s]);
          if (++s == nst) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      // the last (up to nst) copies issued: their phases complete when they land
      for (int back = 1; back <= nst && back <= it; ++back) {
        const int j = it - back;
        mbar_wait(&full_bar[j % nst], (j / nst) & 1, a.err);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issuer ----
      const uint32_t idesc = umma_idesc_bf16(kLBM, kLBN);
      int s = 0, ph = 0;
      bool ok = true;
      for (int i = 0; i < nt && ok; ++i) {
        const int b = i & 1;
        if (i >= 2 && !mbar_wait(&acce_bar[b], ((i >> 1) - 1) & 1, a.err)) {
          record_error(a.err, kDevErrGemm);
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + static_cast<uint32_t>(b * kLBN);
        for (int kb = 0; kb < a.kblocks; ++kb) {
          if (!mbar_wait(&full_bar[s], ph, a.err)) {
            record_error(a.err, kDevErrGemm);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* st = stage0 + size_t(s) * sbytes;
          const uint64_t ad = umma_desc_sw128(st);
          const uint64_t bd = umma_desc_sw128(st + abytes);
#pragma unroll
          for (int k = 0; k < kLBK / 16; ++k)
            umma_bf16(acc, ad + 2 * k, bd + 2 * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          umma_commit(&empty_bar[s]);
          if (++s == nst) {
            s = 0;
            ph ^= 1;
          }
        }
        if (ok) umma_commit(&accf_bar[b]);
      }
      // every MMA this thread issued has completed before TMEM is freed
      umma_commit(done_bar);
      mbar_wait(done_bar, 0, a.err);
    }
    __syncwarp();
  } else {
    // ---- epilogue: TMEM -> per-row running top 16 ----
    const int quarter = warp & 3;        // a warp reads TMEM lanes 32 * (warp % 4) ..
    const int half = (warp - 2) >> 2;    // which 128 columns of each tile
    const int row = m0 + quarter * 32 + lane;
    const bool warp_live = m0 + quarter * 32 < a.R;
    // The running list: values descending, equal values by ascending index;
    // empty slots are (-inf, -1).  Rows past R start "full" at +inf and never
    // take a value.
    float lv[kCand];
    int li[kCand];
#pragma unroll
    for (int q = 0; q < kCand; ++q) {
      lv[q] = row < a.R ? -INFINITY : INFINITY;
      li[q] = -1;
    }
    // The other half's 16th value bounds this row's answer from below too: a
    // value strictly under it has 16 better ones there.  Each half publishes
    // its own after every insertion (a racy read only ever sees a smaller,
    // still valid, bound).
    volatile float* my_thr = thr_s + half * kLBM + quarter * 32 + lane;
    volatile const float* other_thr = thr_s + (half ^ 1) * kLBM + quarter * 32 + lane;
    *my_thr = lv[kCand - 1];
    named_sync(1, kLEpiWarps * 32);
    for (int i = 0; i < nt; ++i) {
      const int b = i & 1;
      // warp-uniform outcome: the TMEM loads below are warp-collective
      if (!__all_sync(kAll, mbar_wait(&accf_bar[b], (i >> 1) & 1, a.err))) {
        record_error(a.err, kDevErrGemm);
        break;
      }
      tc_fence_after();
      if (warp_live) {
        const int vbase = (t_lo + i) * kLBN + half * kLHalf;
        const int lim = a.V - vbase;  // columns at or past V are padding
        const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>(b * kLBN + half * kLHalf);
        uint32_t ra[32], rb[32];
        tmem_ld32_issue(taddr, ra);
        tmem_ld32_wait(ra);
#pragma unroll 1
        for (int c = 0; c < kLHalf; c += 64) {
          tmem_ld32_issue(taddr + static_cast<uint32_t>(c + 32), rb);
          scan_chunk(ra, c, lim, vbase, lv, li, my_thr, other_thr);
          tmem_ld32_wait(rb);
          if (c + 64 < kLHalf) tmem_ld32_issue(taddr + static_cast<uint32_t>(c + 64), ra);
          scan_chunk(rb, c + 32, lim, vbase, lv, li, my_thr, other_thr);
          if (c + 64 < kLHalf) tmem_ld32_wait(ra);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce_bar[b]);
    }
    uint64_t list[kCand];
#pragma unroll
    for (int q = 0; q < kCand; ++q)
      list[q] = li[q] >= 0 ? make_key(lv[q], static_cast<uint32_t>(li[q])) : 0ull;
    // half 1 hands its list to half 0 of the same row, which keeps the top 16
    // of the two (both descending: the elementwise max against the reversed
    // other list is a bitonic sequence holding the top 16, then sorted)
    uint64_t* mine = pair + size_t(quarter * 32 + lane) * kCand;
    if (half == 1) {
#pragma unroll
      for (int q = 0; q < kCand; ++q) mine[q] = list[q];
    }
    named_sync(1, kLEpiWarps * 32);
    if (half == 0 && row < a.R) {
#pragma unroll
      for (int q = 0; q < kCand; ++q) {
        const uint64_t o = mine[kCand - 1 - q];
        list[q] = list[q] > o ? list[q] : o;
      }
#pragma unroll
      for (int j = kCand / 2; j > 0; j >>= 1) {
#pragma unroll
        for (int q = 0; q < kCand; ++q) {
          if ((q & j) == 0) {
            const uint64_t x = list[q], y = list[q + j];
            list[q] = x > y ? x : y;
            list[q + j] = x > y ? y : x;
          }
        }
      }
      ulonglong2* dst =
          reinterpret_cast<ulonglong2*>(a.lists + (size_t(row) * a.vsplits + vs) * kCand);
#pragma unroll
      for (int q = 0; q < kCand / 2; ++q) dst[q] = make_ulonglong2(list[2 * q], list[2 * q + 1]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kLTmemCols);
  }
}

// Top 16 of the union of up to 32 descending lists of 16 unique keys, lane l
// holding list l in k (zeros when it has none): sixteen rounds, each taking
// the largest head across the warp and popping it from its list.  Lane r (< 16)
// returns the key of rank r (0 when the lists hold fewer than r + 1 keys).
__device__ __forceinline__ uint64_t warp_top16_of_lists(uint64_t (&k)[kCand], int lane) {
  uint64_t out = 0ull;
#pragma unroll 1
  for (int r = 0; r < kCand; ++r) {
    // the warp's largest head: the largest high word, then the largest low
    // word among the lanes holding it (one reduction instruction each)
    const uint32_t hi = static_cast<uint32_t>(k[0] >> 32), lo = static_cast<uint32_t>(k[0]);
    const uint32_t mh = __reduce_max_sync(kAll, hi);
    const uint32_t ml = __reduce_max_sync(kAll, hi == mh ? lo : 0u);
    const uint64_t m = (static_cast<uint64_t>(mh) << 32) | ml;
    if (lane == r) out = m;
    if (m != 0ull && k[0] == m) {  // keys are unique: one lane pops
#pragma unroll
      for (int q = 0; q < kCand - 1; ++q) k[q] = k[q + 1];
      k[kCand - 1] = 0ull;
    }
  }
  return out;
}

__device__ __forceinline__ void load_list(const uint64_t* src, bool valid, uint64_t (&k)[kCand]) {
#pragma unroll
  for (int q = 0; q < kCand / 2; ++q) {
    ulonglong2 v = make_ulonglong2(0ull, 0ull);
    if (valid) v = __ldcg(reinterpret_cast<const ulonglong2*>(src) + q);
    k[2 * q] = v.x;
    k[2 * q + 1] = v.y;
  }
}

__device__ __forceinline__ void write_result(uint64_t key, size_t row, int32_t* out_idx,
                                             float* out_val, int lane) {
  if (lane < kCand) {
    out_idx[row * kCand + lane] = static_cast<int32_t>(~static_cast<uint32_t>(key));
    out_val[row * kCand + lane] = unord_f32(static_cast<uint32_t>(key >> 32));
  }
}

// nl <= 32: one warp per row, blockDim.x / 32 rows per block.  nl > 32: one row
// per block, one warp per 32 lists, then warp 0 over the warps' results.
__global__ void __launch_bounds__(1024) lmhead_merge_kernel(const uint64_t* lists, int R, int nl,
                                                            int32_t* out_idx, float* out_val) {
  __shared__ uint64_t wres[32 * kCand];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  pdl_wait();
  uint64_t k[kCand];
  if (nl <= 32) {
    const int row = blockIdx.x * nwarps + warp;
    if (row >= R) return;
    load_list(lists + (size_t(row) * nl + lane) * kCand, lane < nl, k);
    write_result(warp_top16_of_lists(k, lane), row, out_idx, out_val, lane);
    return;
  }
  const int row = blockIdx.x;
  const int l = warp * 32 + lane;
  load_list(lists + (size_t(row) * nl + l) * kCand, l < nl, k);
  const uint64_t top = warp_top16_of_lists(k, lane);
  if (lane < kCand) wres[warp * kCand + lane] = top;
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int q = 0; q < kCand; ++q) k[q] = lane < nwarps ? wres[lane * kCand + q] : 0ull;
    write_result(warp_top16_of_lists(k, lane), row, out_idx, out_val, lane);
  }
}

bool g_lm_attr[64];

}  // namespace

LmheadPlan lmhead_plan(int R, int V, int d) {
  LmheadPlan p{};
  p.R = R;
  p.V = V;
  p.d = d;
  p.rtiles = (R + kLBM - 1) / kLBM;
  p.ntiles = (V + kLBN - 1) / kLBN;
  p.kblocks = (d + kLBK - 1) / kLBK;
  // The workspace holds lists for the most CTAs per row tile any device could
  // use (at most 256 SMs), so its size does not depend on the device.
  p.max_splits = std::max(1, std::min(p.ntiles, kLMaxSplits / p.rtiles));
  p.lists_off = 0;
  p.ws_bytes = align_up(size_t(R) * p.max_splits * kCand * sizeof(uint64_t), 256);
  return p;
}

cudaError_t launch_lmhead_topk(const LmheadPlan& p, const __nv_bfloat16* hidden,
                               const __nv_bfloat16* W_lm, int32_t* idx, float* val, void* ws,
                               cudaStream_t s, bool pdl) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!g_lm_attr[dev & 63]) {
    e = cudaFuncSetAttribute(lmhead_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kLSmemMax));
    if (e != cudaSuccess) return e;
    g_lm_attr[dev & 63] = true;
  }
  const int sms = device_info().sms;
  LmArgs a{};
  a.R = p.R;
  a.V = p.V;
  a.d = p.d;
  a.ntiles = p.ntiles;
  a.kblocks = p.kblocks;
  a.vsplits = std::max(1, std::min(p.max_splits, sms / p.rtiles));
  a.a_rows = p.R >= kLBM ? kLBM : (p.R + 7) / 8 * 8;
  const size_t sbytes = lm_stage_bytes(a.a_rows);
  a.stages = static_cast<int>(std::min<size_t>(kLMaxStages, (kLSmemMax - kLFixedBytes) / sbytes));
  const size_t smem = kLFixedBytes + size_t(a.stages) * sbytes;
  a.lists = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(ws) + p.lists_off);
  a.err = device_error_word();
  alignas(64) CUtensorMap tmH, tmW;
  if (!tensor_map_bf16(hidden, uint64_t(p.R), uint64_t(p.d), static_cast<uint32_t>(a.a_rows), &tmH) ||
      !tensor_map_bf16(W_lm, uint64_t(p.V), uint64_t(p.d), kLBN, &tmW))
    return cudaErrorInvalidValue;
  e = launch_k(lmhead_topk_kernel, dim3(a.vsplits, p.rtiles), dim3(kLThreads), smem, s, pdl,
               a, tmH, tmW);
  if (e != cudaSuccess) return e;
  const int nl = a.vsplits;
  if (nl <= 32) {
    constexpr int kRowsPerBlock = 8;
    return launch_k(lmhead_merge_kernel, dim3((p.R + kRowsPerBlock - 1) / kRowsPerBlock),
                    dim3(kRowsPerBlock * 32), 0, s, true, static_cast<const uint64_t*>(a.lists),
                    p.R, nl, idx, val);
  }
  return launch_k(lmhead_merge_kernel, dim3(p.R), dim3((nl + 31) / 32 * 32), 0, s, true,
                  static_cast<const uint64_t*>(a.lists), p.R, nl, idx, val);
}

}  // namespace dfl2
