// Pair scores of the path selector ("DFlash 2: Keep Drafting Parallel",
// 方法细节 > 轻量级路径选择器, the pair-score equation):
//   S_t(a,b) = U_t(b) + <A(a) ⊙ H(h_t), B(b)>,
//   A(a) = W_A E[a], B(b) = W_B E[b], H(h) = sigmoid(W_H h)  (W_* [256,d]).
//
// Stage 1, one tcgen05 launch with three GEMM problems (C = rows x W^T, K = d):
//   PA: the rows whose A(.) is needed (the verified token, then the 16
//       candidates of positions 0..L-2), gathered from E, times W_A^T;
//   PB: the candidates of positions 0..L-1, gathered from E, times W_B^T;
//   GH: the hidden states times W_H^T (pre-sigmoid).
// Tiles are 128 rows x 256 columns, K in blocks of 64 (a partial last block
// reads zeros past d: TMA out-of-bounds fill for W, zero-fill for the rows).
// W tiles arrive by TMA (128-byte swizzle); the gathered rows by 16-byte
// cp.async written in the same swizzle; the accumulator lives in TMEM (256 columns).  When there are too few
// tiles to fill the GPU (batch 1), K is split over the CTAs of a thread-block
// cluster: each CTA stages its fp32 partial tile in shared memory and stores it
// to the caller's workspace in whole rows (the partials stay in L2), one
// cluster barrier, then every CTA sums one slice of rows over the splits in
// rank order, so the result is deterministic.
//
// Stage 2, the pair scores: a position's 16x16 scores from the previous
// position's A rows, the gate and this position's B rows (2x2 register
// blocking over 16-byte shared-memory reads).  In the fused tail
// (pair_walk_kernel, L <= 32) one thread-block cluster serves each sequence:
// each position takes the walk's decision for every predecessor row and hands
// the choices to the cluster's first CTA through distributed shared memory,
// which follows the chosen slots.  dfl2_select (scores only) and blocks longer
// than 32 positions use pair16_kernel, one CTA per (sequence, position); with
// the walk fused, the last CTA of each sequence (ticket) follows the slots.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "dfl2.h"
#include "dfl2_internal.cuh"

namespace dfl2 {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64, kGStages = 4;
constexpr int kAStage = kBM * kBK * 2;  // 16 KB
constexpr int kBStage = kBN * kBK * 2;  // 32 KB
constexpr int kGemmThreads = 256;       // warps 0-3 load, warp 4 issues MMAs, warps 4-7 drain TMEM
constexpr int kGemmTargetCtas = 148;
constexpr int kMaxClusterSplits = 8;       // portable cluster size
constexpr size_t kGemmSmem = 1024 + size_t(kGStages) * (kAStage + kBStage) + 256;

constexpr uint32_t kTmemCols = 256;

enum RowKind : int { kRowsPA = 0, kRowsPB = 1, kRowsHidden = 2, kRowsE = 3 };

struct GemmProblem {
  const __nv_bfloat16* W;  // [256, d] (the L2 prefetch; the GEMM reads it through the tensor map)
  int kind;     // RowKind
  int M;        // rows
  int mtiles;   // ceil(M / 128)
  float* out;   // [M][256]
  float* part;  // [splits][M][256] split-K partials (split K only)
};

struct GemmArgs {
  GemmProblem prob[3];
  int tiles_before[3];  // tiles of the problems before this one
  int splits, kps, kblocks;  // splits = cluster size along K
  int nsplit;                // CTAs per row tile along N: 1, 2 or 4 (256 / nsplit columns each)
  const __nv_bfloat16* E;
  const __nv_bfloat16* hidden;
  const int32_t* cand_idx;  // [B,L,16]
  const int32_t* verified;  // [B]
  int L, V, d;
  uint32_t* err;
};

// Where row m of a problem comes from, known before the dependency wait (only
// the index arithmetic): direct rows (hidden states, E in order) as `row`, a
// gathered row as the address of its token (the verified token or a
// candidate, read after the wait), nothing past M.
struct RowRef {
  const __nv_bfloat16* row;
  const int32_t* tok;
};
__device__ __forceinline__ RowRef a_row_ref(const GemmArgs& a, int kind, int m, int M) {
  if (m >= M) return RowRef{nullptr, nullptr};
  if (kind == kRowsHidden) return RowRef{a.hidden + size_t(m) * a.d, nullptr};
  if (kind == kRowsE) return RowRef{a.E + size_t(m) * a.d, nullptr};
  if (kind == kRowsPA) {
    const int per = kCand * (a.L - 1) + 1;
    const int b = m / per, q = m % per;
    return RowRef{nullptr, q == 0 ? a.verified + b : a.cand_idx + size_t(b) * a.L * kCand + (q - 1)};
  }
  return RowRef{nullptr, a.cand_idx + m};  // PB: row m is candidate m
}
// The row of a reference, after the wait; nullptr (a zero row) past M or for a
// token outside [0, V), which is recorded.
__device__ __forceinline__ const __nv_bfloat16* a_row_at(const GemmArgs& a, RowRef r) {
  if (!r.tok) return r.row;
  const int32_t tok = *r.tok;
  if (tok < 0 || tok >= a.V) {  // never read outside E: record it and use a zero row
    record_error(a.err, kDevErrBadIndex);
    return nullptr;
  }
  return a.E + size_t(tok) * a.d;
}


// WARP = false: tcgen05 MMAs issued by one thread into a TMEM accumulator.
// WARP = true (CTAs of 128 output columns only): the warp-level engine, each
// of warps 4-7 owning 32 output columns of all 128 rows (its slice of W is read
// by that warp alone), m16n8k16 mma.sync from the same staged tiles through
// ldmatrix, fp32 accumulators in registers.
template <bool WARP>
__global__ void __launch_bounds__(kGemmThreads, 1)
    proj_tc_kernel(const __grid_constant__ GemmArgs a, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmH) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;                                   // kGStages x 16 KB
  uint8_t* sB = smem + size_t(kGStages) * kAStage;      // kGStages x 32 KB
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(sB + size_t(kGStages) * kBStage);
  uint64_t* empty_bar = full_bar + kGStages;
  uint64_t* accum_bar = empty_bar + kGStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum_bar + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // CTA -> (m tile, column part, split); the splits of one (tile, part) form one cluster
  const int split = blockIdx.x % a.splits;
  const int rem = (blockIdx.x / a.splits) / a.nsplit;
  const int bn = kBN / a.nsplit;                                   // output columns of this CTA
  const int n0 = ((blockIdx.x / a.splits) % a.nsplit) * bn;        // the first of them
  const int p = rem >= a.tiles_before[2] ? 2 : (rem >= a.tiles_before[1] ? 1 : 0);
  const GemmProblem& P = a.prob[p];
  const int m0 = (rem - a.tiles_before[p]) * kBM;
  const int kb0 = split * a.kps;
  const int nkb = min(a.kblocks, kb0 + a.kps) - kb0;
  const CUtensorMap* tmap = p == 0 ? &tmA : (p == 1 ? &tmB : &tmH);

  if (tid == 0) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(&full_bar[s], 4 * 32 + 1);  // 128 cp.async arrivals + the TMA expect_tx
      mbar_init(&empty_bar[s], WARP ? 4 : 1);  // one tcgen05.commit, or each MMA warp
    }
    mbar_init(accum_bar, 1);
    fence_mbar_init();
    tma_prefetch_desc(tmap);
  }
  if (!WARP && warp == 4) tmem_alloc(tmem_slot, kTmemCols);
  // This CTA's K range of the 256 W rows into L2 while the previous kernel
  // (the top-16) still runs: a prefetch into L2 is coherent with writes in
  // flight, so it may precede the dependency wait.
  // One CTA per K range (the problem's first row tile) asks for it.
  if (P.W && nkb > 0 && m0 == 0 && tid < bn)
    prefetch_l2_rows(P.W + size_t(n0 + tid) * a.d + size_t(kb0) * kBK,
                     uint32_t(min(nkb * kBK, a.d - kb0 * kBK)) * 2u);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = WARP ? 0u : *tmem_slot;
  // the epilogue's index arithmetic (bn / 4 is a power of two; the K split's
  // row slice of this CTA)
  const int q4 = bn / 4, q4s = 31 - __clz(q4);
  const int per = (kBM + a.splits - 1) / a.splits;
  const int r0 = split * per;
  const int valid_rows = max(0, min(min(per, kBM - r0), P.M - (m0 + r0)));
  // the producers' 8 rows, resolved up to the token reads
  RowRef refs[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) refs[i] = a_row_ref(a, P.kind, m0 + ((tid & 127) >> 3) + 16 * i, P.M);
  pdl_wait();  // candidates may come from the previous kernel

  if (warp < 4) {
    // ---- producers: TMA for the W tile, cp.async for the 128 gathered rows ----
    const int j = tid & 7;  // 16-byte chunk within the 128-byte row
    const __nv_bfloat16* src[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) src[i] = a_row_at(a, refs[i]);
    for (int it = 0; it < nkb; ++it) {
      const int s = it % kGStages;
      if (it >= kGStages && !mbar_wait(&empty_bar[s], ((it / kGStages) - 1) & 1, a.err))
        record_error(a.err, kDevErrGemm);
      const int kelem = (kb0 + it) * kBK;
      if (tid == 0) {
        mbar_arrive_expect_tx(&full_bar[s], uint32_t(bn) * kBK * 2u);
        tma_load_2d(sB + size_t(s) * kBStage, tmap, kelem, n0, &full_bar[s]);
      }
      uint8_t* dstA = sA + size_t(s) * kAStage;
      const bool kin = kelem + j * 8 < a.d;  // chunks past d (the last K block) read as zero
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = (tid >> 3) + 16 * i;
        void* dst = dstA + r * 128 + ((j ^ (r & 7)) << 4);
        const bool ok = src[i] != nullptr && kin;
        cp_async16(dst, ok ? src[i] + kelem + j * 8 : a.E, ok);
      }
      cp_async_commit();
      if (it >= 2) {
        cp_async_wait<2>();
        fence_proxy_async_smem();
        mbar_arrive(&full_bar[(it - 2) % kGStages]);
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    for (int it = max(0, nkb - 2); it < nkb; ++it) mbar_arrive(&full_bar[it % kGStages]);
  } else if constexpr (WARP) {
    // ---- warp-level MMA: this warp's 32 output columns of all 128 rows ----
    const int cw = (warp - 4) * 32;
    const int mi = lane >> 3, rr = lane & 7;
    float acc[kBM / 16][4][4];
#pragma unroll
    for (int mt = 0; mt < kBM / 16; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
    for (int it = 0; it < nkb; ++it) {
      const int s = it % kGStages;
      if (!mbar_wait(&full_bar[s], (it / kGStages) & 1, a.err)) record_error(a.err, kDevErrGemm);
      const uint32_t sa = smem_u32(sA + size_t(s) * kAStage);
      const uint32_t sb = smem_u32(sB + size_t(s) * kBStage);
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        // B fragments of the four n8 tiles: W rows (output columns) x 16 K, two
        // tiles per ldmatrix.x4 (matrices: n 0-7 K lo, n 0-7 K hi, n 8-15 K lo, K hi)
        uint32_t bfr[4][2];
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          const int n = cw + np * 16 + (mi >> 1) * 8 + rr;
          const int ch = 2 * kk + (mi & 1);  // 16-byte chunk of the 128-byte row, swizzled
          uint32_t r[4];
          ldsm_x4(sb + uint32_t(n) * 128u + uint32_t((ch ^ (n & 7)) << 4), r);
          bfr[2 * np][0] = r[0];
          bfr[2 * np][1] = r[1];
          bfr[2 * np + 1][0] = r[2];
          bfr[2 * np + 1][1] = r[3];
        }
#pragma unroll
        for (int mt = 0; mt < kBM / 16; ++mt) {
          // A fragment: rows mt*16.. x 16 K (matrices: rows 0-7 K lo, 8-15 K lo, 0-7 K hi, 8-15 K hi)
          const int row = mt * 16 + (mi & 1) * 8 + rr;
          const int ch = 2 * kk + (mi >> 1);
          uint32_t af[4];
          ldsm_x4(sa + uint32_t(row) * 128u + uint32_t((ch ^ (row & 7)) << 4), af);
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) mma_16816_bf16(acc[mt][nt], af, bfr[nt]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
    // every MMA warp is past its last ldmatrix before the staging overwrites the stages
    named_sync(1, 128);
    // accumulators -> the staged tile (rows kBN + 4 floats apart): c0,c1 at
    // (row g, columns 2t, 2t+1), c2,c3 at row g + 8
    float* stage = reinterpret_cast<float*>(smem);
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int mt = 0; mt < kBM / 16; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int col = cw + nt * 8 + 2 * t;
        *reinterpret_cast<float2*>(stage + size_t(mt * 16 + g) * (kBN + 4) + col) =
            make_float2(acc[mt][nt][0], acc[mt][nt][1]);
        *reinterpret_cast<float2*>(stage + size_t(mt * 16 + g + 8) * (kBN + 4) + col) =
            make_float2(acc[mt][nt][2], acc[mt][nt][3]);
      }
  } else {
    if (warp == 4 && lane == 0) {
      // ---- MMA issuer ----
      const uint32_t idesc = umma_idesc_bf16(kBM, bn);
      for (int it = 0; it < nkb; ++it) {
        const int s = it % kGStages;
        if (!mbar_wait(&full_bar[s], (it / kGStages) & 1, a.err)) record_error(a.err, kDevErrGemm);
        tc_fence_after();
        const uint64_t ad = umma_desc_sw128(sA + size_t(s) * kAStage);
        const uint64_t bd = umma_desc_sw128(sB + size_t(s) * kBStage);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          umma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc, (it > 0 || k > 0) ? 1u : 0u);
        umma_commit(&empty_bar[s]);
      }
      umma_commit(accum_bar);
    }
    __syncwarp();
    if (!mbar_wait(accum_bar, 0, a.err)) record_error(a.err, kDevErrGemm);
    tc_fence_after();
    if (a.splits == 1) {
      // ---- one split: TMEM -> registers -> the output rows ----
      const int quarter = warp & 3;
      const int row = m0 + quarter * 32 + lane;
#pragma unroll 1
      for (int c = 0; c < bn / 32; ++c) {
        float v[32];
        tmem_ld32(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(c * 32), v);
        if (row < P.M) {
          float4* o = reinterpret_cast<float4*>(P.out + size_t(row) * kBN + n0 + c * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
      }
    }
  }
  tc_fence_before();
  if (WARP && a.splits == 1) {
    // ---- one split: the staged tile -> the output rows ----
    __syncthreads();
    const int rows = max(0, min(kBM, P.M - m0));
    const float* stage = reinterpret_cast<const float*>(smem);
    for (int e = tid; e < rows * (bn / 4); e += kGemmThreads) {
      const int lr = e >> q4s, c4 = e & (q4 - 1);
      *reinterpret_cast<float4*>(P.out + size_t(m0 + lr) * kBN + n0 + 4 * c4) =
          *reinterpret_cast<const float4*>(stage + size_t(lr) * (kBN + 4) + 4 * c4);
    }
    pdl_launch_dependents();
    return;
  }
  if (a.splits == 1) {
    __syncthreads();
    pdl_launch_dependents();
    if (warp == 4) {
      tc_fence_after();
      tmem_dealloc(tmem, kTmemCols);
    }
    return;
  }
  // ---- split K over the cluster: every CTA stores its fp32 partial tile to the
  // workspace (L2), then each CTA sums one slice of rows over the splits in rank
  // order (deterministic) and writes the result ----
  // The partial tile goes TMEM -> shared memory (the drained operand stages,
  // rows kStagePitch floats apart) -> global memory in whole rows, so that each
  // warp store covers 512 contiguous bytes.
  constexpr int kStagePitch = kBN + 4;
  static_assert(size_t(kBM) * kStagePitch * 4 <= size_t(kGStages) * (kAStage + kBStage),
                "the partial tile fits the operand stages");
  const int S = a.splits;
  float* mypart = P.part + (size_t(split) * P.M) * kBN;
  float* stage = reinterpret_cast<float*>(smem);
  if (!WARP && warp >= 4) {  // (the warp engine staged its tile already)
    const int quarter = warp & 3;
    const int lrow = quarter * 32 + lane;
#pragma unroll 1
    for (int c = 0; c < bn / 32; ++c) {
      float v[32];
      tmem_ld32(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(c * 32), v);
      float4* o = reinterpret_cast<float4*>(stage + size_t(lrow) * kStagePitch + c * 32);
#pragma unroll
      for (int q = 0; q < 8; ++q) o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  {
    const int rows = max(0, min(kBM, P.M - m0));
    for (int e = tid; e < rows * (bn / 4); e += kGemmThreads) {
      const int lr = e >> q4s, c4 = e & (q4 - 1);
      *reinterpret_cast<float4*>(mypart + size_t(m0 + lr) * kBN + n0 + 4 * c4) =
          *reinterpret_cast<const float4*>(stage + size_t(lr) * kStagePitch + 4 * c4);
    }
  }
  cluster_sync_all();  // every split's partial tile is in the workspace
  if (!WARP && warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // the next launch may start now (it waits for this grid to finish before
  // reading anything, and holds no tensor memory)
  pdl_launch_dependents();
  const int n4 = valid_rows * q4;
  constexpr int kMaxSplitLoads = kMaxClusterSplits;
  constexpr int kPer = 2;  // elements per thread and pass: 2 x 8 loads in flight
  for (int e0 = tid; e0 < n4; e0 += kGemmThreads * kPer) {
    float4 v[kPer][kMaxSplitLoads];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = e0 + u * kGemmThreads;
      const int lr = e >> q4s, c4 = e & (q4 - 1);
      const size_t at = size_t(m0 + r0 + lr) * kBN + n0 + 4 * c4;
#pragma unroll
      for (int k = 0; k < kMaxSplitLoads; ++k)  // every split's value requested first
        v[u][k] = k < S && e < n4
                      ? __ldcg(reinterpret_cast<const float4*>(P.part + size_t(k) * P.M * kBN + at))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = e0 + u * kGemmThreads;
      if (e >= n4) break;
      const int lr = e >> q4s, c4 = e & (q4 - 1);
      float4 acc = v[u][0];
#pragma unroll
      for (int k = 1; k < kMaxSplitLoads; ++k) {  // rank order: deterministic
        acc.x += v[u][k].x; acc.y += v[u][k].y; acc.z += v[u][k].z; acc.w += v[u][k].w;
      }
      *reinterpret_cast<float4*>(P.out + size_t(m0 + r0 + lr) * kBN + n0 + 4 * c4) = acc;
    }
  }
}

// ============================================================================
// Batched projections: each E row gathered once, N = 512.
// ============================================================================
// Per sequence the rows are the verified token, then the 16 L candidates
// (position-major).  A(.) is needed for the verified token and the candidates
// of positions 0..L-2 (the predecessors), B(.) for every candidate; the rows
// overlap, so one GEMM [rows x d] x [d x 512] with [W_A; W_B] as N gathers each
// E row once.  The epilogue writes columns 0..255 to PA for predecessor rows
// and columns 256..511 to PB for candidate rows (the A of the last position's
// candidates and the B of the verified token are computed and dropped: 1/16
// and 1/(16L+1) of the work).  The gate rows (hidden states x W_H, N = 256)
// are further row tiles of the same launch.
//
// A tile is 128 rows by 512 columns: two M=128 N=256 tcgen05 MMAs per K step,
// the 512 float32 columns filling TMEM.  The gathered rows (16 KB per K block,
// cp.async from random E rows) and the W tiles (64 KB per K block by TMA, L2
// hits) travel in separate rings: 4 stages of gathered rows, kAbLag + 1 of
// them requested ahead of the MMAs, and four 32 KB W slots (W_A's or W_B's 256
// rows of one K block), each released as soon as its MMAs complete.  The loop
// runs at about 0.7 us per K block at batch 64 (the MMAs alone take 0.57): the
// gather, 128 random 128-byte pieces of E per K block and CTA, is served at
// about 3 TB/s.  Measured no faster: N=128 MMAs on 16 KB W quarters (at N=128
// the MMAs read shared memory twice as often per flop), 7 gather stages with
// 6 in flight, and an L2 prefetch of the gathered rows (whole rows at once,
// or 1 KB chunks ahead of the gather).
constexpr int kAbAStages = 4, kAbWSlots = 4;
constexpr int kAbLag = kAbAStages - 2;  // cp.async groups left pending behind the newest
constexpr int kAbWQuarter = kBStage;  // one slot: 256 W rows x 64 K (32 KB)
constexpr size_t kAbSmem = 1024 + size_t(kAbAStages) * kAStage + size_t(kAbWSlots) * kAbWQuarter + 256;
constexpr uint32_t kAbTmemCols = 512;

struct AbArgs {
  int M_ab;           // B (16 L + 1) rows of the combined problem
  int tiles_ab;       // ceil(M_ab / 128); the gate's tiles follow
  int M_h;            // B L hidden rows
  int kblocks;
  int L, V, d;
  const __nv_bfloat16* E;
  const __nv_bfloat16* hidden;
  const __nv_bfloat16* W_A;  // L2 prefetch only (the GEMM reads W through the tensor maps)
  const __nv_bfloat16* W_B;
  const __nv_bfloat16* W_H;
  const int32_t* cand_idx;  // [B,L,16]
  const int32_t* verified;  // [B]
  float* PA;  // [B (16 (L-1) + 1)][256]
  float* PB;  // [B 16 L][256]
  float* GH;  // [B L][256]
  uint32_t* err;
};

// Source row of the combined problem (verified token or candidate), or nullptr.
__device__ __forceinline__ const __nv_bfloat16* ab_row(const AbArgs& a, int m) {
  if (m >= a.M_ab) return nullptr;
  const int per = kCand * a.L + 1;
  const int b = m / per, q = m % per;
  const int32_t tok = q == 0 ? a.verified[b] : a.cand_idx[size_t(b) * a.L * kCand + (q - 1)];
  if (tok < 0 || tok >= a.V) {  // never read outside E: record it and use a zero row
    record_error(a.err, kDevErrBadIndex);
    return nullptr;
  }
  return a.E + size_t(tok) * a.d;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    proj_ab_kernel(const __grid_constant__ AbArgs a, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmH) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;                                         // [4][128 rows][128 B]
  uint8_t* sW = smem + size_t(kAbAStages) * kAStage;          // [4 slots][256 W rows][128 B]
  uint64_t* a_full = reinterpret_cast<uint64_t*>(sW + size_t(kAbWSlots) * kAbWQuarter);
  uint64_t* a_empty = a_full + kAbAStages;
  uint64_t* w_full = a_empty + kAbAStages;
  uint64_t* w_empty = w_full + kAbWSlots;
  uint64_t* accum_bar = w_empty + kAbWSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum_bar + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool ab = static_cast<int>(blockIdx.x) < a.tiles_ab;  // else a gate tile
  const int m0 = (ab ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x) - a.tiles_ab) * kBM;
  const int M = ab ? a.M_ab : a.M_h;
  const int nq = ab ? 2 : 1;  // W slots (N = 256 each) per K block
  const int nkb = a.kblocks;

  if (tid == 0) {
    for (int s = 0; s < kAbAStages; ++s) {
      mbar_init(&a_full[s], 4 * 32);  // the 128 gathering threads
      mbar_init(&a_empty[s], 1);      // one tcgen05.commit
    }
    for (int s = 0; s < kAbWSlots; ++s) {
      mbar_init(&w_full[s], 1);       // the TMA expect_tx
      mbar_init(&w_empty[s], 1);
    }
    mbar_init(accum_bar, 1);
    fence_mbar_init();
    if (ab) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
    } else {
      tma_prefetch_desc(&tmH);
    }
  }
  if (warp == 4) tmem_alloc(tmem_slot, kAbTmemCols);
  // The W rows into L2 while the previous kernel (the top-16) still runs: a
  // prefetch into L2 is coherent with writes in flight.  The first tile of
  // each problem asks for its W.
  if (m0 == 0 && tid < 256) {
    const size_t rb = size_t(a.d) * 2;
    if (ab) {
      prefetch_l2_rows(a.W_A + size_t(tid) * a.d, uint32_t(rb));
      prefetch_l2_rows(a.W_B + size_t(tid) * a.d, uint32_t(rb));
    } else {
      prefetch_l2_rows(a.W_H + size_t(tid) * a.d, uint32_t(rb));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // candidates may come from the previous kernel

  if (warp < 4) {
    // ---- gather: 128 rows x 128 B per K block by 16-byte cp.async, written in
    // the 128-byte swizzle; up to kAbLag + 1 K blocks in flight ----
    const int j = tid & 7;  // 16-byte chunk within the 128-byte row
    const __nv_bfloat16* src[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int m = m0 + (tid >> 3) + 16 * i;
      src[i] = ab ? ab_row(a, m) : (m < M ? a.hidden + size_t(m) * a.d : nullptr);
    }
    for (int it = 0; it < nkb; ++it) {
      const int s = it % kAbAStages;
      if (it >= kAbAStages && !mbar_wait(&a_empty[s], ((it / kAbAStages) - 1) & 1, a.err))
        record_error(a.err, kDevErrGemm);
      const int kelem = it * kBK;
      uint8_t* dstA = sA + size_t(s) * kAStage;
      const bool kin = kelem + j * 8 < a.d;  // chunks past d (the last K block) read as zero
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = (tid >> 3) + 16 * i;
        void* dst = dstA + r * 128 + ((j ^ (r & 7)) << 4);
        const bool ok = src[i] != nullptr && kin;
        cp_async16(dst, ok ? src[i] + kelem + j * 8 : a.E, ok);
      }
      cp_async_commit();
      if (it >= kAbLag) {
        cp_async_wait<kAbLag>();
        fence_proxy_async_smem();
        mbar_arrive(&a_full[(it - kAbLag) % kAbAStages]);
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    for (int it = max(0, nkb - kAbLag); it < nkb; ++it) mbar_arrive(&a_full[it % kAbAStages]);
  } else {
    if (warp == 4 && lane == 0) {
      // ---- MMA issuer: per K block, one N=256 MMA per W slot ----
      const uint32_t idesc = umma_idesc_bf16(kBM, kBN);
      for (int it = 0; it < nkb; ++it) {
        const int sa = it % kAbAStages;
        if (!mbar_wait(&a_full[sa], (it / kAbAStages) & 1, a.err)) record_error(a.err, kDevErrGemm);
        const uint64_t ad = umma_desc_sw128(sA + size_t(sa) * kAStage);
        for (int q = 0; q < nq; ++q) {
          const int u = it * nq + q, sw = u % kAbWSlots;
          if (!mbar_wait(&w_full[sw], (u / kAbWSlots) & 1, a.err)) record_error(a.err, kDevErrGemm);
          tc_fence_after();
          const uint64_t bd = umma_desc_sw128(sW + size_t(sw) * kAbWQuarter);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            umma_bf16(tmem + uint32_t(q * kBN), ad + 2 * k, bd + 2 * k, idesc,
                      (it > 0 || k > 0) ? 1u : 0u);
          umma_commit(&w_empty[sw]);
        }
        umma_commit(&a_empty[sa]);
      }
      umma_commit(accum_bar);
    } else if (warp == 5 && lane == 0) {
      // ---- W producer: the K block's W_A then W_B tile (or W_H's) by TMA,
      // one slot each ----
      for (int u = 0; u < nkb * nq; ++u) {
        const int it = u / nq, q = u % nq, sw = u % kAbWSlots;
        if (u >= kAbWSlots && !mbar_wait(&w_empty[sw], ((u / kAbWSlots) - 1) & 1, a.err))
          record_error(a.err, kDevErrGemm);
        mbar_arrive_expect_tx(&w_full[sw], uint32_t(kAbWQuarter));
        const CUtensorMap* tm = !ab ? &tmH : (q == 0 ? &tmA : &tmB);
        tma_load_2d(sW + size_t(sw) * kAbWQuarter, tm, it * kBK, 0, &w_full[sw]);
      }
    }
    __syncwarp();
    // ---- epilogue: TMEM -> the rows' outputs ----
    if (!mbar_wait(accum_bar, 0, a.err)) record_error(a.err, kDevErrGemm);
    tc_fence_after();
    const int quarter = warp & 3;
    const int row = m0 + quarter * 32 + lane;
    float* dst[2] = {nullptr, nullptr};
    if (row < M) {
      if (ab) {
        const int per = kCand * a.L + 1;
        const int b = row / per, q = row % per;
        if (q <= kCand * (a.L - 1)) dst[0] = a.PA + (size_t(b) * (kCand * (a.L - 1) + 1) + q) * kRank;
        if (q >= 1) dst[1] = a.PB + (size_t(b) * kCand * a.L + (q - 1)) * kRank;
      } else {
        dst[0] = a.GH + size_t(row) * kRank;
      }
    }
    for (int h = 0; h < nq; ++h) {
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        float v[32];
        tmem_ld32(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(h * kBN + c * 32), v);
        if (dst[h]) {
          float4* o = reinterpret_cast<float4*>(dst[h] + c * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  pdl_launch_dependents();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kAbTmemCols);
  }
}

struct PairArgs {
  const float* PA;  // [MA][256] (per-cycle projections), or
  const float* PB;  // [MB][256]
  const float* tabA;        // [V][256] precomputed A(.) for every token (table mode), or null
  const float* tabB;        // [V][256] precomputed B(.)
  const int32_t* verified;  // [B] (table mode)
  int V;
  uint32_t* err;
  const float* GH;  // [B*L][256], pre-sigmoid
  const float* cand_val;  // [B,L,16]
  float* scores;          // [B,L,16,16]
  int L;
  // fused walk (walk == 0: scores only)
  int walk;
  float T;
  const uint64_t* seeds;
  uint64_t cycle;
  const int32_t* cand_idx;  // [B,L,16]
  int32_t* tokens;          // [B,L]
  int32_t* slots;           // [B,L] or null
  float* q;                 // [B,L,16] or null
  uint32_t* tickets;        // [B], zero between calls
  int32_t* choice;          // [B*L][16] workspace
  float* qrows;             // [B*L][16][16] workspace
};

// One CTA per (sequence b, position t), 128 threads.  The 16x16 dot products
// of length 256 (bilinear16) read shared memory 16 bytes at a time into 4x4
// register blocks.  Rows sit kPairPitch floats apart (16-byte aligned, and
// eight consecutive rows fall in different bank groups).
constexpr int kPairThreads = 128;
constexpr int kPairPitch = kRank + 4;

// The nearest tf32 value of x (10 explicit mantissa bits), in a 32-bit register.
__device__ __forceinline__ uint32_t tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void mma_1688_tf32(float d[4], const uint32_t a[4], const uint32_t b[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// out[i][j] = sum over the 256 ranks of Gs[i][q] * Bsh[j][q] for the 16 x 16
// pairs, by the 128 threads of a group, on the tensor cores: warp w takes the
// ranks [64 w, 64 w + 64) as eight k8 steps of m16n8k8 MMAs (M = the 16 rows i,
// N = two tiles of 8 columns j), each operand read from shared memory once.
// fp32 accuracy from tf32 MMAs: each value is split into its nearest tf32 and
// the tf32 of the remainder, and a*b is taken as a_hi*b_lo + a_lo*b_hi +
// a_hi*b_hi (the dropped a_lo*b_lo is below 2^-22 of |a*b|), accumulated in
// fp32.  The four warps' partial tiles are added in warp order through the
// bytes of Gs, which the products no longer need (so Gs is overwritten); the
// caller synchronises the group before and after.
template <typename Sync>
__device__ __forceinline__ void bilinear16(float (*Gs)[kPairPitch], const float (*Bsh)[kPairPitch],
                                           float (*out)[kCand + 1], int tid, Sync sync) {
  const int w = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 2
  for (int ks = 0; ks < 8; ++ks) {
    const int k0 = 64 * w + 8 * ks;
    const float av[4] = {Gs[g][k0 + t], Gs[g + 8][k0 + t], Gs[g][k0 + t + 4], Gs[g + 8][k0 + t + 4]};
    uint32_t ahi[4], alo[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      ahi[r] = tf32_rna(av[r]);
      alo[r] = tf32_rna(av[r] - __uint_as_float(ahi[r]));
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const float bv[2] = {Bsh[8 * nt + g][k0 + t], Bsh[8 * nt + g][k0 + t + 4]};
      uint32_t bhi[2], blo[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        bhi[r] = tf32_rna(bv[r]);
        blo[r] = tf32_rna(bv[r] - __uint_as_float(bhi[r]));
      }
      mma_1688_tf32(d[nt], ahi, blo);
      mma_1688_tf32(d[nt], alo, bhi);
      mma_1688_tf32(d[nt], ahi, bhi);
    }
  }
  sync();  // every warp is past its last read of Gs
  // d[nt]: (row g, columns 8 nt + 2t, +1) and (row g + 8, the same columns)
  float* part = &Gs[0][0];  // 4 x 16 x 16 floats, within Gs's 16 x kPairPitch
  float* pw = part + w * kCand * kCand;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    *reinterpret_cast<float2*>(pw + g * kCand + 8 * nt + 2 * t) = make_float2(d[nt][0], d[nt][1]);
    *reinterpret_cast<float2*>(pw + (g + 8) * kCand + 8 * nt + 2 * t) = make_float2(d[nt][2], d[nt][3]);
  }
  sync();
  for (int e = tid; e < kCand * kCand; e += kPairThreads)
    out[e / kCand][e % kCand] = ((part[e] + part[kCand * kCand + e]) + part[2 * kCand * kCand + e]) +
                                part[3 * kCand * kCand + e];
}

__global__ void __launch_bounds__(kPairThreads) pair16_kernel(PairArgs a) {
  __shared__ __align__(16) float Gs[kCand][kPairPitch];   // A(a_i) ⊙ H(h_t)
  __shared__ __align__(16) float Bsh[kCand][kPairPitch];  // B(b_j)
  __shared__ float Hs[kRank];
  __shared__ float U[kCand];
  __shared__ float Srow[kCand][kCand + 1];
  __shared__ int path[128];
  __shared__ uint32_t last;
  pdl_wait();
  const int cell = blockIdx.x;
  const int b = cell / a.L, t = cell % a.L;
  const int npred = t == 0 ? 1 : kCand;
  const size_t rowA0 =
      size_t(b) * (kCand * (a.L - 1) + 1) + (t == 0 ? 0 : 1 + size_t(kCand) * (t - 1));
  const size_t rowB0 = size_t(b) * kCand * a.L + size_t(kCand) * t;
  const int tid = threadIdx.x;
  // Row sources: the per-cycle projections, or (table mode) the precomputed
  // rows of the predecessor and candidate tokens.
  __shared__ const float* rowA[kCand];
  __shared__ const float* rowB[kCand];
  if (tid < 2 * kCand) {
    const int i = tid % kCand;
    const bool isA = tid < kCand;
    const float* src;
    if (a.tabA) {
      int tok = 0;
      if (isA) {
        if (i < npred)
          tok = t == 0 ? a.verified[b] : a.cand_idx[(size_t(b) * a.L + (t - 1)) * kCand + i];
      } else {
        tok = a.cand_idx[(size_t(b) * a.L + t) * kCand + i];
      }
      if (tok < 0 || tok >= a.V) {  // never read outside the tables
        record_error(a.err, kDevErrBadIndex);
        tok = 0;
      }
      src = (isA ? a.tabA : a.tabB) + size_t(tok) * kRank;
    } else {
      src = isA ? a.PA + (rowA0 + i) * kRank : a.PB + (rowB0 + i) * kRank;
    }
    (isA ? rowA : rowB)[i] = src;
  }
  __syncthreads();
  // A and B rows: 16 rows x 64 float4 each; all loads issued before any use.
  float4 va[8], vb[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int e = tid + kPairThreads * k;
    const int i = e >> 6, q4 = e & 63;
    va[k] = i < npred ? reinterpret_cast<const float4*>(rowA[i])[q4] : make_float4(0.f, 0.f, 0.f, 0.f);
    vb[k] = reinterpret_cast<const float4*>(rowB[i])[q4];
  }
  for (int q = tid; q < kRank; q += kPairThreads) {
    const float g = a.GH[size_t(cell) * kRank + q];
    Hs[q] = 1.0f / (1.0f + expf(-g));
  }
  if (tid < kCand) U[tid] = a.cand_val[size_t(cell) * kCand + tid];
  __syncthreads();  // Hs complete
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int e = tid + kPairThreads * k;
    const int i = e >> 6, c = 4 * (e & 63);
    const float4 h = *reinterpret_cast<const float4*>(&Hs[c]);
    *reinterpret_cast<float4*>(&Gs[i][c]) =
        make_float4(va[k].x * h.x, va[k].y * h.y, va[k].z * h.z, va[k].w * h.w);
    *reinterpret_cast<float4*>(&Bsh[i][c]) = vb[k];
  }
  __syncthreads();
  bilinear16(Gs, Bsh, Srow, tid, [] { __syncthreads(); });
  __syncthreads();
  // S = U_t(b_j) + the bilinear term; rows past the predecessors are -inf
  for (int e = tid; e < kCand * kCand; e += kPairThreads) {
    const int i = e / kCand, j = e % kCand;
    const float v = i < npred ? Srow[i][j] + U[j] : -INFINITY;
    Srow[i][j] = v;
    a.scores[size_t(cell) * kCand * kCand + e] = v;
  }
  if (!a.walk) {
    pdl_launch_dependents();
    return;
  }

  // ---- fused walk: the decision of every row of this position ----
  __syncthreads();
  if (tid < npred) {
    const float u = a.T > 0.f ? walk_uniform(a.seeds[b], a.cycle, t) : 0.f;
    float qv[kCand];
    const int c = walk_row_choice(&Srow[tid][0], a.T, u, qv);
    a.choice[size_t(cell) * kCand + tid] = c;
    float4* qo = reinterpret_cast<float4*>(a.qrows + (size_t(cell) * kCand + tid) * kCand);
#pragma unroll
    for (int k = 0; k < 4; ++k) qo[k] = make_float4(qv[4 * k], qv[4 * k + 1], qv[4 * k + 2], qv[4 * k + 3]);
    __threadfence();  // this row's choice and q are visible before the ticket
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t ticket = atomicInc(&a.tickets[b], static_cast<unsigned>(a.L - 1));
    last = ticket == static_cast<uint32_t>(a.L - 1);
  }
  __syncthreads();
  if (!last) {
    pdl_launch_dependents();
    return;
  }
  // ---- last CTA of sequence b: follow the chosen slots from the verified token ----
  __threadfence();
  const int* ch = a.choice + size_t(b) * a.L * kCand;
  int* chs = reinterpret_cast<int*>(&Gs[0][0]);  // L x 16 choices (L <= 128 fits)
  for (int e = tid; e < a.L * kCand; e += kPairThreads) chs[e] = __ldcg(ch + e);
  __syncthreads();
  if (tid == 0) {
    int prev = 0;
    for (int tt = 0; tt < a.L; ++tt) {
      prev = chs[tt * kCand + prev] & (kCand - 1);
      path[tt] = prev;
    }
  }
  __syncthreads();
  for (int tt = tid; tt < a.L; tt += kPairThreads) {
    const size_t c2 = size_t(b) * a.L + tt;
    a.tokens[c2] = a.cand_idx[c2 * kCand + path[tt]];
    if (a.slots) a.slots[c2] = path[tt];
  }
  if (a.q) {
    for (int e = tid; e < a.L * kCand; e += kPairThreads) {
      const int tt = e / kCand, k = e % kCand;
      const size_t c2 = size_t(b) * a.L + tt;
      const int row = tt == 0 ? 0 : path[tt - 1];  // step tt draws from its predecessor's row
      a.q[c2 * kCand + k] = __ldcg(a.qrows + (c2 * kCand + row) * kCand + k);
    }
  }
  pdl_launch_dependents();
}

// ============================================================================
// Pair scores with the walk fused, one thread-block cluster per sequence.
// ============================================================================
// CTA `rank` of the cluster of sequence b takes positions rank*P .. rank*P+P-1,
// one 128-thread group per position (the same computation as pair16_kernel).
// Each group takes the walk's decision for every predecessor row of its
// position and stores the choices, the q rows and its 16 candidate tokens
// straight into the shared memory of the cluster's first CTA (distributed
// shared memory, about 1 KB per position); after one cluster barrier that CTA
// follows the chosen slots from the verified token and writes the path.  No
// global workspace, fence or ticket sits between the positions and the walk.
constexpr int kPwMaxL = 32;  // P <= 4 positions per CTA, clusters of <= 8

struct PairGroupSmem {
  float Gs[kCand][kPairPitch];   // A(a_i) ⊙ H(h_t)
  float Bsh[kCand][kPairPitch];  // B(b_j)
  float Hs[kRank];
  float U[kCand];
  float Srow[kCand][kCand + 1];
  const float* rowA[kCand];
  const float* rowB[kCand];
};
struct PairWalkSmem {  // used in the cluster's first CTA only (same layout in every CTA)
  float q[kPwMaxL][kCand][kCand];
  int choice[kPwMaxL][kCand];
  int tok[kPwMaxL][kCand];
  int path[kPwMaxL];
  uint64_t bar;  // counts the bytes stored by every position
};

// Stores into CTA `rank`'s shared memory at the offsets of `local` / `bar`,
// counted as transaction bytes on that CTA's mbarrier.
__device__ __forceinline__ void st_async_b32(const void* local, uint32_t rank, uint32_t v,
                                             const uint64_t* bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(
                   dsmem_addr(local, rank)),
               "r"(v), "r"(dsmem_addr(bar, rank))
               : "memory");
}
__device__ __forceinline__ void st_async_f32(const void* local, uint32_t rank, float v,
                                             const uint64_t* bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(
                   dsmem_addr(local, rank)),
               "f"(v), "r"(dsmem_addr(bar, rank))
               : "memory");
}
__device__ __forceinline__ void st_async_v4(const void* local, uint32_t rank, float4 v,
                                            const uint64_t* bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
          dsmem_addr(local, rank)),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(dsmem_addr(bar, rank))
      : "memory");
}

// Scores of position t of sequence b into g->Srow (rows past the predecessors
// are -inf) and, when requested, into a.scores.  `sync` is the group's barrier.
template <typename Sync>
__device__ __forceinline__ void pair_position(const PairArgs& a, int b, int t, int tid,
                                              PairGroupSmem* g, Sync sync) {
  const int cell = b * a.L + t;
  const int npred = t == 0 ? 1 : kCand;
  const size_t rowA0 =
      size_t(b) * (kCand * (a.L - 1) + 1) + (t == 0 ? 0 : 1 + size_t(kCand) * (t - 1));
  const size_t rowB0 = size_t(b) * kCand * a.L + size_t(kCand) * t;
  if (tid < 2 * kCand) {
    const int i = tid % kCand;
    const bool isA = tid < kCand;
    const float* src;
    if (a.tabA) {
      int tok = 0;
      if (isA) {
        if (i < npred)
          tok = t == 0 ? a.verified[b] : a.cand_idx[(size_t(b) * a.L + (t - 1)) * kCand + i];
      } else {
        tok = a.cand_idx[(size_t(b) * a.L + t) * kCand + i];
      }
      if (tok < 0 || tok >= a.V) {  // never read outside the tables
        record_error(a.err, kDevErrBadIndex);
        tok = 0;
      }
      src = (isA ? a.tabA : a.tabB) + size_t(tok) * kRank;
    } else {
      src = isA ? a.PA + (rowA0 + i) * kRank : a.PB + (rowB0 + i) * kRank;
    }
    (isA ? g->rowA : g->rowB)[i] = src;
  }
  sync();
  float4 va[8], vb[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int e = tid + kPairThreads * k;
    const int i = e >> 6, q4 = e & 63;
    va[k] = i < npred ? __ldcg(reinterpret_cast<const float4*>(g->rowA[i]) + q4)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    vb[k] = __ldcg(reinterpret_cast<const float4*>(g->rowB[i]) + q4);
  }
  float gh[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) gh[k] = __ldcg(a.GH + size_t(cell) * kRank + tid + kPairThreads * k);
  if (tid < kCand) g->U[tid] = __ldcg(a.cand_val + size_t(cell) * kCand + tid);
#pragma unroll
  for (int k = 0; k < 2; ++k) g->Hs[tid + kPairThreads * k] = 1.0f / (1.0f + expf(-gh[k]));
  sync();  // Hs complete
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int e = tid + kPairThreads * k;
    const int i = e >> 6, c = 4 * (e & 63);
    const float4 h = *reinterpret_cast<const float4*>(&g->Hs[c]);
    *reinterpret_cast<float4*>(&g->Gs[i][c]) =
        make_float4(va[k].x * h.x, va[k].y * h.y, va[k].z * h.z, va[k].w * h.w);
    *reinterpret_cast<float4*>(&g->Bsh[i][c]) = vb[k];
  }
  sync();
  bilinear16(g->Gs, g->Bsh, g->Srow, tid, sync);
  sync();
  for (int e = tid; e < kCand * kCand; e += kPairThreads) {
    const int i = e / kCand, j = e % kCand;
    const float v = i < npred ? g->Srow[i][j] + g->U[j] : -INFINITY;
    g->Srow[i][j] = v;
    if (a.scores) a.scores[size_t(cell) * kCand * kCand + e] = v;
  }
  sync();
}

template <int P>
__global__ void __launch_bounds__(kPairThreads * P) pair_walk_kernel(PairArgs a) {
  extern __shared__ __align__(16) uint8_t pw_smem[];
  const int grp = threadIdx.x / kPairThreads, tid = threadIdx.x % kPairThreads;
  const int CL = (a.L + P - 1) / P;  // the cluster size
  const int b = blockIdx.x / CL;
  const int rank = CL > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int t = rank * P + grp;
  const bool live = t < a.L;
  PairGroupSmem* g = reinterpret_cast<PairGroupSmem*>(pw_smem) + grp;
  PairWalkSmem* w = reinterpret_cast<PairWalkSmem*>(pw_smem + P * sizeof(PairGroupSmem));
  if (threadIdx.x == 0 && CL > 1) {
    mbar_init(&w->bar, 1);
    fence_mbar_init();
    // every position's choices, q rows and tokens, in bytes (stored with st.async)
    if (rank == 0)
      mbar_arrive_expect_tx(&w->bar, uint32_t(kCand * 4 + 1 * (4 + kCand * 4)) +
                                         uint32_t(a.L - 1) * uint32_t(kCand * 4 + kCand * (4 + kCand * 4)));
  }
  if (CL > 1)
    cluster_arrive_release();  // the first CTA's barrier is initialised before any store
  else
    __syncthreads();
  // The walk's random number for this position, before the dependency wait:
  // the Philox keys are the caller's input, and this kernel only starts once
  // the kernel before it has passed its own wait (so everything the caller
  // queued before this library's calls has finished).
  const float u = live && a.T > 0.f ? walk_uniform(__ldcg(a.seeds + b), a.cycle, t) : 0.f;
  pdl_wait();
  pdl_launch_dependents();
  auto sync = [grp]() { named_sync(1 + grp, kPairThreads); };
  if (live) pair_position(a, b, t, tid, g, sync);
  // ---- the walk's decision for every predecessor row of position t, and the
  // candidate tokens, into the first CTA (st.async, counted on its barrier) ----
  if (CL > 1) cluster_wait_acquire();
  if (live) {
    const int npred = t == 0 ? 1 : kCand;
    const int cell = b * a.L + t;
    const int j = tid & 15;
    // 16 lanes per predecessor row, 8 rows per pass
#pragma unroll 1
    for (int i = tid >> 4; i < kCand; i += kPairThreads / 16) {
      float q_j;
      const int c = walk_row_choice16(g->Srow[i][j], a.T, u, q_j);
      if (i < npred) {
        if (CL > 1) {
          st_async_f32(&w->q[t][i][j], 0u, q_j, &w->bar);
          if (j == 0) st_async_b32(&w->choice[t][i], 0u, static_cast<uint32_t>(c), &w->bar);
        } else {  // a single CTA (no cluster launch): plain stores
          w->q[t][i][j] = q_j;
          if (j == 0) w->choice[t][i] = c;
        }
      }
    }
    if (tid < kCand) {
      const int tok = __ldcg(a.cand_idx + size_t(cell) * kCand + tid);
      if (CL > 1)
        st_async_b32(&w->tok[t][tid], 0u, static_cast<uint32_t>(tok), &w->bar);
      else
        w->tok[t][tid] = tok;
    }
  }
  if (CL == 1) __syncthreads();
  if (rank != 0) return;
  // ---- first CTA: follow the chosen slots from the verified token ----
  if (threadIdx.x == 0) {
    if (CL > 1 && !mbar_wait_cluster(&w->bar, 0, a.err)) record_error(a.err, kDevErrGemm);
    int prev = 0;
    for (int tt = 0; tt < a.L; ++tt) {
      prev = w->choice[tt][prev] & (kCand - 1);
      w->path[tt] = prev;
    }
  }
  __syncthreads();
  for (int tt = threadIdx.x; tt < a.L; tt += blockDim.x) {
    const size_t c2 = size_t(b) * a.L + tt;
    a.tokens[c2] = w->tok[tt][w->path[tt]];
    if (a.slots) a.slots[c2] = w->path[tt];
  }
  if (a.q) {
    for (int e = threadIdx.x; e < a.L * kCand; e += blockDim.x) {
      const int tt = e / kCand, k = e % kCand;
      const int row = tt == 0 ? 0 : w->path[tt - 1];  // step tt draws from its predecessor's row
      a.q[(size_t(b) * a.L + tt) * kCand + k] = w->q[tt][row][k];
    }
  }
}

bool g_pw_attr[64][3];

// The fused pair + walk launch: clusters of ceil(L / P) CTAs per sequence, P
// the smallest of 1, 2, 4 that keeps the cluster within 8; L <= 32.
cudaError_t launch_pair_walk(const PairArgs& qa, int B, int L, cudaStream_t s, bool pdl) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int P = L <= 8 ? 1 : (L <= 16 ? 2 : 4);
  const int CL = (L + P - 1) / P;
  const size_t smem = size_t(P) * sizeof(PairGroupSmem) + sizeof(PairWalkSmem);
  const int pi = P == 1 ? 0 : (P == 2 ? 1 : 2);
  auto kern = P == 1 ? pair_walk_kernel<1> : (P == 2 ? pair_walk_kernel<2> : pair_walk_kernel<4>);
  if (!g_pw_attr[dev & 63][pi]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    g_pw_attr[dev & 63][pi] = true;
  }
  return launch_kc(kern, dim3(B * CL), dim3(kPairThreads * P), smem, s, pdl, CL, qa);
}

bool g_gemm_attr[64];
bool g_gemm_warp_attr[64];
std::atomic<int> g_proj_engine{DFL2_PROJ_TENSOR};
bool g_ab_attr[64];

}  // namespace

// K split of the gate projection run alone (the table path): the largest power
// of two <= 8 that keeps its tiles within one wave, every split non-empty.
static void gate_split(int MH, int kblocks, int& splits, int& kps) {
  const int tiles = (MH + kBM - 1) / kBM;
  splits = 1;
  while (splits * 2 <= kMaxClusterSplits && tiles * splits * 2 <= kGemmTargetCtas &&
         splits * 2 <= kblocks)
    splits *= 2;
  kps = (kblocks + splits - 1) / splits;
  splits = (kblocks + kps - 1) / kps;
}

int set_projection_engine(int engine) { return g_proj_engine.exchange(engine); }

SelectPlan select_plan(int B, int L, int d) {
  SelectPlan p{};
  p.B = B;
  p.L = L;
  p.d = d;
  p.MA = B * (kCand * (L - 1) + 1);
  p.MB = B * kCand * L;
  p.MH = B * L;
  p.kblocks = (d + kBK - 1) / kBK;  // the last block may be partial (d % 16 == 0)
  const int tiles = (p.MA + kBM - 1) / kBM + (p.MB + kBM - 1) / kBM + (p.MH + kBM - 1) / kBM;
  // Split K (over a cluster) only when the tiles cannot fill the GPU: the
  // largest power of two <= 8 that keeps tiles*splits within one wave.
  int splits = 1;
  while (splits * 2 <= kMaxClusterSplits && tiles * splits * 2 <= kGemmTargetCtas &&
         splits * 2 <= p.kblocks)
    splits *= 2;
  p.kps = (p.kblocks + splits - 1) / splits;
  p.splits = (p.kblocks + p.kps - 1) / p.kps;  // every split gets at least one K block
  // While there is room for twice the CTAs (batch 1: 5 row tiles x 8 splits),
  // each row tile's 256 outputs go to two (or four) CTAs, which divides the W
  // bytes and the partial tile of each CTA.
  p.nsplit = 1;
  while (p.nsplit < 4 && tiles * p.splits * p.nsplit * 2 <= kGemmTargetCtas) p.nsplit *= 2;
  p.PA_off = 256;
  p.PB_off = align_up(p.PA_off + size_t(p.MA) * kRank * 4, 256);
  p.GH_off = align_up(p.PB_off + size_t(p.MB) * kRank * 4, 256);
  p.part_off = align_up(p.GH_off + size_t(p.MH) * kRank * 4, 256);
  // split-K partials: of the three problems together, or of the gate alone
  // (the table path runs the gate projection by itself, with its own split)
  int gs, gk;
  gate_split(p.MH, p.kblocks, gs, gk);
  const size_t part_bytes = std::max(
      p.splits > 1 ? size_t(p.splits) * (p.MA + p.MB + p.MH) * kRank * 4 : size_t(0),
      gs > 1 ? size_t(gs) * p.MH * kRank * 4 : size_t(0));
  p.ticket_off = align_up(p.part_off + part_bytes, 256);
  p.choice_off = align_up(p.ticket_off + size_t(B) * 4, 256);
  p.q_off = align_up(p.choice_off + size_t(B) * L * kCand * 4, 256);
  p.ws_bytes = align_up(p.q_off + size_t(B) * L * kCand * kCand * 4, 256);
  p.M = p.MA;
  return p;
}

// One proj_tc launch over up to three problems (rows of `kind` times W^T).
struct ProjJob {
  int kind;
  int M;
  float* out;
  const __nv_bfloat16* W;
};

static cudaError_t ensure_gemm_attr() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!g_gemm_attr[dev & 63]) {
    e = cudaFuncSetAttribute(proj_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kGemmSmem));
    if (e != cudaSuccess) return e;
    g_gemm_attr[dev & 63] = true;
  }
  return cudaSuccess;
}

static cudaError_t launch_proj_jobs(const ProjJob* jobs, int njobs, int splits, int kps, int d,
                                    const __nv_bfloat16* E, const __nv_bfloat16* hidden,
                                    const int32_t* cand_idx, const int32_t* verified, int L, int V,
                                    float* part, cudaStream_t s, bool pdl) {
  cudaError_t e = ensure_gemm_attr();
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap tm[3];
  GemmArgs g{};
  int before = 0;
  for (int i = 0; i < 3; ++i) {
    const bool live = i < njobs;
    const __nv_bfloat16* W = live ? jobs[i].W : jobs[0].W;
    if (!tensor_map_bf16(W, kRank, d, kBN, &tm[i])) return cudaErrorInvalidValue;
    g.prob[i].W = W;
    g.prob[i].kind = live ? jobs[i].kind : kRowsHidden;
    g.prob[i].M = live ? jobs[i].M : 0;
    g.prob[i].mtiles = live ? (jobs[i].M + kBM - 1) / kBM : 0;
    g.prob[i].out = live ? jobs[i].out : nullptr;
    g.prob[i].part = part;
    if (live && splits > 1) part += size_t(splits) * jobs[i].M * kRank;
    g.tiles_before[i] = before;
    before += g.prob[i].mtiles;
  }
  g.splits = splits;
  g.nsplit = 1;
  g.kps = kps;
  g.kblocks = (d + kBK - 1) / kBK;
  g.E = E;
  g.hidden = hidden;
  g.cand_idx = cand_idx;
  g.verified = verified;
  g.L = L;
  g.V = V;
  g.d = d;
  g.err = device_error_word();
  if (before == 0) return cudaSuccess;
  return launch_kc(proj_tc_kernel<false>, dim3(before * splits), dim3(kGemmThreads), kGemmSmem, s, pdl,
                   splits, g, tm[0], tm[1], tm[2]);
}

// The pair scores (and the fused walk) over the projections in the workspace.
static cudaError_t launch_pair(const SelectPlan& p, const int32_t* cand_idx, const float* cand_val,
                               const float* PA, const float* PB, const float* GH, int V,
                               float* scores, const WalkFuse* walk, void* ws, cudaStream_t s,
                               bool pdl) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  PairArgs qa{};
  qa.PA = PA;
  qa.PB = PB;
  qa.GH = GH;
  qa.V = V;
  qa.err = device_error_word();
  qa.cand_val = cand_val;
  qa.scores = scores;
  qa.L = p.L;
  if (walk) {
    qa.walk = 1;
    qa.T = walk->T;
    qa.seeds = walk->seeds;
    qa.cycle = walk->cycle;
    qa.cand_idx = cand_idx;
    qa.tokens = walk->tokens;
    qa.slots = walk->slots;
    qa.q = walk->q;
    qa.tickets = reinterpret_cast<uint32_t*>(w + p.ticket_off);
    qa.choice = reinterpret_cast<int32_t*>(w + p.choice_off);
    qa.qrows = reinterpret_cast<float*>(w + p.q_off);
    if (p.L <= kPwMaxL) return launch_pair_walk(qa, p.B, p.L, s, pdl);
  }
  return launch_k(pair16_kernel, dim3(p.B * p.L), dim3(kPairThreads), 0, s, pdl, qa);
}

cudaError_t launch_select(const SelectPlan& p, const int32_t* cand_idx, const float* cand_val,
                          const int32_t* verified, const __nv_bfloat16* hidden,
                          const __nv_bfloat16* E, const __nv_bfloat16* W_A,
                          const __nv_bfloat16* W_B, const __nv_bfloat16* W_H, int V,
                          float* scores, const WalkFuse* walk, void* ws, cudaStream_t s,
                          bool pdl) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!g_gemm_attr[dev & 63]) {
    e = cudaFuncSetAttribute(proj_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kGemmSmem));
    if (e != cudaSuccess) return e;
    g_gemm_attr[dev & 63] = true;
  }
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* PA = reinterpret_cast<float*>(w + p.PA_off);
  float* PB = reinterpret_cast<float*>(w + p.PB_off);
  float* GH = reinterpret_cast<float*>(w + p.GH_off);
  if (p.splits == 1 && p.nsplit == 1) {
    // ---- batched: one gather per E row, [W_A; W_B] as N = 512 ----
    if (!g_ab_attr[dev & 63]) {
      e = cudaFuncSetAttribute(proj_ab_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kAbSmem));
      if (e != cudaSuccess) return e;
      g_ab_attr[dev & 63] = true;
    }
    alignas(64) CUtensorMap tA, tB, tH;  // boxes of 64 K x 256 W rows (one slot)
    if (!tensor_map_bf16(W_A, kRank, p.d, kBN, &tA) || !tensor_map_bf16(W_B, kRank, p.d, kBN, &tB) ||
        !tensor_map_bf16(W_H, kRank, p.d, kBN, &tH))
      return cudaErrorInvalidValue;
    AbArgs g{};
    g.M_ab = p.B * (kCand * p.L + 1);
    g.tiles_ab = (g.M_ab + kBM - 1) / kBM;
    g.M_h = p.MH;
    g.kblocks = p.kblocks;
    g.L = p.L;
    g.V = V;
    g.d = p.d;
    g.E = E;
    g.hidden = hidden;
    g.W_A = W_A;
    g.W_B = W_B;
    g.W_H = W_H;
    g.cand_idx = cand_idx;
    g.verified = verified;
    g.PA = PA;
    g.PB = PB;
    g.GH = GH;
    g.err = device_error_word();
    const int grid = g.tiles_ab + (p.MH + kBM - 1) / kBM;
    e = launch_kc(proj_ab_kernel, dim3(grid), dim3(kGemmThreads), kAbSmem, s, pdl, 1, g, tA, tB, tH);
    if (e != cudaSuccess) return e;
    return launch_pair(p, cand_idx, cand_val, PA, PB, GH, V, scores, walk, ws, s, pdl);
  }
  alignas(64) CUtensorMap tA, tB, tH;
  const uint32_t bn = static_cast<uint32_t>(kBN / p.nsplit);
  if (!tensor_map_bf16(W_A, kRank, p.d, bn, &tA) || !tensor_map_bf16(W_B, kRank, p.d, bn, &tB) ||
      !tensor_map_bf16(W_H, kRank, p.d, bn, &tH))
    return cudaErrorInvalidValue;
  GemmArgs g{};
  const int Ms[3] = {p.MA, p.MB, p.MH};
  float* outs[3] = {PA, PB, GH};
  float* part = reinterpret_cast<float*>(w + p.part_off);
  int before = 0;
  const __nv_bfloat16* Ws[3] = {W_A, W_B, W_H};
  for (int i = 0; i < 3; ++i) {
    g.prob[i].W = Ws[i];
    g.prob[i].kind = i;
    g.prob[i].M = Ms[i];
    g.prob[i].mtiles = (Ms[i] + kBM - 1) / kBM;
    g.prob[i].out = outs[i];
    g.prob[i].part = part;
    part += size_t(p.splits) * Ms[i] * kRank;
    g.tiles_before[i] = before;
    before += g.prob[i].mtiles;
  }
  g.splits = p.splits;
  g.nsplit = p.nsplit;
  g.kps = p.kps;
  g.kblocks = p.kblocks;
  g.E = E;
  g.hidden = hidden;
  g.cand_idx = cand_idx;
  g.verified = verified;
  g.L = p.L;
  g.V = V;
  g.d = p.d;
  g.err = device_error_word();
  // the warp-level engine when asked for and the CTAs hold 128 output columns
  if (g_proj_engine.load(std::memory_order_relaxed) == DFL2_PROJ_WARP && bn == 128) {
    if (!g_gemm_warp_attr[dev & 63]) {
      e = cudaFuncSetAttribute(proj_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kGemmSmem));
      if (e != cudaSuccess) return e;
      g_gemm_warp_attr[dev & 63] = true;
    }
    e = launch_kc(proj_tc_kernel<true>, dim3(before * p.nsplit * p.splits), dim3(kGemmThreads),
                  kGemmSmem, s, pdl, p.splits, g, tA, tB, tH);
  } else {
    e = launch_kc(proj_tc_kernel<false>, dim3(before * p.nsplit * p.splits), dim3(kGemmThreads),
                  kGemmSmem, s, pdl, p.splits, g, tA, tB, tH);
  }
  if (e != cudaSuccess) return e;
  return launch_pair(p, cand_idx, cand_val, PA, PB, GH, V, scores, walk, ws, s, pdl);
}

cudaError_t launch_tables_build(const __nv_bfloat16* E, const __nv_bfloat16* W_A,
                                const __nv_bfloat16* W_B, int V, int d, float* P_A, float* P_B,
                                cudaStream_t s) {
  // every row of E times W_A^T and W_B^T: one launch, two problems, K unsplit
  const ProjJob jobs[2] = {{kRowsE, V, P_A, W_A}, {kRowsE, V, P_B, W_B}};
  return launch_proj_jobs(jobs, 2, 1, (d + kBK - 1) / kBK, d, E, nullptr, nullptr, nullptr, 1, V, nullptr, s,
                          true);
}

cudaError_t launch_gate(const SelectPlan& p, const __nv_bfloat16* hidden, const __nv_bfloat16* W_H,
                        void* ws, cudaStream_t s, bool pdl) {
  // the hidden rows only (GH before the sigmoid), K split over a cluster when
  // the tiles cannot fill the GPU
  uint8_t* w = static_cast<uint8_t*>(ws);
  int splits, kps;
  gate_split(p.MH, p.kblocks, splits, kps);
  const ProjJob job{kRowsHidden, p.MH, reinterpret_cast<float*>(w + p.GH_off), W_H};
  return launch_proj_jobs(&job, 1, splits, kps, p.d, nullptr, hidden, nullptr, nullptr, p.L, 1,
                          reinterpret_cast<float*>(w + p.part_off), s, pdl);
}

cudaError_t launch_pair_tables(const SelectPlan& p, const int32_t* cand_idx, const float* cand_val,
                               const int32_t* verified, const float* P_A, const float* P_B, int V,
                               float* scores, const WalkFuse* walk, void* ws, cudaStream_t s,
                               bool pdl) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  PairArgs qa{};
  qa.tabA = P_A;
  qa.tabB = P_B;
  qa.verified = verified;
  qa.V = V;
  qa.err = device_error_word();
  qa.GH = reinterpret_cast<float*>(w + p.GH_off);
  qa.cand_val = cand_val;
  qa.cand_idx = cand_idx;
  qa.scores = scores;
  qa.L = p.L;
  if (walk) {
    qa.walk = 1;
    qa.T = walk->T;
    qa.seeds = walk->seeds;
    qa.cycle = walk->cycle;
    qa.tokens = walk->tokens;
    qa.slots = walk->slots;
    qa.q = walk->q;
    qa.tickets = reinterpret_cast<uint32_t*>(w + p.ticket_off);
    qa.choice = reinterpret_cast<int32_t*>(w + p.choice_off);
    qa.qrows = reinterpret_cast<float*>(w + p.q_off);
    if (p.L <= kPwMaxL) return launch_pair_walk(qa, p.B, p.L, s, pdl);
  }
  return launch_k(pair16_kernel, dim3(p.B * p.L), dim3(kPairThreads), 0, s, pdl, qa);
}

// ---- tensor maps ------------------------------------------------------------------
namespace {
struct TmapEntry {
  int dev;
  const void* base;
  uint64_t rows, cols;
  uint32_t box_rows;
  CUtensorMap map;
};
std::mutex g_tmap_mu;
constexpr int kTmapCache = 128;
TmapEntry g_tmap_cache[kTmapCache];
int g_tmap_n = 0, g_tmap_next = 0;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
}  // namespace

bool tensor_map_bf16(const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                     void* out128) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(g_tmap_mu);
  for (int i = 0; i < g_tmap_n; ++i) {
    const TmapEntry& t = g_tmap_cache[i];
    if (t.dev == dev && t.base == base && t.rows == rows && t.cols == cols &&
        t.box_rows == box_rows) {
      memcpy(out128, &t.map, sizeof(CUtensorMap));
      return true;
    }
  }
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  CUtensorMap m;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  if (g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  TmapEntry& t = g_tmap_cache[g_tmap_next];
  t = TmapEntry{dev, base, rows, cols, box_rows, m};
  g_tmap_next = (g_tmap_next + 1) % kTmapCache;
  g_tmap_n = std::min(g_tmap_n + 1, kTmapCache);
  memcpy(out128, &m, sizeof(CUtensorMap));
  return true;
}

}  // namespace dfl2
