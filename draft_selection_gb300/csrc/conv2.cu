// Two-tap dynamic depthwise conv ("DFlash 2: Keep Drafting Parallel",
// 方法细节 > 轻量级局部卷积, the Conv_k equation):
//   y_t = k_{t,0} ⊙ x_t + k_{t,1} ⊙ x_{t-1},  x_{-1} = the verified token's representation,
//   k_{t,j,c} = base[j,c] + corr[t,j,c/16],   corr[t,j,g] = sum_c W_c[j*G+g, c] x_t[c].
//
// The corrections are a GEMM, corr = X W_sel^T, with the B*L positions as rows
// and, per CTA, the 2*NG W_c rows of NG correction groups (tap 0 and tap 1 of
// the same groups) as columns.  It runs on tcgen05: 128-row tiles, K in blocks
// of 64, both operands staged by 16-byte cp.async in the 128-byte swizzle
// (zero fill past the ends, so any d that is a multiple of 16 works), the
// accumulator in TMEM.  The epilogue applies the 2-tap mix for the CTA's
// 16*NG channels, reading x_t and x_{t-1} (x_prev at t = 0) and writing y in
// bf16: the corrections never leave the chip.  With few positions (batch 1),
// K is split over a thread-block cluster and the partial corrections are summed
// through distributed shared memory, each CTA then mixing its slice of rows.
//
// For at most 16 positions (batch 1) a CUDA-core GEMV kernel spreads the
// groups over the whole GPU, one group mixed per CTA (conv_gemv_kernel).
// For 17..64 positions a transposed kernel computes
// corr^T = W_sel x^T instead: the 128 W_c rows of 64 groups (both taps) are the
// A operand, loaded by TMA with no padding, and the R positions are N.  K is
// split over a cluster; each CTA pushes its small partial (128 x R) to the CTA
// that owns those groups, which sums the splits in rank order and mixes.
#include <cuda.h>

#include <algorithm>

#include "dfl2_internal.cuh"

namespace dfl2 {
namespace {

constexpr int kCBM = 128, kCBK = 64, kCThreads = 256;
constexpr int kCMaxStages = 8;
constexpr int kCMaxNG = 64;          // groups per CTA: N = 2*NG <= 128
constexpr int kCMaxSplits = 8;       // portable cluster size
constexpr int kCAStage = kCBM * kCBK * 2;  // 16 KB
constexpr size_t kCSmemMax = 227 * 1024;

struct ConvArgs {
  const __nv_bfloat16* x;       // [R, d] (the mix; the GEMM reads x through tmX)
  const __nv_bfloat16* x_prev;  // [B, d]
  const float* base;            // [2, d]
  __nv_bfloat16* y;             // [R, d]
  int R, L, d, G;
  int NG, ntiles, splits, kps, kblocks, stages;
  int side;  // K blocks whose x tile is kept for the mix (the CTA's own channels), or 0
  uint32_t* err;
};

__host__ __device__ constexpr int conv_bstage_bytes(int NG) { return 2 * NG * kCBK * 2; }
__host__ __device__ constexpr int conv_pitch(int NG) { return 2 * NG + 4; }  // fp32 per row
__host__ __device__ constexpr size_t conv_tile_bytes(int NG) {
  return size_t(kCBM) * conv_pitch(NG) * 4;
}
// The corrections tile reuses the operand stages once the mainloop is over.
__host__ __device__ constexpr size_t conv_stage_area(int NG, int stages) {
  return size_t(stages) * (kCAStage + conv_bstage_bytes(NG)) > conv_tile_bytes(NG)
             ? size_t(stages) * (kCAStage + conv_bstage_bytes(NG))
             : conv_tile_bytes(NG);
}
// Receive slots for split K: S slots of ceil(128/S) rows, at most 128 + S rows.
__host__ __device__ constexpr size_t conv_recv_bytes(int NG, int splits) {
  return splits > 1 ? size_t(kCBM + kCMaxSplits) * conv_pitch(NG) * 4 : 0;
}
__host__ __device__ constexpr size_t conv_smem_bytes(int NG, int stages, int splits, int side) {
  // [operand stages | corrections] [kept x tiles] [receive slots] [base slice] [barriers]
  return 1024 + conv_stage_area(NG, stages) + size_t(side) * kCAStage +
         conv_recv_bytes(NG, splits) + size_t(2) * 16 * NG * 4 + 256;
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bf8_unpack(const uint4 v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    f[2 * q] = __uint_as_float(w[q] << 16);
    f[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
  }
}

// Warp roles: 0 = TMA producer (one thread), 1 = TMEM owner and MMA issuer (one
// thread), 2-3 = the base slice, 4-7 = TMEM -> corrections; then all 8 mix.
__global__ void __launch_bounds__(kCThreads) conv_tc_kernel(const __grid_constant__ ConvArgs a,
                                                            const __grid_constant__ CUtensorMap tmX,
                                                            const __grid_constant__ CUtensorMap tmW) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int NG = a.NG, N = 2 * NG, pitch = conv_pitch(NG);
  const int bst = conv_bstage_bytes(NG);
  const int nst = a.stages;
  uint8_t* sA = smem;                                   // [stages][128 rows][128 B]
  uint8_t* sB = smem + size_t(nst) * kCAStage;          // [stages][2*NG rows][128 B]
  float* corr = reinterpret_cast<float*>(smem);         // [128][pitch], after the mainloop
  // x tiles of the K blocks that hold this CTA's own channels, kept for the mix
  uint8_t* sKeep = smem + conv_stage_area(NG, nst);                      // [side][128 rows][128 B]
  float* recv = reinterpret_cast<float*>(sKeep + size_t(a.side) * kCAStage);  // [S][rows_per][pitch]
  float* bslice = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(recv) +
                                           conv_recv_bytes(NG, a.splits));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(bslice + 2 * 16 * NG);
  uint64_t* empty_bar = full_bar + kCMaxStages;
  uint64_t* accum_bar = empty_bar + kCMaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum_bar + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x % a.splits;
  const int tile = blockIdx.x / a.splits;
  const int m0 = (tile / a.ntiles) * kCBM;
  const int g0 = (tile % a.ntiles) * NG;
  const int kb0 = split * a.kps;
  const int nkb = min(a.kblocks, kb0 + a.kps) - kb0;  // >= 1 by construction on the host
  const uint32_t ncols = N < 32 ? 32u : static_cast<uint32_t>(N);
  const int kbk0 = (16 * g0) / kCBK;  // first K block of this CTA's channels

  if (tid == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(accum_bar, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) tmem_alloc(tmem_slot, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {  // ---- producer: x rows and both taps' W_c rows by TMA ----
      const uint32_t tx = static_cast<uint32_t>(kCAStage + bst);
      for (int it = 0, s = 0, ph = 0; it < nkb; ++it) {
        if (it >= nst && !mbar_wait(&empty_bar[s], ph ^ 1, a.err)) record_error(a.err, kDevErrConv);
        const int kb = kb0 + it;
        const int k0 = kb * kCBK;
        const int keep = kb - kbk0;  // in [0, side): this x tile stays for the mix
        mbar_arrive_expect_tx(&full_bar[s], tx);
        tma_load_2d(keep >= 0 && keep < a.side ? sKeep + size_t(keep) * kCAStage
                                               : sA + size_t(s) * kCAStage,
                    &tmX, k0, m0, &full_bar[s]);
        uint8_t* dB = sB + size_t(s) * bst;
        tma_load_2d(dB, &tmW, k0, g0, &full_bar[s]);
        tma_load_2d(dB + NG * 128, &tmW, k0, a.G + g0, &full_bar[s]);
        if (++s == nst) {
          s = 0;
          ph ^= 1;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issuer ----
      const uint32_t idesc = umma_idesc_bf16(kCBM, N);
      for (int it = 0, s = 0, ph = 0; it < nkb; ++it) {
        if (!mbar_wait(&full_bar[s], ph, a.err)) record_error(a.err, kDevErrConv);
        tc_fence_after();
        const int keep = kb0 + it - kbk0;
        const uint64_t ad = umma_desc_sw128(keep >= 0 && keep < a.side ? sKeep + size_t(keep) * kCAStage
                                                                       : sA + size_t(s) * kCAStage);
        const uint64_t bd = umma_desc_sw128(sB + size_t(s) * bst);
#pragma unroll
        for (int k = 0; k < kCBK / 16; ++k)
          umma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc, (it > 0 || k > 0) ? 1u : 0u);
        umma_commit(&empty_bar[s]);
        if (++s == nst) {
          s = 0;
          ph ^= 1;
        }
      }
      umma_commit(accum_bar);
    }
    __syncwarp();
  } else if (warp < 4) {
    // idle during the mainloop: the base slice for the CTA's channels, stored
    // [tap][channel within group][group] so that threads on consecutive groups
    // read consecutive banks in the mix
    for (int e = tid - 64; e < 2 * 16 * NG; e += 64) {
      const int tap = e / (16 * NG), cl = e % (16 * NG), c = 16 * g0 + cl;
      bslice[tap * 16 * NG + (cl % 16) * NG + cl / 16] = c < a.d ? a.base[size_t(tap) * a.d + c] : 0.f;
    }
  } else {
    // ---- TMEM -> the corrections (one split), or push this split's partial rows
    // into the receive slot of the CTA that owns them (split K).  The accumulator
    // is complete only when every MMA, and so every read of the stages, is done. ----
    const int quarter = warp & 3;
    if (!mbar_wait(accum_bar, 0, a.err)) record_error(a.err, kDevErrConv);
    tc_fence_after();
    const int lrow = quarter * 32 + lane;
    const int per = (kCBM + a.splits - 1) / a.splits;
    const int owner = lrow / per;
    const bool live = m0 + lrow < a.R;  // rows past R carry nothing
    for (int c = 0; c < N; c += 32) {
      float v[32];
      tmem_ld32(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(c), v);
      if (a.splits == 1) {
        float* dst = corr + size_t(lrow) * pitch + c;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(dst + 4 * q) =
              make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      } else if (live) {
        const float* slot = recv + (size_t(split) * per + (lrow - owner * per)) * pitch + c;
        const uint32_t dst = dsmem_addr(slot, static_cast<uint32_t>(owner));
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dsmem_st4(dst + 16u * q, make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
      }
    }
  }
  tc_fence_before();
  int r_lo = 0, r_n = kCBM;
  if (a.splits == 1) {
    __syncthreads();
  } else {
    // ---- every slot has arrived: sum this CTA's rows over the splits, in rank order ----
    cluster_sync_all();
    const int S = a.splits;
    const int per = (kCBM + S - 1) / S;
    r_lo = split * per;
    r_n = max(0, min(per, kCBM - r_lo));
    const int valid = max(0, min(r_n, a.R - (m0 + r_lo)));
    const int n4 = N / 4;
    for (int e = tid; e < valid * n4; e += kCThreads) {
      const int lr = e / n4, c4 = e % n4;
      float4 acc = *reinterpret_cast<const float4*>(recv + size_t(lr) * pitch + 4 * c4);
      for (int k = 1; k < S; ++k) {
        const float4 v = *reinterpret_cast<const float4*>(recv + (size_t(k) * per + lr) * pitch + 4 * c4);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      *reinterpret_cast<float4*>(corr + size_t(lr) * pitch + 4 * c4) = acc;
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
  pdl_launch_dependents();

  if (a.side) {
    // ---- the 2-tap mix from the kept tiles: thread = (group, half of its 16
    // channels), base in registers, down a run of consecutive rows (x_{t-1} is
    // the previous row's x_t), four rows at a time so that their arithmetic
    // overlaps.  The host takes this path only when L >= run, so a run holds at
    // most one position t = 0 (x_{t-1} = x_prev); that row and the row above the
    // run are the only loads from global memory, issued before the loop. ----
    const int q = tid % (2 * NG), gl = q >> 1, h = q & 1;
    const int groups = kCThreads / (2 * NG);
    const int run = (kCBM + groups - 1) / groups;
    const int g = g0 + gl;
    const int lr0 = (tid / (2 * NG)) * run;
    const int lend = min(min(lr0 + run, kCBM), a.R - m0);
    if (tid < groups * 2 * NG && g < a.G && lr0 < lend) {
      const int c = 16 * g + 8 * h;  // first of this thread's 8 channels
      const int ch = c - kCBK * kbk0;  // channel within the kept tiles
      const uint8_t* tile = sKeep + size_t(ch / kCBK) * kCAStage;
      const int j = (ch % kCBK) / 8;
      auto kept = [&](int row) {
        return *reinterpret_cast<const uint4*>(tile + row * 128 + ((j ^ (row & 7)) << 4));
      };
      const int t0 = (m0 + lr0) % a.L;
      const int tz = t0 == 0 ? 0 : a.L - t0;  // offset of the run's t = 0 row, if < run
      uint4 xp = make_uint4(0u, 0u, 0u, 0u);
      if (lr0 + tz < lend)
        xp = __ldcg(reinterpret_cast<const uint4*>(a.x_prev + size_t((m0 + lr0 + tz) / a.L) * a.d + c));
      uint4 prev = xp;  // x_{t-1} of the first row
      if (t0 != 0)
        prev = lr0 > 0 ? kept(lr0 - 1)
                       : __ldcg(reinterpret_cast<const uint4*>(a.x + size_t(m0 - 1) * a.d + c));
      float b0[8], b1[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        b0[i] = bslice[(8 * h + i) * NG + gl];
        b1[i] = bslice[16 * NG + (8 * h + i) * NG + gl];
      }
      constexpr int kU = 4;
      for (int lr = lr0; lr < lend; lr += kU) {
        uint4 xt[kU], xm[kU];
        float c0[kU], c1[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int row = min(lr + u, lend - 1);
          xt[u] = kept(row);
          c0[u] = corr[size_t(row) * pitch + gl];
          c1[u] = corr[size_t(row) * pitch + NG + gl];
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          xm[u] = (lr + u - lr0 == tz) ? xp : (u == 0 ? prev : xt[u - 1]);
        }
        prev = xt[kU - 1];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          if (lr + u >= lend) break;
          float ft[8], fm[8];
          bf8_unpack(xt[u], ft);
          bf8_unpack(xm[u], fm);
          uint32_t ow[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float lo =
                fmaf(b0[2 * i] + c0[u], ft[2 * i], (b1[2 * i] + c1[u]) * fm[2 * i]);
            const float hi = fmaf(b0[2 * i + 1] + c0[u], ft[2 * i + 1],
                                  (b1[2 * i + 1] + c1[u]) * fm[2 * i + 1]);
            const __nv_bfloat162 pr = __floats2bfloat162_rn(lo, hi);
            ow[i] = *reinterpret_cast<const uint32_t*>(&pr);
          }
          *reinterpret_cast<uint4*>(a.y + size_t(m0 + lr + u) * a.d + c) =
              make_uint4(ow[0], ow[1], ow[2], ow[3]);
        }
      }
    }
    return;
  }
  // ---- the 2-tap mix: one (row, group) = 16 channels per item, 4 items per pass ----
  constexpr int kBatch = 4;
  const int items = r_n * NG;
  for (int e0 = tid; e0 < items; e0 += kCThreads * kBatch) {
    uint4 vt[kBatch][2], vm[kBatch][2];
    bool ok[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {  // every load of the pass first
      const int e = e0 + u * kCThreads;
      const int lr = e / NG, gl = e % NG;
      const int r = m0 + r_lo + lr, g = g0 + gl;
      ok[u] = e < items && r < a.R && g < a.G;
      if (ok[u]) {
        const int t = r % a.L;
        const uint4* xt = reinterpret_cast<const uint4*>(a.x + size_t(r) * a.d + 16 * g);
        const uint4* xm = reinterpret_cast<const uint4*>(
            (t > 0 ? a.x + size_t(r - 1) * a.d : a.x_prev + size_t(r / a.L) * a.d) + 16 * g);
        vt[u][0] = xt[0];
        vt[u][1] = xt[1];
        vm[u][0] = xm[0];
        vm[u][1] = xm[1];
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (!ok[u]) continue;
      const int e = e0 + u * kCThreads;
      const int lr = e / NG, gl = e % NG;
      const int r = m0 + r_lo + lr, g = g0 + gl;
      const float c0 = corr[size_t(lr) * pitch + gl];
      const float c1 = corr[size_t(lr) * pitch + NG + gl];
      const float* b0 = bslice + gl;            // channel ch at b0[ch * NG]
      const float* b1 = bslice + 16 * NG + gl;
      uint4 out[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t tw[4] = {vt[u][h].x, vt[u][h].y, vt[u][h].z, vt[u][h].w};
        const uint32_t mw[4] = {vm[u][h].x, vm[u][h].y, vm[u][h].z, vm[u][h].w};
        uint32_t ow[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int ch = 8 * h + 2 * q;
          const float lo = fmaf(b0[ch * NG] + c0, __uint_as_float(tw[q] << 16),
                                (b1[ch * NG] + c1) * __uint_as_float(mw[q] << 16));
          const float hi = fmaf(b0[(ch + 1) * NG] + c0, __uint_as_float(tw[q] & 0xFFFF0000u),
                                (b1[(ch + 1) * NG] + c1) * __uint_as_float(mw[q] & 0xFFFF0000u));
          const __nv_bfloat162 pr = __floats2bfloat162_rn(lo, hi);
          ow[q] = *reinterpret_cast<const uint32_t*>(&pr);
        }
        out[h] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
      }
      uint4* yo = reinterpret_cast<uint4*>(a.y + size_t(r) * a.d + 16 * g);
      yo[0] = out[0];
      yo[1] = out[1];
    }
  }
}

bool g_conv_attr[64];

// ============================================================================
// Few positions: corr^T = W_sel x^T (W_c rows as A, positions as N).
// ============================================================================
constexpr int kSStages = 4;
constexpr int kSGroups = 64;  // groups per CTA tile: 128 W_c rows (both taps)
constexpr int kSMaxRows = 64; // positions handled by the transposed kernel (N <= 64)

struct ConvSmallArgs {
  const __nv_bfloat16* x;
  const __nv_bfloat16* x_prev;
  const float* base;
  __nv_bfloat16* y;
  int R, L, d, G, Npad, splits, kps, kblocks;
  uint32_t* err;
};

__host__ __device__ constexpr int small_pitch(int Npad) { return Npad + 4; }
__host__ __device__ size_t small_smem_bytes(int Npad, int S) {
  const size_t stages = size_t(kSStages) * (kCAStage + size_t(Npad) * 128);
  const int owned_rows = 2 * (kSGroups / S);
  const size_t recv = size_t(S) * owned_rows * small_pitch(Npad) * 4;
  const size_t corr = size_t(owned_rows) * small_pitch(Npad) * 4;
  const size_t bsl = size_t(2) * 16 * (kSGroups / S) * 4;
  return 1024 + stages + recv + corr + bsl + 256;
}

__global__ void __launch_bounds__(kCThreads, 1)
    conv_small_kernel(const __grid_constant__ ConvSmallArgs a,
                      const __grid_constant__ CUtensorMap tmW) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int S = a.splits, Np = a.Npad, pitch = small_pitch(Np);
  const int og = kSGroups / S;    // groups this CTA mixes
  const int orows = 2 * og;       // their W_c rows (tap 0, then tap 1)
  uint8_t* sA = smem;                                          // [stages][128 rows][128 B]
  uint8_t* sB = smem + size_t(kSStages) * kCAStage;            // [stages][Np rows][128 B]
  float* recv = reinterpret_cast<float*>(sB + size_t(kSStages) * Np * 128);  // [S][orows][pitch]
  float* corr = recv + size_t(S) * orows * pitch;              // [orows][pitch]
  float* bslice = corr + size_t(orows) * pitch;                // [2][16*og]
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(bslice + 2 * 16 * og);
  uint64_t* empty_bar = full_bar + kSStages;
  uint64_t* accum_bar = empty_bar + kSStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum_bar + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x % S;
  const int g0 = (blockIdx.x / S) * kSGroups;
  const int kb0 = split * a.kps;
  const int nkb = min(a.kblocks, kb0 + a.kps) - kb0;
  const uint32_t ncols = Np <= 32 ? 32u : (Np <= 64 ? 64u : 128u);
  const int gown = g0 + split * og;  // first group this CTA mixes

  if (tid == 0) {
    for (int st = 0; st < kSStages; ++st) {
      mbar_init(&full_bar[st], 1 + 32);  // the TMA expect_tx + the 32 lanes staging x
      mbar_init(&empty_bar[st], 1);
    }
    mbar_init(accum_bar, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) tmem_alloc(tmem_slot, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();

  if (warp == 0) {
    // ---- producer: W_c rows by TMA (two boxes of 64 rows), x rows by cp.async ----
    for (int it = 0; it < nkb; ++it) {
      const int st = it % kSStages;
      if (it >= kSStages && !mbar_wait(&empty_bar[st], ((it / kSStages) - 1) & 1, a.err))
        record_error(a.err, kDevErrConv);
      const int k0 = (kb0 + it) * kCBK;
      uint8_t* dA = sA + size_t(st) * kCAStage;
      if (lane == 0) {
        mbar_arrive_expect_tx(&full_bar[st], kCAStage);
        tma_load_2d(dA, &tmW, k0, g0, &full_bar[st]);
        tma_load_2d(dA + kCAStage / 2, &tmW, k0, a.G + g0, &full_bar[st]);
      }
      uint8_t* dB = sB + size_t(st) * Np * 128;
      for (int ch = lane; ch < Np * 8; ch += 32) {
        const int r = ch >> 3, j = ch & 7;
        const bool ok = r < a.R;
        cp_async16(dB + r * 128 + ((j ^ (r & 7)) << 4),
                   ok ? a.x + size_t(r) * a.d + k0 + j * 8 : a.x, ok);
      }
      cp_async_commit();
      if (it >= 2) {
        cp_async_wait<2>();
        fence_proxy_async_smem();
        mbar_arrive(&full_bar[(it - 2) % kSStages]);
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    for (int it = max(0, nkb - 2); it < nkb; ++it) mbar_arrive(&full_bar[it % kSStages]);
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(kCBM, Np);
      for (int it = 0; it < nkb; ++it) {
        const int st = it % kSStages;
        if (!mbar_wait(&full_bar[st], (it / kSStages) & 1, a.err)) record_error(a.err, kDevErrConv);
        tc_fence_after();
        const uint64_t ad = umma_desc_sw128(sA + size_t(st) * kCAStage);
        const uint64_t bd = umma_desc_sw128(sB + size_t(st) * Np * 128);
#pragma unroll
        for (int k = 0; k < kCBK / 16; ++k)
          umma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc, (it > 0 || k > 0) ? 1u : 0u);
        umma_commit(&empty_bar[st]);
      }
      umma_commit(accum_bar);
    }
    __syncwarp();
  } else if (warp < 4) {
    // idle during the mainloop: the base slice of the channels this CTA mixes
    for (int e = tid - 64; e < 2 * 16 * og; e += 64) {
      const int tap = e / (16 * og), c = 16 * gown + e % (16 * og);
      bslice[e] = c < a.d ? a.base[size_t(tap) * a.d + c] : 0.f;
    }
  } else {
    // ---- TMEM row r = W_c row (tap r/64, group g0 + r%64), columns = positions:
    // push the R values to the CTA that mixes that group ----
    if (!mbar_wait(accum_bar, 0, a.err)) record_error(a.err, kDevErrConv);
    tc_fence_after();
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int tap = r / kSGroups, gl = r % kSGroups;
    const int owner = gl / og;
    const int orow = tap * og + (gl % og);
    const uint32_t dst = dsmem_addr(recv + (size_t(split) * orows + orow) * pitch,
                                    static_cast<uint32_t>(owner));
    for (int c = 0; c < Np; c += 32) {
      float v[32];
      tmem_ld32(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(c), v);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (c + 4 * q < Np)
          dsmem_st4(dst + uint32_t(c + 4 * q) * 4u,
                    make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
    }
  }
  tc_fence_before();
  cluster_sync_all();  // all partials have arrived (also a CTA barrier)
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
  // ---- sum the splits in rank order for this CTA's rows ----
  const int n4 = orows * (Np / 4);
  for (int e = tid; e < n4; e += kCThreads) {
    const int orow = e / (Np / 4), c4 = e % (Np / 4);
    float4 acc = *reinterpret_cast<const float4*>(recv + size_t(orow) * pitch + 4 * c4);
    for (int k = 1; k < S; ++k) {
      const float4 v = *reinterpret_cast<const float4*>(recv + (size_t(k) * orows + orow) * pitch + 4 * c4);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    *reinterpret_cast<float4*>(corr + size_t(orow) * pitch + 4 * c4) = acc;
  }
  __syncthreads();
  pdl_launch_dependents();
  // ---- the 2-tap mix for the owned groups: one (position, group) per item ----
  const int items = a.R * og;
  for (int e = tid; e < items; e += kCThreads) {
    const int p = e / og, gl = e % og;
    const int g = gown + gl;
    if (g >= a.G) continue;
    const int t = p % a.L;
    const float c0 = corr[size_t(gl) * pitch + p];
    const float c1 = corr[size_t(og + gl) * pitch + p];
    const uint4* xt = reinterpret_cast<const uint4*>(a.x + size_t(p) * a.d + 16 * g);
    const uint4* xm = reinterpret_cast<const uint4*>(
        (t > 0 ? a.x + size_t(p - 1) * a.d : a.x_prev + size_t(p / a.L) * a.d) + 16 * g);
    const uint4 vt0 = xt[0], vt1 = xt[1], vm0 = xm[0], vm1 = xm[1];
    const float* b0 = bslice + 16 * gl;
    const float* b1 = bslice + 16 * og + 16 * gl;
    uint4 out[2];
    const uint4 vts[2] = {vt0, vt1}, vms[2] = {vm0, vm1};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t tw[4] = {vts[h].x, vts[h].y, vts[h].z, vts[h].w};
      const uint32_t mw[4] = {vms[h].x, vms[h].y, vms[h].z, vms[h].w};
      uint32_t ow[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int ch = 8 * h + 2 * q;
        const float lo = fmaf(b0[ch] + c0, __uint_as_float(tw[q] << 16),
                              (b1[ch] + c1) * __uint_as_float(mw[q] << 16));
        const float hi = fmaf(b0[ch + 1] + c0, __uint_as_float(tw[q] & 0xFFFF0000u),
                              (b1[ch + 1] + c1) * __uint_as_float(mw[q] & 0xFFFF0000u));
        const __nv_bfloat162 pr = __floats2bfloat162_rn(lo, hi);
        ow[q] = *reinterpret_cast<const uint32_t*>(&pr);
      }
      out[h] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    }
    uint4* yo = reinterpret_cast<uint4*>(a.y + size_t(p) * a.d + 16 * g);
    yo[0] = out[0];
    yo[1] = out[1];
  }
}

bool g_conv_small_attr[64];

// ============================================================================
// Many positions: corr^T tiles of 128 W_c rows x up to 256 positions.
// ============================================================================
// The transposed product of the kernel above, now over tiles of Np <= 256
// positions (the N of one tcgen05.mma at M = 128).  A tile pairs 64 groups
// (their 128 W_c rows, both taps, as A) with Np positions (as B), so a position
// tile's x rows are read once per 64 groups instead of once per narrow group
// slice, and W_c once per position tile.  Both operands arrive by TMA (zero
// fill past the last position and the last W_c row).  When the tiles do not
// cover the GPU, K is split over a cluster of S CTAs and the partial tiles are
// exchanged through a caller workspace in L2: each CTA stores its tile in
// whole 128-byte row pieces, one cluster barrier (release / acquire), and CTA
// s of the cluster sums, in rank order, the S slices of the rows of groups
// [s*64/S, (s+1)*64/S) of the tile, the groups it mixes.  (The same exchange
// over distributed shared memory was measured at about 6 us for the 128 KB
// tiles of a 96-CTA launch, against 4 us for the whole mainloop; L2 delivers
// several times the bandwidth.)  Each thread then mixes a run of 16
// consecutive positions of 8 channels, loading the run's x rows at once and
// carrying x_{t-1} in registers.
constexpr int kPGroups = 64;     // groups per tile: 128 W_c rows (both taps) = M
constexpr int kPMaxStages = 4;
constexpr int kPRun = 16;        // consecutive positions mixed by one thread

struct ConvPtileArgs {
  const __nv_bfloat16* x;       // [R, d] (the mix; the GEMM reads x through tmX)
  const __nv_bfloat16* x_prev;  // [B, d]
  const float* base;            // [2, d]
  __nv_bfloat16* y;             // [R, d]
  float* ws;                    // [tiles][splits][128][Np] partials (splits > 1)
  int R, L, d, G, Np, gtiles, splits, kps, kblocks, stages;
  uint32_t* err;
};

__host__ __device__ constexpr size_t ptile_stage_bytes(int Np) {
  return size_t(kCAStage) + size_t(Np) * 128;  // [128 W_c rows | Np x rows] x 128 B
}
__host__ __device__ constexpr int ptile_pitch(int Np) { return Np + 4; }  // fp32 per slot row
constexpr size_t kPScratch = size_t(8) * 32 * 128;  // a 32 x 32 fp32 block per warp
__host__ __device__ constexpr size_t ptile_max3(size_t a, size_t b, size_t c) {
  return a > b ? (a > c ? a : c) : (b > c ? b : c);
}
// The operand ring; after the mainloop the same bytes hold the warps' transpose
// blocks and, past them, the corrections of the CTA's groups (all 128 rows
// when S = 1).
__host__ __device__ constexpr size_t ptile_area(int Np, int stages) {
  return ptile_max3(size_t(stages) * ptile_stage_bytes(Np),
                    kPScratch + size_t(2 * kPGroups) * ptile_pitch(Np) * 4, 0);
}
// Partial tiles exchanged through the workspace: [tiles][S][128][Np] fp32.
__host__ __device__ constexpr size_t ptile_ws_bytes(long long tiles, int S, int Np) {
  return S > 1 ? size_t(tiles) * S * size_t(2 * kPGroups) * Np * 4 : 0;
}
__host__ __device__ constexpr size_t ptile_smem_bytes(int Np, int stages) {
  // [ring | transpose blocks | corrections] [base slice, 2 x 16 x 64 f32] [barriers, TMEM slot]
  return 1024 + ptile_area(Np, stages) + size_t(2) * 16 * kPGroups * 4 + 256;
}

// Warp roles in the mainloop: 0 = TMA producer (one thread), 1 = TMEM owner and
// MMA issuer (one thread), 2-3 = the base slice.  Then all 8 warps drain TMEM
// (warps w and w+4 share lane quarter w%4, alternate 32-column chunks) and mix.
__global__ void __launch_bounds__(kCThreads, 2)
    conv_ptile_kernel(const __grid_constant__ ConvPtileArgs a,
                      const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmX) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int S = a.splits, Np = a.Np, pitch = ptile_pitch(Np), nst = a.stages;
  const int og = kPGroups / S;  // groups this CTA mixes
  const int orows = 2 * og;     // their W_c rows (tap 0, then tap 1)
  const size_t sbytes = ptile_stage_bytes(Np);
  uint8_t* ring = smem;  // stage s: [W_c 16 KB][x Np x 128 B]
  float* bslice = reinterpret_cast<float*>(smem + ptile_area(Np, nst));  // [2][16*og]
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(bslice + 2 * 16 * kPGroups);
  uint64_t* empty_bar = full_bar + kPMaxStages;
  uint64_t* accum_bar = empty_bar + kPMaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum_bar + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x % S;
  const int tile = blockIdx.x / S;
  const int g0 = (tile % a.gtiles) * kPGroups;
  const int p0 = (tile / a.gtiles) * Np;
  const int kb0 = split * a.kps;
  const int nkb = min(a.kblocks, kb0 + a.kps) - kb0;  // >= 1 by construction on the host
  const uint32_t ncols = Np <= 32 ? 32u : (Np <= 64 ? 64u : (Np <= 128 ? 128u : 256u));
  const int gown = g0 + split * og;  // first group this CTA mixes
  // Index arithmetic of the loops after the mainloop, set up once: og (and so
  // 2 og) is a power of two (S is), and e / (Np / 4) for e < 2^16 is one
  // multiply-high by ceil(2^32 / (Np / 4)) (exact while e * (Np / 4) < 2^32).
  const int ogs = 31 - __clz(og);
  const uint32_t np4 = uint32_t(Np / 4);
  const uint64_t np4_inv = ((uint64_t(1) << 32) + np4 - 1) / np4;
  auto div_np4 = [&](int e) { return int((uint64_t(uint32_t(e)) * np4_inv) >> 32); };

  if (tid == 0) {
    for (int st = 0; st < nst; ++st) {
      mbar_init(&full_bar[st], 1);
      mbar_init(&empty_bar[st], 1);
    }
    mbar_init(accum_bar, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) tmem_alloc(tmem_slot, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {  // ---- producer: both taps' W_c rows and Np x rows by TMA ----
      const uint32_t tx = static_cast<uint32_t>(sbytes);
      for (int it = 0; it < nkb; ++it) {
        const int st = it % nst;
        if (it >= nst && !mbar_wait(&empty_bar[st], ((it / nst) - 1) & 1, a.err))
          record_error(a.err, kDevErrConv);
        const int k0 = (kb0 + it) * kCBK;
        uint8_t* dst = ring + size_t(st) * sbytes;
        mbar_arrive_expect_tx(&full_bar[st], tx);
        tma_load_2d(dst, &tmW, k0, g0, &full_bar[st]);
        tma_load_2d(dst + kCAStage / 2, &tmW, k0, a.G + g0, &full_bar[st]);
        tma_load_2d(dst + kCAStage, &tmX, k0, p0, &full_bar[st]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issuer ----
      const uint32_t idesc = umma_idesc_bf16(kCBM, Np);
      for (int it = 0; it < nkb; ++it) {
        const int st = it % nst;
        if (!mbar_wait(&full_bar[st], (it / nst) & 1, a.err)) record_error(a.err, kDevErrConv);
        tc_fence_after();
        const uint64_t ad = umma_desc_sw128(ring + size_t(st) * sbytes);
        const uint64_t bd = umma_desc_sw128(ring + size_t(st) * sbytes + kCAStage);
#pragma unroll
        for (int k = 0; k < kCBK / 16; ++k)
          umma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc, (it > 0 || k > 0) ? 1u : 0u);
        umma_commit(&empty_bar[st]);
      }
      umma_commit(accum_bar);
    }
    __syncwarp();
  } else if (warp < 4) {
    // idle during the mainloop: the base slice of the channels this CTA mixes
    for (int e = tid - 64; e < 2 * 16 * og; e += 64) {
      const int tap = e / (16 * og), c = 16 * gown + e % (16 * og);
      bslice[e] = c < a.d ? a.base[size_t(tap) * a.d + c] : 0.f;
    }
  }
  // ---- every MMA of this CTA is done: the operand ring is free ----
  if (!mbar_wait(accum_bar, 0, a.err)) record_error(a.err, kDevErrConv);
  tc_fence_after();
  const int quarter = warp & 3;
  // [orows][pitch]: this CTA's groups (all 128 rows when S = 1), past the
  // warps' transpose blocks
  float* corr = reinterpret_cast<float*>(smem + kPScratch);
  if (S == 1) {
    // TMEM lane = W_c row = tap * 64 + group, column = position: all rows are ours
    const int row = quarter * 32 + lane;
    for (int c = warp < 4 ? 32 : 0; c < Np; c += 64) {
      float v[32];
      tmem_ld32(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(c), v);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (c + 4 * q < Np)
          *reinterpret_cast<float4*>(corr + size_t(row) * pitch + c + 4 * q) =
              make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
  } else {
    // The partial tile [128 W_c rows][Np] goes to this split's slice of the
    // workspace (all of it: keeping the CTA's own rows in shared memory instead
    // measured about 1 us slower per call).  Each 32 x 32 block passes through
    // the warp's scratch (16-byte chunks XOR-swizzled by row), so that a store
    // instruction writes four rows of 128 contiguous bytes.
    float* part = a.ws + (size_t(tile) * S + split) * (size_t(2 * kPGroups) * Np);
    float4* blk = reinterpret_cast<float4*>(smem) + warp * 256;
    const int q = lane & 7;
    for (int c = warp < 4 ? 32 : 0; c < Np; c += 64) {
      float v[32];
      tmem_ld32(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(c), v);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        blk[lane * 8 + (k ^ (lane & 7))] =
            make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
      __syncwarp();
      if (c + 4 * q < Np) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int rr = 4 * k + (lane >> 3);  // row of the block
          __stcg(reinterpret_cast<float4*>(part + size_t(quarter * 32 + rr) * Np + c + 4 * q),
                 blk[rr * 8 + (q ^ (rr & 7))]);
        }
      }
      __syncwarp();
    }
  }
  tc_fence_before();
  // every slice of the cluster is written (release / acquire at cluster scope)
  if (S > 1) cluster_sync_all(); else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
  pdl_launch_dependents();
  if (S > 1) {
    // ---- this CTA's rows (tap j, group split*og + i) summed over the S slices
    // in rank order, read through L2; two items per thread at a time so that
    // 2*S loads are in flight ----
    const float* parts = a.ws + size_t(tile) * S * (size_t(2 * kPGroups) * Np);
    const size_t slice = size_t(2 * kPGroups) * Np;
    const int n4 = orows * (Np / 4);
    for (int e0 = tid; e0 < n4; e0 += 2 * kCThreads) {
      float4 v[2][kCMaxSplits];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = min(e0 + h * kCThreads, n4 - 1);
        const int orow = div_np4(e), c4 = e - orow * int(np4);
        const int row = (orow >> ogs) * kPGroups + split * og + (orow & (og - 1));
        const float* src = parts + size_t(row) * Np + 4 * c4;
#pragma unroll
        for (int k = 0; k < kCMaxSplits; ++k)
          if (k < S)
            v[h][k] = __ldcg(reinterpret_cast<const float4*>(src + k * slice));
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = e0 + h * kCThreads;
        if (e >= n4) break;
        float4 acc = v[h][0];
#pragma unroll
        for (int k = 1; k < kCMaxSplits; ++k)
          if (k < S) {
            acc.x += v[h][k].x; acc.y += v[h][k].y; acc.z += v[h][k].z; acc.w += v[h][k].w;
          }
        const int orow = div_np4(e), c4 = e - orow * int(np4);
        *reinterpret_cast<float4*>(corr + size_t(orow) * pitch + 4 * c4) = acc;
      }
    }
    __syncthreads();
  }
  // ---- the 2-tap mix: item = (group, 8 channels, run of kPRun positions) ----
  const int np = min(Np, a.R - p0);
  const int ncolumn = 2 * og;
  const int items = ncolumn * ((np + kPRun - 1) / kPRun);
  for (int item = tid; item < items; item += kCThreads) {
    const int col = item & (ncolumn - 1), i0 = (item >> (ogs + 1)) * kPRun;
    const int gl = col >> 1, h = col & 1, g = gown + gl;
    if (g >= a.G) continue;
    const int ch0 = 16 * g + 8 * h;
    const int pf = p0 + i0;  // the run's first position
    uint4 cur[kPRun];
#pragma unroll
    for (int u = 0; u < kPRun; ++u)
      if (i0 + u < np)
        cur[u] = *reinterpret_cast<const uint4*>(a.x + size_t(pf + u) * a.d + ch0);
    int tl = pf % a.L, bq = pf / a.L;  // position in its sequence, and the sequence
    uint4 prev = *reinterpret_cast<const uint4*>(
        (tl == 0 ? a.x_prev + size_t(bq) * a.d : a.x + size_t(pf - 1) * a.d) + ch0);
    float b0[8], b1[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      b0[j] = bslice[16 * gl + 8 * h + j];
      b1[j] = bslice[16 * og + 16 * gl + 8 * h + j];
    }
    const float* c0p = corr + size_t(gl) * pitch + i0;
    const float* c1p = corr + size_t(og + gl) * pitch + i0;
#pragma unroll
    for (int u = 0; u < kPRun; ++u) {
      if (i0 + u >= np) break;
      const int pp = pf + u;
      if (u > 0 && ++tl == a.L) {  // a sequence starts inside the run
        tl = 0;
        ++bq;
        prev = *reinterpret_cast<const uint4*>(a.x_prev + size_t(bq) * a.d + ch0);
      }
      const float c0 = c0p[u], c1 = c1p[u];
      float xt[8], xm[8];
      bf8_unpack(cur[u], xt);
      bf8_unpack(prev, xm);
      uint32_t ow[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float lo = fmaf(b0[2 * q] + c0, xt[2 * q], (b1[2 * q] + c1) * xm[2 * q]);
        const float hi =
            fmaf(b0[2 * q + 1] + c0, xt[2 * q + 1], (b1[2 * q + 1] + c1) * xm[2 * q + 1]);
        const __nv_bfloat162 pr = __floats2bfloat162_rn(lo, hi);
        ow[q] = *reinterpret_cast<const uint32_t*>(&pr);
      }
      *reinterpret_cast<uint4*>(a.y + size_t(pp) * a.d + ch0) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
      prev = cur[u];
    }
  }
}

bool g_conv_ptile_attr[64];

// Tile width and split for the position-tiled kernel: tiles of 256 positions
// (one CTA per SM) or 128 (two per SM), each with the largest power-of-two
// cluster (<= 8) whose CTAs all fit on the SMs at once; of the two, the one
// whose busiest SM moves the fewest bytes (operand ring, its partial tile out
// and the other splits' slices of its rows back, the mix).  (Tiles of 224
// positions, 120 CTAs at 1,024 positions x d = 2560, measured 14.9 us per
// call against 13.9 for 256, and 128-position tiles in clusters of 4 14.6:
// the partial stores slow down with more writers.  The runtime's count of
// resident clusters of 8 at this shared-memory size is below the 12 that were
// measured to start together, so it is not used.)
// The kernel runs only with a split (splits > 1); otherwise conv_tc_kernel runs.
struct PtilePlan {
  int Np, splits, kps, stages, tiles;
  size_t smem, ws_bytes;
  long long cost;
};
PtilePlan ptile_plan(int R, int G, int kblocks, int sms) {
  PtilePlan best{};
  best.cost = -1;
  for (const int want : {256, 128}) {
    const int Np = std::min(want, (R + 15) / 16 * 16);
    const int stages = Np > 128 ? kPMaxStages : 3;
    const size_t smem = ptile_smem_bytes(Np, stages);
    const long long slots = (long long)sms * (smem <= size_t(113) * 1024 ? 2 : 1);
    const long long tiles = (long long)((R + Np - 1) / Np) * ((G + kPGroups - 1) / kPGroups);
    int S = 1;
    while (S * 2 <= kCMaxSplits && tiles * S * 2 <= slots && S * 2 <= kblocks) S *= 2;
    int kps = (kblocks + S - 1) / S;
    while (S > 1 && (S - 1) * kps >= kblocks) {  // keep every split non-empty
      S >>= 1;
      kps = (kblocks + S - 1) / S;
    }
    const long long busiest = (tiles * S + sms - 1) / sms;
    const long long per_cta = (long long)kps * ptile_stage_bytes(Np) +
                              2LL * (S - 1) * (2 * kPGroups / S) * Np * 4 +
                              (long long)(kPGroups / S) * 16 * Np * 4;
    const long long cost = busiest * per_cta;
    if (tiles * S <= slots && (best.cost < 0 || cost < best.cost))
      best = PtilePlan{Np, S, kps, stages, static_cast<int>(tiles), smem,
                       ptile_ws_bytes(tiles, S, Np), cost};
  }
  return best;
}
// Measured (20 chained calls): at 1,024 positions x d = 2560 the split kernel
// (256-position tiles) took 13.9 us per call against 17.4 for conv_tc_kernel;
// at 128 positions (24 CTAs) 10.6 against 8.4.  So it runs only when its CTAs
// fill half the GPU in one wave of clusters.
bool use_ptile(int R, int d, const PtilePlan& pl, int sms) {
  return R > kSMaxRows && d % kCBK == 0 && d / kGroup >= kPGroups / 2 && pl.splits > 1 &&
         2LL * pl.tiles * pl.splits >= sms;
}

// ============================================================================
// At most 16 positions (batch 1): K split over a cluster, groups mixed per CTA.
// ============================================================================
// A cluster of C CTAs owns NG = C * MG consecutive correction groups, whose
// 2 NG W_c rows (tap 0 then tap 1) form the N of a warp-level MMA.  CTA `rank`
// holds the K slice [rank*d/C, (rank+1)*d/C) of those rows and of every
// position of x; it forms the R x 2NG partial corrections with m16n8k16 bf16
// MMAs (positions as M, float32 accumulators, each warp a share of the K
// steps), adds the warps' partials and sends each group's rows to the CTA that
// mixes the group with st.async, which counts the bytes on the receiver's
// mbarrier: no cluster-wide barrier at the end.  The receiver sums the C
// slices in rank order (deterministic) and applies the 2-tap mix to its MG
// groups.  The contraction is 2 NG x R x d per cluster, far below a tcgen05
// tile, and the call is latency-bound, so the warp-level MMA is the cheaper
// instrument here.
//
// Latency: the kernel lets the next launch on the stream start at once, and
// before waiting on the previous launch it copies its W_c slice into shared
// memory and reads its base slice: these are weights, which no kernel still
// pending on the stream writes (the documented contract of the conv entry
// points), so the copy overlaps the previous kernel.  After the wait only x is
// read: each warp copies just the 16-byte pieces of x its own K steps use
// (cp.async), so no CTA-wide barrier sits between the wait and the MMAs; the
// mixing threads load their x_t and x_{t-1} at the same time.
constexpr int kGvThreads = 256;  // 8 warps
// x pieces (16 bytes) of a lane whose addresses are computed before the
// dependency wait: 16 rows x 2 pieces per K step x up to 6 K steps per warp,
// over 32 lanes (K slices of up to 6 x 8 x 16 = 768: d <= 6144 with clusters of
// 8); a lane with more pieces computes the rest after the wait
constexpr int kGvMaxPieces = 6;
__device__ __forceinline__ void cp_async16_s(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
constexpr int kGvWarps = kGvThreads / 32;
constexpr int kGvMaxR = 16;      // positions = the MMA's 16 rows
constexpr size_t kGvSmemMax = 200 * 1024;

struct ConvGemvArgs {
  const __nv_bfloat16* x;       // [R, d]
  const __nv_bfloat16* x_prev;  // [B, d]
  const float* base;            // [2, d]
  const __nv_bfloat16* W_c;     // [2G, d]
  __nv_bfloat16* y;             // [R, d]
  int R, L, d, G;
  uint32_t* err;
};

// Row pitch in bytes of the x and W_c slices: 16 more than the slice, so that
// pitch / 16 is odd and the eight rows of an ldmatrix fall in distinct banks.
__host__ __device__ constexpr int gemv_pitch(int d, int C) { return 2 * (d / C) + 16; }
__host__ __device__ constexpr int gemv_rows(int C, int MG) { return 2 * C * MG; }
// [16 x rows | max(NR, 8) W_c rows] [warp partials 8 x 16 x NR f32]
// [receive C x 2 x MG x 16 f32] [2 mbarriers]
__host__ __device__ constexpr size_t gemv_smem_bytes(int d, int C, int MG) {
  return size_t(16 + (gemv_rows(C, MG) < 8 ? 8 : gemv_rows(C, MG))) * gemv_pitch(d, C) +
         size_t(kGvWarps) * 16 * gemv_rows(C, MG) * 4 + size_t(C) * 2 * MG * 16 * 4 + 32;
}

// 16-byte store into CTA `rank`'s shared memory, counted as transaction bytes
// on that CTA's mbarrier at the same offset as `bar`.
__device__ __forceinline__ void st_async_v4(const void* local, uint32_t rank, float4 v,
                                            const uint64_t* bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, "
      "[%5];" ::"r"(dsmem_addr(local, rank)),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(dsmem_addr(bar, rank))
      : "memory");
}
__device__ __forceinline__ void bf8_to_f32(const uint4 v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    f[2 * q] = __uint_as_float(w[q] << 16);
    f[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
  }
}

template <int C, int MG>
__global__ void __launch_bounds__(kGvThreads) conv_gemv_kernel(const ConvGemvArgs a) {
  constexpr int NG = C * MG;           // groups of the cluster
  constexpr int NR = 2 * NG;           // their W_c rows: row n = tap * NG + group
  constexpr int NT = (NR + 7) / 8;     // n8 tiles of the MMA
  constexpr int NRS = NT * 8;          // W_c rows staged (rows past NR repeat row 0)
  static_assert(NR <= 32, "the W_c rows are loaded by one warp");
  extern __shared__ __align__(128) uint8_t gsm[];
  const int d = a.d, ks = d / C, pitch = gemv_pitch(d, C), R = a.R;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = C > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int gc0 = (blockIdx.x / C) * NG;  // first group of the cluster
  const int k0 = rank * ks;
  uint8_t* xs = gsm;                                                // [16][pitch]
  uint8_t* wsm = gsm + size_t(16) * pitch;                          // [NRS][pitch]
  float* red = reinterpret_cast<float*>(wsm + size_t(NRS) * pitch);  // [8][16][NR]
  float* recv = red + kGvWarps * 16 * NR;                           // [C][2][MG][16]
  uint64_t* bar = reinterpret_cast<uint64_t*>(recv + C * 2 * MG * 16);  // [0] W_c, [1] receive
  const int nq = (R + 3) / 4;  // four-position pieces sent per W_c row

  pdl_launch_dependents();
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar[0], uint32_t(NR) * uint32_t(ks) * 2u);
    // every CTA of the cluster (this one included) sends 2 MG rows of nq pieces here
    if (C > 1) mbar_arrive_expect_tx(&bar[1], uint32_t(C * 2 * MG * nq * 16));
  }
  __syncthreads();  // the barriers are initialised before any copy completes on them
  // ---- before the dependency wait: weights only ----
  if (warp == 0 && lane < NR) {
    const int tap = lane / NG, gi = lane % NG;
    const int g = gc0 + gi < a.G ? gc0 + gi : 0;  // a missing group reads a real row (never stored)
    bulk_g2s(wsm + size_t(lane) * pitch, a.W_c + (size_t(tap) * a.G + g) * d + k0,
             uint32_t(ks) * 2u, &bar[0]);
  } else if (warp == 1 && lane < R) {
    // x may still be being written: an L2 prefetch is coherent with those writes
    prefetch_l2(a.x + size_t(lane) * d + k0, uint32_t(ks) * 2u);
  }
  // mixing threads: (group m of this CTA, position p, half of the 16 channels)
  const int m_mix = tid / (2 * R), p_mix = (tid % (2 * R)) >> 1, h_mix = tid & 1;
  const int gmix = gc0 + rank * MG + m_mix;
  const bool mixer = tid < 2 * R * MG && gmix < a.G;
  const int cmix = 16 * gmix + 8 * h_mix;
  float4 b0[2], b1[2];
  if (mixer) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      b0[h] = __ldg(reinterpret_cast<const float4*>(a.base + cmix) + h);
      b1[h] = __ldg(reinterpret_cast<const float4*>(a.base + d + cmix) + h);
    }
  }
  // The addresses the steps after the wait use, computed before it (integer
  // divisions among them): the mix's x_t and x_{t-1} rows, and this lane's
  // first kGvMaxPieces pieces of the warp's K steps of every x row.
  const uint4* xt_src = nullptr;
  const uint4* xm_src = nullptr;
  if (mixer) {
    const int t = p_mix % a.L;
    xt_src = reinterpret_cast<const uint4*>(a.x + size_t(p_mix) * d + cmix);
    xm_src = reinterpret_cast<const uint4*>(
        (t > 0 ? a.x + size_t(p_mix - 1) * d : a.x_prev + size_t(p_mix / a.L) * d) + cmix);
  }
  const int steps = ks / 16;
  const int s0 = warp * steps / kGvWarps, s1 = (warp + 1) * steps / kGvWarps;
  const int per_row = (s1 - s0) * 2;  // 16-byte pieces of one x row
  int npieces = 0;
  uint32_t piece_dst[kGvMaxPieces];
  const __nv_bfloat16* piece_src[kGvMaxPieces];
#pragma unroll
  for (int q = 0; q < kGvMaxPieces; ++q) {
    const int e = lane + 32 * q;
    piece_dst[q] = 0u;
    piece_src[q] = a.x;
    if (e < R * per_row) {
      const int p = e / per_row, c = s0 * 16 + (e % per_row) * 8;
      piece_dst[q] = smem_u32(xs + size_t(p) * pitch + 2 * c);
      piece_src[q] = a.x + size_t(p) * d + k0 + c;
      npieces = q + 1;
    }
  }
  if constexpr (C > 1) cluster_arrive_release();  // barrier inits visible to the peers
  pdl_wait();

  // ---- the mix's operands, in flight during the MMAs ----
  uint4 xt = make_uint4(0u, 0u, 0u, 0u), xm = xt;
  if (mixer) {
    xt = __ldcg(xt_src);
    xm = __ldcg(xm_src);
  }
  // ---- partial corrections: this warp's K steps of x_slice (16 x K) * W_slice^T ----
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  if (s0 < s1) {
#pragma unroll
    for (int q = 0; q < kGvMaxPieces; ++q)
      if (q < npieces) cp_async16_s(piece_dst[q], piece_src[q]);
    for (int e = lane + 32 * kGvMaxPieces; e < R * per_row; e += 32) {  // wide K slices only
      const int p = e / per_row, c = s0 * 16 + (e % per_row) * 8;
      cp_async16(xs + size_t(p) * pitch + 2 * c, a.x + size_t(p) * d + k0 + c, true);
    }
    cp_async_commit();
    const int arow = lane & 15, acol = (lane >> 4) * 8;
    const int rb = lane & 7, bcol = ((lane >> 3) & 1) * 8;
    // rows past R read row 0: their products land in entries that are never sent
    const uint32_t abase = smem_u32(xs + size_t(arow < R ? arow : 0) * pitch + 2 * acol);
    if (!mbar_wait(&bar[0], 0, a.err)) record_error(a.err, kDevErrConv);
    cp_async_wait<0>();
    __syncwarp();
#pragma unroll 1
    for (int k = s0; k < s1; ++k) {
      uint32_t af[4];
      ldsm_x4(abase + 32u * k, af);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int n = nt * 8 + rb;
        uint32_t bfr[2];
        ldsm_x2(smem_u32(wsm + size_t(n < NR ? n : 0) * pitch + 2 * bcol) + 32u * k, bfr);
        mma_16816_bf16(acc[nt], af, bfr);
      }
    }
  }
  {
    // acc[nt]: (position g, rows nt*8 + 2t, +1), (position g + 8, the same rows)
    const int g = lane >> 2, t = lane & 3;
    float* rw = red + warp * 16 * NR;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int n = nt * 8 + 2 * t;
      if (n < NR) {
        *reinterpret_cast<float2*>(rw + g * NR + n) = make_float2(acc[nt][0], acc[nt][1]);
        *reinterpret_cast<float2*>(rw + (g + 8) * NR + n) = make_float2(acc[nt][2], acc[nt][3]);
      }
    }
  }
  if constexpr (C > 1) cluster_wait_acquire();  // the peers' barriers are initialised
  __syncthreads();
  // ---- warp partials summed (warp order); four positions of row n sent to the
  // CTA that mixes group gc0 + n % NG ----
  if (tid < nq * NR) {
    const int n = tid % NR, q = tid / NR;
    float v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kGvWarps; ++w) s += red[(w * 16 + 4 * q + k) * NR + n];
      v[k] = s;
    }
    const int tap = n / NG, gi = n % NG;
    float* slot = recv + ((rank * 2 + tap) * MG + gi % MG) * 16 + 4 * q;
    const float4 val = make_float4(v[0], v[1], v[2], v[3]);
    if constexpr (C > 1)
      st_async_v4(slot, static_cast<uint32_t>(gi / MG), val, &bar[1]);
    else
      *reinterpret_cast<float4*>(slot) = val;
  }
  if constexpr (C == 1) {
    __syncthreads();
  } else {
    // every CTA waits for its whole receive before it may exit (peers store into it)
    if ((tid == 0 || mixer) && !mbar_wait_cluster(&bar[1], 0, a.err))
      record_error(a.err, kDevErrConv);
  }
  if (!mixer) return;
  // ---- the 2-tap mix of 8 channels at position p ----
  float c0 = 0.f, c1 = 0.f;
#pragma unroll
  for (int k = 0; k < C; ++k) {  // rank order: deterministic
    c0 += recv[((k * 2 + 0) * MG + m_mix) * 16 + p_mix];
    c1 += recv[((k * 2 + 1) * MG + m_mix) * 16 + p_mix];
  }
  float ft[8], fm[8];
  bf8_to_f32(xt, ft);
  bf8_to_f32(xm, fm);
  const float k0v[8] = {b0[0].x, b0[0].y, b0[0].z, b0[0].w, b0[1].x, b0[1].y, b0[1].z, b0[1].w};
  const float k1v[8] = {b1[0].x, b1[0].y, b1[0].z, b1[0].w, b1[1].x, b1[1].y, b1[1].z, b1[1].w};
  uint32_t ow[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float lo = fmaf(k0v[2 * q] + c0, ft[2 * q], (k1v[2 * q] + c1) * fm[2 * q]);
    const float hi =
        fmaf(k0v[2 * q + 1] + c0, ft[2 * q + 1], (k1v[2 * q + 1] + c1) * fm[2 * q + 1]);
    const __nv_bfloat162 pr = __floats2bfloat162_rn(lo, hi);
    ow[q] = *reinterpret_cast<const uint32_t*>(&pr);
  }
  *reinterpret_cast<uint4*>(a.y + size_t(p_mix) * d + cmix) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
}

// (C, MG) instantiations and their attribute flags.
constexpr int kGvShapes = 5;  // (1,1) (2,1) (4,1) (8,1) (16,1)
bool g_conv_gemv_attr[64][kGvShapes];

// Cluster size of the GEMV kernel: the largest of 8, 4, 2, 1 whose slices fit
// the shared-memory budget and whose K slice is still at least 64 long (each
// CTA reads its slice of every position of x after the wait, so a larger
// cluster cuts the bytes each SM waits for); 0 if none fits.
int gemv_cluster(int d, int G) {
  auto fits = [&](int C) {
    return d % (16 * C) == 0 && G >= C && gemv_smem_bytes(d, C, 1) <= kGvSmemMax;
  };
#ifdef DFL2_GEMV_C
  if (fits(DFL2_GEMV_C)) return DFL2_GEMV_C;
#endif
  for (int C = 8; C >= 1; C >>= 1)
    if (fits(C) && (C == 1 || d / C >= 64)) return C;
  return 0;
}

template <int C>
cudaError_t launch_gemv_c(const ConvGemvArgs& a, cudaStream_t s, int dev) {
  auto k = conv_gemv_kernel<C, 1>;
  constexpr int ci = C == 1 ? 0 : (C == 2 ? 1 : (C == 4 ? 2 : (C == 8 ? 3 : 4)));
  if (!g_conv_gemv_attr[dev & 63][ci]) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kGvSmemMax));
    if (e != cudaSuccess) return e;
    if (C > 8) {  // clusters of 16 are outside the portable size
      e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    g_conv_gemv_attr[dev & 63][ci] = true;
  }
  const int grid = (a.G + C - 1) / C * C;
  return launch_kc(k, dim3(grid), dim3(kGvThreads), gemv_smem_bytes(a.d, C, 1), s, true, C, a);
}

}  // namespace

size_t conv2_ws_bytes(int B, int L, int d) {
  const int R = B * L;
  const int sms = device_info().sms;
  const PtilePlan pl = ptile_plan(R, d / kGroup, d / kCBK, sms);
  return use_ptile(R, d, pl, sms) ? pl.ws_bytes : 0;
}

cudaError_t launch_conv2(const __nv_bfloat16* x, const __nv_bfloat16* x_prev, const float* base,
                         const __nv_bfloat16* W_c, int B, int L, int d, __nv_bfloat16* y,
                         void* ws, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!g_conv_attr[dev & 63]) {
    e = cudaFuncSetAttribute(conv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kCSmemMax));
    if (e != cudaSuccess) return e;
    g_conv_attr[dev & 63] = true;
  }
  const int sms = device_info().sms;
  const int R = B * L;
  const int gv_c = R <= kGvMaxR ? gemv_cluster(d, d / kGroup) : 0;
  if (gv_c > 0) {
    // ---- at most 16 positions: the GEMV kernel, one group per CTA ----
    const ConvGemvArgs g{x, x_prev, base, W_c, y, R, L, d, d / kGroup, device_error_word()};
    switch (gv_c) {
      case 16: return launch_gemv_c<16>(g, s, dev);
      case 8: return launch_gemv_c<8>(g, s, dev);
      case 4: return launch_gemv_c<4>(g, s, dev);
      case 2: return launch_gemv_c<2>(g, s, dev);
      default: return launch_gemv_c<1>(g, s, dev);
    }
  }
  if (R <= kSMaxRows && d % kCBK == 0 && d / kGroup >= kSGroups / 2) {
    // ---- few positions: the transposed kernel ----
    if (!g_conv_small_attr[dev & 63]) {
      e = cudaFuncSetAttribute(conv_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(small_smem_bytes(kSMaxRows, 1)));
      if (e != cudaSuccess) return e;
      g_conv_small_attr[dev & 63] = true;
    }
    ConvSmallArgs c{};
    c.x = x;
    c.x_prev = x_prev;
    c.base = base;
    c.y = y;
    c.R = R;
    c.L = L;
    c.d = d;
    c.G = d / kGroup;
    c.Npad = (R + 15) / 16 * 16;
    c.kblocks = d / kCBK;
    c.err = device_error_word();
    const int tiles = (c.G + kSGroups - 1) / kSGroups;
    int want = 1;
    while (want * 2 <= kCMaxSplits && tiles * want * 2 <= sms && want * 2 <= c.kblocks) want *= 2;
    c.splits = want;  // a power of two: it divides the 64 groups of a tile
    c.kps = (c.kblocks + want - 1) / want;
    if ((c.splits - 1) * c.kps >= c.kblocks) {  // keep every split non-empty
      while (c.splits > 1 && (c.splits - 1) * c.kps >= c.kblocks) c.splits >>= 1;
      c.kps = (c.kblocks + c.splits - 1) / c.splits;
    }
    alignas(64) CUtensorMap tmW;
    if (!tensor_map_bf16(W_c, uint64_t(2) * c.G, uint64_t(d), kSGroups, &tmW))
      return cudaErrorInvalidValue;
    return launch_kc(conv_small_kernel, dim3(tiles * c.splits), dim3(kCThreads),
                     small_smem_bytes(c.Npad, c.splits), s, true, c.splits, c, tmW);
  }
  const PtilePlan pl = ws ? ptile_plan(R, d / kGroup, d / kCBK, sms) : PtilePlan{};
  if (ws && use_ptile(R, d, pl, sms)) {
    // ---- many positions: position tiles x 64 groups, K split over a cluster ----
    if (!g_conv_ptile_attr[dev & 63]) {
      e = cudaFuncSetAttribute(conv_ptile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kCSmemMax));
      if (e != cudaSuccess) return e;
      g_conv_ptile_attr[dev & 63] = true;
    }
    ConvPtileArgs c{};
    c.x = x;
    c.x_prev = x_prev;
    c.base = base;
    c.y = y;
    c.R = R;
    c.L = L;
    c.d = d;
    c.G = d / kGroup;
    c.kblocks = d / kCBK;
    c.ws = static_cast<float*>(ws);
    c.Np = pl.Np;
    c.gtiles = (c.G + kPGroups - 1) / kPGroups;
    c.splits = pl.splits;
    c.kps = pl.kps;
    c.stages = pl.stages;
    c.err = device_error_word();
    const int tiles = pl.tiles;
    alignas(64) CUtensorMap tmW, tmX;
    if (!tensor_map_bf16(W_c, uint64_t(2) * c.G, uint64_t(d), kPGroups, &tmW) ||
        !tensor_map_bf16(x, uint64_t(R), uint64_t(d), static_cast<uint32_t>(c.Np), &tmX))
      return cudaErrorInvalidValue;
    return launch_kc(conv_ptile_kernel, dim3(tiles * c.splits), dim3(kCThreads), pl.smem, s, true,
                     c.splits, c, tmW, tmX);
  }
  ConvArgs a{};
  a.x = x;
  a.x_prev = x_prev;
  a.base = base;
  a.y = y;
  a.R = B * L;
  a.L = L;
  a.d = d;
  a.G = d / kGroup;
  a.kblocks = (d + kCBK - 1) / kCBK;
  a.err = device_error_word();
  const int mtiles = (a.R + kCBM - 1) / kCBM;
  // Widest group slice that still gives a full wave of tiles; otherwise the
  // narrowest slice, with K split over a cluster until the GPU is covered.
  int NG = kCMaxNG;
  while (NG > 16 && (long long)mtiles * ((a.G + NG - 1) / NG) < sms) NG >>= 1;
  a.NG = NG;
  a.ntiles = (a.G + NG - 1) / NG;
  const int tiles = mtiles * a.ntiles;
  int want = 1;
  while (want * 2 <= kCMaxSplits && tiles * want * 2 <= sms) want *= 2;
  want = std::min(want, a.kblocks);
  a.kps = (a.kblocks + want - 1) / want;
  a.splits = (a.kblocks + a.kps - 1) / a.kps;  // every split gets at least one K block
  if (a.splits > 1 && NG != 16) return cudaErrorInvalidConfiguration;  // receive slots need NG 16
  // One CTA per SM without split K: the x tiles of the CTA's own channels stay
  // in shared memory for the mix (at most 4 K blocks, 64 KB).
  a.side = 0;
  if (a.splits == 1 && (long long)tiles <= sms && (16 * NG) % kCBK == 0 && 16 * NG / kCBK <= 4 &&
      a.d % kCBK == 0 && L >= NG)  // L >= the mix's run of rows (NG)
    a.side = 16 * NG / kCBK;
  // As many operand stages as the shared memory of one CTA per SM holds, or of
  // two when the tiles outnumber the SMs; never more than the K blocks.
  const size_t budget = (long long)tiles * a.splits > sms ? size_t(112) * 1024 : kCSmemMax;
  const size_t fixed = conv_smem_bytes(NG, 0, a.splits, a.side) - conv_stage_area(NG, 0);
  const size_t per_stage = size_t(kCAStage) + conv_bstage_bytes(NG);
  int stages = budget > fixed ? static_cast<int>((budget - fixed) / per_stage) : 2;
  stages = std::max(2, std::min({stages, kCMaxStages, std::max(a.kps, 2)}));
  a.stages = stages;
  alignas(64) CUtensorMap tmX, tmW;
  if (!tensor_map_bf16(x, uint64_t(a.R), uint64_t(d), kCBM, &tmX) ||
      !tensor_map_bf16(W_c, uint64_t(2) * a.G, uint64_t(d), static_cast<uint32_t>(NG), &tmW))
    return cudaErrorInvalidValue;
  return launch_kc(conv_tc_kernel, dim3(tiles * a.splits), dim3(kCThreads),
                   conv_smem_bytes(NG, stages, a.splits, a.side), s, true, a.splits, a, tmX,
                   tmW);
}

}  // namespace dfl2
