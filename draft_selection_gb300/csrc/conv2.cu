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
// For few positions (R <= 64, batch 1) a transposed kernel computes
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
__host__ __device__ constexpr size_t conv_smem_bytes(int NG, int stages, int splits) {
  // [operand stages | corrections] [receive slots] [base slice] [barriers]
  return 1024 + conv_stage_area(NG, stages) + conv_recv_bytes(NG, splits) +
         size_t(2) * 16 * NG * 4 + 256;
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
  float* recv = reinterpret_cast<float*>(smem + conv_stage_area(NG, nst));  // [S][rows_per][pitch]
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
        if (it >= nst && !mbar_wait(&empty_bar[s], ph ^ 1)) record_error(a.err, kDevErrConv);
        const int k0 = (kb0 + it) * kCBK;
        mbar_arrive_expect_tx(&full_bar[s], tx);
        tma_load_2d(sA + size_t(s) * kCAStage, &tmX, k0, m0, &full_bar[s]);
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
        if (!mbar_wait(&full_bar[s], ph)) record_error(a.err, kDevErrConv);
        tc_fence_after();
        const uint64_t ad = umma_desc_sw128(sA + size_t(s) * kCAStage);
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
    if (!mbar_wait(accum_bar, 0)) record_error(a.err, kDevErrConv);
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
      if (it >= kSStages && !mbar_wait(&empty_bar[st], ((it / kSStages) - 1) & 1))
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
        if (!mbar_wait(&full_bar[st], (it / kSStages) & 1)) record_error(a.err, kDevErrConv);
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
    if (!mbar_wait(accum_bar, 0)) record_error(a.err, kDevErrConv);
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


}  // namespace

cudaError_t launch_conv2(const __nv_bfloat16* x, const __nv_bfloat16* x_prev, const float* base,
                         const __nv_bfloat16* W_c, int B, int L, int d, __nv_bfloat16* y,
                         cudaStream_t s) {
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
  // As many operand stages as the shared memory of one CTA per SM holds, or of
  // two when the tiles outnumber the SMs; never more than the K blocks.
  const size_t budget = (long long)tiles * a.splits > sms ? size_t(112) * 1024 : kCSmemMax;
  const size_t fixed = conv_smem_bytes(NG, 0, a.splits) - conv_stage_area(NG, 0);
  const size_t per_stage = size_t(kCAStage) + conv_bstage_bytes(NG);
  int stages = budget > fixed ? static_cast<int>((budget - fixed) / per_stage) : 2;
  stages = std::max(2, std::min({stages, kCMaxStages, std::max(a.kps, 2)}));
  a.stages = stages;
  alignas(64) CUtensorMap tmX, tmW;
  if (!tensor_map_bf16(x, uint64_t(a.R), uint64_t(d), kCBM, &tmX) ||
      !tensor_map_bf16(W_c, uint64_t(2) * a.G, uint64_t(d), static_cast<uint32_t>(NG), &tmW))
    return cudaErrorInvalidValue;
  return launch_kc(conv_tc_kernel, dim3(tiles * a.splits), dim3(kCThreads),
                   conv_smem_bytes(NG, stages, a.splits), s, true, a.splits, a, tmX, tmW);
}

}  // namespace dfl2
