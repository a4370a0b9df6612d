// Two-tap dynamic depthwise conv ("DFlash 2: Keep Drafting Parallel",
// 方法细节 > 轻量级局部卷积, the Conv_k equation):
//   y_t = k_{t,0} ⊙ x_t + k_{t,1} ⊙ x_{t-1},  x_{-1} = the verified token's representation,
//   k_{t,j,c} = base[j,c] + corr[t,j,c/16],   corr[t,j,g] = sum_c W_c[j*G+g, c] x_t[c].
//
// One CTA owns NG correction groups (2*NG rows of W_c: both taps) for a tile
// of TL positions of one sequence.  It stages x_{t0-1..t0+TL-1} in shared
// memory, streams its W_c rows once, forms the corrections with fp32 FMAs and
// writes y for the NG*16 channels it owns: correction and mixing are fused,
// so the corrections never reach HBM.
#include "dfl2_internal.cuh"

namespace dfl2 {
namespace {

constexpr int kConvThreads = 256;
constexpr int kConvWarps = kConvThreads / 32;
constexpr int kMaxTL = 16;
constexpr int kMaxNG = 8;
constexpr size_t kConvXBudget = 96 * 1024;  // bytes of staged x per CTA

struct ConvArgs {
  const __nv_bfloat16* x;
  const __nv_bfloat16* x_prev;
  const float* base;
  const __nv_bfloat16* W_c;
  __nv_bfloat16* y;
  int L, d, G;
  int TL, NG;
  uint32_t* err;
};

__device__ __forceinline__ float dot8(const uint4& w, const uint4& x) {
  const uint32_t wr[4] = {w.x, w.y, w.z, w.w}, xr[4] = {x.x, x.y, x.z, x.w};
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    s = fmaf(__uint_as_float(wr[e] << 16), __uint_as_float(xr[e] << 16), s);
    s = fmaf(__uint_as_float(wr[e] & 0xFFFF0000u), __uint_as_float(xr[e] & 0xFFFF0000u), s);
  }
  return s;
}

__global__ void __launch_bounds__(kConvThreads) conv2_fma_kernel(ConvArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int d = a.d, G = a.G, TL = a.TL, NG = a.NG;
  const int g0 = blockIdx.x * NG, t0 = blockIdx.y * TL, b = blockIdx.z;
  const int tl = min(TL, a.L - t0);  // positions in this tile
  const int ng = min(NG, G - g0);    // groups in this CTA
  const int rows = 2 * NG;           // W_c rows (both taps), some unused when ng < NG
  // layout: xs [(TL+1) rows][d] bf16 | red [kConvWarps][rows][TL] f32 | corr [rows][TL] f32 | bar
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem);
  float* red = reinterpret_cast<float*>(smem + size_t(TL + 1) * d * 2);
  float* corr = red + kConvWarps * rows * TL;
  uint64_t* bar = reinterpret_cast<uint64_t*>(corr + rows * TL);

  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  // Stage x_{t0-1} (x_prev at t0 == 0) and x_{t0..t0+tl-1} with bulk copies:
  // the rows are contiguous in x, apart from x_prev.
  const int vec_per_row = d / 8;
  if (threadIdx.x == 0) {
    const uint32_t row_bytes = static_cast<uint32_t>(d) * 2;
    mbar_arrive_expect_tx(bar, row_bytes * (tl + 1));
    if (t0 == 0) {
      bulk_g2s(xs, a.x_prev + size_t(b) * d, row_bytes, bar);
      bulk_g2s(xs + d, a.x + size_t(b) * a.L * d, row_bytes * tl, bar);
    } else {
      bulk_g2s(xs, a.x + (size_t(b) * a.L + t0 - 1) * d, row_bytes * (tl + 1), bar);
    }
  }
  if (!mbar_wait(bar, 0)) record_error(a.err, kDevErrConv);

  // Corrections: warps split the rows; with fewer rows than warps they also split K.
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // rows >= 8: warp w owns rows w, w+8, ... over all of K.
  // rows <  8: warp w owns row w % rows over K part w / rows (ksplit parts).
  const int ksplit = rows >= kConvWarps ? 1 : kConvWarps / rows;
  const int kpart = ksplit == 1 ? 0 : warp / rows;
  const int kchunk = (vec_per_row + ksplit - 1) / ksplit;
  for (int lr = (ksplit == 1 ? warp : warp % rows); lr < rows;
       lr += (ksplit == 1 ? kConvWarps : rows)) {
    const int tap = lr / NG, gl = lr % NG;
    float acc[kMaxTL];
#pragma unroll
    for (int tt = 0; tt < kMaxTL; ++tt) acc[tt] = 0.f;
    if (gl < ng) {
      const uint4* wrow = reinterpret_cast<const uint4*>(a.W_c + (size_t(tap) * G + g0 + gl) * d);
      const int v_lo = kpart * kchunk;
      const int v_hi = min(vec_per_row, v_lo + kchunk);
#pragma unroll 4
      for (int v = v_lo + lane; v < v_hi; v += 32) {
        const uint4 w = __ldg(wrow + v);
#pragma unroll
        for (int tt = 0; tt < kMaxTL; ++tt)
          if (tt < tl)
            acc[tt] += dot8(w, reinterpret_cast<const uint4*>(xs + size_t(tt + 1) * d)[v]);
      }
    }
#pragma unroll
    for (int tt = 0; tt < kMaxTL; ++tt) {
      float v = acc[tt];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0 && tt < TL) red[(size_t(kpart) * rows + lr) * TL + tt] = v;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < rows * TL; e += kConvThreads) {
    float s = 0.f;
    for (int k = 0; k < ksplit; ++k) s += red[size_t(k) * rows * TL + e];
    corr[e] = s;
  }
  __syncthreads();
  pdl_launch_dependents();

  // y for the ng*16 channels of this CTA.
  const int nch = ng * kGroup;
  for (int e = threadIdx.x; e < tl * nch; e += kConvThreads) {
    const int tt = e / nch, cl = e % nch;
    const int c = g0 * kGroup + cl, gl = cl / kGroup;
    const float k0 = a.base[c] + corr[size_t(gl) * TL + tt];
    const float k1 = a.base[d + c] + corr[size_t(NG + gl) * TL + tt];
    const float xt = __bfloat162float(xs[size_t(tt + 1) * d + c]);
    const float xm1 = __bfloat162float(xs[size_t(tt) * d + c]);
    const float v = fmaf(k0, xt, k1 * xm1);
    a.y[(size_t(b) * a.L + t0 + tt) * d + c] = __float2bfloat16_rn(v);
  }
}

size_t conv_smem_bytes(int TL, int NG, int d) {
  return size_t(TL + 1) * d * 2 + size_t(kConvWarps + 1) * 2 * NG * TL * sizeof(float) + 16;
}

bool g_conv_attr_set[64];

}  // namespace

cudaError_t launch_conv2(const __nv_bfloat16* x, const __nv_bfloat16* x_prev, const float* base,
                         const __nv_bfloat16* W_c, int B, int L, int d, __nv_bfloat16* y,
                         cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!g_conv_attr_set[dev & 63]) {
    e = cudaFuncSetAttribute(conv2_fma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             200 * 1024);
    if (e != cudaSuccess) return e;
    g_conv_attr_set[dev & 63] = true;
  }
  const int G = d / kGroup;
  int TL = static_cast<int>(kConvXBudget / (size_t(d) * 2)) - 1;
  TL = max(1, min(TL, min(L, kMaxTL)));
  const int tiles = (L + TL - 1) / TL;
  const int sms = device_info().sms;
  int NG = kMaxNG;
  while (NG > 1 && (long long)((G + NG - 1) / NG) * tiles * B < 2LL * sms) NG >>= 1;
  ConvArgs a{x, x_prev, base, W_c, y, L, d, G, TL, NG, device_error_word()};
  const dim3 grid((G + NG - 1) / NG, tiles, B);
  return launch_k(conv2_fma_kernel, grid, dim3(kConvThreads), conv_smem_bytes(TL, NG, d), s,
                  false, a);
}

}  // namespace dfl2
