// Pair scores of the path selector ("DFlash 2: Keep Drafting Parallel",
// 方法细节 > 轻量级路径选择器, the pair-score equation):
//   S_t(a,b) = U_t(b) + <A(a) ⊙ H(h_t), B(b)>,
//   A(a) = W_A E[a], B(b) = W_B E[b], H(h) = sigmoid(W_H h)  (W_* [256,d]).
//
// Two stages:
//   1. projections: every candidate row (the verified token, then 16 per
//      position) is gathered from E and multiplied by [W_A; W_B]^T into
//      P [M,512] fp32; the hidden states are multiplied by W_H^T and passed
//      through the sigmoid into H [B*L,256].
//   2. pair kernel: one CTA per (sequence, position) forms the 16x16 scores
//      from the previous position's A rows, the gate and this position's B rows.
#include "dfl2_internal.cuh"

namespace dfl2 {
namespace {

constexpr int kProjBM = 64, kProjBN = 64, kProjBK = 32;

struct ProjArgs {
  // A operand rows: gathered from `table` by token id (gather = 1), or the
  // consecutive rows of `table` (gather = 0).
  const __nv_bfloat16* table;
  int gather;
  const int32_t* cand_idx;  // [B,L,16]
  const int32_t* verified;  // [B]
  int L, V;
  int M, N, d;
  uint32_t* err;
  const __nv_bfloat16* W0;  // output columns 0..255
  const __nv_bfloat16* W1;  // output columns 256..511 (N == 512)
  float* out;               // [M, N]
  int sigmoid;
};

__device__ __forceinline__ const __nv_bfloat16* proj_row(const ProjArgs& a, int m) {
  if (!a.gather) return a.table + size_t(m) * a.d;
  const int per_seq = kCand * a.L + 1;
  const int b = m / per_seq, q = m % per_seq;
  const int32_t tok = q == 0 ? a.verified[b] : a.cand_idx[size_t(b) * a.L * kCand + (q - 1)];
  if (tok < 0 || tok >= a.V) {  // never read outside E: record it and use a zero row
    record_error(a.err, kDevErrBadIndex);
    return nullptr;
  }
  return a.table + size_t(tok) * a.d;
}

// Plain smem-tiled fp32-FMA GEMM: out[m,n] = sum_c row_m[c] * W(n)[c].
__global__ void __launch_bounds__(256) proj_fma_kernel(ProjArgs a) {
  __shared__ float As[kProjBK][kProjBM + 4];
  __shared__ float Bs[kProjBK][kProjBN + 4];
  pdl_wait();
  const int tid = threadIdx.x;
  const int m0 = blockIdx.x * kProjBM, n0 = blockIdx.y * kProjBN;
  const int ty = tid / 16, tx = tid % 16;
  const int lr = tid / 4, lc = (tid % 4) * 8;  // loader: row, 8-wide column chunk

  const int am = m0 + lr;
  const __nv_bfloat16* arow = am < a.M ? proj_row(a, am) : nullptr;
  const int bn = n0 + lr;
  const __nv_bfloat16* brow = nullptr;
  if (bn < a.N) brow = bn < kRank ? a.W0 + size_t(bn) * a.d : a.W1 + size_t(bn - kRank) * a.d;

  float acc[4][4] = {};
  for (int k0 = 0; k0 < a.d; k0 += kProjBK) {
    uint4 av = arow ? *reinterpret_cast<const uint4*>(arow + k0 + lc) : make_uint4(0, 0, 0, 0);
    uint4 bv = brow ? *reinterpret_cast<const uint4*>(brow + k0 + lc) : make_uint4(0, 0, 0, 0);
    const uint32_t ar[4] = {av.x, av.y, av.z, av.w}, br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      As[lc + 2 * e][lr] = __uint_as_float(ar[e] << 16);
      As[lc + 2 * e + 1][lr] = __uint_as_float(ar[e] & 0xFFFF0000u);
      Bs[lc + 2 * e][lr] = __uint_as_float(br[e] << 16);
      Bs[lc + 2 * e + 1][lr] = __uint_as_float(br[e] & 0xFFFF0000u);
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kProjBK; ++kk) {
      float av4[4], bv4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av4[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv4[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av4[i], bv4[j], acc[i][j]);
    }
    __syncthreads();
  }
  pdl_launch_dependents();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= a.N) continue;
      float v = acc[i][j];
      if (a.sigmoid) v = 1.0f / (1.0f + expf(-v));
      a.out[size_t(m) * a.N + n] = v;
    }
  }
}

struct PairArgs {
  const float* P;         // [B*(16L+1), 512]
  const float* H;         // [B*L, 256]
  const float* cand_val;  // [B,L,16]
  float* scores;          // [B,L,16,16]
  int L;
};

// One CTA per (sequence b, position t); thread (i, j) forms S_t(a_i, b_j).
__global__ void __launch_bounds__(256) pair16_kernel(PairArgs a) {
  __shared__ float Gs[kCand][kRank + 1];  // A(a_i) ⊙ H(h_t)
  __shared__ float Bsh[kCand][kRank + 1]; // B(b_j)
  __shared__ float U[kCand];
  pdl_wait();
  const int cell = blockIdx.x;
  const int b = cell / a.L, t = cell % a.L;
  const int per_seq = kCand * a.L + 1;
  const size_t seq0 = size_t(b) * per_seq;
  const int npred = t == 0 ? 1 : kCand;
  const float* Hrow = a.H + size_t(cell) * kRank;
  for (int e = threadIdx.x; e < kCand * kRank; e += blockDim.x) {
    const int i = e / kRank, q = e % kRank;
    if (i < npred) {
      const size_t prow = t == 0 ? seq0 : seq0 + 1 + size_t(kCand) * (t - 1) + i;
      Gs[i][q] = a.P[prow * (2 * kRank) + q] * Hrow[q];
    }
    Bsh[i][q] = a.P[(seq0 + 1 + size_t(kCand) * t + i) * (2 * kRank) + kRank + q];
  }
  if (threadIdx.x < kCand) U[threadIdx.x] = a.cand_val[size_t(cell) * kCand + threadIdx.x];
  __syncthreads();
  const int i = threadIdx.x / kCand, j = threadIdx.x % kCand;
  float s;
  if (i < npred) {
    s = 0.f;
#pragma unroll 8
    for (int q = 0; q < kRank; ++q) s = fmaf(Gs[i][q], Bsh[j][q], s);
    s += U[j];
  } else {
    s = -INFINITY;
  }
  pdl_launch_dependents();
  a.scores[size_t(cell) * kCand * kCand + threadIdx.x] = s;
}

}  // namespace

SelectPlan select_plan(int B, int L, int d) {
  SelectPlan p{};
  p.B = B;
  p.L = L;
  p.d = d;
  p.M = B * (kCand * L + 1);
  p.P_off = 256;
  p.H_off = align_up(p.P_off + size_t(p.M) * 2 * kRank * sizeof(float), 256);
  p.ws_bytes = align_up(p.H_off + size_t(B) * L * kRank * sizeof(float), 256);
  return p;
}

cudaError_t launch_select(const SelectPlan& p, const int32_t* cand_idx, const float* cand_val,
                          const int32_t* verified, const __nv_bfloat16* hidden,
                          const __nv_bfloat16* E, const __nv_bfloat16* W_A,
                          const __nv_bfloat16* W_B, const __nv_bfloat16* W_H, int V,
                          float* scores, void* ws, cudaStream_t s, bool pdl) {
  float* P = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + p.P_off);
  float* H = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + p.H_off);
  ProjArgs pa{};
  pa.table = E;
  pa.gather = 1;
  pa.cand_idx = cand_idx;
  pa.verified = verified;
  pa.L = p.L;
  pa.V = V;
  pa.err = device_error_word();
  pa.M = p.M;
  pa.N = 2 * kRank;
  pa.d = p.d;
  pa.W0 = W_A;
  pa.W1 = W_B;
  pa.out = P;
  pa.sigmoid = 0;
  cudaError_t e = launch_k(proj_fma_kernel, dim3((pa.M + kProjBM - 1) / kProjBM, pa.N / kProjBN),
                           dim3(256), 0, s, pdl, pa);
  if (e != cudaSuccess) return e;
  ProjArgs ha = pa;
  ha.table = hidden;
  ha.gather = 0;
  ha.M = p.B * p.L;
  ha.N = kRank;
  ha.W0 = W_H;
  ha.W1 = nullptr;
  ha.out = H;
  ha.sigmoid = 1;
  e = launch_k(proj_fma_kernel, dim3((ha.M + kProjBM - 1) / kProjBM, ha.N / kProjBN), dim3(256),
               0, s, pdl, ha);
  if (e != cudaSuccess) return e;
  PairArgs qa{P, H, cand_val, scores, p.L};
  return launch_k(pair16_kernel, dim3(p.B * p.L), dim3(256), 0, s, pdl, qa);
}

}  // namespace dfl2
