// Verification of a drafted block ("DFlash 2: Keep Drafting Parallel",
// 方法细节 > 轻量级路径选择器, "全并行打分与低延迟路径步进": lossless rejection
// sampling recovers the target's distribution; "DFlash 2: The Drafter Stopped
// Guessing Alone", "One pass to draft, one pass to verify": the accepted prefix
// is kept, the first miss is replaced by the target's own choice).  The step is
// the published speculative-sampling rule (Leviathan et al., ICML 2023; Chen et
// al., 2023).
//
// p [B, L+1, V] holds the target's next-token distributions.  Greedy runs the
// top-16 kernels over the L+1 rows (slot 0 is the argmax, lowest index on
// ties) and a scan kernel keeps the matching prefix.  Sampling runs one CTA per
// sequence:
//   * acceptance of every position at once, in double precision: u0 * q(x) and
//     p(x) are exact there, so the decision is exactly the definition's; the
//     first rejected position j (or L when none) is a ballot;
//   * row j in 512-element tiles, a contiguous run per warp, four tiles in
//     flight per lane: each lane sums its 16 consecutive elements and the warp
//     the lanes in single precision (this GPU's double-precision rate is a
//     small fraction of its single-precision one); the residual max(0, p - q)
//     differs from p only at the 16 candidates, whose corrections are added to
//     their tiles' sums; the tile sums are scanned in double;
//   * a block scan of the tile sums gives the running sum at every tile, the
//     first tile whose running sum passes u1 * Z is found in parallel, and one
//     warp locates the element in it.
#include "dfl2_internal.cuh"

namespace dfl2 {
namespace {

constexpr int kVfThreads = 512;
constexpr int kVfTile = 512;                       // elements per tile (32 lanes x 16)
constexpr int kVfMaxTiles = 1024;                  // V <= 524,288
constexpr unsigned kFullMask = 0xffffffffu;

struct VerifyArgs {
  const float* p;
  const int32_t* tokens;
  const int32_t* slots;
  const float* q;
  const int32_t* cand_idx;
  int L, V;
  const uint64_t* seeds;
  uint64_t cycle;
  int32_t* n_accepted;
  int32_t* out;
  uint32_t* err;
};

__device__ __forceinline__ void verify_uniforms(uint64_t seed, uint64_t cycle, int t, double& u0,
                                                double& u1) {
  const uint2 w = philox4x32_10_w01(static_cast<uint32_t>(t), static_cast<uint32_t>(cycle),
                                    static_cast<uint32_t>(cycle >> 32), 1u,
                                    static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  u0 = static_cast<double>(w.x >> 8) * 0x1p-24;
  u1 = static_cast<double>(w.y >> 8) * 0x1p-24;
}

// The lane's 16 elements [16 lane, 16 lane + 16) of tile k (zero past V).
__device__ __forceinline__ void tile_lane(const float* row, int V, int k, int lane, float (&x)[16]) {
  const int base = k * kVfTile + 16 * lane;
#pragma unroll
  for (int v4 = 0; v4 < 4; ++v4) {
    const int e = base + 4 * v4;
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    if (e < V) f = __ldg(reinterpret_cast<const float4*>(row + e));  // V % 4 == 0
    x[4 * v4] = f.x;
    x[4 * v4 + 1] = f.y;
    x[4 * v4 + 2] = f.z;
    x[4 * v4 + 3] = f.w;
  }
}

// Sum of the lane's 16 elements in single precision (pairwise): this GPU's
// double-precision rate is a small fraction of its single-precision one.
__device__ __forceinline__ float lane_sum(const float (&x)[16]) {
  float v[4];
#pragma unroll
  for (int v4 = 0; v4 < 4; ++v4) v[v4] = (x[4 * v4] + x[4 * v4 + 1]) + (x[4 * v4 + 2] + x[4 * v4 + 3]);
  return (v[0] + v[1]) + (v[2] + v[3]);
}

__global__ void __launch_bounds__(kVfThreads) verify_sample_kernel(VerifyArgs a) {
  __shared__ double tsum[kVfMaxTiles];
  __shared__ double tincl[kVfMaxTiles];  // inclusive running sums of tsum
  __shared__ double wsum[kVfThreads / 32];
  __shared__ int cand_tok[kCand];
  __shared__ float cand_res[kCand];  // max(0, p - q) at the candidate
  __shared__ float cand_p[kCand];    // p at the candidate
  __shared__ int j_s, tile_s;
  __shared__ double start_s, target_s;
  pdl_wait();
  const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = a.L, V = a.V;
  const size_t rowstride = size_t(V);
  const float* P = a.p + size_t(b) * (L + 1) * rowstride;
  const uint64_t seed = a.seeds[b];

  // ---- acceptance of every position; j = the first rejected one (L if none) ----
  if (warp == 0) {
    int j = L;
    for (int t0 = 0; t0 < L; t0 += 32) {
      const int t = t0 + lane;
      bool reject = false;
      if (t < L) {
        const size_t cell = size_t(b) * L + t;
        const int x = a.tokens[cell];
        const int sl = a.slots[cell];
        if (x < 0 || x >= V || sl < 0 || sl >= kCand) {
          record_error(a.err, kDevErrBadIndex);
          reject = true;
        } else {
          double u0, u1;
          verify_uniforms(seed, a.cycle, t, u0, u1);
          const double qx = static_cast<double>(a.q[cell * kCand + sl]);
          reject = !(u0 * qx < static_cast<double>(P[size_t(t) * rowstride + x]));
        }
      }
      const unsigned rj = __ballot_sync(kFullMask, reject);
      if (rj) {
        j = t0 + __ffs(rj) - 1;
        break;
      }
    }
    if (lane == 0) j_s = j;
  }
  __syncthreads();
  const int j = j_s;
  const float* row = P + size_t(j) * rowstride;
  const int ntiles = (V + kVfTile - 1) / kVfTile;
  bool use_res = j < L;  // draw from max(0, p - q); else (bonus row) from p
  if (use_res && tid < kCand) {
    const size_t cell = size_t(b) * L + j;
    const int c = a.cand_idx[cell * kCand + tid];
    const bool ok = c >= 0 && c < V;
    const float pc = ok ? row[c] : 0.f;
    cand_tok[tid] = ok ? c : -1;
    cand_p[tid] = pc;
    cand_res[tid] = ok ? fmaxf(0.f, pc - a.q[cell * kCand + tid]) : 0.f;
  }
  constexpr int kWarps = kVfThreads / 32;
  const int per_warp = (ntiles + kWarps - 1) / kWarps;  // contiguous tiles per warp
  for (int pass = 0; pass < 2; ++pass) {
    // ---- tile sums of p over the row: each warp a contiguous run of tiles,
    // four at a time (16 float4 loads per lane in flight) ----
    const int k_lo = warp * per_warp, k_hi = min(ntiles, k_lo + per_warp);
    for (int k0 = k_lo; k0 < k_hi; k0 += 4) {
      float x[4][16];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (k0 + u < k_hi) tile_lane(row, V, k0 + u, lane, x[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (k0 + u < k_hi) {
          float sv = lane_sum(x[u]);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) sv += __shfl_xor_sync(kFullMask, sv, off);
          if (lane == 0) tsum[k0 + u] = static_cast<double>(sv);
        }
      }
    }
    __syncthreads();
    if (use_res && tid == 0) {  // the residual differs from p at the candidates only
      for (int c = 0; c < kCand; ++c) {  // in slot order: deterministic
        const int v = cand_tok[c];
        if (v >= 0) tsum[v / kVfTile] += static_cast<double>(cand_res[c]) - static_cast<double>(cand_p[c]);
      }
    }
    __syncthreads();
    // ---- inclusive scan of the tile sums (fp64, fixed order): thread t holds
    // tiles 2t and 2t+1 ----
    {
      const int k0 = 2 * tid;
      const double s0 = k0 < ntiles ? tsum[k0] : 0.0;
      const double s1 = k0 + 1 < ntiles ? tsum[k0 + 1] : 0.0;
      double incl = s0 + s1;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const double o = __shfl_up_sync(kFullMask, incl, off);
        if (lane >= off) incl += o;
      }
      if (lane == 31) wsum[warp] = incl;
      __syncthreads();
      if (warp == 0) {
        double w = lane < kWarps ? wsum[lane] : 0.0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const double o = __shfl_up_sync(kFullMask, w, off);
          if (lane >= off) w += o;
        }
        if (lane < kWarps) wsum[lane] = w;  // inclusive over warps
      }
      __syncthreads();
      const double before = (warp > 0 ? wsum[warp - 1] : 0.0) + (incl - (s0 + s1));
      if (k0 < ntiles) tincl[k0] = before + s0;
      if (k0 + 1 < ntiles) tincl[k0 + 1] = before + s0 + s1;
      if (tid == 0) tile_s = ntiles;  // no tile found yet
    }
    __syncthreads();
    const double Z = tincl[ntiles - 1];
    double u0, u1;
    verify_uniforms(seed, a.cycle, j, u0, u1);
    const double T = u1 * Z;
    // the crossing tile: the first k whose inclusive sum exceeds T
    for (int k = tid; k < ntiles; k += kVfThreads)
      if (T < tincl[k] && tsum[k] > 0.0) atomicMin(&tile_s, k);
    __syncthreads();
    if (tid == 0) {
      int kk = tile_s;
      if (kk >= ntiles) {  // rounding left T at or above the total: the last tile with mass
        kk = -1;
        for (int k = ntiles - 1; k >= 0 && kk < 0; --k)
          if (tsum[k] > 0.0) kk = k;
      }
      tile_s = Z > 0.0 ? kk : -2;  // -2: no residual mass anywhere
      start_s = kk >= 0 ? tincl[kk] - tsum[kk] : 0.0;
      target_s = T;
    }
    __syncthreads();
    if (tile_s != -2 || !use_res) break;
    use_res = false;  // p never exceeds q: draw from p itself (second pass)
    __syncthreads();
  }
  const int kk = tile_s;
  // ---- locate the element inside tile kk; write the block's outputs ----
  if (warp == 0) {
    int pick = -1;
    if (kk >= 0) {
      float x[16];
      tile_lane(row, V, kk, lane, x);
      if (use_res) {
        for (int c = 0; c < kCand; ++c) {
          const int v = cand_tok[c] - (kk * kVfTile + 16 * lane);
          if (cand_tok[c] >= 0 && v >= 0 && v < 16) {
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (e == v) x[e] = cand_res[c];
          }
        }
      }
      const double ls = static_cast<double>(lane_sum(x));
      double pre = ls;  // inclusive scan over the lanes
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const double o = __shfl_up_sync(kFullMask, pre, off);
        if (lane >= off) pre += o;
      }
      const double lo = start_s + (pre - ls), T = target_s;
      int mine = -1;
      if (T >= lo && T < lo + ls) {
        const float rel = static_cast<float>(T - lo);  // the target inside this lane's run
        float cum = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          cum += x[e];
          if (mine < 0 && rel < cum) mine = e;
        }
        if (mine < 0)
          for (int e = 15; e >= 0; --e)
            if (x[e] > 0.f) {
              mine = e;
              break;
            }
      }
      const unsigned who = __ballot_sync(kFullMask, mine >= 0);
      if (who) {
        const int src = __ffs(who) - 1;
        pick = kk * kVfTile + 16 * src + __shfl_sync(kFullMask, mine, src);
      } else {  // rounding: the last element of the tile with mass
        int last = -1;
#pragma unroll
        for (int e = 0; e < 16; ++e)
          if (x[e] > 0.f) last = kk * kVfTile + 16 * lane + e;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) last = max(last, __shfl_xor_sync(kFullMask, last, off));
        pick = last;
      }
    }
    int32_t* o = a.out + size_t(b) * (L + 1);
    for (int t = lane; t <= L; t += 32) {
      int32_t v = -1;
      if (t < j) v = a.tokens[size_t(b) * L + t];
      else if (t == j) v = pick < 0 ? 0 : pick;
      o[t] = v;
    }
    if (lane == 0) a.n_accepted[b] = j;
  }
  pdl_launch_dependents();
}

__global__ void __launch_bounds__(128) verify_greedy_kernel(const int32_t* tokens,
                                                            const int32_t* top_idx, int L,
                                                            int32_t* n_accepted, int32_t* out) {
  __shared__ int j_s;
  pdl_wait();
  const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {
    int j = L;
    for (int t0 = 0; t0 < L; t0 += 32) {
      const int t = t0 + lane;
      const bool miss = t < L && tokens[size_t(b) * L + t] != top_idx[(size_t(b) * (L + 1) + t) * kCand];
      const unsigned m = __ballot_sync(kFullMask, miss);
      if (m) {
        j = t0 + __ffs(m) - 1;
        break;
      }
    }
    if (lane == 0) {
      j_s = j;
      n_accepted[b] = j;
    }
  }
  __syncthreads();
  const int j = j_s;
  for (int t = tid; t <= L; t += blockDim.x) {
    int32_t v = -1;
    if (t < j) v = tokens[size_t(b) * L + t];
    else if (t == j) v = top_idx[(size_t(b) * (L + 1) + t) * kCand];
    out[size_t(b) * (L + 1) + t] = v;
  }
  pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_verify_sample(const float* p, const int32_t* tokens, const int32_t* slots,
                                 const float* q, const int32_t* cand_idx, int B, int L, int V,
                                 const uint64_t* seeds, uint64_t cycle, int32_t* n_accepted,
                                 int32_t* out, cudaStream_t s) {
  if ((V + kVfTile - 1) / kVfTile > kVfMaxTiles) return cudaErrorInvalidValue;
  VerifyArgs a{p, tokens, slots, q, cand_idx, L, V, seeds, cycle, n_accepted, out,
               device_error_word()};
  return launch_k(verify_sample_kernel, dim3(B), dim3(kVfThreads), 0, s, true, a);
}

cudaError_t launch_verify_greedy(const int32_t* tokens, const int32_t* top_idx, int B, int L,
                                 int32_t* n_accepted, int32_t* out, cudaStream_t s) {
  return launch_k(verify_greedy_kernel, dim3(B), dim3(128), 0, s, true, tokens, top_idx, L,
                  n_accepted, out);
}

}  // namespace dfl2
