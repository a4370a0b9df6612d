// The walk over precomputed pair scores ("DFlash 2: Keep Drafting Parallel",
// 方法细节 > 轻量级路径选择器, "全并行打分与低延迟路径步进"; "DFlash 2: The
// Drafter Stopped Guessing Alone", "Selection beats correction"): the only
// sequential part of the selector.  One warp per sequence, lane j = slot j.
//   greedy   : the lowest slot holding the row maximum
//   sampling : p_j = exp((S_j - max)/T), the first j with u Z < p_0 + ... + p_j,
//              u from Philox4x32-10 (Salmon et al., SC'11), counter
//              (t, lo32(cycle), hi32(cycle), 0), key = the sequence's seed.
#include "dfl2_internal.cuh"

namespace dfl2 {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWalkWarps = 4;

// Philox4x32-10, word 0 of the output block.
__device__ __forceinline__ uint32_t philox4x32_10_w0(uint32_t c0, uint32_t c1, uint32_t c2,
                                                     uint32_t c3, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c0;
}

struct WalkArgs {
  const float* scores;
  const int32_t* cand_idx;
  int B, L;
  float T;
  const uint64_t* seeds;
  uint64_t cycle;
  int32_t* tokens;
  int32_t* slots;
  float* q;
};

__global__ void __launch_bounds__(kWalkWarps * 32) walk_kernel(WalkArgs a) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * kWalkWarps + (threadIdx.x >> 5);
  if (b >= a.B) return;  // whole warp leaves together
  const uint64_t seed = a.T > 0.f ? a.seeds[b] : 0ull;
  int prev = 0;  // row 0 of position 0: the last verified token
  for (int t = 0; t < a.L; ++t) {
    const size_t cell = size_t(b) * a.L + t;
    const float s = lane < kCand ? a.scores[(cell * kCand + prev) * kCand + lane] : -INFINITY;
    int pick;
    float p = 0.f, Z = 1.f;
    if (a.T == 0.f) {
      float v = s;
      int slot = lane;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(kFull, v, off);
        const int os = __shfl_xor_sync(kFull, slot, off);
        if (ov > v || (ov == v && os < slot)) {
          v = ov;
          slot = os;
        }
      }
      // Every lane follows lane 0's choice (lanes could disagree only on NaN scores).
      pick = __shfl_sync(kFull, slot, 0);
    } else {
      float m = s;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
      p = lane < kCand ? expf((s - m) / a.T) : 0.f;
      float cum = p;  // inclusive prefix sum in slot order
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(kFull, cum, off);
        if (lane >= off) cum += o;
      }
      Z = __shfl_sync(kFull, cum, kCand - 1);
      uint32_t w = 0;
      if (lane == 0)
        w = philox4x32_10_w0(static_cast<uint32_t>(t), static_cast<uint32_t>(a.cycle),
                             static_cast<uint32_t>(a.cycle >> 32), 0u,
                             static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
      w = __shfl_sync(kFull, w, 0);
      const float u = static_cast<float>(w >> 8) * 0x1p-24f;
      const float uZ = u * Z;
      const unsigned hit = __ballot_sync(kFull, lane < kCand && uZ < cum);
      if (hit) {
        pick = __ffs(hit) - 1;
      } else {
        const unsigned live = __ballot_sync(kFull, lane < kCand && p > 0.f);
        pick = live ? 31 - __clz(live) : 0;
      }
    }
    pick &= kCand - 1;  // a slot index whatever the scores held
    if (lane == 0) {
      a.tokens[cell] = a.cand_idx[cell * kCand + pick];
      if (a.slots) a.slots[cell] = pick;
    }
    if (a.q && lane < kCand) {
      a.q[cell * kCand + lane] = a.T == 0.f ? (lane == pick ? 1.f : 0.f) : p / Z;
    }
    prev = pick;
  }
  pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_walk(const float* scores, const int32_t* cand_idx, int B, int L, float T,
                        const uint64_t* seeds, uint64_t cycle, int32_t* tokens, int32_t* slots,
                        float* q, cudaStream_t s, bool pdl) {
  WalkArgs a{scores, cand_idx, B, L, T, seeds, cycle, tokens, slots, q};
  return launch_k(walk_kernel, dim3((B + kWalkWarps - 1) / kWalkWarps), dim3(kWalkWarps * 32), 0,
                  s, pdl, a);
}

}  // namespace dfl2
