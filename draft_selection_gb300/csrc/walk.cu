// The walk over precomputed pair scores ("DFlash 2: Keep Drafting Parallel",
// 方法细节 > 轻量级路径选择器, "全并行打分与低延迟路径步进"; "DFlash 2: The
// Drafter Stopped Guessing Alone", "Selection beats correction").
//
// The walk is the selector's only sequential part, but the decision taken at
// step t from row i of S_t depends only on that row and on step t's draw (the
// Philox counter is t, not the path).  So one CTA per sequence stages the
// sequence's L x 16 x 16 score table in shared memory, takes the decision of
// every row in parallel (walk_row_choice: greedy argmax or the Philox draw from
// softmax(S/T)), and one thread then follows the chosen slots from the verified
// token: L dependent shared-memory reads.
#include "dfl2_internal.cuh"

namespace dfl2 {
namespace {

constexpr int kWalkThreads = 256;

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

__global__ void __launch_bounds__(kWalkThreads) walk_kernel(WalkArgs a) {
  extern __shared__ float4 s_tab4[];  // [L][16][16] scores, then each row's draft distribution
  float* tab = reinterpret_cast<float*>(s_tab4);
  __shared__ int choice[128 * kCand];
  __shared__ int path[128];
  pdl_wait();
  const int tid = threadIdx.x;
  const int b = blockIdx.x;
  const int L = a.L;
  {
    const float4* src = reinterpret_cast<const float4*>(a.scores + size_t(b) * L * kCand * kCand);
    const int n4 = L * kCand * kCand / 4;
    for (int e = tid; e < n4; e += kWalkThreads) s_tab4[e] = src[e];
  }
  __syncthreads();
  const uint64_t seed = a.T > 0.f ? a.seeds[b] : 0ull;
  for (int r = tid; r < L * kCand; r += kWalkThreads) {
    const int t = r / kCand, i = r % kCand;
    if (t == 0 && i > 0) {  // position 0 has only the verified token's row
      choice[r] = 0;
      continue;
    }
    const float u = a.T > 0.f ? walk_uniform(seed, a.cycle, t) : 0.f;
    choice[r] = walk_row_choice(tab + size_t(r) * kCand, a.T, u, tab + size_t(r) * kCand);
  }
  __syncthreads();
  if (tid == 0) {
    int prev = 0;  // row 0 of position 0: the last verified token
    for (int t = 0; t < L; ++t) {
      prev = choice[t * kCand + prev] & (kCand - 1);
      path[t] = prev;
    }
  }
  __syncthreads();
  for (int t = tid; t < L; t += kWalkThreads) {
    const size_t cell = size_t(b) * L + t;
    a.tokens[cell] = a.cand_idx[cell * kCand + path[t]];
    if (a.slots) a.slots[cell] = path[t];
  }
  if (a.q) {
    for (int e = tid; e < L * kCand; e += kWalkThreads) {
      const int t = e / kCand, k = e % kCand;
      const int row = t == 0 ? 0 : path[t - 1];  // step t draws from its predecessor's row
      a.q[(size_t(b) * L + t) * kCand + k] = tab[(size_t(t) * kCand + row) * kCand + k];
    }
  }
  pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_walk(const float* scores, const int32_t* cand_idx, int B, int L, float T,
                        const uint64_t* seeds, uint64_t cycle, int32_t* tokens, int32_t* slots,
                        float* q, cudaStream_t s, bool pdl) {
  WalkArgs a{scores, cand_idx, B, L, T, seeds, cycle, tokens, slots, q};
  const size_t smem = size_t(L) * kCand * kCand * sizeof(float);
  if (smem > 32 * 1024) {  // with the static tables, above the default 48 KB
    cudaError_t e = cudaFuncSetAttribute(walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  return launch_k(walk_kernel, dim3(B), dim3(kWalkThreads), smem, s, pdl, a);
}

}  // namespace dfl2
