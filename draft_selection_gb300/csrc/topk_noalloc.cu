// dfl2_topk_noalloc: the top-16 of dfl2_topk for callers that cannot allocate
// device memory.  The split-row partial lists and per-row tickets that
// dfl2_topk keeps in a caller-provided workspace live here in one fixed array
// of device memory that belongs to the library.
//
// Who needs it: serving engines that reserve almost all of the GPU's memory for
// their own pool (weights, KV cache) when they start and then forbid any later
// cudaMalloc, so that a request can never fail half-way for lack of memory or
// fragment the pool; and plug-ins that are handed only input and output
// pointers, with no allocator to ask for a workspace.
//
// Costs and limits:
//   * kScratchBytes (4 MiB) of device memory is reserved on every GPU that loads
//     the library, from load until the process exits.
//   * Problems whose workspace (dfl2_topk_workspace_size) exceeds that size are
//     rejected with DFL2_ERR_WORKSPACE before anything is launched.
//   * The first call on a device looks up the array's device address (and sets
//     up the kernel); make that first call before any stream capture.
//   * All calls share the one array: two calls whose kernels overlap on the GPU
//     (different streams, or different host threads) race and give wrong
//     results.  Calls on one stream, one after another, are safe: each call
//     clears the tickets it uses before its kernel runs.
#include <cstdio>
#include <mutex>

#include "dfl2.h"
#include "dfl2_internal.cuh"

namespace dfl2 {
dfl2_status check_topk_host(const void* logits, int dtype, int B, int L, int V, int k,
                            const void* cand_idx, const void* cand_val);
dfl2_status check_topk_device(const void* logits, const void* cand_idx, const void* cand_val);
dfl2_status report_error(dfl2_status st, const char* msg);
dfl2_status report_cuda_error(cudaError_t e, const char* what);
}  // namespace dfl2

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;

// The library's own scratch for dfl2_topk_noalloc.  Host code must not use this
// name as an address: it is a host-side stand-in; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_topk_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[64];  // per device, filled on the first call

}  // namespace

extern "C" dfl2_status dfl2_topk_noalloc(const void* logits, dfl2_dtype dtype, int B, int L,
                                         int V, int k, int32_t* cand_idx, float* cand_val,
                                         dfl2_stream stream) {
  dfl2_status st = dfl2::check_topk_host(logits, dtype, B, L, V, k, cand_idx, cand_val);
  if (st != DFL2_OK) return st;
  const int es = dtype == DFL2_F32 ? 4 : 2;
  const dfl2::TopkPlan plan = dfl2::topk_plan(B * L, V, es);
  if (plan.ws_bytes > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "dfl2_topk_noalloc: B=%d L=%d V=%d needs %zu bytes of scratch, more than the "
             "library's fixed %zu; use dfl2_topk with a workspace",
             B, L, V, plan.ws_bytes, kScratchBytes);
    return dfl2::report_error(DFL2_ERR_WORKSPACE, msg);
  }
  st = dfl2::check_topk_device(logits, cand_idx, cand_val);
  if (st != DFL2_OK) return st;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return dfl2::report_cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return dfl2::report_error(DFL2_ERR_UNSUPPORTED, "device ordinal >= 64");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_topk_scratch);
      if (e != cudaSuccess) return dfl2::report_cuda_error(e, "cudaGetSymbolAddress(top-16 scratch)");
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The tickets must start at zero; the partial lists are written before they are read.
  e = cudaMemsetAsync(static_cast<uint8_t*>(scratch) + plan.ticket_off, 0,
                      size_t(plan.rows) * sizeof(uint32_t), s);
  if (e != cudaSuccess) return dfl2::report_cuda_error(e, "clearing the top-16 scratch tickets");
  e = dfl2::launch_topk(plan, logits, cand_idx, cand_val, scratch, s, false);
  if (e != cudaSuccess) return dfl2::report_cuda_error(e, "top-16 launch");
  return DFL2_OK;
}
