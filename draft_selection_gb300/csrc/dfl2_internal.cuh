// Internal declarations shared by the dfl2 translation units: device helpers
// (inline PTX for mbarriers and bulk copies), the kernel launchers and the
// workspace layouts.  Not part of the public ABI (include/dfl2.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dfl2 {

constexpr int kCand = 16;   // candidates kept per position
constexpr int kRank = 256;  // width of A(.), B(.) and H(.)
constexpr int kGroup = 16;  // channels sharing one conv correction

// Codes a kernel records in the per-device error word when a bounded wait runs out.
enum DeviceError : uint32_t {
  kDevErrNone = 0,
  kDevErrTopkFull = 1,   // top-16 consumer waited too long for a staged tile
  kDevErrTopkEmpty = 2,  // top-16 producer waited too long for a free stage
  kDevErrGemm = 3,       // projection GEMM pipeline wait ran out
  kDevErrConv = 4,       // conv GEMM pipeline wait ran out
  kDevErrBadIndex = 5,   // a candidate or verified token id outside [0, V)
};

// About two seconds at the GB300's maximum SM clock: far beyond any legitimate wait.
constexpr long long kWaitCycles = 4000000000LL;

__device__ __forceinline__ void record_error(uint32_t* err, uint32_t code) {
  if (err) atomicCAS(err, 0u, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier (shared::cta) ------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on a phase: false when kWaitCycles pass without completion.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) return false;
  }
  return true;
}

// ---- bulk async copy global -> shared (TMA engine, no tensor map) ---------
// Both addresses 16-byte aligned, bytes a multiple of 16.  Completion is
// signalled as transaction bytes on bar.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---- named barrier for a subset of warps ---------------------------------
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---- programmatic dependent launch ----------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- order-preserving keys for (value desc, index asc) -------------------
// key = (ord(value) << 32) | ~index: a larger key is a better candidate, every
// key is unique, and key 0 sorts below every real candidate (ord(-inf) > 0).
__device__ __forceinline__ uint32_t ord_f32(float v) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;  // -0.0 ties +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unord_f32(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
__device__ __forceinline__ uint64_t make_key(float v, uint32_t idx) {
  return (static_cast<uint64_t>(ord_f32(v)) << 32) | static_cast<uint32_t>(~idx);
}

// ---- launch configuration shared with the host ----------------------------
struct DeviceInfo {
  int sms;
  int max_smem_optin;
};
DeviceInfo device_info();        // cached per device
uint32_t* device_error_word();   // cached per device; device address
void count_launch(int n = 1);

// ---- top-16 -----------------------------------------------------------------
struct TopkPlan {
  int rows;            // B*L
  int V;
  int elem_bytes;      // 4 (float32) or 2 (bf16)
  int tiles_per_row;   // ceil(V*elem_bytes / kTopkTileBytes)
  int grid;            // CTAs (persistent; equal shares of rows*tiles_per_row tiles)
  int max_contrib;     // bound on CTAs contributing partial lists to one row
  size_t partial_off;  // workspace offset of uint64 [rows][max_contrib][16]
  size_t ticket_off;   // workspace offset of uint32 [rows]
  size_t ws_bytes;
};
TopkPlan topk_plan(int rows, int V, int elem_bytes);
cudaError_t launch_topk(const TopkPlan& p, const void* logits, int32_t* idx, float* val,
                        void* ws, cudaStream_t s, bool pdl);

// ---- projections + pair scores ---------------------------------------------
struct SelectPlan {
  int B, L, d;
  int M;               // B*(16L+1) candidate rows (verified token first, then 16 per position)
  size_t P_off;        // float32 [M][512]: A(.) in columns 0..255, B(.) in 256..511
  size_t H_off;        // float32 [B*L][256]
  size_t ws_bytes;
};
SelectPlan select_plan(int B, int L, int d);
cudaError_t launch_select(const SelectPlan& p, const int32_t* cand_idx, const float* cand_val,
                          const int32_t* verified, const __nv_bfloat16* hidden,
                          const __nv_bfloat16* E, const __nv_bfloat16* W_A,
                          const __nv_bfloat16* W_B, const __nv_bfloat16* W_H, int V,
                          float* scores, void* ws, cudaStream_t s, bool pdl);

// ---- walk ---------------------------------------------------------------------
cudaError_t launch_walk(const float* scores, const int32_t* cand_idx, int B, int L, float T,
                        const uint64_t* seeds, uint64_t cycle, int32_t* tokens, int32_t* slots,
                        float* q, cudaStream_t s, bool pdl);

// ---- conv ---------------------------------------------------------------------
cudaError_t launch_conv2(const __nv_bfloat16* x, const __nv_bfloat16* x_prev, const float* base,
                         const __nv_bfloat16* W_c, int B, int L, int d, __nv_bfloat16* y,
                         cudaStream_t s);

// ---- helpers ------------------------------------------------------------------
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Launch with optional programmatic-dependent-launch attribute.
template <typename Kernel, typename... Args>
cudaError_t launch_k(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                     Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  count_launch();
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace dfl2
