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
// A wait that has lasted this long (about half a millisecond) also gives up as
// soon as any kernel has recorded an error in the device's error word: once one
// wait of a launch has run out, the launch's other waits end within about
// kGiveUpCycles each instead of kWaitCycles.
constexpr long long kGiveUpCycles = 1LL << 20;

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
// True when a wait that started at t0 must give up: kWaitCycles have passed,
// or kGiveUpCycles have and the error word `err` (nullable) is set.
__device__ __forceinline__ bool wait_expired(long long t0, const uint32_t* err) {
  const long long dt = clock64() - t0;
  if (dt > kWaitCycles) return true;
  return err && dt > kGiveUpCycles && *reinterpret_cast<const volatile uint32_t*>(err) != 0u;
}
// Bounded wait on a phase: false when it expires (wait_expired) first.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          const uint32_t* err = nullptr) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (wait_expired(t0, err)) return false;
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

// ---- mbarrier signalled from other CTAs of the cluster ----------------------
// Arrive (release at cluster scope) on the barrier at `bar` in CTA `rank`.
__device__ __forceinline__ void mbar_arrive_remote(const uint64_t* bar, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(bar)), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(a) : "memory");
}
// Bounded wait (acquire at cluster scope) on a local barrier that other CTAs arrive on.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  const uint32_t* err = nullptr) {
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if (wait_expired(t0, err)) return false;
  }
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
// 4-byte store into distributed shared memory (an address from mapa).
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---- a counter one thread publishes to the rest of its CTA -----------------
__device__ __forceinline__ void st_release_cta(uint32_t* p, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_cta(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
// Bounded wait until *p > n; false when it expires (wait_expired) first.
__device__ __forceinline__ bool wait_count_above(const uint32_t* p, uint32_t n,
                                                 const uint32_t* err = nullptr) {
  if (ld_acquire_cta(p) > n) return true;
  const long long t0 = clock64();
  while (ld_acquire_cta(p) <= n) {
    if (wait_expired(t0, err)) return false;
  }
  return true;
}

// ---- named barrier for a subset of warps ---------------------------------
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---- warp-level tensor-core MMA (mma.sync) --------------------------------
// ldmatrix: lane i gives the shared-memory address of row i % 8 of matrix i / 8.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t r[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t r[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
__device__ __forceinline__ void mma_16816_bf16(float d[4], const uint32_t a[4], const uint32_t b[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
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
// Block verification (verify.cu).
cudaError_t launch_verify_sample(const float* p, const int32_t* tokens, const int32_t* slots,
                                 const float* q, const int32_t* cand_idx, int B, int L, int V,
                                 const uint64_t* seeds, uint64_t cycle, int32_t* n_accepted,
                                 int32_t* out, cudaStream_t s);
cudaError_t launch_verify_greedy(const int32_t* tokens, const int32_t* top_idx, int B, int L,
                                 int32_t* n_accepted, int32_t* out, cudaStream_t s);
cudaError_t launch_topk(const TopkPlan& p, const void* logits, int32_t* idx, float* val,
                        void* ws, cudaStream_t s, bool pdl);

// ---- projections + pair scores ---------------------------------------------
struct SelectPlan {
  int B, L, d;
  int MA;              // rows needing A(.): per sequence the verified token + 16 (L-1) candidates
  int MB;              // rows needing B(.): per sequence 16 L candidates
  int MH;              // hidden rows: B L
  int M;               // MA (kept for reporting)
  int kblocks;         // d / 64
  int kps, splits;     // K blocks per split; K splits = CTAs of one cluster (reduced on chip)
  int nsplit;          // CTAs per row tile along the 256 outputs (1, 2 or 4)
  size_t PA_off;       // float32 [MA][256]
  size_t PB_off;       // float32 [MB][256]
  size_t GH_off;       // float32 [MH][256], before the sigmoid
  size_t part_off;     // float32 split-K partials [splits][MA|MB|MH][256] (splits > 1)
  size_t ticket_off;   // uint32 [B]: per-sequence tickets of the fused pair + walk kernel
  size_t choice_off;   // int32 [B*L][16]: per-row walk choice
  size_t q_off;        // float32 [B*L][16][16]: per-row draft distribution
  size_t ws_bytes;
};
SelectPlan select_plan(int B, int L, int d);
// Engine of the split-K projection (DFL2_PROJ_TENSOR / DFL2_PROJ_WARP); returns the previous one.
int set_projection_engine(int engine);
// Precomputed token tables P_A = E W_A^T, P_B = E W_B^T (float32 [V][256]).
cudaError_t launch_tables_build(const __nv_bfloat16* E, const __nv_bfloat16* W_A,
                                const __nv_bfloat16* W_B, int V, int d, float* P_A, float* P_B,
                                cudaStream_t s);
// Forward declaration for the table-mode launchers below.
struct WalkFuse;
// The gate projection GH = W_H h (before the sigmoid) into the plan's workspace.
cudaError_t launch_gate(const SelectPlan& p, const __nv_bfloat16* hidden, const __nv_bfloat16* W_H,
                        void* ws, cudaStream_t s, bool pdl);
// Pair scores (and, with walk, the fused walk) reading A(.) and B(.) rows from
// the tables by token; GH must be in the workspace.
cudaError_t launch_pair_tables(const SelectPlan& p, const int32_t* cand_idx, const float* cand_val,
                               const int32_t* verified, const float* P_A, const float* P_B, int V,
                               float* scores, const WalkFuse* walk, void* ws, cudaStream_t s,
                               bool pdl);
// The walk, when it runs inside the pair kernel (the fused tail).
struct WalkFuse {
  float T;
  const uint64_t* seeds;
  uint64_t cycle;
  int32_t* tokens;
  int32_t* slots;  // nullable
  float* q;        // nullable
};
cudaError_t launch_select(const SelectPlan& p, const int32_t* cand_idx, const float* cand_val,
                          const int32_t* verified, const __nv_bfloat16* hidden,
                          const __nv_bfloat16* E, const __nv_bfloat16* W_A,
                          const __nv_bfloat16* W_B, const __nv_bfloat16* W_H, int V,
                          float* scores, const WalkFuse* walk, void* ws, cudaStream_t s,
                          bool pdl);

// ---- walk ---------------------------------------------------------------------
cudaError_t launch_walk(const float* scores, const int32_t* cand_idx, int B, int L, float T,
                        const uint64_t* seeds, uint64_t cycle, int32_t* tokens, int32_t* slots,
                        float* q, cudaStream_t s, bool pdl);

// ---- conv ---------------------------------------------------------------------
// ws: NULL, or conv2_ws_bytes(B, L, d) bytes of device memory (the position-
// tiled split-K kernel exchanges its partial tiles there).
size_t conv2_ws_bytes(int B, int L, int d);
cudaError_t launch_conv2(const __nv_bfloat16* x, const __nv_bfloat16* x_prev, const float* base,
                         const __nv_bfloat16* W_c, int B, int L, int d, __nv_bfloat16* y,
                         void* ws, cudaStream_t s);

// ---- LM head + top-16 (lmhead.cu) ---------------------------------------------
struct LmheadPlan {
  int R, V, d;
  int rtiles;          // ceil(R / 128)
  int ntiles;          // ceil(V / 256)
  int kblocks;         // ceil(d / 64)
  int max_splits;      // CTAs per row tile the workspace has room for
  size_t lists_off;    // uint64 [R][splits][16] partial lists, one per row and CTA
  size_t ws_bytes;
};
LmheadPlan lmhead_plan(int R, int V, int d);
cudaError_t launch_lmhead_topk(const LmheadPlan& p, const __nv_bfloat16* hidden,
                               const __nv_bfloat16* W_lm, int32_t* idx, float* val, void* ws,
                               cudaStream_t s, bool pdl);

// ---- helpers ------------------------------------------------------------------
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Launch with optional programmatic-dependent-launch attribute and an optional
// thread-block cluster of `cluster` CTAs along x.
template <typename Kernel, typename... Args>
cudaError_t launch_kc(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                      int cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}
template <typename Kernel, typename... Args>
cudaError_t launch_k(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                     Args... args) {
  return launch_kc(kernel, grid, block, smem, s, pdl, 1, args...);
}

}  // namespace dfl2

// ============================================================================
// Blackwell tensor-core helpers (tcgen05, TMEM, TMA tensor maps), sm_100+.
// ============================================================================
namespace dfl2 {

// ---- cp.async (16 B, L2 only) with zero fill, and proxy fence -------------
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Makes this thread's generic-proxy shared-memory writes (st.shared, cp.async)
// visible to the async proxy (tensor cores, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- TMA tiled 2D load -------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void prefetch_l2_rows(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ---- TMEM allocation (one warp, .sync.aligned) -------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---- UMMA descriptors ------------------------------------------------------------
// Shared-memory matrix descriptor, K-major operand in the 128-byte swizzle
// layout: rows of 64 bf16 (128 B), 8-row atoms of 1024 B (stride byte offset),
// descriptor version 1, layout type 2 (SWIZZLE_128B).
__device__ __forceinline__ uint64_t umma_desc_sw128(const void* smem_tile) {
  const uint64_t addr = smem_u32(smem_tile);
  uint64_t d = 0;
  d |= (addr >> 4) & 0x3FFFull;          // start address
  d |= uint64_t(1) << 16;                // leading byte offset (unused for swizzled K-major)
  d |= uint64_t(1024 >> 4) << 32;        // stride byte offset: next 8-row atom
  d |= uint64_t(1) << 46;                // descriptor version (sm_100)
  d |= uint64_t(2) << 61;                // SWIZZLE_128B
  return d;
}
// Instruction descriptor, kind::f16: bf16 A and B (K-major), fp32 accumulator.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4)                 // D format: f32
         | (1u << 7)               // A format: bf16
         | (1u << 10)              // B format: bf16
         | (uint32_t(N >> 3) << 17)
         | (uint32_t(M >> 4) << 24);
}
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on bar when all previously issued tcgen05.mma of this thread complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// 32 lanes x 32 consecutive fp32 columns: thread i of the warp gets lane (base+i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ---- thread-block clusters (distributed shared memory) -----------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// Shared-memory address of the same variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(local)), "r"(rank));
  return out;
}
__device__ __forceinline__ void dsmem_st4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ float4 dsmem_ld4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Host: 2D bf16 tensor map over a row-major [rows, cols] matrix, box
// {64 cols, box_rows rows}, 128-byte swizzle.  Cached per (pointer, shape).
// Returns false if the driver entry point is unavailable or encoding fails.
bool tensor_map_bf16(const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                     void* out128);

}  // namespace dfl2

// ============================================================================
// The walk's per-row decision ("DFlash 2: Keep Drafting Parallel", 方法细节 >
// 轻量级路径选择器, "全并行打分与低延迟路径步进").  The step-t draw does not
// depend on the path (its Philox counter is t), so the decision for every row
// of every position can be made in parallel; the walk itself then only follows
// the chosen slots from the verified token.
// ============================================================================
namespace dfl2 {

// Philox4x32-10 (Salmon et al., SC'11), word 0 of the output block.
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

// Philox4x32-10, words 0 and 1 of the output block.
__device__ __forceinline__ uint2 philox4x32_10_w01(uint32_t c0, uint32_t c1, uint32_t c2,
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
  return make_uint2(c0, c1);
}

// Uniform in [0,1) of step t: counter (t, lo32(cycle), hi32(cycle), 0), key = seed.
__device__ __forceinline__ float walk_uniform(uint64_t seed, uint64_t cycle, int t) {
  const uint32_t w = philox4x32_10_w0(static_cast<uint32_t>(t), static_cast<uint32_t>(cycle),
                                      static_cast<uint32_t>(cycle >> 32), 0u,
                                      static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  return static_cast<float>(w >> 8) * 0x1p-24f;
}

// The successor slot chosen from one score row of 16, and (if q) the row's draft
// distribution.  T == 0: the lowest slot holding the maximum, q one-hot.
// T > 0: p_j = exp((S_j - max)/T), Z = sum in slot order, the first j with
// u Z < p_0 + ... + p_j (else the last j with p_j > 0), q = p / Z.  `row` may
// alias `q` (the row is read completely first).
// The same decision taken by the 16 lanes of a half-warp together, lane j
// holding entry j of the row: the same operations in the same order as
// walk_row_choice (the running sum is carried lane to lane in slot order, so Z
// and every partial sum are bit for bit the sequential ones), with short
// dependency chains and little code.  Every lane of the warp must call it
// (both halves, same T).  Returns the pick; q_j is lane j's probability.
__device__ __forceinline__ int walk_row_choice16(float v, float T, float u, float& q_j) {
  const int lane = threadIdx.x & 31, j = lane & 15, hbase = lane & 16;
  float m = v;
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off, 16));
  if (T == 0.f) {
    const uint32_t eq = (__ballot_sync(0xffffffffu, v == m) >> hbase) & 0xFFFFu;
    const int pick = __ffs(eq) - 1;  // the first maximum, as the sequential scan keeps
    q_j = j == pick ? 1.f : 0.f;
    return pick;
  }
  const float p = expf((v - m) / T);
  float cum = p;
#pragma unroll 1
  for (int s = 1; s < kCand; ++s) {  // cum_s = cum_{s-1} + p_s, in slot order
    const float prev = __shfl_up_sync(0xffffffffu, cum, 1, 16);
    if (j == s) cum = prev + p;
  }
  const float Z = __shfl_sync(0xffffffffu, cum, 15, 16);
  const float uZ = u * Z;
  // both votes by every lane (the halves may take different branches below)
  const uint32_t hit = (__ballot_sync(0xffffffffu, uZ < cum) >> hbase) & 0xFFFFu;
  const uint32_t pos = (__ballot_sync(0xffffffffu, p > 0.f) >> hbase) & 0xFFFFu;
  // the first crossing; if rounding left none, the last slot with mass
  const int pick = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
  q_j = p / Z;
  return pick;
}
__device__ __forceinline__ int walk_row_choice(const float* row, float T, float u, float* q) {
  float v[kCand];
#pragma unroll
  for (int j = 0; j < kCand; ++j) v[j] = row[j];
  int pick = 0;
  if (T == 0.f) {
    float best = v[0];
#pragma unroll
    for (int j = 1; j < kCand; ++j)
      if (v[j] > best) {
        best = v[j];
        pick = j;
      }
    if (q)
#pragma unroll
      for (int j = 0; j < kCand; ++j) q[j] = j == pick ? 1.f : 0.f;
    return pick;
  }
  float m = v[0];
#pragma unroll
  for (int j = 1; j < kCand; ++j) m = fmaxf(m, v[j]);
  float Z = 0.f;
#pragma unroll
  for (int j = 0; j < kCand; ++j) {
    v[j] = expf((v[j] - m) / T);
    Z += v[j];
  }
  const float uZ = u * Z;
  float cum = 0.f;
  pick = -1;
#pragma unroll
  for (int j = 0; j < kCand; ++j) {
    cum += v[j];
    if (pick < 0 && uZ < cum) pick = j;
  }
  if (pick < 0) {
    pick = 0;
#pragma unroll
    for (int j = 0; j < kCand; ++j)
      if (v[j] > 0.f) pick = j;
  }
  if (q)
#pragma unroll
    for (int j = 0; j < kCand; ++j) q[j] = v[j] / Z;
  return pick;
}

}  // namespace dfl2
