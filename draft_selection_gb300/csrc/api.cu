// The C ABI of include/dfl2.h: argument validation, workspace carving and
// dispatch to the kernels.  Nothing here touches the data: every step of the
// draft tail runs in the CUDA kernels of this directory.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <string>

#include "dfl2.h"
#include "dfl2_internal.cuh"

namespace {

thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches{0};
std::mutex g_mu;

// Per-device error word for bounded in-kernel waits and out-of-range indices.
__device__ uint32_t g_device_error;

struct DevState {
  bool ready = false;
  dfl2::DeviceInfo info{};
  uint32_t* err = nullptr;
};
DevState g_dev[64];
thread_local int g_cur_dev = 0;

dfl2_status fail(dfl2_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

dfl2_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DFL2_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Make sure this device's cached state exists; sets g_cur_dev.
dfl2_status ensure_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(DFL2_ERR_UNSUPPORTED, "device ordinal %d >= 64", dev);
  g_cur_dev = dev;
  DevState& s = g_dev[dev];
  if (s.ready) return DFL2_OK;
  std::lock_guard<std::mutex> lock(g_mu);
  if (s.ready) return DFL2_OK;
  int sms = 0, smem = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
  e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(shared memory)");
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_device_error);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
  s.info.sms = sms;
  s.info.max_smem_optin = smem;
  s.err = static_cast<uint32_t*>(p);
  s.ready = true;
  return DFL2_OK;
}

#define DFL2_TRY(expr)               \
  do {                               \
    dfl2_status _st = (expr);        \
    if (_st != DFL2_OK) return _st;  \
  } while (0)
#define DFL2_TRY_EARLY DFL2_TRY

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-side pointer checks that need no CUDA call: non-NULL and 16-byte aligned.
dfl2_status check_ptr(const void* p, const char* name) {
  if (!p) return fail(DFL2_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(DFL2_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return DFL2_OK;
}

// Device (or managed) memory of the current device's address space.
dfl2_status check_device_ptr(const void* p, const char* name) {
  DFL2_TRY_EARLY(check_ptr(p, name));
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(DFL2_ERR_INVALID_ARG, "%s is not a CUDA pointer (%s)", name, cudaGetErrorName(e));
  }
  if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
    return fail(DFL2_ERR_INVALID_ARG, "%s must be device memory", name);
  return DFL2_OK;
}


struct PtrSpec {
  const void* p;
  const char* name;
  bool optional = false;
};
using Ptrs = std::initializer_list<PtrSpec>;

// Checks that need no CUDA call (run before the device is touched).
dfl2_status check_host(Ptrs ptrs) {
  for (const PtrSpec& s : ptrs) {
    if (s.optional && !s.p) continue;
    DFL2_TRY(check_ptr(s.p, s.name));
  }
  return DFL2_OK;
}

dfl2_status check_device(Ptrs ptrs) {
  for (const PtrSpec& s : ptrs) {
    if (s.optional && !s.p) continue;
    DFL2_TRY(check_device_ptr(s.p, s.name));
  }
  return DFL2_OK;
}

dfl2_status check_temperature(float T) {
  if (!(T >= 0.f) || !std::isfinite(T))
    return fail(DFL2_ERR_INVALID_ARG, "temperature %g must be finite and >= 0", double(T));
  return DFL2_OK;
}


dfl2_status check_shape(int B, int L) {
  if (B < 1 || L < 1) return fail(DFL2_ERR_INVALID_ARG, "B=%d and L=%d must be >= 1", B, L);
  if ((long long)B * (16LL * L + 1) > (1LL << 30))
    return fail(DFL2_ERR_INVALID_ARG, "B*(16L+1) = %lld is too large",
                (long long)B * (16LL * L + 1));
  return DFL2_OK;
}

// The walk keeps a sequence's L x 16 x 16 score table in shared memory.
dfl2_status check_block_len(int L) {
  if (L > 128) return fail(DFL2_ERR_UNSUPPORTED, "L=%d: draft blocks of at most 128 positions", L);
  return DFL2_OK;
}

dfl2_status check_topk_args(int dtype, int B, int L, int V, int k) {
  DFL2_TRY(check_shape(B, L));
  if (dtype != DFL2_F32 && dtype != DFL2_BF16)
    return fail(DFL2_ERR_UNSUPPORTED, "logits dtype %d is not float32 or bf16", dtype);
  if (k != dfl2::kCand) return fail(DFL2_ERR_UNSUPPORTED, "k=%d: only 16 candidates", k);
  if (V < dfl2::kCand) return fail(DFL2_ERR_INVALID_ARG, "V=%d < 16", V);
  return DFL2_OK;
}

dfl2_status check_ws(const void* ws, size_t have, size_t need) {
  if (!ws) return fail(DFL2_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", need);
  if (have < need)
    return fail(DFL2_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", have, need);
  return check_ptr(ws, "workspace");
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return pa < pb + nb && pb < pa + na;
}

const __nv_bfloat16* bf(const uint16_t* p) { return reinterpret_cast<const __nv_bfloat16*>(p); }

struct TailLayout {
  dfl2::TopkPlan topk;
  dfl2::SelectPlan sel;
  size_t topk_off, idx_off, val_off, sel_off, scores_off, bytes;
};

TailLayout tail_layout(int B, int L, int V, int d, int elem_bytes) {
  TailLayout t;
  t.topk = dfl2::topk_plan(B * L, V, elem_bytes);
  t.sel = dfl2::select_plan(B, L, d);
  const size_t rows = size_t(B) * L;
  t.topk_off = 0;
  t.idx_off = dfl2::align_up(t.topk.ws_bytes, 256);
  t.val_off = dfl2::align_up(t.idx_off + rows * dfl2::kCand * 4, 256);
  t.sel_off = dfl2::align_up(t.val_off + rows * dfl2::kCand * 4, 256);
  t.scores_off = dfl2::align_up(t.sel_off + t.sel.ws_bytes, 256);
  t.bytes = dfl2::align_up(t.scores_off + rows * dfl2::kCand * dfl2::kCand * 4, 256);
  return t;
}

dfl2_status check_select_args(int B, int L, int V, int d, int r) {
  DFL2_TRY(check_shape(B, L));
  if (r != dfl2::kRank) return fail(DFL2_ERR_UNSUPPORTED, "r=%d: only rank 256", r);
  if (V < dfl2::kCand) return fail(DFL2_ERR_INVALID_ARG, "V=%d < 16", V);
  if (d < 16 || d % 16 != 0)
    return fail(DFL2_ERR_UNSUPPORTED, "d=%d: the selector needs a multiple of 16", d);
  return DFL2_OK;
}

}  // namespace

namespace dfl2 {
void count_launch(int n) { g_launches.fetch_add(static_cast<uint64_t>(n)); }
DeviceInfo device_info() { return g_dev[g_cur_dev].info; }
uint32_t* device_error_word() { return g_dev[g_cur_dev].err; }

// The checks of dfl2_topk apart from the workspace, for entry points that live
// in other translation units: first those that need no CUDA call, then the
// device ones (which also set up this device's cached state).
dfl2_status check_topk_host(const void* logits, int dtype, int B, int L, int V, int k,
                            const void* cand_idx, const void* cand_val) {
  DFL2_TRY(check_topk_args(dtype, B, L, V, k));
  return check_host({{logits, "logits"}, {cand_idx, "cand_idx"}, {cand_val, "cand_val"}});
}
dfl2_status check_topk_device(const void* logits, const void* cand_idx, const void* cand_val) {
  DFL2_TRY(ensure_device());
  return check_device({{logits, "logits"}, {cand_idx, "cand_idx"}, {cand_val, "cand_val"}});
}
// Records the calling thread's error message; returns st.
dfl2_status report_error(dfl2_status st, const char* msg) { return fail(st, "%s", msg); }
dfl2_status report_cuda_error(cudaError_t e, const char* what) { return cuda_fail(e, what); }
}  // namespace dfl2

extern "C" {

const char* dfl2_version(void) { return "dfl2 0.1 sm_103a"; }

size_t dfl2_last_error(char* buf, size_t len) {
  if (buf && len) {
    size_t n = g_last_error.size() < len - 1 ? g_last_error.size() : len - 1;
    memcpy(buf, g_last_error.data(), n);
    buf[n] = '\0';
  }
  return g_last_error.size();
}

uint64_t dfl2_launch_count(void) { return g_launches.load(); }

int dfl2_set_projection_engine(int engine) {
  if (engine != DFL2_PROJ_TENSOR && engine != DFL2_PROJ_WARP) return -1;
  return dfl2::set_projection_engine(engine);
}

dfl2_status dfl2_workspace_init(void* ws, size_t ws_bytes, dfl2_stream stream) {
  DFL2_TRY(ensure_device());
  if (!ws || ws_bytes == 0) return fail(DFL2_ERR_INVALID_ARG, "empty workspace");
  DFL2_TRY(check_device_ptr(ws, "workspace"));
  cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace)");
  return DFL2_OK;
}

dfl2_status dfl2_device_error(uint32_t* code, int clear) {
  DFL2_TRY(ensure_device());
  if (!code) return fail(DFL2_ERR_INVALID_ARG, "code is NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  e = cudaMemcpyFromSymbol(code, g_device_error, sizeof(uint32_t));
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  if (clear) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
  }
  return DFL2_OK;
}

size_t dfl2_topk_workspace_size(int B, int L, int V) {
  if (B < 1 || L < 1 || V < dfl2::kCand) return 0;
  return dfl2::topk_plan(B * L, V, 4).ws_bytes;
}

dfl2_status dfl2_topk(const void* logits, dfl2_dtype dtype, int B, int L, int V, int k,
                      int32_t* cand_idx, float* cand_val, void* ws, size_t ws_bytes,
                      dfl2_stream stream) {
  DFL2_TRY(check_topk_args(dtype, B, L, V, k));
  const int es = dtype == DFL2_F32 ? 4 : 2;
  const dfl2::TopkPlan plan = dfl2::topk_plan(B * L, V, es);
  const Ptrs ptrs = {{logits, "logits"}, {cand_idx, "cand_idx"}, {cand_val, "cand_val"}};
  DFL2_TRY(check_host(ptrs));
  DFL2_TRY(check_ws(ws, ws_bytes, plan.ws_bytes));
  DFL2_TRY(ensure_device());
  DFL2_TRY(check_device(ptrs));
  DFL2_TRY(check_device_ptr(ws, "workspace"));
  cudaError_t e = dfl2::launch_topk(plan, logits, cand_idx, cand_val, ws,
                                    reinterpret_cast<cudaStream_t>(stream), true);
  if (e != cudaSuccess) return cuda_fail(e, "top-16 launch");
  return DFL2_OK;
}

size_t dfl2_lmhead_topk_workspace_size(int B, int L, int V, int d) {
  if (B < 1 || L < 1 || V < dfl2::kCand || d < 1) return 0;
  return dfl2::lmhead_plan(B * L, V, d).ws_bytes;
}

dfl2_status dfl2_lmhead_topk(const uint16_t* hidden, const uint16_t* W_lm, int B, int L, int V,
                             int d, int k, int32_t* cand_idx, float* cand_val, void* ws,
                             size_t ws_bytes, dfl2_stream stream) {
  DFL2_TRY(check_shape(B, L));
  if (k != dfl2::kCand) return fail(DFL2_ERR_UNSUPPORTED, "k=%d: only 16 candidates", k);
  if (V < dfl2::kCand) return fail(DFL2_ERR_INVALID_ARG, "V=%d < 16", V);
  if (d < 8 || d % 8 != 0)
    return fail(DFL2_ERR_UNSUPPORTED, "d=%d: rows of hidden and W_lm must be 16-byte multiples", d);
  const dfl2::LmheadPlan plan = dfl2::lmhead_plan(B * L, V, d);
  const Ptrs ptrs = {{hidden, "hidden"}, {W_lm, "W_lm"}, {cand_idx, "cand_idx"},
                     {cand_val, "cand_val"}};
  DFL2_TRY(check_host(ptrs));
  DFL2_TRY(check_ws(ws, ws_bytes, plan.ws_bytes));
  DFL2_TRY(ensure_device());
  DFL2_TRY(check_device(ptrs));
  DFL2_TRY(check_device_ptr(ws, "workspace"));
  cudaError_t e = dfl2::launch_lmhead_topk(plan, bf(hidden), bf(W_lm), cand_idx, cand_val, ws,
                                           reinterpret_cast<cudaStream_t>(stream), true);
  if (e != cudaSuccess) return cuda_fail(e, "LM head + top-16 launch");
  return DFL2_OK;
}

size_t dfl2_select_workspace_size(int B, int L, int d) {
  if (B < 1 || L < 1 || d < 1) return 0;
  return dfl2::select_plan(B, L, d).ws_bytes;
}

dfl2_status dfl2_select(const int32_t* cand_idx, const float* cand_val,
                        const int32_t* verified_tok, const uint16_t* hidden, const uint16_t* E,
                        const uint16_t* W_A, const uint16_t* W_B, const uint16_t* W_H, int B,
                        int L, int V, int d, int r, float* scores, void* ws, size_t ws_bytes,
                        dfl2_stream stream) {
  DFL2_TRY(check_select_args(B, L, V, d, r));
  const dfl2::SelectPlan plan = dfl2::select_plan(B, L, d);
  const Ptrs ptrs = {{cand_idx, "cand_idx"}, {cand_val, "cand_val"},
                     {verified_tok, "verified_tok"}, {hidden, "hidden"}, {E, "E"},
                     {W_A, "W_A"}, {W_B, "W_B"}, {W_H, "W_H"}, {scores, "scores"}};
  DFL2_TRY(check_host(ptrs));
  DFL2_TRY(check_ws(ws, ws_bytes, plan.ws_bytes));
  DFL2_TRY(ensure_device());
  DFL2_TRY(check_device(ptrs));
  DFL2_TRY(check_device_ptr(ws, "workspace"));
  cudaError_t e = dfl2::launch_select(plan, cand_idx, cand_val, verified_tok, bf(hidden), bf(E),
                                      bf(W_A), bf(W_B), bf(W_H), V, scores, nullptr, ws,
                                      reinterpret_cast<cudaStream_t>(stream), true);
  if (e != cudaSuccess) return cuda_fail(e, "selector launch");
  return DFL2_OK;
}

// ---- precomputed token tables --------------------------------------------------

size_t dfl2_tables_bytes(int V) {
  if (V < dfl2::kCand) return 0;
  return size_t(V) * dfl2::kRank * 4;
}

dfl2_status dfl2_tables_build(const uint16_t* E, const uint16_t* W_A, const uint16_t* W_B, int V,
                              int d, float* P_A, float* P_B, dfl2_stream stream) {
  DFL2_TRY(check_select_args(1, 1, V, d, dfl2::kRank));
  const Ptrs ptrs = {{E, "E"}, {W_A, "W_A"}, {W_B, "W_B"}, {P_A, "P_A"}, {P_B, "P_B"}};
  DFL2_TRY(check_host(ptrs));
  DFL2_TRY(ensure_device());
  DFL2_TRY(check_device(ptrs));
  cudaError_t e = dfl2::launch_tables_build(bf(E), bf(W_A), bf(W_B), V, d, P_A, P_B,
                                            reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "token table launch");
  return DFL2_OK;
}

dfl2_status dfl2_select_tables(const int32_t* cand_idx, const float* cand_val,
                               const int32_t* verified_tok, const uint16_t* hidden,
                               const uint16_t* W_H, const float* P_A, const float* P_B, int B,
                               int L, int V, int d, int r, float* scores, void* ws,
                               size_t ws_bytes, dfl2_stream stream) {
  DFL2_TRY(check_select_args(B, L, V, d, r));
  const dfl2::SelectPlan plan = dfl2::select_plan(B, L, d);
  const Ptrs ptrs = {{cand_idx, "cand_idx"}, {cand_val, "cand_val"}, {verified_tok, "verified_tok"},
                     {hidden, "hidden"}, {W_H, "W_H"}, {P_A, "P_A"}, {P_B, "P_B"},
                     {scores, "scores"}};
  DFL2_TRY(check_host(ptrs));
  DFL2_TRY(check_ws(ws, ws_bytes, plan.ws_bytes));
  DFL2_TRY(ensure_device());
  DFL2_TRY(check_device(ptrs));
  DFL2_TRY(check_device_ptr(ws, "workspace"));
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = dfl2::launch_gate(plan, bf(hidden), bf(W_H), ws, s, true);
  if (e != cudaSuccess) return cuda_fail(e, "gate projection launch");
  e = dfl2::launch_pair_tables(plan, cand_idx, cand_val, verified_tok, P_A, P_B, V, scores,
                               nullptr, ws, s, true);
  if (e != cudaSuccess) return cuda_fail(e, "pair score launch");
  return DFL2_OK;
}

namespace {
// A side stream and two events per device for each host thread: the table
// tail runs the gate projection beside the top-16 (they share no data).
struct SideStream {
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
thread_local SideStream t_side[64];

cudaError_t side_stream(SideStream*& out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  SideStream& ss = t_side[dev & 63];
  if (!ss.side) {
    e = cudaStreamCreateWithFlags(&ss.side, cudaStreamNonBlocking);
    if (e != cudaSuccess) return e;
    e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
    e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
  }
  out = &ss;
  return cudaSuccess;
}
}  // namespace

dfl2_status dfl2_tail_tables(const void* logits, dfl2_dtype dtype, const int32_t* verified_tok,
                             const uint16_t* hidden, const uint16_t* W_H, const float* P_A,
                             const float* P_B, int B, int L, int V, int d, float temperature,
                             const uint64_t* seeds, uint64_t cycle_offset, int32_t* tokens,
                             int32_t* slots, float* q, int32_t* cand_idx, float* cand_val,
                             float* scores, void* ws, size_t ws_bytes, dfl2_stream stream) {
  DFL2_TRY(check_topk_args(dtype, B, L, V, dfl2::kCand));
  DFL2_TRY(check_select_args(B, L, V, d, dfl2::kRank));
  DFL2_TRY(check_block_len(L));
  DFL2_TRY(check_temperature(temperature));
  const int es = dtype == DFL2_F32 ? 4 : 2;
  const TailLayout t = tail_layout(B, L, V, d, es);
  const Ptrs ptrs = {{logits, "logits"}, {verified_tok, "verified_tok"}, {hidden, "hidden"},
                     {W_H, "W_H"}, {P_A, "P_A"}, {P_B, "P_B"},
                     {tokens, "tokens"}, {slots, "slots", true}, {q, "q", true},
                     {cand_idx, "cand_idx", true}, {cand_val, "cand_val", true},
                     {scores, "scores", true}, {seeds, "seeds", !(temperature > 0.f)}};
  DFL2_TRY(check_host(ptrs));
  DFL2_TRY(check_ws(ws, ws_bytes, t.bytes));
  DFL2_TRY(ensure_device());
  DFL2_TRY(check_device(ptrs));
  DFL2_TRY(check_device_ptr(ws, "workspace"));
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* idx = cand_idx ? cand_idx : reinterpret_cast<int32_t*>(w + t.idx_off);
  float* val = cand_val ? cand_val : reinterpret_cast<float*>(w + t.val_off);
  float* S = scores ? scores : reinterpret_cast<float*>(w + t.scores_off);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  SideStream* ss = nullptr;
  cudaError_t e = side_stream(ss);
  if (e != cudaSuccess) return cuda_fail(e, "side stream");
  // fork: the gate projection on the side stream, the top-16 on the caller's
  if ((e = cudaEventRecord(ss->fork, s)) != cudaSuccess) return cuda_fail(e, "fork");
  if ((e = cudaStreamWaitEvent(ss->side, ss->fork, 0)) != cudaSuccess) return cuda_fail(e, "fork");
  e = dfl2::launch_gate(t.sel, bf(hidden), bf(W_H), w + t.sel_off, ss->side, false);
  if (e != cudaSuccess) return cuda_fail(e, "gate projection launch");
  if ((e = cudaEventRecord(ss->join, ss->side)) != cudaSuccess) return cuda_fail(e, "join");
  e = dfl2::launch_topk(t.topk, logits, idx, val, w + t.topk_off, s, true);
  if (e != cudaSuccess) return cuda_fail(e, "top-16 launch");
  if ((e = cudaStreamWaitEvent(s, ss->join, 0)) != cudaSuccess) return cuda_fail(e, "join");
  const dfl2::WalkFuse wf{temperature, seeds, cycle_offset, tokens, slots, q};
  e = dfl2::launch_pair_tables(t.sel, idx, val, verified_tok, P_A, P_B, V, S, &wf,
                               w + t.sel_off, s, true);
  if (e != cudaSuccess) return cuda_fail(e, "pair score + walk launch");
  return DFL2_OK;
}

// Greedy verification ranks the L+1 target rows with the top-16 kernels; its
// workspace is their top-16 workspace followed by the ranked indices and values.
static dfl2::TopkPlan verify_topk_plan(int B, int L, int V) {
  return dfl2::topk_plan(B * (L + 1), V, 4);
}
static size_t verify_idx_off(const dfl2::TopkPlan& plan) {
  return (plan.ws_bytes + 255) / 256 * 256;
}

size_t dfl2_verify_workspace_size(int B, int L, int V) {
  if (B < 1 || L < 1 || V < dfl2::kCand) return 0;
  const dfl2::TopkPlan plan = verify_topk_plan(B, L, V);
  const size_t rows = size_t(B) * (L + 1);
  return verify_idx_off(plan) + (rows * dfl2::kCand * 4 + 255) / 256 * 256 + rows * dfl2::kCand * 4;
}

dfl2_status dfl2_verify(const float* p, const int32_t* tokens, const int32_t* slots,
                        const float* q, const int32_t* cand_idx, int B, int L, int V, int greedy,
                        const uint64_t* seeds, uint64_t cycle_offset, int32_t* n_accepted,
                        int32_t* out_tokens, void* ws, size_t ws_bytes, dfl2_stream stream) {
  DFL2_TRY(check_shape(B, L));
  DFL2_TRY(check_block_len(L));
  if (V < dfl2::kCand) return fail(DFL2_ERR_INVALID_ARG, "V=%d < 16", V);
  if (V % 4 != 0) return fail(DFL2_ERR_UNSUPPORTED, "V=%d: rows of p must be a multiple of 16 bytes", V);
  if (V > 524288) return fail(DFL2_ERR_UNSUPPORTED, "V=%d: verification supports V <= 524288", V);
  const bool sampling = greedy == 0;
  const Ptrs ptrs = {{p, "p"}, {tokens, "tokens"}, {slots, "slots", !sampling},
                     {q, "q", !sampling}, {cand_idx, "cand_idx", !sampling},
                     {seeds, "seeds", !sampling}, {n_accepted, "n_accepted"},
                     {out_tokens, "out_tokens"}};
  DFL2_TRY(check_host(ptrs));
  const dfl2::TopkPlan plan = verify_topk_plan(B, L, V);
  if (!sampling) DFL2_TRY(check_ws(ws, ws_bytes, dfl2_verify_workspace_size(B, L, V)));
  DFL2_TRY(ensure_device());
  DFL2_TRY(check_device(ptrs));
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (sampling) {
    cudaError_t e = dfl2::launch_verify_sample(p, tokens, slots, q, cand_idx, B, L, V, seeds,
                                               cycle_offset, n_accepted, out_tokens, s);
    if (e != cudaSuccess) return cuda_fail(e, "verification launch");
    return DFL2_OK;
  }
  DFL2_TRY(check_device_ptr(ws, "workspace"));
  uint8_t* w = static_cast<uint8_t*>(ws);
  const size_t rows = size_t(B) * (L + 1);
  int32_t* top_idx = reinterpret_cast<int32_t*>(w + verify_idx_off(plan));
  float* top_val = reinterpret_cast<float*>(w + verify_idx_off(plan) +
                                            (rows * dfl2::kCand * 4 + 255) / 256 * 256);
  cudaError_t e = dfl2::launch_topk(plan, p, top_idx, top_val, ws, s, true);
  if (e != cudaSuccess) return cuda_fail(e, "verification top-16 launch");
  e = dfl2::launch_verify_greedy(tokens, top_idx, B, L, n_accepted, out_tokens, s);
  if (e != cudaSuccess) return cuda_fail(e, "verification launch");
  return DFL2_OK;
}

dfl2_status dfl2_walk(const float* scores, const int32_t* cand_idx, int B, int L,
                      float temperature, const uint64_t* seeds, uint64_t cycle_offset,
                      int32_t* tokens, int32_t* slots, float* q, dfl2_stream stream) {
  DFL2_TRY(check_shape(B, L));
  DFL2_TRY(check_block_len(L));
  DFL2_TRY(check_temperature(temperature));
  const Ptrs ptrs = {{scores, "scores"}, {cand_idx, "cand_idx"}, {tokens, "tokens"},
                     {slots, "slots", true}, {q, "q", true},
                     {seeds, "seeds", !(temperature > 0.f)}};
  DFL2_TRY(check_host(ptrs));
  DFL2_TRY(ensure_device());
  DFL2_TRY(check_device(ptrs));
  cudaError_t e = dfl2::launch_walk(scores, cand_idx, B, L, temperature, seeds, cycle_offset,
                                    tokens, slots, q, reinterpret_cast<cudaStream_t>(stream),
                                    true);
  if (e != cudaSuccess) return cuda_fail(e, "walk launch");
  return DFL2_OK;
}

namespace {
dfl2_status conv2_common(const uint16_t* x, const uint16_t* x_prev, const float* base,
                         const uint16_t* W_c, int B, int L, int d, uint16_t* y, void* ws,
                         size_t ws_bytes, bool with_ws, dfl2_stream stream) {
  DFL2_TRY(check_shape(B, L));
  if (d < dfl2::kGroup || d % dfl2::kGroup != 0 || d > 65536)
    return fail(DFL2_ERR_UNSUPPORTED, "d=%d: the conv needs a multiple of 16 up to 65536", d);
  const Ptrs ptrs = {{x, "x"}, {x_prev, "x_prev"}, {base, "base"}, {W_c, "W_c"}, {y, "y"}};
  DFL2_TRY(check_host(ptrs));
  const size_t ybytes = size_t(B) * L * d * 2;
  if (overlaps(y, ybytes, x, ybytes) || overlaps(y, ybytes, x_prev, size_t(B) * d * 2))
    return fail(DFL2_ERR_INVALID_ARG, "y overlaps x or x_prev");
  DFL2_TRY(ensure_device());
  DFL2_TRY(check_device(ptrs));
  void* use_ws = nullptr;
  if (with_ws) {
    const size_t need = dfl2::conv2_ws_bytes(B, L, d);
    if (need > 0) {
      DFL2_TRY(check_ws(ws, ws_bytes, need));
      const Ptrs wp = {{ws, "ws"}};
      DFL2_TRY(check_host(wp));
      DFL2_TRY(check_device(wp));
      if (overlaps(ws, need, y, ybytes) || overlaps(ws, need, x, ybytes))
        return fail(DFL2_ERR_INVALID_ARG, "ws overlaps x or y");
      use_ws = ws;
    }
  }
  cudaError_t e = dfl2::launch_conv2(bf(x), bf(x_prev), base, bf(W_c), B, L, d,
                                     reinterpret_cast<__nv_bfloat16*>(y), use_ws,
                                     reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "conv launch");
  return DFL2_OK;
}
}  // namespace

dfl2_status dfl2_conv2(const uint16_t* x, const uint16_t* x_prev, const float* base,
                       const uint16_t* W_c, int B, int L, int d, uint16_t* y,
                       dfl2_stream stream) {
  return conv2_common(x, x_prev, base, W_c, B, L, d, y, nullptr, 0, false, stream);
}

size_t dfl2_conv2_workspace_size(int B, int L, int d) {
  if (B < 1 || L < 1 || d < dfl2::kGroup || d % dfl2::kGroup != 0 || d > 65536) return 0;
  if (ensure_device() != DFL2_OK) return 0;
  return dfl2::conv2_ws_bytes(B, L, d);
}

dfl2_status dfl2_conv2_ws(const uint16_t* x, const uint16_t* x_prev, const float* base,
                          const uint16_t* W_c, int B, int L, int d, uint16_t* y, void* ws,
                          size_t ws_bytes, dfl2_stream stream) {
  return conv2_common(x, x_prev, base, W_c, B, L, d, y, ws, ws_bytes, true, stream);
}

size_t dfl2_tail_workspace_size(int B, int L, int V, int d) {
  if (B < 1 || L < 1 || V < dfl2::kCand || d < 1) return 0;
  return tail_layout(B, L, V, d, 4).bytes;
}

dfl2_status dfl2_tail(const void* logits, dfl2_dtype dtype, const int32_t* verified_tok,
                      const uint16_t* hidden, const uint16_t* E, const uint16_t* W_A,
                      const uint16_t* W_B, const uint16_t* W_H, int B, int L, int V, int d,
                      float temperature, const uint64_t* seeds, uint64_t cycle_offset,
                      int32_t* tokens, int32_t* slots, float* q, int32_t* cand_idx,
                      float* cand_val, float* scores, void* ws, size_t ws_bytes,
                      dfl2_stream stream) {
  DFL2_TRY(check_topk_args(dtype, B, L, V, dfl2::kCand));
  DFL2_TRY(check_select_args(B, L, V, d, dfl2::kRank));
  DFL2_TRY(check_block_len(L));
  DFL2_TRY(check_temperature(temperature));
  const int es = dtype == DFL2_F32 ? 4 : 2;
  const TailLayout t = tail_layout(B, L, V, d, es);
  const Ptrs ptrs = {{logits, "logits"}, {verified_tok, "verified_tok"}, {hidden, "hidden"},
                     {E, "E"}, {W_A, "W_A"}, {W_B, "W_B"}, {W_H, "W_H"},
                     {tokens, "tokens"}, {slots, "slots", true}, {q, "q", true},
                     {cand_idx, "cand_idx", true}, {cand_val, "cand_val", true},
                     {scores, "scores", true}, {seeds, "seeds", !(temperature > 0.f)}};
  DFL2_TRY(check_host(ptrs));
  DFL2_TRY(check_ws(ws, ws_bytes, t.bytes));
  DFL2_TRY(ensure_device());
  DFL2_TRY(check_device(ptrs));
  DFL2_TRY(check_device_ptr(ws, "workspace"));
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* idx = cand_idx ? cand_idx : reinterpret_cast<int32_t*>(w + t.idx_off);
  float* val = cand_val ? cand_val : reinterpret_cast<float*>(w + t.val_off);
  float* S = scores ? scores : reinterpret_cast<float*>(w + t.scores_off);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = dfl2::launch_topk(t.topk, logits, idx, val, w + t.topk_off, s, true);
  if (e != cudaSuccess) return cuda_fail(e, "top-16 launch");
  const dfl2::WalkFuse wf{temperature, seeds, cycle_offset, tokens, slots, q};
  e = dfl2::launch_select(t.sel, idx, val, verified_tok, bf(hidden), bf(E), bf(W_A), bf(W_B),
                          bf(W_H), V, S, &wf, w + t.sel_off, s, true);
  if (e != cudaSuccess) return cuda_fail(e, "selector + walk launch");
  return DFL2_OK;
}

}  // extern "C"
