/*
 * dfl2: the DFlash 2 draft tail on one GB300 (sm_103a), as a C ABI.
 *
 * The tail runs once per draft-verify cycle, after the drafter's one-pass
 * forward and before the target's verify pass:
 *
 *   logits U [B,L,V] --top-16--> candidates --pair scores S_t(a,b)--> walk --> draft tokens
 *
 * plus the two-tap dynamic conv that the drafter applies before and after each
 * attention and feed-forward sublayer (5 layers x 4 insertion points).
 *
 * Sources (page title, section):
 *   [SEL]  "DFlash 2: Keep Drafting Parallel" (papercache.org digest of the
 *          Inco AI post), 方法细节 > 轻量级路径选择器 (Lightweight Path Selector):
 *          top-16 candidates per position, the pair-score equation
 *          S_t(a,b) = U_t(b) + <A(a) ⊙ H(h_t), B(b)>, and the walk over the
 *          precomputed scores starting from the last verified token.
 *   [CONV] same page, 方法细节 > 轻量级局部卷积 (Lightweight Local Convolution):
 *          Conv_k(x)_t = k_{t,0} ⊙ x_t + k_{t,1} ⊙ x_{t-1}, a learned base
 *          kernel plus a correction from the hidden state shared by every 16
 *          channels, and position 0 reading the last verified token.
 *   [TAB2] same page, Table 2 (+2.0M selector parameters) and the conv's
 *          "+16.5M" paragraph; these fix A(a) = W_A E[a], B(b) = W_B E[b],
 *          H(h) = sigmoid(W_H h) with W_* in R^{256 x d}, and a correction map
 *          of 2 d/16 rows for both taps.
 *   [WALK] "DFlash 2: The Drafter Stopped Guessing Alone" (rohitghumare.com),
 *          "Selection beats correction": greedy follows the best successor;
 *          sampling draws from the same scores.
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE memory owned by the caller, row-major and
 *     contiguous, 16-byte aligned.  bf16 tensors are passed as uint16_t bit
 *     patterns.  Nothing is allocated by the library; scratch memory is a
 *     caller-provided workspace of at least *_workspace_size() bytes.
 *   - Work is enqueued on the caller's stream; no call synchronises the host
 *     (except dfl2_device_error, which says so).
 *   - Arguments are validated on the host before anything is launched; a bad
 *     argument returns a status and launches nothing.  Launch failures return
 *     DFL2_ERR_CUDA.  No call throws, aborts or prints.  dfl2_last_error()
 *     returns a thread-local message for the last failing call.
 *   - Fixed method sizes: k = 16 candidates, r = 256 selector rank; d must be a
 *     multiple of 16; V >= 16 (any V: logits rows need not start on 16 bytes),
 *     L >= 1, B >= 1.  The entry points of the NEXT rows keep narrower limits,
 *     stated at each (dfl2_verify: V % 4 == 0; dfl2_lmhead_topk: d % 8 == 0).
 *   - Every wait inside a kernel is bounded.  A wait that runs out (about 2 s
 *     of SM clock) records a code in a per-device error word
 *     (dfl2_device_error) and the kernel carries on without the data it
 *     waited for, so that launch's outputs are undefined; it still ends and
 *     leaves the context usable.  Once the error word is set, every other wait
 *     that has lasted about 0.5 ms gives up too, so a launch whose pipeline
 *     stalls ends within a few seconds, not one full timeout per wait.
 *   - Workspaces must be zero-filled once before their first use (for example
 *     with dfl2_workspace_init); the library keeps them valid afterwards.
 */
#ifndef DFL2_H
#define DFL2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (NULL = the legacy default stream). */
typedef struct CUstream_st* dfl2_stream;

typedef enum dfl2_status {
  DFL2_OK = 0,
  DFL2_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, T < 0 ... */
  DFL2_ERR_UNSUPPORTED = 2, /* k != 16, r != 256, d or V not of a supported multiple */
  DFL2_ERR_WORKSPACE = 3,   /* workspace missing or smaller than *_workspace_size() */
  DFL2_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  DFL2_ERR_TIMEOUT = 5      /* a bounded in-kernel wait ran out (see dfl2_device_error) */
} dfl2_status;

typedef enum dfl2_dtype { DFL2_F32 = 0, DFL2_BF16 = 1 } dfl2_dtype;

/* Library version string, e.g. "dfl2 0.1 sm_103a". */
const char* dfl2_version(void);

/* Copies the calling thread's last error message (NUL-terminated, truncated to
 * len) and returns its full length. */
size_t dfl2_last_error(char* buf, size_t len);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t dfl2_launch_count(void);

/* Engine of the projection GEMM (A = W_A E[a], B = W_B E[b], the gate's W_H h)
 * on its split-K path, the one that runs when the rows are few (batch 1 on the
 * drafter shapes: 241 + 256 gathered rows, 16 hidden rows); the batched path
 * always uses tcgen05.
 *   DFL2_PROJ_TENSOR (default): tcgen05 MMAs into a tensor-memory accumulator.
 *   DFL2_PROJ_WARP: the warp-level engine, each warp owning 32 output columns of
 *     its CTA's rows and computing them with mma.sync (m16n8k16, bf16 in, fp32
 *     accumulate) from the same shared-memory tiles.  It applies where a CTA
 *     holds 128 output columns (the batch-1 plans); elsewhere the tensor engine
 *     runs.
 * Process-wide (every device and thread), read when a call is enqueued; a
 * captured CUDA graph keeps the engine it was captured with.  Returns the
 * previous setting; an unknown value returns -1 and changes nothing. */
#define DFL2_PROJ_TENSOR 0
#define DFL2_PROJ_WARP 1
int dfl2_set_projection_engine(int engine);

/* Zero-fills a workspace on the stream (one cudaMemsetAsync). */
dfl2_status dfl2_workspace_init(void* ws, size_t ws_bytes, dfl2_stream stream);

/* Reads, and if clear != 0 resets, the current device's error word.  0 means no
 * kernel recorded a failed wait.  SYNCHRONISES the current device. */
dfl2_status dfl2_device_error(uint32_t* code, int clear);

/* ------------------------------------------------------------------ top-16
 * [SEL] "每个位置提取并保留 Top-16": for each of the B*L rows of logits [B,L,V]
 * (dtype float32 or bf16), the k = 16 largest logits, ordered by value
 * descending and then index ascending (-0.0 ties +0.0; NaN is not supported).
 * Writes cand_idx int32 [B,L,16] and cand_val float32 [B,L,16] (the logit,
 * widened exactly; a zero is written as +0.0).  ws: dfl2_topk_workspace_size
 * bytes (split-row partial lists and per-row tickets).
 */
size_t dfl2_topk_workspace_size(int B, int L, int V);
dfl2_status dfl2_topk(const void* logits, dfl2_dtype dtype, int B, int L, int V, int k,
                      int32_t* cand_idx, float* cand_val, void* ws, size_t ws_bytes,
                      dfl2_stream stream);

/* ------------------------------------------------------------------ LM head + top-16
 * The logits the top-16 step reads are the drafter's LM head applied to its
 * last hidden state ("DFlash 2: Keep Drafting Parallel", 方法细节 >
 * 轻量级路径选择器: U_t(.) is the drafter's own logit at position t).  This
 * entry point computes U_t(v) = sum_c hidden[t, c] * W_lm[v, c] (bf16 inputs,
 * float32 accumulation on the tensor cores) and keeps only the 16 largest per
 * row, inside the GEMM's epilogue: the [B*L, V] logits are never written.
 *   hidden  bf16 [B, L, d] row-major, device, 16-byte aligned.
 *   W_lm    bf16 [V, d] row-major, device, 16-byte aligned (a tied embedding
 *           table E may be passed).
 *   d       a multiple of 8 (16-byte rows); any V >= 16, any B*L >= 1.
 *   k       must be 16.
 *   Writes cand_idx int32 [B,L,16] and cand_val float32 [B,L,16] in the order
 *   of dfl2_topk (value descending, index ascending).  cand_val is the float32
 *   accumulator, so rows whose 16th and 17th logits differ by less than the
 *   accumulation error may pick either; with inputs whose partial sums are
 *   exact in float32 (e.g. small integers) the result equals dfl2_topk on the
 *   exact logits.  NaN/Inf inputs are not supported.
 *   ws: dfl2_lmhead_topk_workspace_size bytes (partial lists, not needing
 *   initialisation).  Two kernel launches on `stream`.
 * Errors: DFL2_ERR_INVALID_ARG (NULL/unaligned/host pointers, V < 16, B or L
 * < 1), DFL2_ERR_UNSUPPORTED (k != 16, d % 8 != 0), DFL2_ERR_WORKSPACE.
 */
size_t dfl2_lmhead_topk_workspace_size(int B, int L, int V, int d);
dfl2_status dfl2_lmhead_topk(const uint16_t* hidden, const uint16_t* W_lm, int B, int L, int V,
                             int d, int k, int32_t* cand_idx, float* cand_val, void* ws,
                             size_t ws_bytes, dfl2_stream stream);

/* ------------------------------------------------------------------ top-16, no allocation
 * No counterpart on the pages: a convenience of this library.  The same result
 * as dfl2_topk, for callers that cannot allocate device memory, such as serving
 * engines that reserve the GPU's memory for their own pool at start-up and
 * forbid later cudaMalloc, or plug-ins that get only input and output pointers.
 * The scratch dfl2_topk keeps in its workspace lives instead in a fixed 4 MiB
 * array of library-owned device memory (held on every GPU that loads the
 * library until the process exits); problems whose dfl2_topk_workspace_size
 * exceeds 4 MiB return DFL2_ERR_WORKSPACE without launching.  The first call on
 * a device looks up that array's address; make it before any stream capture.
 * All calls share the array, so calls whose kernels overlap on the GPU (other
 * streams or threads) race; calls in order on one stream are safe.
 */
dfl2_status dfl2_topk_noalloc(const void* logits, dfl2_dtype dtype, int B, int L, int V, int k,
                              int32_t* cand_idx, float* cand_val, dfl2_stream stream);

/* ------------------------------------------------------------------ pair scores
 * [SEL equation], [TAB2] reading:
 *   A(a) = W_A E[a], B(b) = W_B E[b], H(h_t) = sigmoid(W_H h_t)   (W_* [256,d], E [V,d])
 *   S[b,t,i,j] = cand_val[b,t,j] + sum_q A_q(a_i) H_q(h_{b,t}) B_q(cand_idx[b,t,j])
 * where a_i = cand_idx[b,t-1,i] for t >= 1, and for t = 0 only row i = 0 is
 * defined, with a_0 = verified_tok[b] (rows 1..15 of t = 0 are -inf).
 * hidden [B,L,d] bf16 is the drafter's final hidden state at each position.
 * scores float32 [B,L,16,16]; projections accumulate in float32.
 * ws: dfl2_select_workspace_size bytes (projected candidates and gates).
 */
size_t dfl2_select_workspace_size(int B, int L, int d);
dfl2_status dfl2_select(const int32_t* cand_idx, const float* cand_val,
                        const int32_t* verified_tok, const uint16_t* hidden, const uint16_t* E,
                        const uint16_t* W_A, const uint16_t* W_B, const uint16_t* W_H, int B,
                        int L, int V, int d, int r, float* scores, void* ws, size_t ws_bytes,
                        dfl2_stream stream);

/* ------------------------------------------------------------------ walk
 * [SEL "全并行打分与低延迟路径步进"], [WALK].  One sequential pass per
 * sequence over scores [B,L,16,16]: prev starts at row 0 of position 0 (the
 * verified token); at each t the step reads row prev of S[b,t] and picks
 *   temperature == 0: the lowest slot holding the row maximum (greedy);
 *   temperature  > 0: p_j = exp((S_j - max)/T), Z = sum_j p_j, u uniform in
 *                     [0,1), the first j with u Z < p_0 + ... + p_j.
 * u = (w >> 8) * 2^-24, w = word 0 of Philox4x32-10 (Salmon et al., SC'11)
 * with counter (t, lo32(cycle_offset), hi32(cycle_offset), 0) and key
 * (lo32(seeds[b]), hi32(seeds[b])).  Then prev = j*.
 * Writes tokens [B,L] = cand_idx[b,t,j*]; slots [B,L] = j* (nullable);
 * q [B,L,16] = p/Z, the draft distribution the verifier's rejection sampling
 * needs (one-hot when greedy; nullable).  seeds: device uint64 [B], may be NULL
 * when temperature == 0.
 */
dfl2_status dfl2_walk(const float* scores, const int32_t* cand_idx, int B, int L,
                      float temperature, const uint64_t* seeds, uint64_t cycle_offset,
                      int32_t* tokens, int32_t* slots, float* q, dfl2_stream stream);

/* ------------------------------------------------------------------ conv
 * [CONV equation], [TAB2] reading.  G = d/16 correction groups.
 *   corr[b,t,j,g] = sum_c W_c[j*G + g, c] x[b,t,c]          (j = tap 0, 1)
 *   k_j[c]        = base[j,c] + corr[b,t,j,c/16]
 *   y[b,t,c]      = k_0[c] x[b,t,c] + k_1[c] x[b,t-1,c],   x[b,-1,:] = x_prev[b,:]
 * x, y [B,L,d] bf16; x_prev [B,d] bf16 (the verified token's representation
 * at this insertion point); base float32 [2,d]; W_c bf16 [2G, d] with rows
 * [tap-0 groups; tap-1 groups].  float32 arithmetic, y rounded once to bf16
 * (nearest even).  y must not overlap x or x_prev.  No workspace.
 * base and W_c are weights: the call may read them before it waits for the
 * work queued ahead of it on `stream` (so that loading them overlaps that
 * work), hence no kernel still pending on `stream` may write them (set them,
 * e.g. with a copy, and let that copy complete or order it on another stream
 * that the caller synchronises, before the call).  x and x_prev are read only
 * after the earlier work on `stream` has finished.
 */
dfl2_status dfl2_conv2(const uint16_t* x, const uint16_t* x_prev, const float* base,
                       const uint16_t* W_c, int B, int L, int d, uint16_t* y,
                       dfl2_stream stream);

/* The same conv with a workspace.  With many positions (B*L > 64, d a multiple
 * of 64 and at least 512) the correction product is split over K across a
 * thread-block cluster and the partial products are exchanged through the
 * workspace, which lets the call spread over the whole GPU; otherwise the
 * call is the same as dfl2_conv2.  y is the same as dfl2_conv2's up to the
 * order of the float32 additions (each partial sum is added in a fixed
 * order, so a given shape always gives the same bits).
 * dfl2_conv2_workspace_size: bytes of device memory the call needs for this
 * shape on the current device (0: none, ws may be NULL); 0 also for an
 * unsupported shape or when no device is usable.
 * ws: device memory owned by the caller, at least that many bytes, not
 * overlapping x or y; its contents are scratch (no state is kept between
 * calls), and two calls that may run at the same time need separate
 * workspaces.  Errors: DFL2_ERR_WORKSPACE if ws is NULL or ws_bytes is too
 * small when bytes are needed; the argument errors of dfl2_conv2.
 */
size_t dfl2_conv2_workspace_size(int B, int L, int d);
dfl2_status dfl2_conv2_ws(const uint16_t* x, const uint16_t* x_prev, const float* base,
                          const uint16_t* W_c, int B, int L, int d, uint16_t* y, void* ws,
                          size_t ws_bytes, dfl2_stream stream);

/* ------------------------------------------------------------------ fused tail
 * top-16 -> pair scores -> walk in one call on one stream, with no host
 * synchronisation: the same results as dfl2_topk, dfl2_select and dfl2_walk
 * called in sequence.  cand_idx, cand_val, scores, slots and q are optional
 * outputs (NULL: kept in the workspace / not written).
 */
size_t dfl2_tail_workspace_size(int B, int L, int V, int d);
dfl2_status dfl2_tail(const void* logits, dfl2_dtype dtype, const int32_t* verified_tok,
                      const uint16_t* hidden, const uint16_t* E, const uint16_t* W_A,
                      const uint16_t* W_B, const uint16_t* W_H, int B, int L, int V, int d,
                      float temperature, const uint64_t* seeds, uint64_t cycle_offset,
                      int32_t* tokens, int32_t* slots, float* q, int32_t* cand_idx,
                      float* cand_val, float* scores, void* ws, size_t ws_bytes,
                      dfl2_stream stream);

/* ---------------------------------------------------------------------------
 * Precomputed token tables (a variant of the projections; the pages compute
 * A(a) = W_A E[a] and B(b) = W_B E[b] per candidate, "DFlash 2: Keep Drafting
 * Parallel", 方法细节 > 轻量级路径选择器, the definitions under the pair-score
 * equation).  Both maps are linear in E[.], so P_A = E W_A^T and P_B = E W_B^T,
 * built once per set of weights, give the same values per token (float32, the
 * accumulation order of the GEMM aside), and the per-cycle work shrinks to
 * gathering 1 KB rows instead of d-wide embedding rows.
 *
 * dfl2_tables_bytes(V): bytes of ONE table (float32 [V, 256]).
 * dfl2_tables_build: P_A, P_B (caller-owned device memory, dfl2_tables_bytes(V)
 *   each) from E [V, d] and W_A, W_B [256, d] (bf16, device).  d % 64 == 0.
 *   One tcgen05 GEMM launch; rebuild whenever E, W_A or W_B change.
 * dfl2_select_tables: as dfl2_select, with A(.) and B(.) read from the tables
 *   (E, W_A, W_B are not needed); the gate H = sigmoid(W_H h) is still computed
 *   per call.  Workspace: dfl2_select_workspace_size(B, L, d).
 * dfl2_tail_tables: as dfl2_tail with the tables.  The gate projection runs on
 *   a library-owned side stream (one per device and host thread), forked from
 *   and joined back to `stream` with events, beside the top-16; under CUDA
 *   graph capture the fork and join become graph edges.  Workspace:
 *   dfl2_tail_workspace_size(B, L, V, d).
 * Errors as for dfl2_select / dfl2_tail; a token outside [0, V) is recorded in
 * the device error word and read as row 0.
 * ------------------------------------------------------------------------- */
size_t dfl2_tables_bytes(int V);
dfl2_status dfl2_tables_build(const uint16_t* E, const uint16_t* W_A, const uint16_t* W_B, int V,
                              int d, float* P_A, float* P_B, dfl2_stream stream);
dfl2_status dfl2_select_tables(const int32_t* cand_idx, const float* cand_val,
                               const int32_t* verified_tok, const uint16_t* hidden,
                               const uint16_t* W_H, const float* P_A, const float* P_B, int B,
                               int L, int V, int d, int r, float* scores, void* ws,
                               size_t ws_bytes, dfl2_stream stream);
dfl2_status dfl2_tail_tables(const void* logits, dfl2_dtype dtype, const int32_t* verified_tok,
                             const uint16_t* hidden, const uint16_t* W_H, const float* P_A,
                             const float* P_B, int B, int L, int V, int d, float temperature,
                             const uint64_t* seeds, uint64_t cycle_offset, int32_t* tokens,
                             int32_t* slots, float* q, int32_t* cand_idx, float* cand_val,
                             float* scores, void* ws, size_t ws_bytes, dfl2_stream stream);

/* ---------------------------------------------------------------------------
 * dfl2_verify: verification of the drafted block against the target's
 * distributions, the step after the walk ("DFlash 2: Keep Drafting Parallel",
 * 方法细节 > 轻量级路径选择器, "全并行打分与低延迟路径步进": lossless rejection
 * sampling recovers the target's distribution; "DFlash 2: The Drafter Stopped
 * Guessing Alone", "One pass to draft, one pass to verify": the accepted prefix
 * is kept, the first miss is replaced by the target's own choice and the rest
 * dropped).  The sampling rule is the published speculative-sampling step
 * (Leviathan et al., ICML 2023; Chen et al., 2023).
 *
 *   p          [B, L+1, V] float32, device: the target's next-token
 *              probabilities; row t < L follows the verified token and the first
 *              t drafted tokens, row L follows the whole block.
 *   tokens     [B, L] int32: the drafted tokens (dfl2_walk / dfl2_tail).
 *   greedy     non-zero: keep tokens[t] while it is the lowest index holding the
 *              maximum of row t; the first miss is replaced by that index; when
 *              all L match, row L's argmax is appended.
 *              zero (sampling): with x = tokens[t] and q(x) = q[b,t,slots[t]],
 *              keep x iff u0 * q(x) < p_t(x); otherwise draw the replacement
 *              from max(0, p_t - q_t) (q_t is zero off cand_idx[b,t,:]): the
 *              first index, in order, whose running sum exceeds u1 * total (the
 *              last index with mass if rounding leaves none; p_t itself if the
 *              residual is zero).  When all L are kept, one token is drawn from
 *              row L the same way with u1.  u0, u1 = words 0 and 1 of
 *              Philox4x32-10 with counter (t, lo32(cycle), hi32(cycle), 1) and
 *              key = seeds[b], each (w >> 8) * 2^-24.
 *   slots, q, cand_idx, seeds: the walk's outputs [B,L], [B,L,16], the top-16
 *              candidates [B,L,16] and the per-sequence keys [B]; unused (may
 *              be NULL) when greedy.
 *   n_accepted [B] int32: drafted tokens kept (0..L).
 *   out_tokens [B, L+1] int32: the kept tokens, then the replacement or
 *              appended token, then -1.
 *   ws, ws_bytes: dfl2_verify_workspace_size(B, L, V) bytes of device memory
 *              (used by greedy; sampling may pass NULL and 0).
 * Constraints: L <= 128, 16 <= V <= 524288, V % 4 == 0.  Decisions are exact
 * (double precision); the replacement draw sums the row in single precision
 * within 512-element tiles and in double across tiles, so it can differ from
 * an exact sum only when u1 * total lies within rounding of a boundary.
 * Errors: DFL2_ERR_INVALID_ARG / UNSUPPORTED before any launch; a token or
 * slot out of range is recorded in the device error word (dfl2_device_error).
 * ------------------------------------------------------------------------- */
size_t dfl2_verify_workspace_size(int B, int L, int V);
dfl2_status dfl2_verify(const float* p, const int32_t* tokens, const int32_t* slots,
                        const float* q, const int32_t* cand_idx, int B, int L, int V, int greedy,
                        const uint64_t* seeds, uint64_t cycle_offset, int32_t* n_accepted,
                        int32_t* out_tokens, void* ws, size_t ws_bytes, dfl2_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* DFL2_H */
