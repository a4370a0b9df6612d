/*
 * dfl2 oracle: TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, obviously correct CPU restatement of the DFlash 2 draft tail,
 * evaluated in double precision.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table
 * or helper with the CUDA library; the two meet only through seeded inputs.
 *
 * Sources (page title, section):
 *   [SEL]  "DFlash 2: Keep Drafting Parallel" (papercache.org digest of the
 *          Inco AI post), 方法细节 > 轻量级路径选择器: the adjacent-pair score
 *          S_t(a,b) = U_t(b) + <A(a) ⊙ H(h_t), B(b)>, the top-16 candidates per
 *          position, and the walk from the last verified token (greedy: best
 *          successor; sampling: draw from the score distribution).
 *   [CONV] same page, 方法细节 > 轻量级局部卷积: Conv_k(x)_t = k_{t,0}⊙x_t +
 *          k_{t,1}⊙x_{t-1}; base kernel plus a hidden-state correction shared by
 *          every 16 channels; position 0 reads the last verified token.
 *   [TAB2] same page, Table 2 (selector: +2.0M parameters) and the conv
 *          paragraph "结构特性与衰减消除验证" (+16.5M parameters over 5 layers).
 *   [WALK] "DFlash 2: The Drafter Stopped Guessing Alone" (rohitghumare.com),
 *          section "Selection beats correction": start from the last verified
 *          token, follow the best successor; under sampling draw from the same
 *          scores.
 *   [PHILOX] Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
 *          1, 2, 3", SC'11: the Philox4x32-10 bijection.
 *   [VERIFY] [SEL] "全并行打分与低延迟路径步进" (sampling recovers the target's
 *          distribution by lossless rejection sampling) and [WALK] "One pass to
 *          draft, one pass to verify" (the accepted prefix is kept, the first
 *          miss is replaced by the target's own choice, the rest is dropped;
 *          greedy output equals the target's own).  The rejection rule is the
 *          published speculative-sampling step: Leviathan, Kalman, Matias,
 *          "Fast Inference from Transformers via Speculative Decoding", ICML
 *          2023, and Chen et al., "Accelerating Large Language Model Decoding
 *          with Speculative Sampling", 2023.
 *
 * Readings where the pages are silent are stated at each function.
 * bf16 arguments are raw 16-bit patterns (uint16_t); bf16 -> double is exact.
 */
#ifndef DFL2_ORACLE_H
#define DFL2_ORACLE_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 0 = logits are float32, 1 = logits are bf16 bit patterns. */
#define ORACLE_F32 0
#define ORACLE_BF16 1

/* Number of OpenMP threads the oracle uses (<= 0: leave the runtime default). */
void oracle_set_threads(int n);
int oracle_get_threads(void);

/* Philox4x32-10 [PHILOX]: out = bijection(ctr) under key. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* The uniform the sampling walk draws at step t of a cycle (reading, since the
 * pages only say "seeded"): word 0 of Philox4x32-10 with counter
 * (t, lo32(cycle), hi32(cycle), 0) and key (lo32(seed), hi32(seed)),
 * u = (word >> 8) * 2^-24 in [0, 1). */
double oracle_walk_uniform(uint64_t seed, uint64_t cycle, int t);

/* Top-k per row [SEL, "每个位置提取并保留 Top-16"]: rows = B*L, each of V logits.
 * Full sort by (value descending, index ascending); -0.0 ties +0.0.
 * Writes idx [rows,k] and val [rows,k] (the logit, exact).  Returns 0, or -1 on
 * a bad argument. */
int oracle_topk(const void* logits, int dtype, int B, int L, int V, int k,
                int32_t* idx, float* val);

/* Projections [SEL]: A(tok) = W_A E[tok], B(tok) = W_B E[tok] (W [r,d] row
 * major, E [V,d]), H(h) = sigmoid(W_H h).  One row each, written as doubles. */
void oracle_proj_token(const uint16_t* E, const uint16_t* W, int d, int r,
                       int32_t tok, double* out /*[r]*/);
void oracle_gate(const uint16_t* W_H, const uint16_t* h, int d, int r, double* out /*[r]*/);

/* Pair scores [SEL equation].  For t >= 1, a ranges over cand_idx[b,t-1,:]
 * (row i = slot of the predecessor); for t = 0 only row 0 is defined and uses
 * the verified token; rows 1..15 of t = 0 are -inf.  b ranges over
 * cand_idx[b,t,:] (column j).  scores [B,L,16,16].  U_t(b) is the candidate's
 * raw logit cand_val[b,t,j].  Returns 0, or -1 on a bad argument. */
int oracle_select(const int32_t* cand_idx, const float* cand_val, const int32_t* verified,
                  const uint16_t* hidden, const uint16_t* E, const uint16_t* W_A,
                  const uint16_t* W_B, const uint16_t* W_H, int B, int L, int V, int d,
                  int r, double* scores);

/* The walk [SEL "全并行打分与低延迟路径步进"; WALK].  prev starts at row 0 of
 * t = 0 (the verified token).  Greedy (T == 0): the lowest slot holding the
 * row maximum.  Sampling (T > 0): p_j = exp((S_j - max)/T), Z = sum in slot
 * order, j* = first j with u*Z < p_0 + ... + p_j (u from oracle_walk_uniform),
 * else the last j with p_j > 0.  Writes tokens [B,L] = cand_idx[b,t,j*],
 * slots [B,L] (nullable) and q [B,L,16] = p/Z (one-hot when greedy; nullable).
 * Returns 0, or -1 on a bad argument. */
int oracle_walk(const double* scores, const int32_t* cand_idx, int B, int L, double T,
                const uint64_t* seeds, uint64_t cycle, int32_t* tokens, int32_t* slots,
                double* q);

/* Two-tap dynamic depthwise conv [CONV equation].  G = d/16 groups.
 * corr_{t,j,g} = sum_c W_c[j*G+g, c] * x_t[c]; k_{t,j,c} = base[j,c] +
 * corr_{t,j,c/16}; y_t = k_{t,0} x_t + k_{t,1} x_{t-1}, x_{-1} = x_prev[b].
 * y_exact [B,L,d] double (nullable); y_bf16 [B,L,d] rounded once, to nearest
 * even (nullable).  Returns 0, or -1 on a bad argument. */
int oracle_conv2(const uint16_t* x, const uint16_t* x_prev, const float* base,
                 const uint16_t* W_c, int B, int L, int d, double* y_exact, uint16_t* y_bf16);

/* Top-k of the LM head's logits [SEL "每个位置提取并保留 Top-16" applied to
 * the drafter's LM-head output]: logits[r, v] = sum_c hidden[r, c] * W_lm[v, c]
 * in double (bf16 inputs, exact), then the full sort of oracle_topk.  idx/val
 * [R, k].  Returns 0, or -1 on a bad argument. */
int oracle_lmhead_topk(const uint16_t* hidden, const uint16_t* W_lm, int R, int V, int d, int k,
                       int32_t* idx, double* val);

/* The two uniforms verification draws at block position t (reading, the pages
 * name no generator): words 0 and 1 of Philox4x32-10 with counter
 * (t, lo32(cycle), hi32(cycle), 1) and key = the sequence's seed, each
 * (w >> 8) * 2^-24.  u[0] decides acceptance, u[1] the replacement draw. */
void oracle_verify_uniforms(uint64_t seed, uint64_t cycle, int t, double u[2]);

/* Verification of a drafted block [VERIFY].  p [B, L+1, V] holds the target's
 * next-token distributions: row t (t < L) follows the verified token and the
 * first t drafted tokens, row L follows the whole block.  For t = 0..L-1:
 *   greedy: accept iff tokens[t] is the lowest index holding the row's maximum;
 *           otherwise emit that index and stop;
 *   sampling: with x = tokens[t] and its draft probability q(x) =
 *           q[b,t,slots[t]], accept iff u0 * q(x) < p_t(x); otherwise draw from
 *           r(v) = max(0, p_t(v) - q_t(v)) (q_t is zero off the 16 candidates
 *           cand_idx[b,t,:]): the first v, in index order, whose running sum of
 *           r exceeds u1 * sum(r) (the last v with r > 0 if rounding leaves
 *           none; p_t itself if sum(r) = 0), emit it and stop.
 * When all L are accepted, one more token comes from row L (its argmax, or a
 * draw from p_L with u1 of t = L).  Writes n_accepted [B] (0..L) and out
 * [B, L+1]: the accepted draft tokens, then the emitted token, then -1.
 * q, slots, cand_idx and seeds may be NULL when greedy.  Returns 0, or -1 on a
 * bad argument. */
int oracle_verify(const float* p, const int32_t* tokens, const int32_t* slots, const float* q,
                  const int32_t* cand_idx, int B, int L, int V, int greedy,
                  const uint64_t* seeds, uint64_t cycle, int32_t* n_accepted, int32_t* out);

/* Round a double to the nearest bf16 (ties to even), as a bit pattern. */
uint16_t oracle_round_bf16(double v);

#ifdef __cplusplus
}
#endif
#endif
