/*
 * dfl2 oracle: TEST INFRASTRUCTURE, not part of the product.
 *
 * Plain C11, double precision, literal loops.  The only parallelism is an
 * OpenMP loop over independent rows / sequences; no blocking, fusion or
 * reordering of any sum beyond what each definition states.  Sources and the
 * readings taken where the pages are silent are listed in dfl2_oracle.h.
 */
#include "dfl2_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

uint16_t oracle_round_bf16(double v) {
  if (isnan(v)) return 0x7FC0;
  if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
  int neg = v < 0.0;
  double a = fabs(v);
  /* Halfway between the largest finite bf16, (2 - 2^-7) 2^127, and 2^128. */
  if (a >= ldexp(2.0 - ldexp(1.0, -8), 127)) return neg ? 0xFF80 : 0x7F80;
  int ex;
  frexp(a, &ex);              /* a = m 2^ex, m in [0.5, 1) */
  int e = ex - 1;             /* a in [2^e, 2^(e+1)) */
  if (e < -126) e = -126;     /* subnormal range: fixed quantum 2^-133 */
  double quantum = ldexp(1.0, e - 7); /* 8 significant bits */
  double n = nearbyint(a / quantum);  /* ties to even (default rounding mode) */
  float f = (float)(n * quantum);     /* exactly representable */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint16_t bits = (uint16_t)(u >> 16);
  return neg ? (uint16_t)(bits | 0x8000u) : bits;
}

/* ---------------------------------------------------------------- Philox */

/* Philox4x32-10 as published by Salmon et al. (SC'11): ten rounds of two
 * 32x32->64 multiplies with the round keys bumped by the Weyl constants. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    uint64_t p0 = (uint64_t)M0 * c0;
    uint64_t p1 = (uint64_t)M1 * c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    k0 += W0;
    k1 += W1;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

double oracle_walk_uniform(uint64_t seed, uint64_t cycle, int t) {
  uint32_t ctr[4] = {(uint32_t)t, (uint32_t)cycle, (uint32_t)(cycle >> 32), 0u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  return (double)(out[0] >> 8) * ldexp(1.0, -24);
}

/* ---------------------------------------------------------------- top-k */

typedef struct {
  double v;
  int32_t i;
} vi_pair;

/* (value descending, index ascending).  Comparing doubles makes -0.0 == +0.0,
 * so the two zeros are ordered by index, like any other tie. */
static int cmp_value_desc_index_asc(const void* pa, const void* pb) {
  const vi_pair* a = (const vi_pair*)pa;
  const vi_pair* b = (const vi_pair*)pb;
  if (a->v > b->v) return -1;
  if (a->v < b->v) return 1;
  return (a->i < b->i) ? -1 : (a->i > b->i);
}

int oracle_topk(const void* logits, int dtype, int B, int L, int V, int k,
                int32_t* idx, float* val) {
  if (!logits || !idx || !val || B < 0 || L < 0 || V < 1 || k < 1 || k > V) return -1;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return -1;
  long rows = (long)B * L;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (long row = 0; row < rows; ++row) {
    vi_pair* p = (vi_pair*)malloc(sizeof(vi_pair) * (size_t)V);
    if (!p) {
#pragma omp atomic write
      bad = 1;
      continue;
    }
    for (int i = 0; i < V; ++i) {
      size_t at = (size_t)row * (size_t)V + (size_t)i;
      double v = dtype == ORACLE_F32 ? (double)((const float*)logits)[at]
                                     : bf16_to_double(((const uint16_t*)logits)[at]);
      p[i].v = v;
      p[i].i = i;
    }
    qsort(p, (size_t)V, sizeof(vi_pair), cmp_value_desc_index_asc);
    for (int j = 0; j < k; ++j) {
      idx[row * k + j] = p[j].i;
      val[row * k + j] = (float)p[j].v;
    }
    free(p);
  }
  return bad ? -1 : 0;
}

/* ---------------------------------------------------------------- selector */

/* out[q] = sum_c W[q,c] * E[tok,c]: one row of A(.) or B(.) [SEL, "A 和 B 将
 * 离散 Token 映射至 256 维"], read as a linear map of the token embedding. */
void oracle_proj_token(const uint16_t* E, const uint16_t* W, int d, int r, int32_t tok,
                       double* out) {
  const uint16_t* e = E + (size_t)tok * (size_t)d;
  for (int q = 0; q < r; ++q) {
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += bf16_to_double(W[(size_t)q * d + c]) * bf16_to_double(e[c]);
    out[q] = s;
  }
}

/* out[q] = sigmoid(sum_c W_H[q,c] h[c]): the context gate H(h_t) [SEL,
 * "门控向量用于动态决定哪些嵌入维度在当前上下文中生效"], read as a sigmoid gate. */
void oracle_gate(const uint16_t* W_H, const uint16_t* h, int d, int r, double* out) {
  for (int q = 0; q < r; ++q) {
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += bf16_to_double(W_H[(size_t)q * d + c]) * bf16_to_double(h[c]);
    out[q] = 1.0 / (1.0 + exp(-s));
  }
}

#define NCAND 16

int oracle_select(const int32_t* cand_idx, const float* cand_val, const int32_t* verified,
                  const uint16_t* hidden, const uint16_t* E, const uint16_t* W_A,
                  const uint16_t* W_B, const uint16_t* W_H, int B, int L, int V, int d,
                  int r, double* scores) {
  if (!cand_idx || !cand_val || !verified || !hidden || !E || !W_A || !W_B || !W_H || !scores)
    return -1;
  if (B < 0 || L < 0 || V < 1 || d < 1 || r < 1) return -1;
  for (long i = 0; i < (long)B * L * NCAND; ++i)
    if (cand_idx[i] < 0 || cand_idx[i] >= V) return -1;
  for (int b = 0; b < B; ++b)
    if (verified[b] < 0 || verified[b] >= V) return -1;
  long cells = (long)B * L;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (long cell = 0; cell < cells; ++cell) {
    int b = (int)(cell / L), t = (int)(cell % L);
    double* H = (double*)malloc(sizeof(double) * (size_t)r);
    double* A = (double*)malloc(sizeof(double) * (size_t)r * NCAND);
    double* Bv = (double*)malloc(sizeof(double) * (size_t)r * NCAND);
    if (!H || !A || !Bv) {
#pragma omp atomic write
      bad = 1;
      free(H); free(A); free(Bv);
      continue;
    }
    /* H(h_t): the drafter's hidden state at position t. */
    oracle_gate(W_H, hidden + ((size_t)b * L + t) * (size_t)d, d, r, H);
    /* Predecessors: the verified token at t = 0, else the 16 candidates of t-1. */
    int npred = t == 0 ? 1 : NCAND;
    for (int i = 0; i < npred; ++i) {
      int32_t a = t == 0 ? verified[b] : cand_idx[((size_t)b * L + (t - 1)) * NCAND + i];
      oracle_proj_token(E, W_A, d, r, a, A + (size_t)i * r);
    }
    for (int j = 0; j < NCAND; ++j) {
      int32_t tok = cand_idx[((size_t)b * L + t) * NCAND + j];
      oracle_proj_token(E, W_B, d, r, tok, Bv + (size_t)j * r);
    }
    double* S = scores + (size_t)cell * NCAND * NCAND;
    for (int i = 0; i < NCAND; ++i) {
      for (int j = 0; j < NCAND; ++j) {
        if (i >= npred) {
          S[i * NCAND + j] = -INFINITY;
          continue;
        }
        /* S_t(a,b) = U_t(b) + sum_q A_q(a) H_q(h_t) B_q(b). */
        double s = 0.0;
        for (int q = 0; q < r; ++q) s += A[(size_t)i * r + q] * H[q] * Bv[(size_t)j * r + q];
        S[i * NCAND + j] = (double)cand_val[((size_t)b * L + t) * NCAND + j] + s;
      }
    }
    free(H); free(A); free(Bv);
  }
  return bad ? -1 : 0;
}

int oracle_walk(const double* scores, const int32_t* cand_idx, int B, int L, double T,
                const uint64_t* seeds, uint64_t cycle, int32_t* tokens, int32_t* slots,
                double* q) {
  if (!scores || !cand_idx || !tokens || B < 0 || L < 0 || !(T >= 0.0)) return -1;
  if (T > 0.0 && !seeds) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int b = 0; b < B; ++b) {
    int prev = 0; /* row 0 of position 0 is the last verified token */
    for (int t = 0; t < L; ++t) {
      const double* row = scores + (((size_t)b * L + t) * NCAND + (size_t)prev) * NCAND;
      double p[NCAND];
      int pick = 0;
      if (T == 0.0) {
        for (int j = 1; j < NCAND; ++j)
          if (row[j] > row[pick]) pick = j; /* strict: the lowest slot wins a tie */
        for (int j = 0; j < NCAND; ++j) p[j] = j == pick ? 1.0 : 0.0;
      } else {
        double m = row[0];
        for (int j = 1; j < NCAND; ++j)
          if (row[j] > m) m = row[j];
        double Z = 0.0;
        for (int j = 0; j < NCAND; ++j) {
          p[j] = exp((row[j] - m) / T);
          Z += p[j];
        }
        double uZ = oracle_walk_uniform(seeds[b], cycle, t) * Z;
        double cum = 0.0;
        pick = -1;
        for (int j = 0; j < NCAND; ++j) {
          cum += p[j];
          if (uZ < cum) {
            pick = j;
            break;
          }
        }
        if (pick < 0) /* rounding left u*Z above the total: take the last live slot */
          for (int j = NCAND - 1; j >= 0; --j)
            if (p[j] > 0.0) {
              pick = j;
              break;
            }
        for (int j = 0; j < NCAND; ++j) p[j] /= Z;
      }
      tokens[(size_t)b * L + t] = cand_idx[((size_t)b * L + t) * NCAND + pick];
      if (slots) slots[(size_t)b * L + t] = pick;
      if (q)
        for (int j = 0; j < NCAND; ++j) q[((size_t)b * L + t) * NCAND + j] = p[j];
      prev = pick;
    }
  }
  return 0;
}

/* ---------------------------------------------------------------- conv */

int oracle_conv2(const uint16_t* x, const uint16_t* x_prev, const float* base,
                 const uint16_t* W_c, int B, int L, int d, double* y_exact, uint16_t* y_bf16) {
  if (!x || !x_prev || !base || !W_c || B < 0 || L < 0 || d < 16 || d % 16 != 0) return -1;
  const int G = d / 16;
  long cells = (long)B * L;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (long cell = 0; cell < cells; ++cell) {
    int b = (int)(cell / L), t = (int)(cell % L);
    const uint16_t* xt = x + (size_t)cell * d;
    const uint16_t* xm1 = t == 0 ? x_prev + (size_t)b * d : x + (size_t)(cell - 1) * d;
    double* corr = (double*)malloc(sizeof(double) * 2 * (size_t)G);
    if (!corr) {
#pragma omp atomic write
      bad = 1;
      continue;
    }
    /* Correction from the current hidden state, one per 16-channel group and tap. */
    for (int j = 0; j < 2; ++j)
      for (int g = 0; g < G; ++g) {
        double s = 0.0;
        const uint16_t* w = W_c + ((size_t)j * G + g) * (size_t)d;
        for (int c = 0; c < d; ++c) s += bf16_to_double(w[c]) * bf16_to_double(xt[c]);
        corr[j * G + g] = s;
      }
    for (int c = 0; c < d; ++c) {
      double k0 = (double)base[c] + corr[c / 16];
      double k1 = (double)base[d + c] + corr[G + c / 16];
      double y = k0 * bf16_to_double(xt[c]) + k1 * bf16_to_double(xm1[c]);
      if (y_exact) y_exact[(size_t)cell * d + c] = y;
      if (y_bf16) y_bf16[(size_t)cell * d + c] = oracle_round_bf16(y);
    }
    free(corr);
  }
  return bad ? -1 : 0;
}

/* ---------------------------------------------------------------- verify */

void oracle_verify_uniforms(uint64_t seed, uint64_t cycle, int t, double u[2]) {
  uint32_t ctr[4] = {(uint32_t)t, (uint32_t)cycle, (uint32_t)(cycle >> 32), 1u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  u[0] = (double)(out[0] >> 8) * ldexp(1.0, -24);
  u[1] = (double)(out[1] >> 8) * ldexp(1.0, -24);
}

static int32_t row_argmax(const float* row, int V) {
  int32_t best = 0;
  for (int v = 1; v < V; ++v)
    if ((double)row[v] > (double)row[best]) best = v;
  return best;
}

/* First v whose running sum of w exceeds target; the last v with w > 0 when
 * rounding leaves none. */
static int32_t draw_index(const double* w, int V, double target) {
  double cum = 0.0;
  for (int v = 0; v < V; ++v) {
    cum += w[v];
    if (target < cum) return v;
  }
  for (int v = V - 1; v >= 0; --v)
    if (w[v] > 0.0) return v;
  return 0;
}

int oracle_verify(const float* p, const int32_t* tokens, const int32_t* slots, const float* q,
                  const int32_t* cand_idx, int B, int L, int V, int greedy,
                  const uint64_t* seeds, uint64_t cycle, int32_t* n_accepted, int32_t* out) {
  if (!p || !tokens || !n_accepted || !out || B < 1 || L < 1 || V < 1) return -1;
  if (!greedy && (!slots || !q || !cand_idx || !seeds)) return -1;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int b = 0; b < B; ++b) {
    double* w = (double*)malloc(sizeof(double) * (size_t)V);
    if (!w) {
      bad = 1;
      continue;
    }
    int32_t* o = out + (size_t)b * (L + 1);
    for (int t = 0; t <= L; ++t) o[t] = -1;
    int n = L;
    int32_t emit = -1;
    for (int t = 0; t < L; ++t) {
      const float* row = p + ((size_t)b * (L + 1) + t) * V;
      const int32_t x = tokens[(size_t)b * L + t];
      if (greedy) {
        const int32_t a = row_argmax(row, V);
        if (x == a) {
          o[t] = x;
          continue;
        }
        n = t;
        emit = a;
        break;
      }
      double u[2];
      oracle_verify_uniforms(seeds[b], cycle, t, u);
      const size_t cell = (size_t)b * L + t;
      const double qx = (double)q[cell * 16 + slots[cell]];
      if (u[0] * qx < (double)row[x]) {
        o[t] = x;
        continue;
      }
      /* rejected: draw from the residual max(0, p - q) */
      double Z = 0.0;
      for (int v = 0; v < V; ++v) w[v] = (double)row[v];
      for (int k = 0; k < 16; ++k) {
        const int32_t c = cand_idx[cell * 16 + k];
        if (c >= 0 && c < V) w[c] -= (double)q[cell * 16 + k];
      }
      for (int v = 0; v < V; ++v) {
        if (w[v] < 0.0) w[v] = 0.0;
        Z += w[v];
      }
      if (Z <= 0.0) { /* p does not exceed q anywhere: draw from p itself */
        for (int v = 0; v < V; ++v) Z += (w[v] = (double)row[v]);
      }
      n = t;
      emit = draw_index(w, V, u[1] * Z);
      break;
    }
    if (n == L) { /* every draft token accepted: one more from row L */
      const float* row = p + ((size_t)b * (L + 1) + L) * V;
      if (greedy) {
        emit = row_argmax(row, V);
      } else {
        double u[2], Z = 0.0;
        oracle_verify_uniforms(seeds[b], cycle, L, u);
        for (int v = 0; v < V; ++v) Z += (w[v] = (double)row[v]);
        emit = draw_index(w, V, u[1] * Z);
      }
    }
    n_accepted[b] = n;
    o[n] = emit;
    free(w);
  }
  return bad ? -1 : 0;
}

/* ---------------------------------------------------------------- LM head + top-k */

int oracle_lmhead_topk(const uint16_t* hidden, const uint16_t* W_lm, int R, int V, int d, int k,
                       int32_t* idx, double* val) {
  if (!hidden || !W_lm || !idx || !val || R < 1 || V < k || d < 1 || k < 1) return -1;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int r = 0; r < R; ++r) {
    double* h = (double*)malloc(sizeof(double) * (size_t)d);
    vi_pair* all = (vi_pair*)malloc(sizeof(vi_pair) * (size_t)V);
    if (!h || !all) {
      bad = 1;
      free(h);
      free(all);
      continue;
    }
    for (int c = 0; c < d; ++c) h[c] = bf16_to_double(hidden[(size_t)r * d + c]);
    for (int v = 0; v < V; ++v) {
      const uint16_t* w = W_lm + (size_t)v * d;
      double acc = 0.0;
      for (int c = 0; c < d; ++c) acc += h[c] * bf16_to_double(w[c]);
      all[v].v = acc;
      all[v].i = v;
    }
    qsort(all, (size_t)V, sizeof(vi_pair), cmp_value_desc_index_asc);
    for (int j = 0; j < k; ++j) {
      idx[(size_t)r * k + j] = all[j].i;
      val[(size_t)r * k + j] = all[j].v;
    }
    free(h);
    free(all);
  }
  return bad ? -1 : 0;
}
