/*
 * gqa_oracle.c -- plain, slow, fp64 CPU oracle for grouped-query attention
 * forward and backward.  TEST INFRASTRUCTURE ONLY: only the test-suite, the
 * smoke check and the benchmark's CPU-baseline leg may load this library.  It
 * shares no code, header or constant with the CUDA path.
 *
 * What it computes (notation of the pages; h = query head, g = kv head,
 * i = query row, j = key row, d = feature):
 *
 *   g          = h / (Hq / Hkv)                        ("bx // groups", tilelang
 *                                                       PR #1093, Additional comments)
 *   A(i)       = { j in the same sequence as i, j <= i + (Lk - Lq) if causal,
 *                  i + (Lk - Lq) - j < W if a window W > 0 is set,
 *                  j - (i + (Lk - Lq)) < Wr if a right window Wr > 0 is set (not causal) }
 *                with i, j local to their sequence, Lq / Lk its query / key lengths:
 *                the causal diagonal is aligned at the bottom right (the last query sees
 *                the last key), which is the top-left j <= i when Lq == Lk
 *   S_ij       = scale * sum_d Q[h,i,d] K[g,j,d]       (tilelang-ascend PR #1638,
 *                                                       review thread, k1/k2)
 *   LSE_i      = log( [e^{sink_h}] + sum_{j in A(i)} e^{S_ij} )
 *                                                      (forward with attention sink,
 *                                                       PR #1638 commit "4->2 kernels")
 *   P_ij       = exp(S_ij - LSE_i),  p_sink_i = exp(sink_h - LSE_i)
 *   O_i        = sum_j P_ij V[g,j]
 *   Delta_i    = sum_d dO[h,i,d] O[h,i,d]              (PR #1638, Phase0(Delta))
 *   dP_ij      = sum_d dO[h,i,d] V[g,j,d]              (PR #1638, k3)
 *   dS_ij      = P_ij (dP_ij - Delta_i) * scale        (PR #1638, k4)
 *   dQ_i       = sum_j dS_ij K[g,j]                    (PR #1638, k5)
 *   dK_j       = sum_{h in group g} sum_i dS_ij Q[h,i] (PR #1638, k5; the group
 *                                                       sum: PR #1093 comments)
 *   dV_j       = sum_{h in group g} sum_i P_ij dO[h,i] (PR #1638, k3)
 *   dsink_h    = - sum_{b,i} p_sink_i Delta_i          (PR #1638, "Kernel 9: Dsink")
 *
 * The sink is one extra logit per query head that enters the softmax
 * denominator and has no value vector; it is in scaled-logit units.
 *
 * Layout: every tensor is dense row-major [B, H, S, D] in fp64 (S is the
 * per-batch length, or the packed token count T when cu_seqlens is given, in
 * which case B == 1); k, v, dk, dv have Sk rows per (b, h) instead (Sk = S
 * unless set).  LSE / Delta are [B, Hq, S].
 *
 * Evaluation order is the plain definition: a row pass over (b, h, i) and a
 * column pass over (b, g, j) that revisits every (h, i) which sees key j, so no
 * output is ever written by two threads.  OpenMP only splits independent rows.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int B, Hq, Hkv, S, Dqk, Dv;
  int causal;          /* 1: key j visible to query i only if j <= i (top-left) */
  int window;          /* > 0: additionally i - j < window; <= 0: no window */
  double scale;        /* softmax scale applied to Q.K */
  int nseq;            /* number of packed sequences when cu_seqlens != NULL */
  const int32_t* cu_seqlens; /* [nseq+1] token offsets, or NULL (dense) */
  const double* sink;  /* [Hq] or NULL */
  int Sk;              /* key rows per batch (or packed key tokens); 0: the same as S */
  const int32_t* cu_seqlens_k; /* [nseq+1] key offsets, or NULL: the same as cu_seqlens */
  int window_right;    /* > 0 (not causal): keys at most window_right - 1 right of the diagonal */
} oracle_problem;

static inline int key_len(const oracle_problem* p) { return p->Sk > 0 ? p->Sk : p->S; }

/* Range of key rows visible to query row i (both in absolute token index
 * within the S axis), returned as [lo, hi) ; empty if lo >= hi. */
static void key_range(const oracle_problem* p, int i, int* lo, int* hi) {
  int qs = 0, ql = p->S, ks = 0, kl = key_len(p);
  if (p->cu_seqlens) {
    const int32_t* ck = p->cu_seqlens_k ? p->cu_seqlens_k : p->cu_seqlens;
    for (int s = 0; s < p->nseq; ++s) {
      if (i >= p->cu_seqlens[s] && i < p->cu_seqlens[s + 1]) {
        qs = p->cu_seqlens[s];
        ql = p->cu_seqlens[s + 1] - qs;
        ks = ck[s];
        kl = ck[s + 1] - ks;
        break;
      }
    }
  }
  const int il = i - qs, off = kl - ql;  /* query il sits on key diagonal il + off */
  int a = 0, b = kl;
  if (p->causal && il + off + 1 < b) b = il + off + 1;
  if (!p->causal && p->window_right > 0 && il + off + p->window_right < b) b = il + off + p->window_right;
  if (p->window > 0 && il + off - p->window + 1 > a) a = il + off - p->window + 1;
  *lo = ks + a;
  *hi = ks + b;  /* empty when b <= a */
}

static inline const double* row(const double* t, int H, int S, int D, int b, int h, int i) {
  return t + (((size_t)b * H + h) * S + i) * D;
}

static double dot(const double* x, const double* y, int n) {
  double s = 0.0;
  for (int d = 0; d < n; ++d) s += x[d] * y[d];
  return s;
}

/* Scaled logit S_ij. */
static double logit(const oracle_problem* p, const double* q, const double* k, int b, int h, int i, int j) {
  const int g = h / (p->Hq / p->Hkv);
  return p->scale * dot(row(q, p->Hq, p->S, p->Dqk, b, h, i), row(k, p->Hkv, key_len(p), p->Dqk, b, g, j), p->Dqk);
}

/* LSE_i from its definition, with the row maximum subtracted for stability. */
static double row_lse(const oracle_problem* p, const double* q, const double* k, int b, int h, int i) {
  int lo, hi;
  key_range(p, i, &lo, &hi);
  double m = -INFINITY;
  if (p->sink) m = p->sink[h];
  for (int j = lo; j < hi; ++j) {
    double s = logit(p, q, k, b, h, i, j);
    if (s > m) m = s;
  }
  if (m == -INFINITY) return -INFINITY;
  double z = p->sink ? exp(p->sink[h] - m) : 0.0;
  for (int j = lo; j < hi; ++j) z += exp(logit(p, q, k, b, h, i, j) - m);
  return m + log(z);
}

/* Forward: O and LSE for every (b, h, i). */
void oracle_forward(const oracle_problem* p, const double* q, const double* k, const double* v, double* o,
                    double* lse) {
  const int G = p->Hq / p->Hkv;
  const long nrows = (long)p->B * p->Hq * p->S;
#pragma omp parallel for schedule(dynamic, 16)
  for (long r = 0; r < nrows; ++r) {
    const int i = (int)(r % p->S), h = (int)((r / p->S) % p->Hq), b = (int)(r / ((long)p->S * p->Hq));
    const int g = h / G;
    const double L = row_lse(p, q, k, b, h, i);
    lse[r] = L;
    double* orow = o + (size_t)r * p->Dv;
    for (int d = 0; d < p->Dv; ++d) orow[d] = 0.0;
    int lo, hi;
    key_range(p, i, &lo, &hi);
    for (int j = lo; j < hi; ++j) {
      const double pij = exp(logit(p, q, k, b, h, i, j) - L);
      const double* vj = row(v, p->Hkv, key_len(p), p->Dv, b, g, j);
      for (int d = 0; d < p->Dv; ++d) orow[d] += pij * vj[d];
    }
  }
}

/* Delta_i = rowsum(dO * O) for every row. */
void oracle_delta(const oracle_problem* p, const double* o, const double* dout, double* delta) {
  const long nrows = (long)p->B * p->Hq * p->S;
#pragma omp parallel for schedule(static)
  for (long r = 0; r < nrows; ++r) delta[r] = dot(dout + (size_t)r * p->Dv, o + (size_t)r * p->Dv, p->Dv);
}

/* dS_ij (with the scale) given the row statistics LSE_i and Delta_i. */
static double grad_logit(const oracle_problem* p, const double* q, const double* k, const double* v,
                         const double* dout, double L, double D_i, int b, int h, int i, int j, double* pij_out) {
  const int g = h / (p->Hq / p->Hkv);
  const double pij = exp(logit(p, q, k, b, h, i, j) - L);
  const double dpij = dot(row(dout, p->Hq, p->S, p->Dv, b, h, i), row(v, p->Hkv, key_len(p), p->Dv, b, g, j), p->Dv);
  if (pij_out) *pij_out = pij;
  return pij * (dpij - D_i) * p->scale;
}

/*
 * Backward.  Inputs: q, k, v, dout, and the forward's lse and o (Delta is
 * formed from o and dout).  Outputs: delta [B,Hq,S], dq [B,Hq,S,Dqk],
 * dk [B,Hkv,Sk,Dqk], dv [B,Hkv,Sk,Dv], dsink [Hq] (only if p->sink).
 */
void oracle_backward(const oracle_problem* p, const double* q, const double* k, const double* v,
                     const double* o, const double* lse, const double* dout, double* delta, double* dq,
                     double* dk, double* dv, double* dsink) {
  const int G = p->Hq / p->Hkv;
  oracle_delta(p, o, dout, delta);
  const long nrows = (long)p->B * p->Hq * p->S;

  /* row pass: dQ_i */
#pragma omp parallel for schedule(dynamic, 16)
  for (long r = 0; r < nrows; ++r) {
    const int i = (int)(r % p->S), h = (int)((r / p->S) % p->Hq), b = (int)(r / ((long)p->S * p->Hq));
    const int g = h / G;
    double* dqi = dq + (size_t)r * p->Dqk;
    for (int d = 0; d < p->Dqk; ++d) dqi[d] = 0.0;
    int lo, hi;
    key_range(p, i, &lo, &hi);
    for (int j = lo; j < hi; ++j) {
      const double ds = grad_logit(p, q, k, v, dout, lse[r], delta[r], b, h, i, j, NULL);
      const double* kj = row(k, p->Hkv, key_len(p), p->Dqk, b, g, j);
      for (int d = 0; d < p->Dqk; ++d) dqi[d] += ds * kj[d];
    }
  }

  /* column pass: dK_j, dV_j summed over every query head of the group */
  const int SK = key_len(p);
  const long ncols = (long)p->B * p->Hkv * SK;
#pragma omp parallel for schedule(dynamic, 16)
  for (long c = 0; c < ncols; ++c) {
    const int j = (int)(c % SK), g = (int)((c / SK) % p->Hkv), b = (int)(c / ((long)SK * p->Hkv));
    double* dkj = dk + (size_t)c * p->Dqk;
    double* dvj = dv + (size_t)c * p->Dv;
    for (int d = 0; d < p->Dqk; ++d) dkj[d] = 0.0;
    for (int d = 0; d < p->Dv; ++d) dvj[d] = 0.0;
    for (int h = g * G; h < (g + 1) * G; ++h) {
      for (int i = 0; i < p->S; ++i) {
        int lo, hi;
        key_range(p, i, &lo, &hi);
        if (j < lo || j >= hi) continue;
        const long r = ((long)b * p->Hq + h) * p->S + i;
        double pij;
        const double ds = grad_logit(p, q, k, v, dout, lse[r], delta[r], b, h, i, j, &pij);
        const double* qi = row(q, p->Hq, p->S, p->Dqk, b, h, i);
        const double* doi = row(dout, p->Hq, p->S, p->Dv, b, h, i);
        for (int d = 0; d < p->Dqk; ++d) dkj[d] += ds * qi[d];
        for (int d = 0; d < p->Dv; ++d) dvj[d] += pij * doi[d];
      }
    }
  }

  /* dsink_h = - sum over b, i of p_sink_i * Delta_i */
  if (p->sink && dsink) {
    for (int h = 0; h < p->Hq; ++h) {
      double acc = 0.0;
      for (int b = 0; b < p->B; ++b)
        for (int i = 0; i < p->S; ++i) {
          const long r = ((long)b * p->Hq + h) * p->S + i;
          acc += exp(p->sink[h] - lse[r]) * delta[r];
        }
      dsink[h] = -acc;
    }
  }
}

/*
 * Sampled evaluation for problems too large for the full passes.
 *
 * Query side: for each listed (b, h, i) it computes LSE_i, O_i, Delta_i and
 * dQ_i exactly (Delta from its own O).  Outputs are packed in list order:
 * lse[n], o[n*Dv], delta[n], dq[n*Dqk].
 *
 * Key side: for each listed (b, g, j) it computes dK_j and dV_j exactly.  Each
 * query row that sees j needs its own LSE and Delta, which are recomputed from
 * the definition here (so the cost grows with the number of such rows).
 */
void oracle_sample_rows(const oracle_problem* p, const double* q, const double* k, const double* v,
                        const double* dout, int n, const int32_t* bs, const int32_t* hs, const int32_t* is,
                        double* lse, double* o, double* delta, double* dq) {
  const int G = p->Hq / p->Hkv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < n; ++t) {
    const int b = bs[t], h = hs[t], i = is[t], g = h / G;
    const double L = row_lse(p, q, k, b, h, i);
    double* orow = o + (size_t)t * p->Dv;
    for (int d = 0; d < p->Dv; ++d) orow[d] = 0.0;
    int lo, hi;
    key_range(p, i, &lo, &hi);
    for (int j = lo; j < hi; ++j) {
      const double pij = exp(logit(p, q, k, b, h, i, j) - L);
      const double* vj = row(v, p->Hkv, key_len(p), p->Dv, b, g, j);
      for (int d = 0; d < p->Dv; ++d) orow[d] += pij * vj[d];
    }
    const double Di = dot(row(dout, p->Hq, p->S, p->Dv, b, h, i), orow, p->Dv);
    lse[t] = L;
    delta[t] = Di;
    double* dqi = dq + (size_t)t * p->Dqk;
    for (int d = 0; d < p->Dqk; ++d) dqi[d] = 0.0;
    for (int j = lo; j < hi; ++j) {
      const double ds = grad_logit(p, q, k, v, dout, L, Di, b, h, i, j, NULL);
      const double* kj = row(k, p->Hkv, key_len(p), p->Dqk, b, g, j);
      for (int d = 0; d < p->Dqk; ++d) dqi[d] += ds * kj[d];
    }
  }
}

void oracle_sample_cols(const oracle_problem* p, const double* q, const double* k, const double* v,
                        const double* dout, int n, const int32_t* bs, const int32_t* gs, const int32_t* js,
                        double* dk, double* dv) {
  const int G = p->Hq / p->Hkv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < n; ++t) {
    const int b = bs[t], g = gs[t], j = js[t];
    double* dkj = dk + (size_t)t * p->Dqk;
    double* dvj = dv + (size_t)t * p->Dv;
    for (int d = 0; d < p->Dqk; ++d) dkj[d] = 0.0;
    for (int d = 0; d < p->Dv; ++d) dvj[d] = 0.0;
    double* orow = (double*)malloc(sizeof(double) * (size_t)p->Dv);
    for (int h = g * G; h < (g + 1) * G; ++h) {
      for (int i = 0; i < p->S; ++i) {
        int lo, hi;
        key_range(p, i, &lo, &hi);
        if (j < lo || j >= hi) continue;
        /* this query row's own statistics, from the definition */
        const double L = row_lse(p, q, k, b, h, i);
        for (int d = 0; d < p->Dv; ++d) orow[d] = 0.0;
        for (int jj = lo; jj < hi; ++jj) {
          const double pw = exp(logit(p, q, k, b, h, i, jj) - L);
          const double* vj = row(v, p->Hkv, key_len(p), p->Dv, b, g, jj);
          for (int d = 0; d < p->Dv; ++d) orow[d] += pw * vj[d];
        }
        const double Di = dot(row(dout, p->Hq, p->S, p->Dv, b, h, i), orow, p->Dv);
        double pij;
        const double ds = grad_logit(p, q, k, v, dout, L, Di, b, h, i, j, &pij);
        const double* qi = row(q, p->Hq, p->S, p->Dqk, b, h, i);
        const double* doi = row(dout, p->Hq, p->S, p->Dv, b, h, i);
        for (int d = 0; d < p->Dqk; ++d) dkj[d] += ds * qi[d];
        for (int d = 0; d < p->Dv; ++d) dvj[d] += pij * doi[d];
      }
    }
    free(orow);
  }
}

/*
 * Row statistics at listed query rows (b, h, i): LSE_i from its definition and
 * Delta_i = dO_i . O_i with O_i = sum_j P_ij V_j -- the values oracle_forward
 * and oracle_delta give for those rows.  The row's logits are formed once and
 * kept for the maximum, the sum and the O passes (the same values and the same
 * order of every sum as row_lse and oracle_forward), so large problems can be
 * sampled row by row in parallel.  Outputs in list order: lse[n], delta[n].
 */
void oracle_row_stats(const oracle_problem* p, const double* q, const double* k, const double* v,
                      const double* dout, int n, const int32_t* bs, const int32_t* hs, const int32_t* is,
                      double* lse, double* delta) {
  const int G = p->Hq / p->Hkv;
#pragma omp parallel for schedule(dynamic, 4)
  for (int t = 0; t < n; ++t) {
    const int b = bs[t], h = hs[t], i = is[t], g = h / G;
    int lo, hi;
    key_range(p, i, &lo, &hi);
    const int nk = hi > lo ? hi - lo : 0;
    double* s = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
    double* orow = (double*)malloc(sizeof(double) * (size_t)p->Dv);
    double m = p->sink ? p->sink[h] : -INFINITY;
    for (int j = lo; j < hi; ++j) {
      s[j - lo] = logit(p, q, k, b, h, i, j);
      if (s[j - lo] > m) m = s[j - lo];
    }
    double L = -INFINITY;
    if (m != -INFINITY) {
      double z = p->sink ? exp(p->sink[h] - m) : 0.0;
      for (int j = lo; j < hi; ++j) z += exp(s[j - lo] - m);
      L = m + log(z);
    }
    for (int d = 0; d < p->Dv; ++d) orow[d] = 0.0;
    for (int j = lo; j < hi; ++j) {
      const double pij = exp(s[j - lo] - L);
      const double* vj = row(v, p->Hkv, key_len(p), p->Dv, b, g, j);
      for (int d = 0; d < p->Dv; ++d) orow[d] += pij * vj[d];
    }
    lse[t] = L;
    delta[t] = dot(row(dout, p->Hq, p->S, p->Dv, b, h, i), orow, p->Dv);
    free(orow);
    free(s);
  }
}

/*
 * dK_j and dV_j at listed key rows (b, g, j) given LSE and Delta of the query
 * rows in full [B, Hq, S] arrays: the column pass of oracle_backward restricted
 * to the listed keys.  Only the entries of rows that see a listed key are read.
 */
void oracle_cols_with_stats(const oracle_problem* p, const double* q, const double* k, const double* v,
                            const double* dout, const double* lse, const double* delta, int n,
                            const int32_t* bs, const int32_t* gs, const int32_t* js, double* dk, double* dv) {
  const int G = p->Hq / p->Hkv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < n; ++t) {
    const int b = bs[t], g = gs[t], j = js[t];
    double* dkj = dk + (size_t)t * p->Dqk;
    double* dvj = dv + (size_t)t * p->Dv;
    for (int d = 0; d < p->Dqk; ++d) dkj[d] = 0.0;
    for (int d = 0; d < p->Dv; ++d) dvj[d] = 0.0;
    for (int h = g * G; h < (g + 1) * G; ++h) {
      for (int i = 0; i < p->S; ++i) {
        int lo, hi;
        key_range(p, i, &lo, &hi);
        if (j < lo || j >= hi) continue;
        const long r = ((long)b * p->Hq + h) * p->S + i;
        double pij;
        const double ds = grad_logit(p, q, k, v, dout, lse[r], delta[r], b, h, i, j, &pij);
        const double* qi = row(q, p->Hq, p->S, p->Dqk, b, h, i);
        const double* doi = row(dout, p->Hq, p->S, p->Dv, b, h, i);
        for (int d = 0; d < p->Dqk; ++d) dkj[d] += ds * qi[d];
        for (int d = 0; d < p->Dv; ++d) dvj[d] += pij * doi[d];
      }
    }
  }
}

/* dsink_h = - sum over b, i of exp(sink_h - LSE_i) * Delta_i, given full
 * [B, Hq, S] LSE and Delta ("Kernel 9: Dsink", tilelang-ascend PR #1638). */
void oracle_dsink(const oracle_problem* p, const double* lse, const double* delta, double* dsink) {
  if (!p->sink) {
    for (int h = 0; h < p->Hq; ++h) dsink[h] = 0.0;
    return;
  }
#pragma omp parallel for schedule(static)
  for (int h = 0; h < p->Hq; ++h) {
    double acc = 0.0;
    for (int b = 0; b < p->B; ++b)
      for (int i = 0; i < p->S; ++i) {
        const long r = ((long)b * p->Hq + h) * p->S + i;
        acc += exp(p->sink[h] - lse[r]) * delta[r];
      }
    dsink[h] = -acc;
  }
}
