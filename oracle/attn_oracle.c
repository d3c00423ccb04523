/*
 * attn_oracle.c -- plain fp64 CPU oracle for exact softmax attention and
 * its analytic gradients.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the yardstick the CUDA path is
 * checked against.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header, table or helper
 * with the CUDA library, and it never calls it.
 *
 * What it computes.  The pages this project follows ("Training Transformers
 * and Hybrid models on AMD Instinct MI300X Accelerators", section "Flash
 * Attention" and section "Harnessing the MI300 Hardware Specs") name the
 * FlashAttention-2 forward and backward kernels and say the backward
 * recomputes activations; they print no formula.  FlashAttention computes
 * exact softmax attention, so this oracle is the textbook definition of that
 * quantity and of its gradient, written out with no tiling:
 *
 *   per head, with s = scale and mask M_ij = 0 if (not causal or j <= i)
 *   else -inf:
 *     S_ij  = s * <q_i, k_j> + M_ij
 *     L_i   = max_j S_ij + ln sum_j exp(S_ij - max_j S_ij)   (log-sum-exp)
 *     P_ij  = exp(S_ij - L_i)
 *     O_i   = sum_j P_ij v_j
 *     D_i   = <dO_i, O_i>
 *     dP_ij = <dO_i, v_j>
 *     dS_ij = P_ij (dP_ij - D_i)
 *     dQ_i  = s * sum_j dS_ij k_j
 *     dK_j  = s * sum_i dS_ij q_i
 *     dV_j  = sum_i P_ij dO_i
 *
 * The causal mask is the square, top-left aligned one ("Training - CUDA Moat
 * Still Alive", section on the model-FLOP formula, calls causal attention a
 * mask of 50% density).  Every row keeps at least its diagonal entry, so no
 * row is empty.
 *
 * Sliding window.  With causal and a window W > 0, key j is visible to query
 * i when i - W < j <= i: each query sees itself and the W - 1 keys before it
 * (the banded causal mask of sliding-window attention, named in "Training -
 * CUDA Moat Still Alive", section on attention variants, as the Mistral 7B
 * mask).  M_ij = -inf outside the band; W >= N is the plain causal mask.
 *
 * Documents.  With causal and a document map (several sequences packed into
 * one), key j is visible to query i only when both belong to the same
 * document: doc[i] <= j <= i, where doc[i] is the first position of the
 * document holding position i (FlexAttention's document mask, named in the
 * same section).  A window and documents combine: j >= max(doc[i], i - W + 1).
 *
 * How.  Three passes over the rows of each head, each a direct evaluation of
 * the definition above, all in double precision:
 *   pass 1, over query rows i:   L_i, O_i, D_i
 *   pass 2, over query rows i:   dQ_i   (needs L_i, D_i of its own row)
 *   pass 3, over key rows j:     dK_j, dV_j (needs L_i, D_i of every row)
 * Each pass keeps one length-N scratch row per thread, so no N x N matrix is
 * ever stored.  Threads (OpenMP, when built with it) split the rows; every
 * output element is written by exactly one thread, so the result does not
 * depend on the thread count.
 *
 * Layout.  All tensors are contiguous row-major doubles: Q, K, V, dO, O, dQ,
 * dK, dV are [BH][N][d]; L and D are [BH][N].  BH is the number of
 * independent heads (batch times heads).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NOMEM 2

static double dot(const double *a, const double *b, long d) {
  double acc = 0.0;
  for (long c = 0; c < d; ++c) acc += a[c] * b[c];
  return acc;
}

/* The mask of one head: causal or not, a sliding window (0 = none), and the
 * document map of the head ([N], NULL = one document). */
typedef struct {
  int causal;
  long window;
  const long *doc;
} Mask;

/* One past the last key row i may attend to. */
static long row_len(long i, long N, int causal) { return causal ? i + 1 : N; }

/* The first key row i may attend to: under a sliding window W, i - W + 1;
 * with documents, no earlier than the start of i's document. */
static long row_start(long i, const Mask *mk) {
  long window = mk->window;
  long lo = (mk->causal && window > 0 && i - window + 1 > 0) ? i - window + 1 : 0;
  if (mk->causal && mk->doc && mk->doc[i] > lo) lo = mk->doc[i];
  return lo;
}

/* Fill srow[j] = scale * <q_i, k_j> for the unmasked keys j of row i, which
 * are lo <= j < n; set *lo and return n. */
static long scores_row(const double *Qh, const double *Kh, long i, long N,
                       long d, const Mask *mk, double scale, double *srow, long *lo) {
  long n = row_len(i, N, mk->causal);
  const double *qi = Qh + i * d;
  *lo = row_start(i, mk);
  for (long j = *lo; j < n; ++j) srow[j] = scale * dot(qi, Kh + j * d, d);
  return n;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

/* L_i, O_i and (when dOh is given) D_i = <dO_i, O_i> for one query row i of
 * one head. */
static void fwd_row(const double *Qh, const double *Kh, const double *Vh,
                    const double *dOh, long N, long d, const Mask *mk,
                    double scale, long i, double *srow, double *Li_out, double *Oi,
                    double *Di_out) {
  long lo;
  long n = scores_row(Qh, Kh, i, N, d, mk, scale, srow, &lo);
  double m = -INFINITY;
  for (long j = lo; j < n; ++j) m = srow[j] > m ? srow[j] : m;
  double l = 0.0;
  for (long j = lo; j < n; ++j) l += exp(srow[j] - m);
  double Li = m + log(l);
  *Li_out = Li;
  for (long c = 0; c < d; ++c) Oi[c] = 0.0;
  for (long j = lo; j < n; ++j) {
    double p = exp(srow[j] - Li);
    const double *vj = Vh + j * d;
    for (long c = 0; c < d; ++c) Oi[c] += p * vj[c];
  }
  if (dOh && Di_out) *Di_out = dot(dOh + i * d, Oi, d);
}

/* Pass 1: L, O and D for every query row. */
static int pass_forward(const double *Q, const double *K, const double *V,
                        const double *dO, long BH, long N, long d, int causal,
                        long window, const long *doc, double scale, double *O, double *L,
                        double *D) {
  int failed = 0;
#pragma omp parallel
  {
    double *srow = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    if (!srow) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for collapse(2) schedule(dynamic, 16)
    for (long h = 0; h < BH; ++h) {
      for (long i = 0; i < N; ++i) {
        if (!srow) continue;
        const Mask mk = {causal, window, doc ? doc + h * N : NULL};
        fwd_row(Q + h * N * d, K + h * N * d, V + h * N * d,
                dO ? dO + h * N * d : NULL, N, d, &mk, scale, i, srow,
                L + h * N + i, O + (h * N + i) * d, D ? D + h * N + i : NULL);
      }
    }
    free(srow);
  }
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* dQ_i = s * sum_j P_ij (dP_ij - D_i) k_j for one query row i of one head. */
static void dq_row(const double *Qh, const double *Kh, const double *Vh,
                   const double *dOh, double Li, double Di, long N, long d,
                   const Mask *mk, double scale, long i, double *srow, double *dQi) {
  const double *dOi = dOh + i * d;
  long lo;
  long n = scores_row(Qh, Kh, i, N, d, mk, scale, srow, &lo);
  for (long c = 0; c < d; ++c) dQi[c] = 0.0;
  for (long j = lo; j < n; ++j) {
    double p = exp(srow[j] - Li);
    double dp = dot(dOi, Vh + j * d, d);
    double ds = p * (dp - Di);
    const double *kj = Kh + j * d;
    for (long c = 0; c < d; ++c) dQi[c] += ds * kj[c];
  }
  for (long c = 0; c < d; ++c) dQi[c] *= scale;
}

/* dK_j = s * sum_i dS_ij q_i and dV_j = sum_i P_ij dO_i for one key row j of
 * one head.  Under the causal mask, key j is seen by query rows i >= j only;
 * under a sliding window W also only by rows i < j + W; with documents only
 * by rows of its own document. */
static void dkdv_row(const double *Qh, const double *Kh, const double *Vh,
                     const double *dOh, const double *Lh, const double *Dh, long N,
                     long d, const Mask *mk, double scale, long j, double *dKj,
                     double *dVj) {
  const double *kj = Kh + j * d, *vj = Vh + j * d;
  const int causal = mk->causal;
  const long window = mk->window;
  for (long c = 0; c < d; ++c) dKj[c] = dVj[c] = 0.0;
  long i0 = causal ? j : 0;
  long i1 = (causal && window > 0 && j + window < N) ? j + window : N;
  for (long i = i0; i < i1; ++i) {
    if (row_start(i, mk) > j) continue;  /* j is outside row i's document */
    const double *qi = Qh + i * d, *dOi = dOh + i * d;
    double sij = scale * dot(qi, kj, d);
    double p = exp(sij - Lh[i]);
    double dp = dot(dOi, vj, d);
    double ds = p * (dp - Dh[i]);
    for (long c = 0; c < d; ++c) {
      dKj[c] += ds * qi[c];
      dVj[c] += p * dOi[c];
    }
  }
  for (long c = 0; c < d; ++c) dKj[c] *= scale;
}

/* Pass 2: dQ for every query row. */
static int pass_dq(const double *Q, const double *K, const double *V,
                   const double *dO, const double *L, const double *D, long BH,
                   long N, long d, int causal, long window, const long *doc, double scale,
                   double *dQ) {
  int failed = 0;
#pragma omp parallel
  {
    double *srow = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    if (!srow) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for collapse(2) schedule(dynamic, 16)
    for (long h = 0; h < BH; ++h) {
      for (long i = 0; i < N; ++i) {
        if (!srow) continue;
        const Mask mk = {causal, window, doc ? doc + h * N : NULL};
        dq_row(Q + h * N * d, K + h * N * d, V + h * N * d, dO + h * N * d,
               L[h * N + i], D[h * N + i], N, d, &mk, scale, i, srow,
               dQ + (h * N + i) * d);
      }
    }
    free(srow);
  }
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* Pass 3: dK and dV for every key row. */
static int pass_dkdv(const double *Q, const double *K, const double *V,
                     const double *dO, const double *L, const double *D,
                     long BH, long N, long d, int causal, long window, const long *doc,
                     double scale, double *dK, double *dV) {
#pragma omp parallel for collapse(2) schedule(dynamic, 16)
  for (long h = 0; h < BH; ++h) {
    for (long j = 0; j < N; ++j) {
      const Mask mk = {causal, window, doc ? doc + h * N : NULL};
      dkdv_row(Q + h * N * d, K + h * N * d, V + h * N * d, dO + h * N * d,
               L + h * N, D + h * N, N, d, &mk, scale, j,
               dK + (h * N + j) * d, dV + (h * N + j) * d);
    }
  }
  return ORACLE_OK;
}

static int check_args(const void *a, const void *b, const void *c, long BH,
                      long N, long d, int causal, long window, const long *doc,
                      double scale) {
  if (BH < 0 || N < 0 || d < 0) return ORACLE_ERR_ARG;
  if (window < 0 || (window > 0 && !causal)) return ORACLE_ERR_ARG; /* the band is causal */
  if (doc && !causal) return ORACLE_ERR_ARG;                         /* so are documents */
  /* a document map: doc[i] = i (a document starts) or doc[i - 1] */
  for (long h = 0; doc && h < BH; ++h)
    for (long i = 0; i < N; ++i) {
      long v = doc[h * N + i];
      if (!(v == i || (i > 0 && v == doc[h * N + i - 1]))) return ORACLE_ERR_ARG;
    }
  if (BH * N * d > 0 && (!a || !b || !c)) return ORACLE_ERR_ARG;
  if (!(scale == scale)) return ORACLE_ERR_ARG; /* NaN */
  return ORACLE_OK;
}

/* Forward only: O [BH][N][d] and L [BH][N]. */
int oracle_attn_fwd(const double *Q, const double *K, const double *V, long BH,
                    long N, long d, int causal, long window, const long *doc,
                    double scale, double *O, double *L, int nthreads) {
  int st = check_args(Q, K, V, BH, N, d, causal, window, doc, scale);
  if (st) return st;
  if (BH * N == 0) return ORACLE_OK;
  if (!O || !L) return ORACLE_ERR_ARG;
  set_threads(nthreads);
  return pass_forward(Q, K, V, NULL, BH, N, d, causal, window, doc, scale, O, L, NULL);
}

/* Forward and backward: O, L, D = rowsum(dO * O), dQ, dK, dV. */
int oracle_attn_fwd_bwd(const double *Q, const double *K, const double *V,
                        const double *dO, long BH, long N, long d, int causal,
                        long window, const long *doc, double scale, double *O, double *L,
                        double *D, double *dQ, double *dK, double *dV, int nthreads) {
  int st = check_args(Q, K, V, BH, N, d, causal, window, doc, scale);
  if (st) return st;
  if (BH * N == 0) return ORACLE_OK;
  if (!dO || !O || !L || !D || !dQ || !dK || !dV) return ORACLE_ERR_ARG;
  set_threads(nthreads);
  st = pass_forward(Q, K, V, dO, BH, N, d, causal, window, doc, scale, O, L, D);
  if (st) return st;
  st = pass_dq(Q, K, V, dO, L, D, BH, N, d, causal, window, doc, scale, dQ);
  if (st) return st;
  return pass_dkdv(Q, K, V, dO, L, D, BH, N, d, causal, window, doc, scale, dK, dV);
}

/* Threads the oracle would use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Sampled rows of one head, for shapes too large to evaluate in full.
 * Pass 1 runs over every query row (dK_j and dV_j need L_i and D_i of all
 * rows); passes 2 and 3 run only over the requested query rows qrows[0..nq)
 * and key rows krows[0..nk).  Outputs: O_rows, dQ_rows [nq][d], L_rows [nq],
 * dK_rows, dV_rows [nk][d].  Q, K, V, dO are one head, [N][d]. */
int oracle_attn_head_rows(const double *Q, const double *K, const double *V,
                          const double *dO, long N, long d, int causal, long window,
                          const long *doc, double scale, long nq, const long *qrows, long nk,
                          const long *krows, double *O_rows, double *L_rows,
                          double *dQ_rows, double *dK_rows, double *dV_rows,
                          int nthreads) {
  int st = check_args(Q, K, V, 1, N, d, causal, window, doc, scale);
  if (st) return st;
  if (nq < 0 || nk < 0 || (nq && (!qrows || !O_rows || !L_rows || !dQ_rows)) ||
      (nk && (!krows || !dK_rows || !dV_rows)) || !dO)
    return ORACLE_ERR_ARG;
  for (long t = 0; t < nq; ++t)
    if (qrows[t] < 0 || qrows[t] >= N) return ORACLE_ERR_ARG;
  for (long t = 0; t < nk; ++t)
    if (krows[t] < 0 || krows[t] >= N) return ORACLE_ERR_ARG;
  if (N == 0) return ORACLE_OK;
  set_threads(nthreads);
  const Mask mk = {causal, window, doc};
  if (nk == 0) {
    /* Query rows only: O_i, L_i, D_i and dQ_i depend on row i alone. */
    int failed = 0;
#pragma omp parallel
    {
      double *srow = (double *)malloc(sizeof(double) * (size_t)N);
      double Li = 0.0, Di = 0.0;
      if (!srow) {
#pragma omp atomic write
        failed = 1;
      }
#pragma omp for schedule(dynamic, 1)
      for (long t = 0; t < nq; ++t) {
        if (!srow) continue;
        long i = qrows[t];
        fwd_row(Q, K, V, dO, N, d, &mk, scale, i, srow, &Li, O_rows + t * d, &Di);
        L_rows[t] = Li;
        dq_row(Q, K, V, dO, Li, Di, N, d, &mk, scale, i, srow, dQ_rows + t * d);
      }
      free(srow);
    }
    return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
  }
  double *O = (double *)malloc(sizeof(double) * (size_t)(N * d));
  double *L = (double *)malloc(sizeof(double) * (size_t)N);
  double *D = (double *)malloc(sizeof(double) * (size_t)N);
  if (!O || !L || !D) {
    free(O); free(L); free(D);
    return ORACLE_ERR_NOMEM;
  }
  st = pass_forward(Q, K, V, dO, 1, N, d, causal, window, doc, scale, O, L, D);
  if (!st) {
    int failed = 0;
#pragma omp parallel
    {
      double *srow = (double *)malloc(sizeof(double) * (size_t)N);
      if (!srow) {
#pragma omp atomic write
        failed = 1;
      }
#pragma omp for schedule(dynamic, 1)
      for (long t = 0; t < nq; ++t) {
        if (!srow) continue;
        long i = qrows[t];
        memcpy(O_rows + t * d, O + i * d, sizeof(double) * (size_t)d);
        L_rows[t] = L[i];
        dq_row(Q, K, V, dO, L[i], D[i], N, d, &mk, scale, i, srow, dQ_rows + t * d);
      }
#pragma omp for schedule(dynamic, 1)
      for (long t = 0; t < nk; ++t)
        dkdv_row(Q, K, V, dO, L, D, N, d, &mk, scale, krows[t], dK_rows + t * d,
                 dV_rows + t * d);
      free(srow);
    }
    if (failed) st = ORACLE_ERR_NOMEM;
  }
  free(O); free(L); free(D);
  return st;
}

/* Rounding budget of a backward whose P and dS are rounded to 8 bits.
 *
 * For the fp8 backward the test needs, per output element, the sums that
 * the rounding errors of P and dS are multiplied by:
 *   vP[j][c]  = sum_i P_ij^2 dO_ic^2      (dV_jc = sum_i P_ij dO_ic)
 *   vK[j][c]  = sum_i dS_ij^2 q_ic^2      (dK_jc = s sum_i dS_ij q_ic)
 *   vQ[i][c]  = sum_j dS_ij^2 k_jc^2      (dQ_ic = s sum_j dS_ij k_jc)
 *   nvis[j]   = number of query rows that see key j (for the absolute error
 *               of values below the 8-bit format's normal range)
 * and the largest |dS_ij| of each head, dsmax[h].  P and dS are the same
 * quantities as in the backward above (plain masks: causal or none), from
 * the L and D that oracle_attn_fwd_bwd returned. */
static void budget_query_row(const double *Qh, const double *Kh, const double *Vh,
                             const double *dOh, double Lrow, double Drow, long N, long d,
                             int causal, double scale, long i, double *vQi, double *dsmax_row) {
  const double *qrow = Qh + i * d, *dorow = dOh + i * d;
  const long nk = causal ? i + 1 : N;
  double mx = 0.0;
  for (long c = 0; c < d; ++c) vQi[c] = 0.0;
  for (long j = 0; j < nk; ++j) {
    const double prob = exp(scale * dot(qrow, Kh + j * d, d) - Lrow);
    const double dsv = prob * (dot(dorow, Vh + j * d, d) - Drow);
    const double *krow = Kh + j * d;
    for (long c = 0; c < d; ++c) vQi[c] += dsv * dsv * krow[c] * krow[c];
    if (fabs(dsv) > mx) mx = fabs(dsv);
  }
  *dsmax_row = mx;
}

static void budget_key_row(const double *Qh, const double *Kh, const double *Vh,
                           const double *dOh, const double *Lh, const double *Dh, long N,
                           long d, int causal, double scale, long j, double *vPj, double *vKj,
                           double *nvis) {
  const double *krow = Kh + j * d, *vrow = Vh + j * d;
  for (long c = 0; c < d; ++c) vPj[c] = vKj[c] = 0.0;
  const long first = causal ? j : 0;
  for (long i = first; i < N; ++i) {
    const double *qrow = Qh + i * d, *dorow = dOh + i * d;
    const double prob = exp(scale * dot(qrow, krow, d) - Lh[i]);
    const double dsv = prob * (dot(dorow, vrow, d) - Dh[i]);
    for (long c = 0; c < d; ++c) {
      vPj[c] += prob * prob * dorow[c] * dorow[c];
      vKj[c] += dsv * dsv * qrow[c] * qrow[c];
    }
  }
  *nvis = (double)(N - first);
}

int oracle_attn_bwd_budget(const double *Q, const double *K, const double *V, const double *dO,
                           const double *L, const double *D, long BH, long N, long d,
                           int causal, double scale, double *vP, double *vK, double *vQ,
                           double *nvis, double *dsmax, int nthreads) {
  if (BH < 0 || N < 0 || d < 0) return ORACLE_ERR_ARG;
  if (BH * N == 0) return ORACLE_OK;
  if (!Q || !K || !V || !dO || !L || !D || !vP || !vK || !vQ || !nvis || !dsmax)
    return ORACLE_ERR_ARG;
  set_threads(nthreads);
  double *rowmax = (double *)malloc(sizeof(double) * (size_t)(BH * N));
  if (!rowmax) return ORACLE_ERR_NOMEM;
#pragma omp parallel for collapse(2) schedule(dynamic, 16)
  for (long h = 0; h < BH; ++h)
    for (long r = 0; r < N; ++r) {
      const double *Qh = Q + h * N * d, *Kh = K + h * N * d, *Vh = V + h * N * d;
      const double *dOh = dO + h * N * d;
      budget_query_row(Qh, Kh, Vh, dOh, L[h * N + r], D[h * N + r], N, d, causal, scale, r,
                       vQ + (h * N + r) * d, rowmax + h * N + r);
      budget_key_row(Qh, Kh, Vh, dOh, L + h * N, D + h * N, N, d, causal, scale, r,
                     vP + (h * N + r) * d, vK + (h * N + r) * d, nvis + h * N + r);
    }
  for (long h = 0; h < BH; ++h) {
    double m = 0.0;
    for (long r = 0; r < N; ++r) m = rowmax[h * N + r] > m ? rowmax[h * N + r] : m;
    dsmax[h] = m;
  }
  free(rowmax);
  return ORACLE_OK;
}
