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

/* Number of keys row i may attend to. */
static long row_len(long i, long N, int causal) { return causal ? i + 1 : N; }

/* Fill srow[j] = scale * <q_i, k_j> for the unmasked keys j of row i and
 * return how many there are. */
static long scores_row(const double *Qh, const double *Kh, long i, long N,
                       long d, int causal, double scale, double *srow) {
  long n = row_len(i, N, causal);
  const double *qi = Qh + i * d;
  for (long j = 0; j < n; ++j) srow[j] = scale * dot(qi, Kh + j * d, d);
  return n;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

/* Pass 1: L, O and D for every query row. */
static int pass_forward(const double *Q, const double *K, const double *V,
                        const double *dO, long BH, long N, long d, int causal,
                        double scale, double *O, double *L, double *D) {
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
        const double *Qh = Q + h * N * d, *Kh = K + h * N * d;
        const double *Vh = V + h * N * d;
        long n = scores_row(Qh, Kh, i, N, d, causal, scale, srow);
        double m = -INFINITY;
        for (long j = 0; j < n; ++j) m = srow[j] > m ? srow[j] : m;
        double l = 0.0;
        for (long j = 0; j < n; ++j) l += exp(srow[j] - m);
        double Li = m + log(l);
        L[h * N + i] = Li;
        double *Oi = O + (h * N + i) * d;
        for (long c = 0; c < d; ++c) Oi[c] = 0.0;
        for (long j = 0; j < n; ++j) {
          double p = exp(srow[j] - Li);
          const double *vj = Vh + j * d;
          for (long c = 0; c < d; ++c) Oi[c] += p * vj[c];
        }
        if (D) D[h * N + i] = dot(dO + (h * N + i) * d, Oi, d);
      }
    }
    free(srow);
  }
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* Pass 2: dQ_i = s * sum_j P_ij (dP_ij - D_i) k_j for every query row. */
static int pass_dq(const double *Q, const double *K, const double *V,
                   const double *dO, const double *L, const double *D, long BH,
                   long N, long d, int causal, double scale, double *dQ) {
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
        const double *Qh = Q + h * N * d, *Kh = K + h * N * d;
        const double *Vh = V + h * N * d;
        const double *dOi = dO + (h * N + i) * d;
        long n = scores_row(Qh, Kh, i, N, d, causal, scale, srow);
        double Li = L[h * N + i], Di = D[h * N + i];
        double *dQi = dQ + (h * N + i) * d;
        for (long c = 0; c < d; ++c) dQi[c] = 0.0;
        for (long j = 0; j < n; ++j) {
          double p = exp(srow[j] - Li);
          double dp = dot(dOi, Vh + j * d, d);
          double ds = p * (dp - Di);
          const double *kj = Kh + j * d;
          for (long c = 0; c < d; ++c) dQi[c] += ds * kj[c];
        }
        for (long c = 0; c < d; ++c) dQi[c] *= scale;
      }
    }
    free(srow);
  }
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* Pass 3: dK_j = s * sum_i dS_ij q_i and dV_j = sum_i P_ij dO_i for every key
 * row j.  Under the causal mask, key j is seen by query rows i >= j only. */
static int pass_dkdv(const double *Q, const double *K, const double *V,
                     const double *dO, const double *L, const double *D,
                     long BH, long N, long d, int causal, double scale,
                     double *dK, double *dV) {
#pragma omp parallel for collapse(2) schedule(dynamic, 16)
  for (long h = 0; h < BH; ++h) {
    for (long j = 0; j < N; ++j) {
      const double *Qh = Q + h * N * d, *Kh = K + h * N * d;
      const double *Vh = V + h * N * d, *dOh = dO + h * N * d;
      const double *kj = Kh + j * d, *vj = Vh + j * d;
      double *dKj = dK + (h * N + j) * d, *dVj = dV + (h * N + j) * d;
      for (long c = 0; c < d; ++c) dKj[c] = dVj[c] = 0.0;
      long i0 = causal ? j : 0;
      for (long i = i0; i < N; ++i) {
        const double *qi = Qh + i * d, *dOi = dOh + i * d;
        double sij = scale * dot(qi, kj, d);
        double p = exp(sij - L[h * N + i]);
        double dp = dot(dOi, vj, d);
        double ds = p * (dp - D[h * N + i]);
        for (long c = 0; c < d; ++c) {
          dKj[c] += ds * qi[c];
          dVj[c] += p * dOi[c];
        }
      }
      for (long c = 0; c < d; ++c) dKj[c] *= scale;
    }
  }
  return ORACLE_OK;
}

static int check_args(const void *a, const void *b, const void *c, long BH,
                      long N, long d, double scale) {
  if (BH < 0 || N < 0 || d < 0) return ORACLE_ERR_ARG;
  if (BH * N * d > 0 && (!a || !b || !c)) return ORACLE_ERR_ARG;
  if (!(scale == scale)) return ORACLE_ERR_ARG; /* NaN */
  return ORACLE_OK;
}

/* Forward only: O [BH][N][d] and L [BH][N]. */
int oracle_attn_fwd(const double *Q, const double *K, const double *V, long BH,
                    long N, long d, int causal, double scale, double *O,
                    double *L, int nthreads) {
  int st = check_args(Q, K, V, BH, N, d, scale);
  if (st) return st;
  if (BH * N == 0) return ORACLE_OK;
  if (!O || !L) return ORACLE_ERR_ARG;
  set_threads(nthreads);
  return pass_forward(Q, K, V, NULL, BH, N, d, causal, scale, O, L, NULL);
}

/* Forward and backward: O, L, D = rowsum(dO * O), dQ, dK, dV. */
int oracle_attn_fwd_bwd(const double *Q, const double *K, const double *V,
                        const double *dO, long BH, long N, long d, int causal,
                        double scale, double *O, double *L, double *D,
                        double *dQ, double *dK, double *dV, int nthreads) {
  int st = check_args(Q, K, V, BH, N, d, scale);
  if (st) return st;
  if (BH * N == 0) return ORACLE_OK;
  if (!dO || !O || !L || !D || !dQ || !dK || !dV) return ORACLE_ERR_ARG;
  set_threads(nthreads);
  st = pass_forward(Q, K, V, dO, BH, N, d, causal, scale, O, L, D);
  if (st) return st;
  st = pass_dq(Q, K, V, dO, L, D, BH, N, d, causal, scale, dQ);
  if (st) return st;
  return pass_dkdv(Q, K, V, dO, L, D, BH, N, d, causal, scale, dK, dV);
}

/* Threads the oracle would use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
