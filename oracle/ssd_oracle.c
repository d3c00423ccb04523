/*
 * ssd_oracle.c -- plain fp64 CPU oracle for the Mamba-2 state-space layer
 * (the scalar-decay selective SSM) and its backward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the yardstick the CUDA SSD kernels
 * are checked against.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table
 * or helper with the CUDA library, and it never calls it.
 *
 * What it computes.  "Training Transformers and Hybrid models on AMD Instinct
 * MI300X Accelerators" (section "Mamba-2") names the Mamba-2 backward kernel
 * of a hybrid model and describes it by its prefix scan, its reverse scan and
 * its buffers (the decays exp(delta A), the running suffix of the state
 * gradient, dA, dB/dC); it prints no formula.  The plainest reading is the
 * Mamba-2 selective state-space recurrence with a scalar decay per head and
 * its adjoint, written out here step by step.  Per batch element b and head
 * h (group g = h / (H / G) supplies B and C), with state h_t in R^{N x P}:
 *
 *   a_t   = exp(dt_t * A)                              (decay, A < 0)
 *   h_t   = a_t h_{t-1} + dt_t B_t x_t^T,  h_{-1} = 0  (prefix scan)
 *   y_t   = h_t^T C_t + D x_t
 *
 * and, for the loss <dy, y>, the reverse scan of the state gradient
 *
 *   g_t   = C_t dy_t^T + a_{t+1} g_{t+1},  g_T = 0     (running suffix)
 *   dx_t  = dt_t g_t^T B_t + D dy_t
 *   dB_t  = dt_t g_t x_t                (summed over the heads of the group)
 *   dC_t  = h_t dy_t                    (summed over the heads of the group)
 *   ddt_t = < g_t, A a_t h_{t-1} + B_t x_t^T >
 *   dA    = sum_t < g_t, dt_t a_t h_{t-1} >
 *   dD    = sum_t < dy_t, x_t >
 *
 * How.  Pass 1 runs the recurrence forward and keeps every h_t of the head
 * (T x N x P doubles); pass 2 runs the suffix recurrence backward and forms
 * the gradients from it.  Threads (OpenMP) take (batch, head) pairs; every
 * per-head quantity is written by one thread, and the sums over heads (dB,
 * dC of a group) and over batches (dA, dD) are taken afterwards in a fixed
 * order, so results do not depend on the thread count.
 *
 * Layout (contiguous, row-major doubles):
 *   x, y, dy, dx    [Bt][T][H][P]
 *   dt, ddt         [Bt][T][H]
 *   A, D, dA, dD    [H]
 *   B, C, dB, dC    [Bt][T][G][N]
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define SSD_OK 0
#define SSD_ERR_ARG 1
#define SSD_ERR_NOMEM 2

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

static int check(long Bt, long T, long H, long G, long N, long P) {
  if (Bt < 0 || T < 0 || H < 0 || G <= 0 || N < 0 || P < 0) return SSD_ERR_ARG;
  if (H % G != 0) return SSD_ERR_ARG;
  return SSD_OK;
}

/* Pass 1 for one (b, h): every state h_t into hs [T][N][P]; y when given. */
static void scan_forward(const double *x, const double *dt, double A, const double *Bm,
                         const double *Cm, double Dh, long b, long h, long g, long T, long H,
                         long G, long N, long P, double *hs, double *y) {
  for (long t = 0; t < T; ++t) {
    const double d = dt[(b * T + t) * H + h];
    const double a = exp(d * A);
    const double *xt = x + ((b * T + t) * H + h) * P;
    const double *Bt = Bm + ((b * T + t) * G + g) * N;
    const double *Ct = Cm + ((b * T + t) * G + g) * N;
    double *cur = hs + t * N * P;
    const double *prev = t > 0 ? hs + (t - 1) * N * P : NULL;
    for (long n = 0; n < N; ++n)
      for (long p = 0; p < P; ++p)
        cur[n * P + p] = (prev ? a * prev[n * P + p] : 0.0) + d * Bt[n] * xt[p];
    if (y) {
      double *yt = y + ((b * T + t) * H + h) * P;
      for (long p = 0; p < P; ++p) {
        double acc = 0.0;
        for (long n = 0; n < N; ++n) acc += cur[n * P + p] * Ct[n];
        yt[p] = acc + Dh * xt[p];
      }
    }
  }
}

/* Forward only: y. */
int oracle_ssd_fwd(const double *x, const double *dt, const double *A, const double *Bm,
                   const double *Cm, const double *D, long Bt, long T, long H, long G, long N,
                   long P, double *y, int nthreads) {
  int st = check(Bt, T, H, G, N, P);
  if (st) return st;
  if (Bt * T * H == 0) return SSD_OK;
  if (!x || !dt || !A || !Bm || !Cm || !D || !y) return SSD_ERR_ARG;
  set_threads(nthreads);
  int failed = 0;
  const long hpg = H / G;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (long b = 0; b < Bt; ++b)
    for (long h = 0; h < H; ++h) {
      double *hs = (double *)malloc(sizeof(double) * (size_t)(T * N * P > 0 ? T * N * P : 1));
      if (!hs) {
#pragma omp atomic write
        failed = 1;
        continue;
      }
      scan_forward(x, dt, A[h], Bm, Cm, D[h], b, h, h / hpg, T, H, G, N, P, hs, y);
      free(hs);
    }
  return failed ? SSD_ERR_NOMEM : SSD_OK;
}

/* Forward and backward for the loss <dy, y>: y and every gradient. */
int oracle_ssd_fwd_bwd(const double *x, const double *dt, const double *A, const double *Bm,
                       const double *Cm, const double *D, const double *dy, long Bt, long T,
                       long H, long G, long N, long P, double *y, double *dx, double *ddt,
                       double *dA, double *dB, double *dC, double *dD, int nthreads) {
  int st = check(Bt, T, H, G, N, P);
  if (st) return st;
  if (H > 0) {
    if (!dA || !dD) return SSD_ERR_ARG;
    memset(dA, 0, sizeof(double) * (size_t)H);
    memset(dD, 0, sizeof(double) * (size_t)H);
  }
  if (Bt * T * H == 0) return SSD_OK;
  if (!x || !dt || !A || !Bm || !Cm || !D || !dy || !y || !dx || !ddt || !dB || !dC)
    return SSD_ERR_ARG;
  set_threads(nthreads);
  const long hpg = H / G;
  /* per (b, h) partials: dA, dD, and dB, dC [Bt][H][T][N], summed over the
   * heads of each group (and dA, dD over batches) in a fixed order below */
  double *pA = (double *)calloc((size_t)(Bt * H), sizeof(double));
  double *pD = (double *)calloc((size_t)(Bt * H), sizeof(double));
  double *pB = (double *)calloc((size_t)(Bt * H * T * N > 0 ? Bt * H * T * N : 1),
                                sizeof(double));
  double *pC = (double *)calloc((size_t)(Bt * H * T * N > 0 ? Bt * H * T * N : 1),
                                sizeof(double));
  if (!pA || !pD || !pB || !pC) {
    free(pA);
    free(pD);
    free(pB);
    free(pC);
    return SSD_ERR_NOMEM;
  }
  int failed = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (long b = 0; b < Bt; ++b)
    for (long h = 0; h < H; ++h) {
      const long g = h / hpg;
      double *hs = (double *)malloc(sizeof(double) * (size_t)(T * N * P > 0 ? T * N * P : 1));
      double *gs = (double *)malloc(sizeof(double) * (size_t)(N * P > 0 ? N * P : 1));
      if (!hs || !gs) {
        free(hs);
        free(gs);
#pragma omp atomic write
        failed = 1;
        continue;
      }
      const double Ah = A[h], Dh = D[h];
      scan_forward(x, dt, Ah, Bm, Cm, Dh, b, h, g, T, H, G, N, P, hs, y);
      memset(gs, 0, sizeof(double) * (size_t)(N * P)); /* g_T = 0 */
      double sumA = 0.0, sumD = 0.0;
      double a_next = 0.0; /* a_{t+1}; unused at t = T - 1 (g_T = 0) */
      for (long t = T - 1; t >= 0; --t) {
        const double d = dt[(b * T + t) * H + h];
        const double a = exp(d * Ah);
        const double *xt = x + ((b * T + t) * H + h) * P;
        const double *dyt = dy + ((b * T + t) * H + h) * P;
        const double *Bt_ = Bm + ((b * T + t) * G + g) * N;
        const double *Ct = Cm + ((b * T + t) * G + g) * N;
        const double *ht = hs + t * N * P;
        const double *hp = t > 0 ? hs + (t - 1) * N * P : NULL;
        /* g_t = C_t dy_t^T + a_{t+1} g_{t+1} */
        for (long n = 0; n < N; ++n)
          for (long p = 0; p < P; ++p) gs[n * P + p] = Ct[n] * dyt[p] + a_next * gs[n * P + p];
        double *dxt = dx + ((b * T + t) * H + h) * P;
        for (long p = 0; p < P; ++p) {
          double acc = 0.0;
          for (long n = 0; n < N; ++n) acc += gs[n * P + p] * Bt_[n];
          dxt[p] = d * acc + Dh * dyt[p];
        }
        double *dBt = pB + ((b * H + h) * T + t) * N;
        double *dCt = pC + ((b * H + h) * T + t) * N;
        for (long n = 0; n < N; ++n) {
          double accb = 0.0, accc = 0.0;
          for (long p = 0; p < P; ++p) {
            accb += gs[n * P + p] * xt[p];
            accc += ht[n * P + p] * dyt[p];
          }
          dBt[n] = d * accb;
          dCt[n] = accc;
        }
        double dd = 0.0, da = 0.0;
        for (long n = 0; n < N; ++n)
          for (long p = 0; p < P; ++p) {
            const double prev = hp ? hp[n * P + p] : 0.0;
            dd += gs[n * P + p] * (Ah * a * prev + Bt_[n] * xt[p]);
            da += gs[n * P + p] * d * a * prev;
          }
        ddt[(b * T + t) * H + h] = dd;
        sumA += da;
        for (long p = 0; p < P; ++p) sumD += dyt[p] * xt[p];
        a_next = a;
      }
      pA[b * H + h] = sumA;
      pD[b * H + h] = sumD;
      free(hs);
      free(gs);
    }
  /* dB, dC: the sum over the heads of each group, in head order */
#pragma omp parallel for collapse(2) schedule(static)
  for (long b = 0; b < Bt; ++b)
    for (long t = 0; t < T; ++t)
      for (long g = 0; g < G; ++g)
        for (long n = 0; n < N; ++n) {
          double sb = 0.0, sc = 0.0;
          for (long h = g * hpg; h < (g + 1) * hpg; ++h) {
            sb += pB[((b * H + h) * T + t) * N + n];
            sc += pC[((b * H + h) * T + t) * N + n];
          }
          dB[((b * T + t) * G + g) * N + n] = sb;
          dC[((b * T + t) * G + g) * N + n] = sc;
        }
  for (long h = 0; h < H; ++h)
    for (long b = 0; b < Bt; ++b) {
      dA[h] += pA[b * H + h];
      dD[h] += pD[b * H + h];
    }
  free(pA);
  free(pD);
  free(pB);
  free(pC);
  return failed ? SSD_ERR_NOMEM : SSD_OK;
}

int oracle_ssd_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
