/*
 * Oracle for the Mamba-3 SSM layer core -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, sequential fp64 CPU recurrence.  Only tests/, the smoke
 * check and the benchmark's CPU-baseline / reference leg may load it.  It
 * shares no code with the CUDA path and is not part of the product.
 *
 * What it computes, step by step, for one sequence (one batch row, one head),
 * in the notation of the Mamba-3 paper ("Mamba-3: Improved Sequence Modeling
 * using State Space Principles"):
 *
 *   Discretisation, Proposition 1 (exponential-trapezoidal rule, as printed on
 *   the yunpan.plus explanatory post, section "first improvement", and in the
 *   aipaper.cc summary, "Mathematical formulas", item 1):
 *       alpha_t = exp(dt_t * A)
 *       beta_t  = (1 - lambda_t) * dt_t * alpha_t
 *       gamma_t = lambda_t * dt_t
 *       h_t = alpha_t h_{t-1} + beta_t B_{t-1} x_{t-1} + gamma_t B_t x_t
 *
 *   Complex state as data-dependent RoPE, Proposition 3 (aipaper.cc summary,
 *   "Mathematical formulas", item 2; paper section 3.2): B and C are rotated
 *   by the cumulative product of the transposed 2x2 rotations R_i^T,
 *   i = 0..t inclusive.  Pair k of the state is (2k, 2k+1) and its angle
 *   is phi_k(t) = sum_{i<=t} dt_i * theta_{i,k}.  R(phi)^T maps (u, v) to
 *   (cos(phi) u + sin(phi) v, -sin(phi) u + cos(phi) v).
 *
 *   Proposition 4 (paper section 3.2.2; the equation body is missing from
 *   the pages) combines the two.  Reading taken here: the previous-token term
 *   uses B_{t-1} rotated by its own cumulative angle phi(t-1).  That is the
 *   trapezoid's left endpoint carried through the complex transition
 *   exp(dt (A + i theta)) and then moved into the rotating frame.
 *
 *   MIMO, paper section 3.3 and the aipaper.cc summary item 3: x_t becomes a
 *   P x R matrix X_t and B_t, C_t become N x R.  Each input term is the
 *   matrix product B_t X_t^T (N x P), and the output is y_t = h_t^T C~_t
 *   (P x R).  Remark 6 of section 3.3 says the three-term trapezoidal case
 *   is analogous, so both input terms become rank-R products.
 *
 * Storage.  Per sequence, row-major, innermost index last:
 *   x     [T][R][P]   (X_t stored column by column: x[t][r][p] = X_t[p, r])
 *   Bm    [T][R][N]   (Bm[t][r][n] = B_t[n, r]);  Cm likewise
 *   dt    [T], lam [T], theta [T][N/2]
 *   h     [N][P]      state, in/out
 *   phi   [N/2]       cumulative angle of the last token seen, in/out
 *   prevB [R][N], prevx [R][P]  the last token's raw B and x, in/out
 *   y     [T][R][P]   output (y[t][r][p] = y_t[p, r])
 * A fresh sequence starts from h = 0, phi = 0, prevB = 0, prevx = 0.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* (u, v) -> R(phi)^T (u, v): rotation by -phi. */
static void rot_t(double c, double s, double u, double v, double* ou, double* ov) {
  *ou = c * u + s * v;
  *ov = -s * u + c * v;
}

void m3o_scan(int T, int N, int P, int R, const double* x, const double* Bm, const double* Cm,
              const double* dt, double A, const double* lam, const double* theta, double* h,
              double* phi, double* prevB, double* prevx, double* y) {
  const int K = N / 2;
  double* Bp = (double*)malloc(sizeof(double) * (size_t)R * N); /* B~_{t-1} */
  double* Bt = (double*)malloc(sizeof(double) * (size_t)R * N); /* B~_t */
  double* Ct = (double*)malloc(sizeof(double) * (size_t)R * N); /* C~_t */

  for (int t = 0; t < T; ++t) {
    /* 1. discretisation (Proposition 1) */
    const double a = dt[t] * A;
    const double alpha = exp(a);
    const double beta = (1.0 - lam[t]) * dt[t] * alpha;
    const double gamma = lam[t] * dt[t];

    /* 2. previous token, rotated by its own cumulative angle phi(t-1) */
    for (int k = 0; k < K; ++k) {
      const double c = cos(phi[k]), s = sin(phi[k]);
      for (int r = 0; r < R; ++r)
        rot_t(c, s, prevB[r * N + 2 * k], prevB[r * N + 2 * k + 1], &Bp[r * N + 2 * k],
              &Bp[r * N + 2 * k + 1]);
    }

    /* 3. advance the cumulative angle (inclusive of token t) */
    for (int k = 0; k < K; ++k) phi[k] += dt[t] * theta[(size_t)t * K + k];

    /* 4. rotate the current B_t and C_t (Proposition 3) */
    const double* Bcur = Bm + (size_t)t * R * N;
    const double* Ccur = Cm + (size_t)t * R * N;
    for (int k = 0; k < K; ++k) {
      const double c = cos(phi[k]), s = sin(phi[k]);
      for (int r = 0; r < R; ++r) {
        rot_t(c, s, Bcur[r * N + 2 * k], Bcur[r * N + 2 * k + 1], &Bt[r * N + 2 * k],
              &Bt[r * N + 2 * k + 1]);
        rot_t(c, s, Ccur[r * N + 2 * k], Ccur[r * N + 2 * k + 1], &Ct[r * N + 2 * k],
              &Ct[r * N + 2 * k + 1]);
      }
    }

    /* 5. state update: h <- alpha h + beta B~_{t-1} X_{t-1}^T + gamma B~_t X_t^T */
    const double* xcur = x + (size_t)t * R * P;
    for (int n = 0; n < N; ++n) {
      for (int p = 0; p < P; ++p) {
        double prev_term = 0.0, cur_term = 0.0;
        for (int r = 0; r < R; ++r) {
          prev_term += Bp[r * N + n] * prevx[r * P + p];
          cur_term += Bt[r * N + n] * xcur[r * P + p];
        }
        h[(size_t)n * P + p] = alpha * h[(size_t)n * P + p] + beta * prev_term + gamma * cur_term;
      }
    }

    /* 6. output y_t = h_t^T C~_t  (P x R) */
    double* ycur = y + (size_t)t * R * P;
    for (int r = 0; r < R; ++r) {
      for (int p = 0; p < P; ++p) {
        double acc = 0.0;
        for (int n = 0; n < N; ++n) acc += h[(size_t)n * P + p] * Ct[r * N + n];
        ycur[r * P + p] = acc;
      }
    }

    /* 7. remember the raw token for the next step's trapezoid term */
    memcpy(prevB, Bcur, sizeof(double) * (size_t)R * N);
    memcpy(prevx, xcur, sizeof(double) * (size_t)R * P);
  }

  free(Bp);
  free(Bt);
  free(Ct);
}

/*
 * S independent sequences, each laid out as in m3o_scan and stacked along a
 * leading slice index.  Slices are spread over `nthreads` OpenMP threads
 * (nthreads <= 0: the runtime default).  Returns the number of threads used.
 */
int m3o_scan_batch(int S, int T, int N, int P, int R, const double* x, const double* Bm,
                   const double* Cm, const double* dt, const double* A, const double* lam,
                   const double* theta, double* h, double* phi, double* prevB, double* prevx,
                   double* y, int nthreads) {
  int used = 1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
  {
#pragma omp single
    used = omp_get_num_threads();
#pragma omp for schedule(dynamic, 1)
    for (int s = 0; s < S; ++s) {
#else
  (void)nthreads;
  {
    for (int s = 0; s < S; ++s) {
#endif
      const size_t tx = (size_t)T * R * P, tb = (size_t)T * R * N, tt = (size_t)T,
                   tth = (size_t)T * (N / 2);
      m3o_scan(T, N, P, R, x + s * tx, Bm + s * tb, Cm + s * tb, dt + s * tt, A[s], lam + s * tt,
               theta + s * tth, h + (size_t)s * N * P, phi + (size_t)s * (N / 2),
               prevB + (size_t)s * R * N, prevx + (size_t)s * R * P, y + s * tx);
    }
  }
  return used;
}
