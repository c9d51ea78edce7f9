/*
 * Reference oracle for elu(x)+1 linear attention -- TEST INFRASTRUCTURE ONLY.
 *
 * This file is the plain, slow, fp64 CPU statement of what the method computes.
 * It exists so that the CUDA library can be checked against it.  It is not part
 * of the product: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header or constant with the
 * CUDA library.
 *
 * Sources (cited by page title and section/equation):
 *   [TR2]  "Transformers are RNNs: Fast Autoregressive Transformers with Linear
 *          Attention -- part 2/3": eq. 7 (feature map), §3.3 eq. 8-12 (causal
 *          masking), §3.3.1 eq. 13-15 (cumulative-sum gradients), §3.4
 *          eq. 16-20 (RNN form).
 *   [TRN]  papercache note "Transformers are RNNs" (Chinese summary), appendix A
 *          "gradient derivation" (numerator gradients; the denominator is left
 *          to automatic differentiation there).
 *   [LA]   "Linear Attention/zh": "kernel reformulation" section (non-causal form
 *          with a shared S and z), "recurrent form and autoregressive
 *          inference" section, and the RetNet item of "variants and
 *          extensions" (a decay factor gamma in (0, 1): S_t = gamma S_{t-1} +
 *          phi(k_t) v_t^T).
 *
 * Layout: every array is a dense row-major double array.  Heads are flattened:
 * head index hh in [0, B*H) addresses q[hh][n][d], v[hh][n][m] and so on.
 * Decode inputs are stored per step: q[t][hh][d].
 *
 * Readings taken where the pages are silent (each also listed in the design
 * notes): ELU alpha = 1; no 1/sqrt(D) temperature; no epsilon in the
 * denominator; the denominator gradient follows the same cumulative-sum
 * structure as eq. 13-15 with V_j replaced by the constant 1; decode updates the
 * state before reading it (eq. 18-20 use s_i, not s_{i-1}); padded positions of
 * the non-causal form contribute nothing and receive zero output and gradient;
 * with the RetNet decay the normaliser z decays with S (z_t = gamma z_{t-1} +
 * phi(k_t)), so that V'_i stays a convex combination of the values, and
 * gamma = 1 is the undecayed method.
 *
 * Parity status: every function here is pinned by tests that do not retype its
 * formulas (two independent forms, closed forms, invariants, central finite
 * differences, library GEMMs); see tests/test_oracle.py.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- feature map */

/* [TR2] eq. 7: phi(x) = elu(x) + 1 with the standard ELU (alpha = 1):
 * elu(x) = x for x > 0 and exp(x) - 1 otherwise, so phi(x) = x + 1 or exp(x). */
static double phi(double x) { return x > 0.0 ? x + 1.0 : exp(x); }

/* Derivative of eq. 7: 1 for x > 0, exp(x) otherwise (never zero, which is the
 * reason the pages give for preferring elu over relu). */
static double dphi(double x) { return x > 0.0 ? 1.0 : exp(x); }

void orc_phi(long n, const double* x, double* y, double* dy) {
  for (long i = 0; i < n; ++i) {
    y[i] = phi(x[i]);
    if (dy) dy[i] = dphi(x[i]);
  }
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

int orc_openmp_enabled(void) {
#ifdef _OPENMP
  return 1;
#else
  return 0;
#endif
}

/* ------------------------------------------------ causal, quadratic form (Q) */

/* [TR2] §3.3 eq. 8 with sim(q, k) = phi(q)^T phi(k) (the similarity of eq. 9):
 *   A_ij  = phi(Q_i) . phi(K_j)                 for j <= i
 *   den_i = sum_{j<=i} A_ij
 *   V'_i  = sum_{j<=i} A_ij V_j / den_i
 * The N x N matrix is built explicitly, one row at a time.  With the RetNet
 * decay of [LA] every pair is weighted by gamma^(i-j) in both sums (A_ij ->
 * gamma^(i-j) A_ij); gamma = 1 is eq. 8 itself. */
void orc_causal_fwd_quadratic_decay(int BH, int N, int D, int M, const double* q,
                                    const double* k, const double* v, double gamma,
                                    double* out, double* den, int nthreads) {
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
  for (int hh = 0; hh < BH; ++hh) {
    const double* Q = q + (size_t)hh * N * D;
    const double* K = k + (size_t)hh * N * D;
    const double* V = v + (size_t)hh * N * M;
    double* O = out + (size_t)hh * N * M;
    double* row = (double*)malloc(sizeof(double) * (size_t)N);
    for (int i = 0; i < N; ++i) {
      double s = 0.0;
      for (int j = 0; j <= i; ++j) {
        double a = 0.0;
        for (int d = 0; d < D; ++d) a += phi(Q[(size_t)i * D + d]) * phi(K[(size_t)j * D + d]);
        a *= pow(gamma, (double)(i - j)); /* the decay of the pair: gamma^(i-j), 1 when gamma = 1 */
        row[j] = a;
        s += a;
      }
      if (den) den[(size_t)hh * N + i] = s;
      for (int m = 0; m < M; ++m) {
        double acc = 0.0;
        for (int j = 0; j <= i; ++j) acc += row[j] * V[(size_t)j * M + m];
        O[(size_t)i * M + m] = acc / s;
      }
    }
    free(row);
  }
}

void orc_causal_fwd_quadratic(int BH, int N, int D, int M, const double* q,
                              const double* k, const double* v, double* out,
                              double* den, int nthreads) {
  orc_causal_fwd_quadratic_decay(BH, N, D, M, q, k, v, 1.0, out, den, nthreads);
}

/* --------------------------------------------- causal, recurrent form (R) */

/* [TR2] §3.3 eq. 10-12: walk i = 1..N,
 *   S_i = S_{i-1} + phi(K_i) V_i^T      (D x M)
 *   Z_i = Z_{i-1} + phi(K_i)            (D)
 *   V'_i = phi(Q_i)^T S_i / phi(Q_i)^T Z_i
 * Only the running S, Z are kept: linear time, constant state.  With the
 * RetNet decay of [LA] the update is S_i = gamma S_{i-1} + phi(K_i) V_i^T and
 * Z_i = gamma Z_{i-1} + phi(K_i) (multiplying by gamma = 1 changes nothing). */
void orc_causal_fwd_recurrent_decay(int BH, int N, int D, int M, const double* q,
                                    const double* k, const double* v, double gamma,
                                    double* out, double* den, int nthreads) {
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
  for (int hh = 0; hh < BH; ++hh) {
    const double* Q = q + (size_t)hh * N * D;
    const double* K = k + (size_t)hh * N * D;
    const double* V = v + (size_t)hh * N * M;
    double* O = out + (size_t)hh * N * M;
    double* S = (double*)calloc((size_t)D * M, sizeof(double));
    double* Z = (double*)calloc((size_t)D, sizeof(double));
    double* fq = (double*)malloc(sizeof(double) * (size_t)D);
    for (int i = 0; i < N; ++i) {
      for (int d = 0; d < D; ++d) {
        double fk = phi(K[(size_t)i * D + d]);
        for (int m = 0; m < M; ++m)
          S[(size_t)d * M + m] = gamma * S[(size_t)d * M + m] + fk * V[(size_t)i * M + m];
        Z[d] = gamma * Z[d] + fk;
      }
      double s = 0.0;
      for (int d = 0; d < D; ++d) {
        fq[d] = phi(Q[(size_t)i * D + d]);
        s += fq[d] * Z[d];
      }
      if (den) den[(size_t)hh * N + i] = s;
      for (int m = 0; m < M; ++m) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += fq[d] * S[(size_t)d * M + m];
        O[(size_t)i * M + m] = acc / s;
      }
    }
    free(S);
    free(Z);
    free(fq);
  }
}

void orc_causal_fwd_recurrent(int BH, int N, int D, int M, const double* q,
                              const double* k, const double* v, double* out,
                              double* den, int nthreads) {
  orc_causal_fwd_recurrent_decay(BH, N, D, M, q, k, v, 1.0, out, den, nthreads);
}

/* ----------------------------------------- causal gradients, recurrent form */

/* Gradients of L = sum_i G_i . V'_i with respect to Q, K, V.
 *
 * V'_i = Vbar_i / den_i with the numerator Vbar_i = phi(Q_i)^T S_i and
 * den_i = phi(Q_i)^T Z_i.  By the quotient rule the loss reaches the numerator
 * through gt_i = G_i / den_i and the denominator through the scalar
 * gam_i = -(G_i . V'_i) / den_i.  The denominator is the numerator with every
 * V_j replaced by the constant 1, so its gradients follow eq. 13-15 with
 * (V_j, grad Vbar_j) -> (1, gam_j).
 *
 * [TR2] §3.3.1 eq. 13:  grad phi(Q_i) = S_i gt_i (+ gam_i Z_i)      forward sweep
 * [TR2] §3.3.1 eq. 14:  grad phi(K_i) = R_i V_i (+ r_i)              reverse sweep
 * [TR2] §3.3.1 eq. 15:  grad V_i      = R_i^T phi(K_i)
 *   with R_i = sum_{j>=i} phi(Q_j) gt_j^T and r_i = sum_{j>=i} gam_j phi(Q_j),
 *   the reverse cumulative sums ([TRN] appendix A compares them to BPTT).
 * Finally dQ = grad phi(Q) * phi'(Q) and dK = grad phi(K) * phi'(K) (eq. 7).
 * With the RetNet decay of [LA] the sums carry the same factor both ways:
 * S_i, Z_i as in the decayed forward, and R_i = gamma R_{i+1} + phi(Q_i) gt_i^T,
 * r_i = gamma r_{i+1} + gam_i phi(Q_i) (token j reaches query i >= j through
 * gamma^(i-j) in either direction). */
void orc_causal_bwd_recurrent_decay(int BH, int N, int D, int M, const double* q,
                                    const double* k, const double* v, const double* g,
                                    double gamma, double* dq, double* dk, double* dv,
                                    int nthreads) {
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
  for (int hh = 0; hh < BH; ++hh) {
    const double* Q = q + (size_t)hh * N * D;
    const double* K = k + (size_t)hh * N * D;
    const double* V = v + (size_t)hh * N * M;
    const double* G = g + (size_t)hh * N * M;
    double* dQ = dq + (size_t)hh * N * D;
    double* dK = dk + (size_t)hh * N * D;
    double* dV = dv + (size_t)hh * N * M;
    double* S = (double*)calloc((size_t)D * M, sizeof(double));
    double* Z = (double*)calloc((size_t)D, sizeof(double));
    double* R = (double*)calloc((size_t)D * M, sizeof(double));
    double* r = (double*)calloc((size_t)D, sizeof(double));
    double* fq = (double*)malloc(sizeof(double) * (size_t)D);
    double* vp = (double*)malloc(sizeof(double) * (size_t)M);
    double* gt = (double*)malloc(sizeof(double) * (size_t)N * M); /* gt_i */
    double* gam = (double*)malloc(sizeof(double) * (size_t)N);     /* gam_i */

    /* forward sweep: S_i, Z_i (eq. 10-11), V'_i, den_i (eq. 12), then eq. 13 */
    for (int i = 0; i < N; ++i) {
      for (int d = 0; d < D; ++d) {
        double fk = phi(K[(size_t)i * D + d]);
        for (int m = 0; m < M; ++m)
          S[(size_t)d * M + m] = gamma * S[(size_t)d * M + m] + fk * V[(size_t)i * M + m];
        Z[d] = gamma * Z[d] + fk;
      }
      double s = 0.0;
      for (int d = 0; d < D; ++d) {
        fq[d] = phi(Q[(size_t)i * D + d]);
        s += fq[d] * Z[d];
      }
      double gv = 0.0;
      for (int m = 0; m < M; ++m) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += fq[d] * S[(size_t)d * M + m];
        vp[m] = acc / s;
        gv += G[(size_t)i * M + m] * vp[m];
      }
      for (int m = 0; m < M; ++m) gt[(size_t)i * M + m] = G[(size_t)i * M + m] / s;
      gam[i] = -gv / s;
      for (int d = 0; d < D; ++d) {
        double acc = gam[i] * Z[d];
        for (int m = 0; m < M; ++m) acc += S[(size_t)d * M + m] * gt[(size_t)i * M + m];
        dQ[(size_t)i * D + d] = acc * dphi(Q[(size_t)i * D + d]);
      }
    }
    /* reverse sweep: R_i, r_i, then eq. 14-15 */
    for (int i = N - 1; i >= 0; --i) {
      for (int d = 0; d < D; ++d) {
        double fqd = phi(Q[(size_t)i * D + d]);
        for (int m = 0; m < M; ++m)
          R[(size_t)d * M + m] = gamma * R[(size_t)d * M + m] + fqd * gt[(size_t)i * M + m];
        r[d] = gamma * r[d] + gam[i] * fqd;
      }
      for (int d = 0; d < D; ++d) {
        double acc = r[d];
        for (int m = 0; m < M; ++m) acc += R[(size_t)d * M + m] * V[(size_t)i * M + m];
        dK[(size_t)i * D + d] = acc * dphi(K[(size_t)i * D + d]);
      }
      for (int m = 0; m < M; ++m) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += R[(size_t)d * M + m] * phi(K[(size_t)i * D + d]);
        dV[(size_t)i * M + m] = acc;
      }
    }
    free(S); free(Z); free(R); free(r); free(fq); free(vp); free(gt); free(gam);
  }
}

void orc_causal_bwd_recurrent(int BH, int N, int D, int M, const double* q,
                              const double* k, const double* v, const double* g,
                              double* dq, double* dk, double* dv, int nthreads) {
  orc_causal_bwd_recurrent_decay(BH, N, D, M, q, k, v, g, 1.0, dq, dk, dv, nthreads);
}

/* ----------------------------------------- causal gradients, quadratic form */

/* Differentiates eq. 8 directly through the explicit masked matrix:
 *   dA_ij   = gt_i . V_j + gam_i                    (j <= i)
 *   grad phi(Q_i) = sum_{j<=i} dA_ij phi(K_j)
 *   grad phi(K_j) = sum_{i>=j} dA_ij phi(Q_i)
 *   grad V_j      = sum_{i>=j} A_ij gt_i
 * with gt_i, gam_i as in the recurrent form.  Independent of the cumulative
 * sums: it touches every (i, j) pair.  With the RetNet decay the pair's
 * weight A_ij and its gradient dA_ij both carry gamma^(i-j). */
void orc_causal_bwd_quadratic_decay(int BH, int N, int D, int M, const double* q,
                                    const double* k, const double* v, const double* g,
                                    double gamma, double* dq, double* dk, double* dv,
                                    int nthreads) {
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
  for (int hh = 0; hh < BH; ++hh) {
    const double* Q = q + (size_t)hh * N * D;
    const double* K = k + (size_t)hh * N * D;
    const double* V = v + (size_t)hh * N * M;
    const double* G = g + (size_t)hh * N * M;
    double* dQ = dq + (size_t)hh * N * D;
    double* dK = dk + (size_t)hh * N * D;
    double* dV = dv + (size_t)hh * N * M;
    double* A = (double*)malloc(sizeof(double) * (size_t)N * N);
    double* gt = (double*)malloc(sizeof(double) * (size_t)N * M);
    double* gam = (double*)malloc(sizeof(double) * (size_t)N);
    double* gfq = (double*)calloc((size_t)N * D, sizeof(double));
    double* gfk = (double*)calloc((size_t)N * D, sizeof(double));
    memset(dV, 0, sizeof(double) * (size_t)N * M);
    for (int i = 0; i < N; ++i) {
      double s = 0.0;
      for (int j = 0; j < N; ++j) {
        double a = 0.0;
        if (j <= i) {
          for (int d = 0; d < D; ++d) a += phi(Q[(size_t)i * D + d]) * phi(K[(size_t)j * D + d]);
          a *= pow(gamma, (double)(i - j));
        }
        A[(size_t)i * N + j] = a;
        s += a;
      }
      double gv = 0.0;
      for (int m = 0; m < M; ++m) {
        double acc = 0.0;
        for (int j = 0; j <= i; ++j) acc += A[(size_t)i * N + j] * V[(size_t)j * M + m];
        gv += G[(size_t)i * M + m] * (acc / s);
        gt[(size_t)i * M + m] = G[(size_t)i * M + m] / s;
      }
      gam[i] = -gv / s;
    }
    for (int i = 0; i < N; ++i) {
      for (int j = 0; j <= i; ++j) {
        double da = gam[i];
        for (int m = 0; m < M; ++m) da += gt[(size_t)i * M + m] * V[(size_t)j * M + m];
        da *= pow(gamma, (double)(i - j)); /* d(loss)/d(phi(Q_i) . phi(K_j)) */
        for (int d = 0; d < D; ++d) {
          gfq[(size_t)i * D + d] += da * phi(K[(size_t)j * D + d]);
          gfk[(size_t)j * D + d] += da * phi(Q[(size_t)i * D + d]);
        }
        for (int m = 0; m < M; ++m) dV[(size_t)j * M + m] += A[(size_t)i * N + j] * gt[(size_t)i * M + m];
      }
    }
    for (int i = 0; i < N; ++i)
      for (int d = 0; d < D; ++d) {
        dQ[(size_t)i * D + d] = gfq[(size_t)i * D + d] * dphi(Q[(size_t)i * D + d]);
        dK[(size_t)i * D + d] = gfk[(size_t)i * D + d] * dphi(K[(size_t)i * D + d]);
      }
    free(A); free(gt); free(gam); free(gfq); free(gfk);
  }
}

void orc_causal_bwd_quadratic(int BH, int N, int D, int M, const double* q,
                              const double* k, const double* v, const double* g,
                              double* dq, double* dk, double* dv, int nthreads) {
  orc_causal_bwd_quadratic_decay(BH, N, D, M, q, k, v, g, 1.0, dq, dk, dv, nthreads);
}

/* --------------------------------- causal, degree-2 polynomial kernel */

/* [TR2] the feature-map discussion that opens part 2/3 (§3.2.1): the
 * polynomial kernel has an exact finite feature map, and linear attention
 * with the degree-2 one costs O(N D^2 M).  Read as the homogeneous kernel
 * sim(Q_i, K_j) = (Q_i . K_j)^2 in place of phi(Q_i) . phi(K_j) in eq. 8 and
 * 12 (no feature map is applied to Q or K first):
 *   A_ij = (Q_i . K_j)^2 for j <= i,  den_i = sum_j A_ij,
 *   out_i = sum_j A_ij V_j / den_i.
 * Written as the plain quadratic form: every (i, j) pair. */
void orc_causal_fwd_poly(int BH, int N, int D, int M, const double* q, const double* k,
                         const double* v, double* out, double* den, int nthreads) {
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
  for (int hh = 0; hh < BH; ++hh) {
    const double* Q = q + (size_t)hh * N * D;
    const double* K = k + (size_t)hh * N * D;
    const double* V = v + (size_t)hh * N * M;
    double* O = out + (size_t)hh * N * M;
    double* row = (double*)malloc(sizeof(double) * (size_t)N);
    for (int i = 0; i < N; ++i) {
      double s = 0.0;
      for (int j = 0; j <= i; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += Q[(size_t)i * D + d] * K[(size_t)j * D + d];
        row[j] = dot * dot;
        s += row[j];
      }
      if (den) den[(size_t)hh * N + i] = s;
      for (int m = 0; m < M; ++m) {
        double acc = 0.0;
        for (int j = 0; j <= i; ++j) acc += row[j] * V[(size_t)j * M + m];
        O[(size_t)i * M + m] = acc / s;
      }
    }
    free(row);
  }
}

/* Gradients of L = sum_i G_i . out_i for the degree-2 polynomial kernel, by
 * the pairwise rule: with gt_i = G_i / den_i and gam_i = -(G_i . out_i) /
 * den_i as for eq. 13-15, dL/dA_ij = gt_i . V_j + gam_i (j <= i), and
 * A_ij = (Q_i . K_j)^2 gives dA_ij/dQ_i = 2 (Q_i . K_j) K_j, dA_ij/dK_j =
 * 2 (Q_i . K_j) Q_i:
 *   dQ_i = sum_{j<=i} dA_ij 2 (Q_i . K_j) K_j,
 *   dK_j = sum_{i>=j} dA_ij 2 (Q_i . K_j) Q_i,
 *   dV_j = sum_{i>=j} A_ij gt_i. */
void orc_causal_bwd_poly(int BH, int N, int D, int M, const double* q, const double* k,
                         const double* v, const double* g, double* dq, double* dk, double* dv,
                         int nthreads) {
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
  for (int hh = 0; hh < BH; ++hh) {
    const double* Q = q + (size_t)hh * N * D;
    const double* K = k + (size_t)hh * N * D;
    const double* V = v + (size_t)hh * N * M;
    const double* G = g + (size_t)hh * N * M;
    double* dQ = dq + (size_t)hh * N * D;
    double* dK = dk + (size_t)hh * N * D;
    double* dV = dv + (size_t)hh * N * M;
    double* dots = (double*)malloc(sizeof(double) * (size_t)N);
    double* gt = (double*)malloc(sizeof(double) * (size_t)M);
    memset(dQ, 0, sizeof(double) * (size_t)N * D);
    memset(dK, 0, sizeof(double) * (size_t)N * D);
    memset(dV, 0, sizeof(double) * (size_t)N * M);
    for (int i = 0; i < N; ++i) {
      double s = 0.0;
      for (int j = 0; j <= i; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += Q[(size_t)i * D + d] * K[(size_t)j * D + d];
        dots[j] = dot;
        s += dot * dot;
      }
      double gv = 0.0;
      for (int m = 0; m < M; ++m) {
        double acc = 0.0;
        for (int j = 0; j <= i; ++j) acc += dots[j] * dots[j] * V[(size_t)j * M + m];
        gv += G[(size_t)i * M + m] * (acc / s);
        gt[m] = G[(size_t)i * M + m] / s;
      }
      const double gam = -gv / s;
      for (int j = 0; j <= i; ++j) {
        double da = gam;
        for (int m = 0; m < M; ++m) da += gt[m] * V[(size_t)j * M + m];
        const double w = 2.0 * da * dots[j];
        for (int d = 0; d < D; ++d) {
          dQ[(size_t)i * D + d] += w * K[(size_t)j * D + d];
          dK[(size_t)j * D + d] += w * Q[(size_t)i * D + d];
        }
        for (int m = 0; m < M; ++m) dV[(size_t)j * M + m] += dots[j] * dots[j] * gt[m];
      }
    }
    free(dots);
    free(gt);
  }
}

/* ---------------------------------------------------------- non-causal form */

/* Valid length of batch entry b: lengths[b] if given, else N. */
static int valid_len(const int* lengths, int b, int N) {
  if (!lengths) return N;
  int L = lengths[b];
  return L < 0 ? 0 : (L > N ? N : L);
}

/* [LA] "kernel reformulation": with a shared
 *   S = sum_{j<L} phi(K_j) V_j^T,   Z = sum_{j<L} phi(K_j)
 * every query reads  V'_i = phi(Q_i)^T S / phi(Q_i)^T Z  (the non-causal
 * counterpart of [TR2] eq. 9-12).  L is the batch entry's valid length; rows
 * i >= L are padding and get V' = 0, den = 0.  S_out / Z_out (optional) receive
 * the shared state, [BH][D][M] and [BH][D]. */
void orc_noncausal_fwd(int B, int H, int N, int D, int M, const int* lengths,
                       const double* q, const double* k, const double* v,
                       double* out, double* den, double* S_out, double* Z_out,
                       int nthreads) {
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
  for (int hh = 0; hh < B * H; ++hh) {
    int L = valid_len(lengths, hh / H, N);
    const double* Q = q + (size_t)hh * N * D;
    const double* K = k + (size_t)hh * N * D;
    const double* V = v + (size_t)hh * N * M;
    double* O = out + (size_t)hh * N * M;
    double* S = (double*)calloc((size_t)D * M, sizeof(double));
    double* Z = (double*)calloc((size_t)D, sizeof(double));
    double* fq = (double*)malloc(sizeof(double) * (size_t)D);
    for (int j = 0; j < L; ++j)
      for (int d = 0; d < D; ++d) {
        double fk = phi(K[(size_t)j * D + d]);
        for (int m = 0; m < M; ++m) S[(size_t)d * M + m] += fk * V[(size_t)j * M + m];
        Z[d] += fk;
      }
    for (int i = 0; i < N; ++i) {
      if (i >= L) {
        for (int m = 0; m < M; ++m) O[(size_t)i * M + m] = 0.0;
        if (den) den[(size_t)hh * N + i] = 0.0;
        continue;
      }
      double s = 0.0;
      for (int d = 0; d < D; ++d) {
        fq[d] = phi(Q[(size_t)i * D + d]);
        s += fq[d] * Z[d];
      }
      if (den) den[(size_t)hh * N + i] = s;
      for (int m = 0; m < M; ++m) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += fq[d] * S[(size_t)d * M + m];
        O[(size_t)i * M + m] = acc / s;
      }
    }
    if (S_out) memcpy(S_out + (size_t)hh * D * M, S, sizeof(double) * (size_t)D * M);
    if (Z_out) memcpy(Z_out + (size_t)hh * D, Z, sizeof(double) * (size_t)D);
    free(S); free(Z); free(fq);
  }
}

/* Non-causal, quadratic form: the unmasked analogue of eq. 8 over the valid
 * rows, A_ij = phi(Q_i) . phi(K_j) for i, j < L, V'_i = sum_j A_ij V_j / sum_j A_ij. */
void orc_noncausal_fwd_quadratic(int B, int H, int N, int D, int M, const int* lengths,
                                 const double* q, const double* k, const double* v,
                                 double* out, double* den, int nthreads) {
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
  for (int hh = 0; hh < B * H; ++hh) {
    int L = valid_len(lengths, hh / H, N);
    const double* Q = q + (size_t)hh * N * D;
    const double* K = k + (size_t)hh * N * D;
    const double* V = v + (size_t)hh * N * M;
    double* O = out + (size_t)hh * N * M;
    double* row = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    for (int i = 0; i < N; ++i) {
      if (i >= L) {
        for (int m = 0; m < M; ++m) O[(size_t)i * M + m] = 0.0;
        if (den) den[(size_t)hh * N + i] = 0.0;
        continue;
      }
      double s = 0.0;
      for (int j = 0; j < L; ++j) {
        double a = 0.0;
        for (int d = 0; d < D; ++d) a += phi(Q[(size_t)i * D + d]) * phi(K[(size_t)j * D + d]);
        row[j] = a;
        s += a;
      }
      if (den) den[(size_t)hh * N + i] = s;
      for (int m = 0; m < M; ++m) {
        double acc = 0.0;
        for (int j = 0; j < L; ++j) acc += row[j] * V[(size_t)j * M + m];
        O[(size_t)i * M + m] = acc / s;
      }
    }
    free(row);
  }
}

/* Non-causal gradients: eq. 13-15 with every cumulative sum replaced by the
 * full sum over the valid rows (no mask), plus the denominator terms:
 *   grad phi(Q_i) = S gt_i + gam_i Z
 *   R = sum_{i<L} phi(Q_i) gt_i^T,   r = sum_{i<L} gam_i phi(Q_i)
 *   grad phi(K_j) = R V_j + r,        grad V_j = R^T phi(K_j)
 * Padded rows get zero gradients. */
void orc_noncausal_bwd(int B, int H, int N, int D, int M, const int* lengths,
                       const double* q, const double* k, const double* v,
                       const double* g, double* dq, double* dk, double* dv,
                       int nthreads) {
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
  for (int hh = 0; hh < B * H; ++hh) {
    int L = valid_len(lengths, hh / H, N);
    const double* Q = q + (size_t)hh * N * D;
    const double* K = k + (size_t)hh * N * D;
    const double* V = v + (size_t)hh * N * M;
    const double* G = g + (size_t)hh * N * M;
    double* dQ = dq + (size_t)hh * N * D;
    double* dK = dk + (size_t)hh * N * D;
    double* dV = dv + (size_t)hh * N * M;
    double* S = (double*)calloc((size_t)D * M, sizeof(double));
    double* Z = (double*)calloc((size_t)D, sizeof(double));
    double* R = (double*)calloc((size_t)D * M, sizeof(double));
    double* r = (double*)calloc((size_t)D, sizeof(double));
    double* fq = (double*)malloc(sizeof(double) * (size_t)D);
    double* gt = (double*)malloc(sizeof(double) * (size_t)M);
    memset(dQ, 0, sizeof(double) * (size_t)N * D);
    memset(dK, 0, sizeof(double) * (size_t)N * D);
    memset(dV, 0, sizeof(double) * (size_t)N * M);
    for (int j = 0; j < L; ++j)
      for (int d = 0; d < D; ++d) {
        double fk = phi(K[(size_t)j * D + d]);
        for (int m = 0; m < M; ++m) S[(size_t)d * M + m] += fk * V[(size_t)j * M + m];
        Z[d] += fk;
      }
    for (int i = 0; i < L; ++i) {
      double s = 0.0;
      for (int d = 0; d < D; ++d) {
        fq[d] = phi(Q[(size_t)i * D + d]);
        s += fq[d] * Z[d];
      }
      double gv = 0.0;
      for (int m = 0; m < M; ++m) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += fq[d] * S[(size_t)d * M + m];
        gv += G[(size_t)i * M + m] * (acc / s);
        gt[m] = G[(size_t)i * M + m] / s;
      }
      double gam = -gv / s;
      for (int d = 0; d < D; ++d) {
        double acc = gam * Z[d];
        for (int m = 0; m < M; ++m) acc += S[(size_t)d * M + m] * gt[m];
        dQ[(size_t)i * D + d] = acc * dphi(Q[(size_t)i * D + d]);
        for (int m = 0; m < M; ++m) R[(size_t)d * M + m] += fq[d] * gt[m];
        r[d] += gam * fq[d];
      }
    }
    for (int j = 0; j < L; ++j) {
      for (int d = 0; d < D; ++d) {
        double acc = r[d];
        for (int m = 0; m < M; ++m) acc += R[(size_t)d * M + m] * V[(size_t)j * M + m];
        dK[(size_t)j * D + d] = acc * dphi(K[(size_t)j * D + d]);
      }
      for (int m = 0; m < M; ++m) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += R[(size_t)d * M + m] * phi(K[(size_t)j * D + d]);
        dV[(size_t)j * M + m] = acc;
      }
    }
    free(S); free(Z); free(R); free(r); free(fq); free(gt);
  }
}

/* Non-causal gradients through the explicit unmasked matrix (quadratic form),
 * the same pairwise rules as the causal quadratic gradient without the mask. */
void orc_noncausal_bwd_quadratic(int B, int H, int N, int D, int M, const int* lengths,
                                 const double* q, const double* k, const double* v,
                                 const double* g, double* dq, double* dk, double* dv,
                                 int nthreads) {
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
  for (int hh = 0; hh < B * H; ++hh) {
    int L = valid_len(lengths, hh / H, N);
    const double* Q = q + (size_t)hh * N * D;
    const double* K = k + (size_t)hh * N * D;
    const double* V = v + (size_t)hh * N * M;
    const double* G = g + (size_t)hh * N * M;
    double* dQ = dq + (size_t)hh * N * D;
    double* dK = dk + (size_t)hh * N * D;
    double* dV = dv + (size_t)hh * N * M;
    size_t n1 = (size_t)(N > 0 ? N : 1);
    double* A = (double*)malloc(sizeof(double) * n1 * n1);
    double* gt = (double*)malloc(sizeof(double) * n1 * (size_t)M);
    double* gam = (double*)malloc(sizeof(double) * n1);
    double* gfq = (double*)calloc(n1 * (size_t)D, sizeof(double));
    double* gfk = (double*)calloc(n1 * (size_t)D, sizeof(double));
    memset(dQ, 0, sizeof(double) * (size_t)N * D);
    memset(dK, 0, sizeof(double) * (size_t)N * D);
    memset(dV, 0, sizeof(double) * (size_t)N * M);
    for (int i = 0; i < L; ++i) {
      double s = 0.0;
      for (int j = 0; j < L; ++j) {
        double a = 0.0;
        for (int d = 0; d < D; ++d) a += phi(Q[(size_t)i * D + d]) * phi(K[(size_t)j * D + d]);
        A[(size_t)i * N + j] = a;
        s += a;
      }
      double gv = 0.0;
      for (int m = 0; m < M; ++m) {
        double acc = 0.0;
        for (int j = 0; j < L; ++j) acc += A[(size_t)i * N + j] * V[(size_t)j * M + m];
        gv += G[(size_t)i * M + m] * (acc / s);
        gt[(size_t)i * M + m] = G[(size_t)i * M + m] / s;
      }
      gam[i] = -gv / s;
    }
    for (int i = 0; i < L; ++i)
      for (int j = 0; j < L; ++j) {
        double da = gam[i];
        for (int m = 0; m < M; ++m) da += gt[(size_t)i * M + m] * V[(size_t)j * M + m];
        for (int d = 0; d < D; ++d) {
          gfq[(size_t)i * D + d] += da * phi(K[(size_t)j * D + d]);
          gfk[(size_t)j * D + d] += da * phi(Q[(size_t)i * D + d]);
        }
        for (int m = 0; m < M; ++m) dV[(size_t)j * M + m] += A[(size_t)i * N + j] * gt[(size_t)i * M + m];
      }
    for (int i = 0; i < L; ++i)
      for (int d = 0; d < D; ++d) {
        dQ[(size_t)i * D + d] = gfq[(size_t)i * D + d] * dphi(Q[(size_t)i * D + d]);
        dK[(size_t)i * D + d] = gfk[(size_t)i * D + d] * dphi(K[(size_t)i * D + d]);
      }
    free(A); free(gt); free(gam); free(gfq); free(gfk);
  }
}

/* -------------------------------------------- prefill: the causal form from a state */

/* [TR2] §3.4 eq. 16-19 run over a whole prompt: the causal form of §3.3
 * eq. 10-12 with its sums started from a given state instead of zero,
 *   S_i = S_0 + sum_{j<=i} phi(K_j) V_j^T,   Z_i = Z_0 + sum_{j<=i} phi(K_j),
 *   out_i = phi(Q_i)^T S_i / phi(Q_i)^T Z_i,   den_i = phi(Q_i)^T Z_i,
 * so that a prompt's state feeds the RNN form (eq. 16-19) of the tokens that
 * follow it.  S [BH][D][M] and Z [BH][D] hold S_0, Z_0 on entry and S_N, Z_N
 * on exit; q, k: [BH][N][D]; v, out: [BH][N][M]; den: [BH][N]. */
void orc_causal_prefill(int BH, int N, int D, int M, const double* q, const double* k,
                        const double* v, double* S, double* Z, double* out, double* den,
                        int nthreads) {
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
  for (int hh = 0; hh < BH; ++hh) {
    const double* Qh = q + (size_t)hh * N * D;
    const double* Kh = k + (size_t)hh * N * D;
    const double* Vh = v + (size_t)hh * N * M;
    double* Oh = out + (size_t)hh * N * M;
    double* st = S + (size_t)hh * D * M;
    double* zt = Z + (size_t)hh * D;
    double* sl = (double*)malloc(sizeof(double) * (size_t)D * M);
    double* zl = (double*)malloc(sizeof(double) * (size_t)D);
    double* fq = (double*)malloc(sizeof(double) * (size_t)D);
    memcpy(sl, st, sizeof(double) * (size_t)D * M);
    for (int d = 0; d < D; ++d) zl[d] = zt[d];
    for (int i = 0; i < N; ++i) {
      for (int d = 0; d < D; ++d) {
        const double fkp = phi(Kh[(size_t)i * D + d]);
        for (int m = 0; m < M; ++m) sl[(size_t)d * M + m] += fkp * Vh[(size_t)i * M + m];
        zl[d] += fkp;
      }
      double dsum = 0.0;
      for (int d = 0; d < D; ++d) {
        fq[d] = phi(Qh[(size_t)i * D + d]);
        dsum += fq[d] * zl[d];
      }
      den[(size_t)hh * N + i] = dsum;
      for (int m = 0; m < M; ++m) {
        double num = 0.0;
        for (int d = 0; d < D; ++d) num += fq[d] * sl[(size_t)d * M + m];
        Oh[(size_t)i * M + m] = num / dsum;
      }
    }
    for (size_t e = 0; e < (size_t)D * M; ++e) st[e] = sl[e];
    for (int d = 0; d < D; ++d) zt[d] = zl[d];
    free(sl);
    free(zl);
    free(fq);
  }
}

/* ------------------------------------------------------------ RNN-form decode */

/* [TR2] §3.4 eq. 16-19 (and [LA] "recurrent form"): for each step t and each
 * independent stream hh,
 *   s <- s + phi(k_t) v_t^T,   z <- z + phi(k_t),
 *   y_t = phi(q_t)^T s / phi(q_t)^T z
 * The state is updated before it is read, as in eq. 18-20.  The layer's f_l and
 * residual of eq. 20 are outside the attention and are not applied.  S [BH][D][M]
 * and Z [BH][D] hold the state on entry (zero for eq. 16-17) and on exit.
 * q, k: [T][BH][D]; v, y: [T][BH][M].  With the RetNet decay of [LA]:
 * s <- gamma s + phi(k_t) v_t^T and z <- gamma z + phi(k_t). */
void orc_decode_decay(int T, int BH, int D, int M, const double* q, const double* k,
                      const double* v, double gamma, double* S, double* Z, double* y,
                      int nthreads) {
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
  for (int hh = 0; hh < BH; ++hh) {
    double* s = S + (size_t)hh * D * M;
    double* z = Z + (size_t)hh * D;
    double* fq = (double*)malloc(sizeof(double) * (size_t)D);
    for (int t = 0; t < T; ++t) {
      const double* qt = q + ((size_t)t * BH + hh) * D;
      const double* kt = k + ((size_t)t * BH + hh) * D;
      const double* vt = v + ((size_t)t * BH + hh) * M;
      double* yt = y + ((size_t)t * BH + hh) * M;
      for (int d = 0; d < D; ++d) {
        double fk = phi(kt[d]);
        for (int m = 0; m < M; ++m) s[(size_t)d * M + m] = gamma * s[(size_t)d * M + m] + fk * vt[m];
        z[d] = gamma * z[d] + fk;
      }
      double den = 0.0;
      for (int d = 0; d < D; ++d) {
        fq[d] = phi(qt[d]);
        den += fq[d] * z[d];
      }
      for (int m = 0; m < M; ++m) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += fq[d] * s[(size_t)d * M + m];
        yt[m] = acc / den;
      }
    }
    free(fq);
  }
}

void orc_decode(int T, int BH, int D, int M, const double* q, const double* k,
                const double* v, double* S, double* Z, double* y, int nthreads) {
  orc_decode_decay(T, BH, D, M, q, k, v, 1.0, S, Z, y, nthreads);
}
