/*
 * oracle.c -- plain float64 CPU oracle for the Matryoshka contrastive losses.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline /
 * "--impl reference" leg use it.  It shares no code, header or constant with the
 * CUDA library.
 *
 * What it computes (written out from the definitions, no blocking or fusion):
 *   Inputs are bf16 bit patterns, widened exactly to double.  For every prefix p of
 *   the Matryoshka ladder (UForm README, "Matryoshka" paragraph: the leading 64,
 *   128, 256, 512 and 1024 dimensions must each work as an embedding; blog post
 *   "Scaling-Up Contrastive Learning over NVLink Multicast", section "One Set or
 *   Two": five grids, not one) the vectors a_i[:p], b_j[:p] are compared by cosine
 *   (each prefix normalised on its own), scaled, and fed to
 *     CLIP   symmetric InfoNCE: L = 1/2 [ mean_i CE(row i) + mean_j CE(column j) ],
 *            logits s = scale * cos, positives on the diagonal (blog, "One Set or
 *            Two": CLIP turns each row of cosines into a softmax over the batch);
 *     SIGLIP pairwise sigmoid: L = -(1/N) sum_i sum_j log sigmoid(z_ij (t cos + b)),
 *            N the rows of A, z = +1 for a positive pair and -1 for every negative
 *            (blog, "One Set or Two", the SigLIP equation).  The positives are the
 *            diagonal cells (i, i), i < Na, unless a label matrix names them (the
 *            *_labels entry points: Z[i * Nb + j] != 0 marks (i, j) positive; a row may
 *            have several positives or none).  Nb >= Na: the columns past Na are
 *            extra negatives (the blog's "explicit hard negatives ... gathered as
 *            extra band columns", section "Scaling-Up");
 *     ROWS   row-direction InfoNCE: L = mean_{i<Nq} CE(row i) over all Nk keys,
 *            the positive of query i being key i.
 *   Gradients are taken by the chain rule, prefix by prefix, and summed with the
 *   caller's per-prefix weights:
 *     G_ij = dL/dcos_ij,  dcos_ij/da_i = (bhat_j - cos_ij * ahat_i) / |a_i|,
 *     dcos_ij/db_j = (ahat_i - cos_ij * bhat_j) / |b_j|.
 *   A zero-norm prefix uses 1/max(|x|, 1e-30) as its inverse norm (the pages are
 *   silent; this is the reading the library documents as well).
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC oracle.c -o liboracle.so -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_CLIP = 0, ORC_SIGLIP = 1, ORC_ROWS = 2 };

static double widen(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double softplus(double y) { /* log(1 + e^y), evaluated without overflow */
  return (y > 0 ? y : 0.0) + log1p(exp(-fabs(y)));
}

static double sigmoid(double y) {
  if (y >= 0) return 1.0 / (1.0 + exp(-y));
  double e = exp(y);
  return e / (1.0 + e);
}

static double inv_norm(const double* x, int p) {
  double ss = 0;
  for (int d = 0; d < p; ++d) ss += x[d] * x[d];
  double n = sqrt(ss);
  return 1.0 / (n > 1e-30 ? n : 1e-30);
}

static double* widen_matrix(const uint16_t* X, int64_t rows, int D) {
  double* W = (double*)malloc((size_t)rows * D * sizeof(double));
  if (!W) return NULL;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < rows; ++i)
    for (int d = 0; d < D; ++d) W[i * D + d] = widen(X[i * D + d]);
  return W;
}

static int check_args(int kind, int64_t Na, int64_t Nb, int D, const int* prefixes, int n) {
  if (Na <= 0 || Nb <= 0 || D <= 0 || n <= 0 || !prefixes) return -1;
  for (int k = 0; k < n; ++k) {
    if (prefixes[k] <= 0 || prefixes[k] > D) return -1;
    if (k && prefixes[k] <= prefixes[k - 1]) return -1;
  }
  if (kind == ORC_CLIP && Na != Nb) return -1;
  if ((kind == ORC_ROWS || kind == ORC_SIGLIP) && Nb < Na) return -1;
  if (kind < 0 || kind > 2) return -1;
  return 0;
}

/* Is (i, j) a positive pair?  The label matrix when there is one, else the diagonal. */
static int positive(const unsigned char* Z, int64_t Nb, int64_t i, int64_t j) {
  return Z ? Z[i * Nb + j] != 0 : i == j;
}

/*
 * Full forward and backward over the whole Na x Nb grid, on float64 inputs.
 *   loss[k]            unweighted loss of prefix k
 *   dA (Na x D), dB (Nb x D)   gradients of sum_k weights[k] * L_k (NULL to skip;
 *                      weights NULL means all ones); columns >= the last prefix are 0
 *   row_terms[k][i]    per-row term: CLIP/ROWS: LSE_j(s_ij) - s_ii (every row of A is
 *                      a query in ROWS); SIGLIP: sum_j softplus(-z_ij x_ij)
 *   col_terms[k][j]    CLIP: LSE_i(s_ij) - s_jj; SIGLIP: sum_i softplus(-z_ij x_ij);
 *                      ROWS: 0
 * Returns 0, or -1 on bad arguments, -2 when out of memory.
 */
static int fwd_bwd(int kind, const double* A, const double* B, int64_t Na, int64_t Nb, int D,
                   const int* prefixes, int n, double scale, double bias, const double* weights,
                   const unsigned char* Z, double* loss, double* dA, double* dB, double* row_terms,
                   double* col_terms) {
  if (check_args(kind, Na, Nb, D, prefixes, n)) return -1;
  if (Z && kind != ORC_SIGLIP) return -1;
  double* C = (double*)malloc((size_t)Na * Nb * sizeof(double));  /* cosines */
  double* G = (double*)malloc((size_t)Na * Nb * sizeof(double));  /* dL/dcos */
  double* ra = (double*)malloc((size_t)Na * sizeof(double));
  double* rb = (double*)malloc((size_t)Nb * sizeof(double));
  double* lse_r = (double*)malloc((size_t)Na * sizeof(double));
  double* lse_c = (double*)malloc((size_t)Nb * sizeof(double));
  if (!C || !G || !ra || !rb || !lse_r || !lse_c) {
    free(C); free(G); free(ra); free(rb); free(lse_r); free(lse_c);
    return -2;
  }
  if (dA) memset(dA, 0, (size_t)Na * D * sizeof(double));
  if (dB) memset(dB, 0, (size_t)Nb * D * sizeof(double));

  for (int k = 0; k < n; ++k) {
    const int p = prefixes[k];
    const double w = weights ? weights[k] : 1.0;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < Na; ++i) ra[i] = inv_norm(A + i * D, p);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < Nb; ++j) rb[j] = inv_norm(B + j * D, p);

    /* cosine of every pair, on the first p dimensions */
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < Na; ++i)
      for (int64_t j = 0; j < Nb; ++j) {
        double dot = 0;
        for (int d = 0; d < p; ++d) dot += A[i * D + d] * B[j * D + d];
        C[i * Nb + j] = dot * ra[i] * rb[j];
      }

    double L = 0;
    if (kind == ORC_CLIP || kind == ORC_ROWS) {
      const double tau = scale;
      /* row log-sum-exp of the logits s = tau * cos, shifted by the row maximum */
#pragma omp parallel for schedule(static)
      for (int64_t i = 0; i < Na; ++i) {
        double m = -INFINITY, s = 0;
        for (int64_t j = 0; j < Nb; ++j) m = fmax(m, tau * C[i * Nb + j]);
        for (int64_t j = 0; j < Nb; ++j) s += exp(tau * C[i * Nb + j] - m);
        lse_r[i] = m + log(s);
      }
      if (kind == ORC_CLIP) {
#pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < Nb; ++j) {
          double m = -INFINITY, s = 0;
          for (int64_t i = 0; i < Na; ++i) m = fmax(m, tau * C[i * Nb + j]);
          for (int64_t i = 0; i < Na; ++i) s += exp(tau * C[i * Nb + j] - m);
          lse_c[j] = m + log(s);
        }
        const double N = (double)Na;
        double Lr = 0, Lc = 0;
        for (int64_t i = 0; i < Na; ++i) {
          double t = lse_r[i] - tau * C[i * Nb + i];
          Lr += t;
          if (row_terms) row_terms[(int64_t)k * Na + i] = t;
        }
        for (int64_t j = 0; j < Nb; ++j) {
          double t = lse_c[j] - tau * C[j * Nb + j];
          Lc += t;
          if (col_terms) col_terms[(int64_t)k * Nb + j] = t;
        }
        L = 0.5 * (Lr / N + Lc / N);
        /* dL/ds_ij = (softmax_row + softmax_col - 2 [i==j]) / (2N); dL/dcos = tau * that */
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < Na; ++i)
          for (int64_t j = 0; j < Nb; ++j) {
            double s = tau * C[i * Nb + j];
            double g = exp(s - lse_r[i]) + exp(s - lse_c[j]) - (i == j ? 2.0 : 0.0);
            G[i * Nb + j] = tau * g / (2.0 * N);
          }
      } else {
        const double Nq = (double)Na;
        for (int64_t i = 0; i < Na; ++i) {
          double t = lse_r[i] - tau * C[i * Nb + i];
          L += t;
          if (row_terms) row_terms[(int64_t)k * Na + i] = t;
        }
        if (col_terms)
          for (int64_t j = 0; j < Nb; ++j) col_terms[(int64_t)k * Nb + j] = 0.0;
        L /= Nq;
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < Na; ++i)
          for (int64_t j = 0; j < Nb; ++j) {
            double s = tau * C[i * Nb + j];
            double g = exp(s - lse_r[i]) - (i == j ? 1.0 : 0.0);
            G[i * Nb + j] = tau * g / Nq;
          }
      }
    } else { /* SIGLIP */
      const double t = scale, b = bias, N = (double)Na;
      if (row_terms)
        for (int64_t i = 0; i < Na; ++i) row_terms[(int64_t)k * Na + i] = 0.0;
      if (col_terms)
        for (int64_t j = 0; j < Nb; ++j) col_terms[(int64_t)k * Nb + j] = 0.0;
      for (int64_t i = 0; i < Na; ++i)
        for (int64_t j = 0; j < Nb; ++j) {
          double x = t * C[i * Nb + j] + b;
          const int pos = positive(Z, Nb, i, j);
          double z = pos ? 1.0 : -1.0;
          double l = softplus(-z * x); /* -log sigmoid(z x) */
          L += l;
          if (row_terms) row_terms[(int64_t)k * Na + i] += l;
          if (col_terms) col_terms[(int64_t)k * Nb + j] += l;
          /* d/dx softplus(-z x) = -z sigmoid(-z x) = sigmoid(x) - [z == +1] */
          G[i * Nb + j] = t * (sigmoid(x) - (pos ? 1.0 : 0.0)) / N;
        }
      L /= N;
    }
    loss[k] = L;

    /* chain rule through the cosine: dA_i += w sum_j G_ij (bhat_j - cos_ij ahat_i) / |a_i| */
    if (dA) {
#pragma omp parallel for schedule(dynamic, 4)
      for (int64_t i = 0; i < Na; ++i) {
        double* out = dA + i * D;
        for (int64_t j = 0; j < Nb; ++j) {
          const double g = w * G[i * Nb + j], c = C[i * Nb + j];
          if (g == 0.0) continue;
          for (int d = 0; d < p; ++d)
            out[d] += g * (B[j * D + d] * rb[j] - c * A[i * D + d] * ra[i]) * ra[i];
        }
      }
    }
    if (dB) {
#pragma omp parallel for schedule(dynamic, 4)
      for (int64_t j = 0; j < Nb; ++j) {
        double* out = dB + j * D;
        for (int64_t i = 0; i < Na; ++i) {
          const double g = w * G[i * Nb + j], c = C[i * Nb + j];
          if (g == 0.0) continue;
          for (int d = 0; d < p; ++d)
            out[d] += g * (A[i * D + d] * ra[i] - c * B[j * D + d] * rb[j]) * rb[j];
        }
      }
    }
  }
  free(C); free(G); free(ra); free(rb); free(lse_r); free(lse_c);
  return 0;
}

int orc_fwd_bwd_f64(int kind, const double* A, const double* B, int64_t Na, int64_t Nb, int D,
                    const int* prefixes, int n, double scale, double bias, const double* weights,
                    double* loss, double* dA, double* dB, double* row_terms, double* col_terms) {
  return fwd_bwd(kind, A, B, Na, Nb, D, prefixes, n, scale, bias, weights, NULL, loss, dA, dB, row_terms,
                 col_terms);
}

/* SIGLIP with the positives named by the label matrix Z (Na x Nb bytes, nonzero = positive). */
int orc_fwd_bwd_labels_f64(const double* A, const double* B, int64_t Na, int64_t Nb, int D,
                           const int* prefixes, int n, double scale, double bias, const double* weights,
                           const unsigned char* Z, double* loss, double* dA, double* dB, double* row_terms,
                           double* col_terms) {
  if (!Z) return -1;
  return fwd_bwd(ORC_SIGLIP, A, B, Na, Nb, D, prefixes, n, scale, bias, weights, Z, loss, dA, dB, row_terms,
                 col_terms);
}

/* The same on bf16 inputs (the form every test and the library consume): widen, then compute. */
static int fwd_bwd_bf16(int kind, const uint16_t* A16, const uint16_t* B16, int64_t Na, int64_t Nb, int D,
                        const int* prefixes, int n, double scale, double bias, const double* weights,
                        const unsigned char* Z, double* loss, double* dA, double* dB, double* row_terms,
                        double* col_terms) {
  if (check_args(kind, Na, Nb, D, prefixes, n)) return -1;
  double* A = widen_matrix(A16, Na, D);
  double* B = widen_matrix(B16, Nb, D);
  int rc = (A && B) ? fwd_bwd(kind, A, B, Na, Nb, D, prefixes, n, scale, bias, weights, Z, loss, dA, dB,
                              row_terms, col_terms)
                    : -2;
  free(A);
  free(B);
  return rc;
}

int orc_fwd_bwd(int kind, const uint16_t* A16, const uint16_t* B16, int64_t Na, int64_t Nb, int D,
                const int* prefixes, int n, double scale, double bias, const double* weights,
                double* loss, double* dA, double* dB, double* row_terms, double* col_terms) {
  return fwd_bwd_bf16(kind, A16, B16, Na, Nb, D, prefixes, n, scale, bias, weights, NULL, loss, dA, dB,
                      row_terms, col_terms);
}

int orc_fwd_bwd_labels(const uint16_t* A16, const uint16_t* B16, int64_t Na, int64_t Nb, int D,
                       const int* prefixes, int n, double scale, double bias, const double* weights,
                       const unsigned char* Z, double* loss, double* dA, double* dB, double* row_terms,
                       double* col_terms) {
  if (!Z) return -1;
  return fwd_bwd_bf16(ORC_SIGLIP, A16, B16, Na, Nb, D, prefixes, n, scale, bias, weights, Z, loss, dA, dB,
                      row_terms, col_terms);
}

/*
 * One-set SigLIP (blog, section "One Set or Two": the loss scores one set against itself,
 * with the same labels for mirrored cells; an image and its caption are two rows of the
 * set marked as a positive pair).  For the N x D set X and the N x N label matrix Z
 * (symmetric; the diagonal is ignored):
 *   L_k = -(1/N) sum_i sum_{j != i} log sigmoid(z_ij (t cos_ij + b)),
 * cos_ij between x_i[:p] and x_j[:p].  Every cell depends on both of its rows, so
 *   dX_i += w G_ij (xhat_j - cos_ij xhat_i) / |x_i|   (x_i as the first argument)
 *   dX_j += w G_ij (xhat_i - cos_ij xhat_j) / |x_j|   (x_j as the second),
 * G_ij = dL/dcos_ij = t (sigmoid(x_ij) - [z_ij = +1]) / N.  Also dL/dt = sum_ij G_ij cos_ij / t
 * written as (1/N) sum (sigmoid - [z = +1]) cos, and dL/db = (1/N) sum (sigmoid - [z = +1]).
 * row_terms[k][i] = sum_{j != i} softplus(-z_ij x_ij).  dX, row_terms, dscale, dbias may be NULL.
 */
int orc_oneset_f64(const double* X, int64_t N, int D, const int* prefixes, int n, double t, double b,
                   const double* weights, const unsigned char* Z, double* loss, double* dX, double* row_terms,
                   double* dscale, double* dbias) {
  if (check_args(ORC_SIGLIP, N, N, D, prefixes, n) || !Z) return -1;
  double* C = (double*)malloc((size_t)N * N * sizeof(double));
  double* G = (double*)malloc((size_t)N * N * sizeof(double));
  double* r = (double*)malloc((size_t)N * sizeof(double));
  if (!C || !G || !r) {
    free(C); free(G); free(r);
    return -2;
  }
  if (dX) memset(dX, 0, (size_t)N * D * sizeof(double));
  double ds = 0, db = 0;
  for (int k = 0; k < n; ++k) {
    const int p = prefixes[k];
    const double w = weights ? weights[k] : 1.0;
    for (int64_t i = 0; i < N; ++i) r[i] = inv_norm(X + i * D, p);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < N; ++i)
      for (int64_t j = 0; j < N; ++j) {
        double dot = 0;
        for (int d = 0; d < p; ++d) dot += X[i * D + d] * X[j * D + d];
        C[i * N + j] = dot * r[i] * r[j];
      }
    double L = 0, gk = 0, bk = 0;
    for (int64_t i = 0; i < N; ++i) {
      double row = 0;
      for (int64_t j = 0; j < N; ++j) {
        if (j == i) { /* a row is not paired with itself */
          G[i * N + j] = 0;
          continue;
        }
        const double x = t * C[i * N + j] + b;
        const int pos = Z[i * N + j] != 0;
        const double zij = pos ? 1.0 : -1.0;  /* the label z_ij */
        row += softplus(-zij * x);
        const double g = sigmoid(x) - (pos ? 1.0 : 0.0);
        G[i * N + j] = t * g / (double)N;
        gk += g * C[i * N + j];
        bk += g;
      }
      L += row;
      if (row_terms) row_terms[(int64_t)k * N + i] = row;
    }
    loss[k] = L / (double)N;
    ds += w * gk / (double)N;
    db += w * bk / (double)N;
    if (dX) {
#pragma omp parallel for schedule(dynamic, 4)
      for (int64_t i = 0; i < N; ++i) {
        double* out = dX + i * D;
        for (int64_t j = 0; j < N; ++j) {
          /* cell (i, j) through its first argument, and cell (j, i) through its second */
          const double g1 = w * G[i * N + j], g2 = w * G[j * N + i], c = C[i * N + j];
          if (g1 == 0.0 && g2 == 0.0) continue;
          for (int d = 0; d < p; ++d)
            out[d] += (g1 + g2) * (X[j * D + d] * r[j] - c * X[i * D + d] * r[i]) * r[i];
        }
      }
    }
  }
  if (dscale) *dscale = ds;
  if (dbias) *dbias = db;
  free(C); free(G); free(r);
  return 0;
}

int orc_oneset(const uint16_t* X16, int64_t N, int D, const int* prefixes, int n, double t, double b,
               const double* weights, const unsigned char* Z, double* loss, double* dX, double* row_terms,
               double* dscale, double* dbias) {
  if (check_args(ORC_SIGLIP, N, N, D, prefixes, n) || !Z) return -1;
  double* X = widen_matrix(X16, N, D);
  int rc = X ? orc_oneset_f64(X, N, D, prefixes, n, t, b, weights, Z, loss, dX, row_terms, dscale, dbias) : -2;
  free(X);
  return rc;
}

/*
 * Derivatives of the weighted total sum_k weights[k] * L_k with respect to the logit scale
 * and (SIGLIP) the bias, taken directly from the loss definitions on float64 inputs:
 *   CLIP   dL_k/dtau = 1/2 [ (1/N) sum_i (sum_j Prow_ij cos_ij - cos_ii)
 *                          + (1/N) sum_j (sum_i Pcol_ij cos_ij - cos_jj) ],
 *          Prow / Pcol the softmax of tau * cos over the row / the column;
 *   ROWS   dL_k/dtau = (1/Nq) sum_i (sum_j Prow_ij cos_ij - cos_ii);
 *   SIGLIP with x = t cos + b and d/dx softplus(-z x) = sigmoid(x) - [z = +1]:
 *          dL_k/dt = (1/N) sum_ij (sigmoid(x_ij) - [(i, j) positive]) cos_ij,
 *          dL_k/db = (1/N) sum_ij (sigmoid(x_ij) - [(i, j) positive]);  dbias = 0 for CLIP / ROWS.
 * Returns 0, or -1 on bad arguments, -2 when out of memory.
 */
static int scale_grads(int kind, const double* A, const double* B, int64_t Na, int64_t Nb, int D,
                       const int* prefixes, int n, double scale, double bias, const double* weights,
                       const unsigned char* Z, double* dscale, double* dbias) {
  if (check_args(kind, Na, Nb, D, prefixes, n)) return -1;
  if (Z && kind != ORC_SIGLIP) return -1;
  double* C = (double*)malloc((size_t)Na * Nb * sizeof(double));
  double* ra = (double*)malloc((size_t)Na * sizeof(double));
  double* rb = (double*)malloc((size_t)Nb * sizeof(double));
  if (!C || !ra || !rb) {
    free(C); free(ra); free(rb);
    return -2;
  }
  double ds = 0, db = 0;
  for (int k = 0; k < n; ++k) {
    const int p = prefixes[k];
    const double w = weights ? weights[k] : 1.0;
    for (int64_t i = 0; i < Na; ++i) ra[i] = inv_norm(A + i * D, p);
    for (int64_t j = 0; j < Nb; ++j) rb[j] = inv_norm(B + j * D, p);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < Na; ++i)
      for (int64_t j = 0; j < Nb; ++j) {
        double dot = 0;
        for (int d = 0; d < p; ++d) dot += B[j * D + d] * A[i * D + d];
        C[i * Nb + j] = dot * ra[i] * rb[j];
      }
    double gk = 0, bk = 0;
    if (kind == ORC_CLIP || kind == ORC_ROWS) {
      const double tau = scale;
      double rows = 0;  /* sum_i (E_row[cos] - cos_ii) */
      for (int64_t i = 0; i < Na; ++i) {
        double m = -INFINITY, z = 0, zc = 0;
        for (int64_t j = 0; j < Nb; ++j) m = fmax(m, tau * C[i * Nb + j]);
        for (int64_t j = 0; j < Nb; ++j) {
          const double e = exp(tau * C[i * Nb + j] - m);
          z += e;
          zc += e * C[i * Nb + j];
        }
        rows += zc / z - C[i * Nb + i];
      }
      if (kind == ORC_CLIP) {
        double cols = 0;
        for (int64_t j = 0; j < Nb; ++j) {
          double m = -INFINITY, z = 0, zc = 0;
          for (int64_t i = 0; i < Na; ++i) m = fmax(m, tau * C[i * Nb + j]);
          for (int64_t i = 0; i < Na; ++i) {
            const double e = exp(tau * C[i * Nb + j] - m);
            z += e;
            zc += e * C[i * Nb + j];
          }
          cols += zc / z - C[j * Nb + j];
        }
        gk = 0.5 * (rows / (double)Na + cols / (double)Nb);
      } else {
        gk = rows / (double)Na;
      }
    } else {
      const double t = scale, N = (double)Na;
      for (int64_t i = 0; i < Na; ++i)
        for (int64_t j = 0; j < Nb; ++j) {
          const double g = sigmoid(t * C[i * Nb + j] + bias) - (positive(Z, Nb, i, j) ? 1.0 : 0.0);
          gk += g * C[i * Nb + j];
          bk += g;
        }
      gk /= N;
      bk /= N;
    }
    ds += w * gk;
    db += w * bk;
  }
  *dscale = ds;
  *dbias = db;
  free(C); free(ra); free(rb);
  return 0;
}

int orc_scale_grads_f64(int kind, const double* A, const double* B, int64_t Na, int64_t Nb, int D,
                        const int* prefixes, int n, double scale, double bias, const double* weights,
                        double* dscale, double* dbias) {
  return scale_grads(kind, A, B, Na, Nb, D, prefixes, n, scale, bias, weights, NULL, dscale, dbias);
}

int orc_scale_grads_labels_f64(const double* A, const double* B, int64_t Na, int64_t Nb, int D,
                               const int* prefixes, int n, double scale, double bias, const double* weights,
                               const unsigned char* Z, double* dscale, double* dbias) {
  if (!Z) return -1;
  return scale_grads(ORC_SIGLIP, A, B, Na, Nb, D, prefixes, n, scale, bias, weights, Z, dscale, dbias);
}

static int scale_grads_bf16(int kind, const uint16_t* A16, const uint16_t* B16, int64_t Na, int64_t Nb, int D,
                            const int* prefixes, int n, double scale, double bias, const double* weights,
                            const unsigned char* Z, double* dscale, double* dbias) {
  if (check_args(kind, Na, Nb, D, prefixes, n)) return -1;
  double* A = widen_matrix(A16, Na, D);
  double* B = widen_matrix(B16, Nb, D);
  int rc = (A && B) ? scale_grads(kind, A, B, Na, Nb, D, prefixes, n, scale, bias, weights, Z, dscale, dbias)
                    : -2;
  free(A);
  free(B);
  return rc;
}

int orc_scale_grads(int kind, const uint16_t* A16, const uint16_t* B16, int64_t Na, int64_t Nb, int D,
                    const int* prefixes, int n, double scale, double bias, const double* weights,
                    double* dscale, double* dbias) {
  return scale_grads_bf16(kind, A16, B16, Na, Nb, D, prefixes, n, scale, bias, weights, NULL, dscale, dbias);
}

int orc_scale_grads_labels(const uint16_t* A16, const uint16_t* B16, int64_t Na, int64_t Nb, int D,
                           const int* prefixes, int n, double scale, double bias, const double* weights,
                           const unsigned char* Z, double* dscale, double* dbias) {
  if (!Z) return -1;
  return scale_grads_bf16(ORC_SIGLIP, A16, B16, Na, Nb, D, prefixes, n, scale, bias, weights, Z, dscale, dbias);
}

/*
 * Row statistics for selected rows of X against every row of Y, one row at a time
 * (for batches too large for the full grid).  The positive of row i of X is row i
 * of Y.  For each selected row and prefix k:
 *   CLIP/ROWS:  lse[r][k] = log sum_j exp(scale * cos_ij)   (max-shifted)
 *               pos[r][k] = scale * cos_ii  (0 if i >= Ny)
 *   SIGLIP:     lse[r][k] = sum_j softplus(-z_ij (scale * cos_ij + bias)),  pos = 0
 * So the CLIP/ROWS row term is lse - pos and the SIGLIP row term is lse.
 */
int orc_row_stats(int kind, const uint16_t* X16, const uint16_t* Y16, int64_t Nx, int64_t Ny, int D,
                  const int* prefixes, int n, double scale, double bias, const int64_t* rows,
                  int64_t nrows, double* lse, double* pos) {
  if (Nx <= 0 || Ny <= 0 || D <= 0 || n <= 0 || !prefixes || nrows < 0) return -1;
  for (int k = 0; k < n; ++k)
    if (prefixes[k] <= 0 || prefixes[k] > D || (k && prefixes[k] <= prefixes[k - 1])) return -1;
  for (int64_t r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= Nx) return -1;
  double* Y = widen_matrix(Y16, Ny, D);
  double* ryk = (double*)malloc((size_t)n * Ny * sizeof(double)); /* inverse norms of Y per prefix */
  if (!Y || !ryk) { free(Y); free(ryk); return -2; }
  for (int k = 0; k < n; ++k) {
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < Ny; ++j) ryk[(int64_t)k * Ny + j] = inv_norm(Y + j * D, prefixes[k]);
  }
  int err = 0;
#pragma omp parallel
  {
    double* x = (double*)malloc((size_t)D * sizeof(double));
    double* cs = (double*)malloc((size_t)Ny * sizeof(double));
    if (!x || !cs) {
#pragma omp atomic write
      err = -2;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows[r];
        for (int d = 0; d < D; ++d) x[d] = widen(X16[i * D + d]);
        for (int k = 0; k < n; ++k) {
          const int p = prefixes[k];
          const double rx = inv_norm(x, p);
          for (int64_t j = 0; j < Ny; ++j) {
            const double* y = Y + j * D;
            double dot = 0;
            for (int d = 0; d < p; ++d) dot += x[d] * y[d];
            cs[j] = dot * rx * ryk[(int64_t)k * Ny + j];
          }
          if (kind == ORC_SIGLIP) {
            double s = 0;
            for (int64_t j = 0; j < Ny; ++j) {
              double xx = scale * cs[j] + bias;
              s += softplus(j == i ? -xx : xx);
            }
            lse[r * n + k] = s;
            pos[r * n + k] = 0;
          } else {
            double m = -INFINITY, s = 0;
            for (int64_t j = 0; j < Ny; ++j) m = fmax(m, scale * cs[j]);
            for (int64_t j = 0; j < Ny; ++j) s += exp(scale * cs[j] - m);
            lse[r * n + k] = m + log(s);
            pos[r * n + k] = (i < Ny) ? scale * cs[i] : 0.0;
          }
        }
      }
    }
    free(x);
    free(cs);
  }
  free(Y);
  free(ryk);
  return err;
}

/*
 * Gradient rows for selected rows of X (X is A when x_is_a, else B) against all
 * rows of Y, given the log-normalisers the loss needs:
 *   lse_x[k][Nx]  log-normaliser of X's own rows   (CLIP, and ROWS with X = queries)
 *   lse_y[k][Ny]  log-normaliser of Y's rows       (CLIP, and ROWS with X = keys)
 * (SIGLIP needs neither; arrays not needed may be NULL.)  out[r][D] receives the
 * gradient of sum_k weights[k] * L_k with respect to X's row rows[r].
 * Na and Nb are the batch sizes of A and B (for the loss normalisers).
 */
int orc_grad_rows(int kind, int x_is_a, const uint16_t* X16, const uint16_t* Y16, int64_t Nx, int64_t Ny,
                  int D, const int* prefixes, int n, double scale, double bias, const double* weights,
                  const double* lse_x, const double* lse_y, const int64_t* rows, int64_t nrows,
                  double* out) {
  if (Nx <= 0 || Ny <= 0 || D <= 0 || n <= 0 || !prefixes || nrows < 0) return -1;
  for (int64_t r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= Nx) return -1;
  const int64_t Na = x_is_a ? Nx : Ny, Nb = x_is_a ? Ny : Nx;
  if (check_args(kind, Na, Nb, D, prefixes, n)) return -1;
  double* Y = widen_matrix(Y16, Ny, D);
  double* ryk = (double*)malloc((size_t)n * Ny * sizeof(double)); /* inverse norms of Y per prefix */
  if (!Y || !ryk) { free(Y); free(ryk); return -2; }
  for (int k = 0; k < n; ++k) {
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < Ny; ++j) ryk[(int64_t)k * Ny + j] = inv_norm(Y + j * D, prefixes[k]);
  }
  int err = 0;
#pragma omp parallel
  {
    double* x = (double*)malloc((size_t)D * sizeof(double));
    if (!x) {
#pragma omp atomic write
      err = -2;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows[r];
        double* o = out + r * D;
        for (int d = 0; d < D; ++d) { x[d] = widen(X16[i * D + d]); o[d] = 0; }
        for (int k = 0; k < n; ++k) {
          const int p = prefixes[k];
          const double w = weights ? weights[k] : 1.0;
          const double rx = inv_norm(x, p);
          const double* ry = ryk + (int64_t)k * Ny;
          for (int64_t j = 0; j < Ny; ++j) {
            const double* y = Y + j * D;
            double dot = 0;
            for (int d = 0; d < p; ++d) dot += x[d] * y[d];
            const double c = dot * rx * ry[j];
            const int diag = (j == i);
            double g; /* dL/dcos for the pair (x_i, y_j) */
            if (kind == ORC_CLIP) {
              const double s = scale * c;
              g = scale * (exp(s - lse_x[(int64_t)k * Nx + i]) + exp(s - lse_y[(int64_t)k * Ny + j]) -
                           (diag ? 2.0 : 0.0)) / (2.0 * (double)Na);
            } else if (kind == ORC_ROWS) {
              const double s = scale * c;
              /* the query of the pair is row i of X when X holds the queries, else row j of Y */
              const double lq = x_is_a ? lse_x[(int64_t)k * Nx + i] : lse_y[(int64_t)k * Ny + j];
              g = scale * (exp(s - lq) - (diag ? 1.0 : 0.0)) / (double)Na;
            } else {
              const double xx = scale * c + bias;
              g = scale * (sigmoid(xx) - (diag ? 1.0 : 0.0)) / (double)Na;
            }
            g *= w;
            for (int d = 0; d < p; ++d) o[d] += g * (y[d] * ry[j] - c * x[d] * rx) * rx;
          }
        }
      }
    }
    free(x);
  }
  free(Y);
  free(ryk);
  return err;
}
