/*
 * tpmlp_oracle.c -- plain fp64 CPU oracle for the t-sharded Megatron MLP block.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA path and must never be used as a
 * fallback for it.
 *
 * What it computes (row convention, every matrix row-major):
 *   X  [T x d]      tokens x hidden
 *   W1 [d x dff]    first linear (SwiGLU: the gate projection)
 *   W3 [d x dff]    SwiGLU up projection (unused for GeLU)
 *   W2 [dff x d]    second linear
 *   GeLU  : A = X W1,          H = GeLU(A),            Y = H W2
 *   SwiGLU: G = X W1, U = X W3, H = U * Swish(G),      Y = H W2
 * Sources:
 *   - "Parallelism" tag page of Jiang Yi's homepage, post "megatron-lm",
 *     Method / FFN: the Linear-GeLU-Linear FFN Y = GeLU(X W1) W2 with
 *     X in R^{bs x d}, W1 in R^{d x dff}, W2 in R^{dff x d}; the column split of
 *     W1, the row split of W2 and the SwiGLU form Y = (X W3 . Swish(X W1)) W2.
 *   - "Tensor parallelism" (brunomaga.github.io), section "Megatron-LM tensor
 *     parallelism": Megatron_FeedForward calls F.gelu (the exact, erf-based
 *     GeLU) and the f/g operators.
 *   - "Parallelism" page, Implementation / SwiGLU listing: the gate is
 *     silu(w1(x)) multiplied by w3(x), i.e. Swish with beta = 1.
 * The backward pass is the chain rule applied to the definitions above;
 * the backward of the seed is an input dY (no loss is formed).
 *
 * Unsharded functions compute the block directly.  The sharded functions
 * follow the pages' per-shard formulation (column shard i owns columns
 * [o_i, o_i + d_i) of W1/W3 and rows [o_i, o_i + d_i) of W2; forward partial
 * outputs Z_i are summed by the g operator, backward partial input gradients
 * dX_i are summed by the f operator) and exist so the tests can check the
 * identities the pages state.
 *
 * Biases (optional, NULL = none): b1 [dff] (and b3 [dff] for SwiGLU) are
 * added to the first linear's output before the activation, b2 [d] to Y once
 * after the g-sum -- "Tensor parallelism" (brunomaga.github.io),
 * Megatron_FeedForward: fc1 carries its bias, fc2 has none and fc2_bias is
 * added after the all-reduce so that it is not counted once per shard.
 * Their gradients are column sums over tokens: db1 = sum_r dA[r, :],
 * db3 = sum_r dU[r, :], db2 = sum_r dY[r, :].
 *
 * The sequence-parallel layout (forward_sp / backward_sp) takes X and dY as
 * stripes of tokens and returns Y and dX as stripes, gathering before the
 * block and reduce-scattering after it.
 *
 * The attention block's two projections (QKV, column-split by heads, and the
 * output projection, row-split with the g-sum) have their own functions
 * below; the attention core between them is a different operation and is an
 * input here (O, and dQ/dK/dV in the backward).
 *
 * Two extra activations, identity and ReLU, are test hooks: they keep
 * small-integer inputs integral so sharded and unsharded results can be
 * compared exactly.
 *
 * Every loop is a plain definition: no blocking, no reordering beyond the
 * OpenMP split of independent output rows.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_ACT_GELU 0
#define ORACLE_ACT_SWIGLU 1
#define ORACLE_ACT_IDENTITY 2 /* test hook */
#define ORACLE_ACT_RELU 3     /* test hook */

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NOMEM 2

/* ---- activations and their derivatives (scalar, fp64) ------------------ */

/* Standard normal CDF and density. */
static double norm_cdf(double a) { return 0.5 * (1.0 + erf(a / sqrt(2.0))); }
static double norm_pdf(double a) { return exp(-0.5 * a * a) / sqrt(2.0 * M_PI); }

/* GeLU(a) = a * Phi(a) (erf form). */
static double gelu(double a) { return a * norm_cdf(a); }
/* d/da GeLU(a) = Phi(a) + a * phi(a). */
static double gelu_grad(double a) { return norm_cdf(a) + a * norm_pdf(a); }

static double sigmoid(double g) { return 1.0 / (1.0 + exp(-g)); }
/* Swish_1(g) = g * sigmoid(g). */
static double swish(double g) { return g * sigmoid(g); }
/* d/dg Swish_1(g) = s + g s (1 - s), s = sigmoid(g). */
static double swish_grad(double g) {
  double s = sigmoid(g);
  return s + g * s * (1.0 - s);
}

/* Elementwise act for the single-input activations (GeLU and the hooks). */
static double act_value(int act, double a) {
  switch (act) {
    case ORACLE_ACT_GELU: return gelu(a);
    case ORACLE_ACT_IDENTITY: return a;
    case ORACLE_ACT_RELU: return a > 0.0 ? a : 0.0;
    default: return NAN;
  }
}
static double act_grad(int act, double a) {
  switch (act) {
    case ORACLE_ACT_GELU: return gelu_grad(a);
    case ORACLE_ACT_IDENTITY: return 1.0;
    case ORACLE_ACT_RELU: return a > 0.0 ? 1.0 : 0.0;
    default: return NAN;
  }
}

/* ---- plain matrix product ------------------------------------------------
 * C[m][n] = sum_k A(m,k) * B(k,n) for m < M, n < N, k < K in increasing k.
 * A(m,k) = A[m*sam + k*sak], B(k,n) = B[k*sbk + n*sbn], C[m*ldc + n].
 * The strides express transposed operands without copies.                   */
static void matmul(int64_t M, int64_t N, int64_t K,
                   const double* A, int64_t sam, int64_t sak,
                   const double* B, int64_t sbk, int64_t sbn,
                   double* C, int64_t ldc) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      double s = 0.0;
      for (int64_t k = 0; k < K; ++k) s += A[m * sam + k * sak] * B[k * sbk + n * sbn];
      C[m * ldc + n] = s;
    }
  }
}

static int valid_act(int act) {
  return act == ORACLE_ACT_GELU || act == ORACLE_ACT_SWIGLU || act == ORACLE_ACT_IDENTITY ||
         act == ORACLE_ACT_RELU;
}

/* M[r][c] += b[c] for every row (no-op for b == NULL). */
static void add_row_bias(int64_t rows, int64_t cols, double* M, const double* b) {
  if (!b) return;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) M[r * cols + c] += b[c];
}

/* out[c] = sum over rows r of M[r][c] (r increasing). */
static void col_sums(int64_t rows, int64_t cols, const double* M, double* out) {
  if (!out) return;
  for (int64_t c = 0; c < cols; ++c) out[c] = 0.0;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) out[c] += M[r * cols + c];
}

/* ---- unsharded forward ----------------------------------------------------
 * Outputs: A (SwiGLU: G) [T x dff], U [T x dff] (SwiGLU only, may be NULL
 * otherwise), H [T x dff], Y [T x d].                                        */
int oracle_forward(int64_t T, int64_t d, int64_t dff, int act, const double* X, const double* W1,
                   const double* W3, const double* W2, const double* b1, const double* b3, const double* b2,
                   double* A, double* U, double* H, double* Y) {
  if (T < 0 || d < 1 || dff < 1 || !valid_act(act) || !X || !W1 || !W2 || !A || !H || !Y)
    return ORACLE_ERR_ARG;
  if (act == ORACLE_ACT_SWIGLU && (!W3 || !U)) return ORACLE_ERR_ARG;
  /* A = X W1 + b1 */
  matmul(T, dff, d, X, d, 1, W1, dff, 1, A, dff);
  add_row_bias(T, dff, A, b1);
  if (act == ORACLE_ACT_SWIGLU) {
    /* U = X W3 + b3; H = U * Swish(G) */
    matmul(T, dff, d, X, d, 1, W3, dff, 1, U, dff);
    add_row_bias(T, dff, U, b3);
    for (int64_t i = 0; i < T * dff; ++i) H[i] = U[i] * swish(A[i]);
  } else {
    for (int64_t i = 0; i < T * dff; ++i) H[i] = act_value(act, A[i]);
  }
  /* Y = H W2 + b2 */
  matmul(T, d, dff, H, dff, 1, W2, d, 1, Y, d);
  add_row_bias(T, d, Y, b2);
  return ORACLE_OK;
}

/* ---- unsharded backward ---------------------------------------------------
 * Given dY = dL/dY, returns dX, dW1, dW3 (SwiGLU only), dW2, the bias
 * gradients db1, db3, db2 (each may be NULL) and the activation gradient dA
 * (SwiGLU: dG) / dU, recomputing the forward from X.  Any of dAct/dUo may be
 * NULL if not wanted.                                                        */
int oracle_backward(int64_t T, int64_t d, int64_t dff, int act, const double* X, const double* W1,
                    const double* W3, const double* W2, const double* b1, const double* b3, const double* b2,
                    const double* dY, double* dX, double* dW1, double* dW3, double* dW2, double* db1,
                    double* db3, double* db2, double* dAct, double* dUo) {
  if (T < 0 || d < 1 || dff < 1 || !valid_act(act) || !X || !W1 || !W2 || !dY || !dX || !dW1 || !dW2)
    return ORACLE_ERR_ARG;
  int swiglu = act == ORACLE_ACT_SWIGLU;
  if (swiglu && (!W3 || !dW3)) return ORACLE_ERR_ARG;
  size_t n = (size_t)(T * dff);
  size_t nb = n ? n : 1;
  double* A = (double*)malloc(nb * sizeof(double));
  double* U = swiglu ? (double*)malloc(nb * sizeof(double)) : NULL;
  double* H = (double*)malloc(nb * sizeof(double));
  double* dH = (double*)malloc(nb * sizeof(double));
  double* dA = (double*)malloc(nb * sizeof(double));
  double* dU = swiglu ? (double*)malloc(nb * sizeof(double)) : NULL;
  double* Y = (double*)malloc((size_t)(T * d ? T * d : 1) * sizeof(double));
  int rc = ORACLE_ERR_NOMEM;
  if (!A || !H || !dH || !dA || !Y || (swiglu && (!U || !dU))) goto done;
  rc = oracle_forward(T, d, dff, act, X, W1, W3, W2, b1, b3, b2, A, U, H, Y);
  if (rc) goto done;
  /* dH = dY W2^T : dH[r][j] = sum_n dY[r][n] W2[j][n] */
  matmul(T, dff, d, dY, d, 1, W2, 1, d, dH, dff);
  if (swiglu) {
    /* H = U * Swish(G): dU = dH * Swish(G), dG = dH * U * Swish'(G) */
    for (size_t i = 0; i < n; ++i) {
      dU[i] = dH[i] * swish(A[i]);
      dA[i] = dH[i] * U[i] * swish_grad(A[i]);
    }
  } else {
    for (size_t i = 0; i < n; ++i) dA[i] = dH[i] * act_grad(act, A[i]);
  }
  /* dW2 = H^T dY : dW2[j][n] = sum_r H[r][j] dY[r][n] */
  matmul(dff, d, T, H, 1, dff, dY, d, 1, dW2, d);
  /* dW1 = X^T dA : dW1[k][j] = sum_r X[r][k] dA[r][j] */
  matmul(d, dff, T, X, 1, d, dA, dff, 1, dW1, dff);
  /* dX = dA W1^T (+ dU W3^T) */
  matmul(T, d, dff, dA, dff, 1, W1, 1, dff, dX, d);
  if (swiglu) {
    matmul(d, dff, T, X, 1, d, dU, dff, 1, dW3, dff);
    double* dX3 = (double*)malloc((size_t)(T * d ? T * d : 1) * sizeof(double));
    if (!dX3) { rc = ORACLE_ERR_NOMEM; goto done; }
    matmul(T, d, dff, dU, dff, 1, W3, 1, dff, dX3, d);
    for (int64_t i = 0; i < T * d; ++i) dX[i] += dX3[i];
    free(dX3);
  }
  col_sums(T, dff, dA, db1);
  if (swiglu) col_sums(T, dff, dU, db3);
  col_sums(T, d, dY, db2);
  if (dAct) memcpy(dAct, dA, n * sizeof(double));
  if (dUo && swiglu) memcpy(dUo, dU, n * sizeof(double));
  rc = ORACLE_OK;
done:
  free(A); free(U); free(H); free(dH); free(dA); free(dU); free(Y);
  return rc;
}

/* ---- sharded forward (the pages' per-shard formulation) ------------------
 * Shard i: A_i = X W1_i, H_i = act(A_i) (SwiGLU: U_i * Swish(X W1_i) with
 * U_i = X W3_i), Z_i = H_i W2_i; the g operator (forward all-reduce) gives
 * Y = sum_i Z_i, summed in shard order.  W1_i, W3_i are [d x d_i], W2_i is
 * [d_i x d], H_i is [T x d_i] (optional output; pass NULL to skip).          */
int oracle_forward_sharded(int64_t T, int64_t d, int32_t t, const int64_t* d_i, int act,
                           const double* X, const double* const* W1_i, const double* const* W3_i,
                           const double* const* W2_i, const double* const* b1_i, const double* const* b3_i,
                           const double* b2, double* Y, double* const* H_i) {
  if (T < 0 || d < 1 || t < 1 || !d_i || !valid_act(act) || !X || !W1_i || !W2_i || !Y)
    return ORACLE_ERR_ARG;
  int swiglu = act == ORACLE_ACT_SWIGLU;
  if (swiglu && !W3_i) return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < T * d; ++i) Y[i] = 0.0;
  for (int32_t s = 0; s < t; ++s) {
    int64_t di = d_i[s];
    if (di < 1) return ORACLE_ERR_ARG;
    size_t n = (size_t)(T * di ? T * di : 1);
    double* A = (double*)malloc(n * sizeof(double));
    double* U = swiglu ? (double*)malloc(n * sizeof(double)) : NULL;
    double* H = (double*)malloc(n * sizeof(double));
    double* Z = (double*)malloc((size_t)(T * d ? T * d : 1) * sizeof(double));
    if (!A || !H || !Z || (swiglu && !U)) {
      free(A); free(U); free(H); free(Z);
      return ORACLE_ERR_NOMEM;
    }
    matmul(T, di, d, X, d, 1, W1_i[s], di, 1, A, di);
    add_row_bias(T, di, A, b1_i ? b1_i[s] : NULL);
    if (swiglu) {
      matmul(T, di, d, X, d, 1, W3_i[s], di, 1, U, di);
      add_row_bias(T, di, U, b3_i ? b3_i[s] : NULL);
      for (int64_t i = 0; i < T * di; ++i) H[i] = U[i] * swish(A[i]);
    } else {
      for (int64_t i = 0; i < T * di; ++i) H[i] = act_value(act, A[i]);
    }
    matmul(T, d, di, H, di, 1, W2_i[s], d, 1, Z, d);
    for (int64_t i = 0; i < T * d; ++i) Y[i] += Z[i]; /* g: sum of partial outputs */
    if (H_i && H_i[s]) memcpy(H_i[s], H, (size_t)(T * di) * sizeof(double));
    free(A); free(U); free(H); free(Z);
  }
  add_row_bias(T, d, Y, b2); /* once, after the g-sum */
  return ORACLE_OK;
}

/* ---- sharded backward ------------------------------------------------------
 * g backward is the identity (every shard receives the same dY); each shard
 * forms dH_i = dY W2_i^T, dA_i, dW2_i = H_i^T dY, dW1_i = X^T dA_i
 * (SwiGLU: dW3_i = X^T dU_i) and its partial input gradient
 * dX_i = dA_i W1_i^T (+ dU_i W3_i^T); f backward (all-reduce) gives
 * dX = sum_i dX_i, summed in shard order.                                    */
int oracle_backward_sharded(int64_t T, int64_t d, int32_t t, const int64_t* d_i, int act,
                            const double* X, const double* const* W1_i, const double* const* W3_i,
                            const double* const* W2_i, const double* const* b1_i, const double* const* b3_i,
                            const double* dY, double* dX, double* const* dW1_i, double* const* dW3_i,
                            double* const* dW2_i, double* const* db1_i, double* const* db3_i, double* db2) {
  if (T < 0 || d < 1 || t < 1 || !d_i || !valid_act(act) || !X || !W1_i || !W2_i || !dY || !dX ||
      !dW1_i || !dW2_i)
    return ORACLE_ERR_ARG;
  int swiglu = act == ORACLE_ACT_SWIGLU;
  if (swiglu && (!W3_i || !dW3_i)) return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < T * d; ++i) dX[i] = 0.0;
  for (int32_t s = 0; s < t; ++s) {
    int64_t di = d_i[s];
    if (di < 1) return ORACLE_ERR_ARG;
    size_t n = (size_t)(T * di ? T * di : 1);
    size_t nx = (size_t)(T * d ? T * d : 1);
    double* A = (double*)malloc(n * sizeof(double));
    double* U = swiglu ? (double*)malloc(n * sizeof(double)) : NULL;
    double* H = (double*)malloc(n * sizeof(double));
    double* dH = (double*)malloc(n * sizeof(double));
    double* dA = (double*)malloc(n * sizeof(double));
    double* dU = swiglu ? (double*)malloc(n * sizeof(double)) : NULL;
    double* dXs = (double*)malloc(nx * sizeof(double));
    double* dX3 = swiglu ? (double*)malloc(nx * sizeof(double)) : NULL;
    int bad = !A || !H || !dH || !dA || !dXs || (swiglu && (!U || !dU || !dX3));
    if (!bad) {
      matmul(T, di, d, X, d, 1, W1_i[s], di, 1, A, di);
      add_row_bias(T, di, A, b1_i ? b1_i[s] : NULL);
      if (swiglu) {
        matmul(T, di, d, X, d, 1, W3_i[s], di, 1, U, di);
        add_row_bias(T, di, U, b3_i ? b3_i[s] : NULL);
        for (int64_t i = 0; i < T * di; ++i) H[i] = U[i] * swish(A[i]);
      } else {
        for (int64_t i = 0; i < T * di; ++i) H[i] = act_value(act, A[i]);
      }
      matmul(T, di, d, dY, d, 1, W2_i[s], 1, d, dH, di);
      if (swiglu) {
        for (int64_t i = 0; i < T * di; ++i) {
          dU[i] = dH[i] * swish(A[i]);
          dA[i] = dH[i] * U[i] * swish_grad(A[i]);
        }
      } else {
        for (int64_t i = 0; i < T * di; ++i) dA[i] = dH[i] * act_grad(act, A[i]);
      }
      matmul(di, d, T, H, 1, di, dY, d, 1, dW2_i[s], d);
      matmul(d, di, T, X, 1, d, dA, di, 1, dW1_i[s], di);
      matmul(T, d, di, dA, di, 1, W1_i[s], 1, di, dXs, d);
      if (swiglu) {
        matmul(d, di, T, X, 1, d, dU, di, 1, dW3_i[s], di);
        matmul(T, d, di, dU, di, 1, W3_i[s], 1, di, dX3, d);
        for (int64_t i = 0; i < T * d; ++i) dXs[i] += dX3[i];
      }
      for (int64_t i = 0; i < T * d; ++i) dX[i] += dXs[i]; /* f: sum of partial dX */
      col_sums(T, di, dA, db1_i ? db1_i[s] : NULL);
      if (swiglu) col_sums(T, di, dU, db3_i ? db3_i[s] : NULL);
    }
    free(A); free(U); free(H); free(dH); free(dA); free(dU); free(dXs); free(dX3);
    if (bad) return ORACLE_ERR_NOMEM;
  }
  col_sums(T, d, dY, db2); /* g backward is the identity: b2 sees dY once */
  return ORACLE_OK;
}

/* ---- sampled outputs for large problems -----------------------------------
 * oracle_rows: Y[r, :] and dX[r, :] for the listed token rows r, each from
 * its own definition (a token's forward and input gradient depend only on
 * that token's row of X and dY).  Y_rows and dX_rows are [nrows x d].
 * Optionally (NULL = not wanted) the same rows of the per-token
 * intermediates, each [nrows x dff]: A_rows = X W1 (+ b1) (SwiGLU: G),
 * U_rows = X W3 (+ b3) (SwiGLU only), H_rows = act(A) (SwiGLU: U Swish(G)),
 * dA_rows = the gradient of A (SwiGLU: of G), dU_rows = the gradient of U
 * (SwiGLU only).                                                             */
int oracle_rows(int64_t T, int64_t d, int64_t dff, int act, const double* X, const double* W1,
                const double* W3, const double* W2, const double* b1, const double* b3, const double* b2,
                const double* dY, int64_t nrows, const int64_t* rows, double* Y_rows, double* dX_rows,
                double* A_rows, double* U_rows, double* H_rows, double* dA_rows, double* dU_rows) {
  if (T < 1 || d < 1 || dff < 1 || !valid_act(act) || nrows < 0 || !rows || !X || !W1 || !W2 ||
      !dY || !Y_rows || !dX_rows)
    return ORACLE_ERR_ARG;
  int swiglu = act == ORACLE_ACT_SWIGLU;
  if (swiglu && !W3) return ORACLE_ERR_ARG;
  for (int64_t q = 0; q < nrows; ++q)
    if (rows[q] < 0 || rows[q] >= T) return ORACLE_ERR_ARG;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t q = 0; q < nrows; ++q) {
    const double* x = X + rows[q] * d;
    const double* g = dY + rows[q] * d;
    double* a = (double*)malloc((size_t)dff * 5 * sizeof(double));
    if (!a) { err = 1; continue; }
    double* u = a + dff;
    double* h = a + 2 * dff;
    double* dh = a + 3 * dff;
    double* da = a + 4 * dff;
    for (int64_t j = 0; j < dff; ++j) {
      double s = 0.0, s3 = 0.0, sg = 0.0;
      for (int64_t k = 0; k < d; ++k) {
        s += x[k] * W1[k * dff + j];
        if (swiglu) s3 += x[k] * W3[k * dff + j];
      }
      if (b1) s += b1[j];
      if (swiglu && b3) s3 += b3[j];
      for (int64_t n = 0; n < d; ++n) sg += g[n] * W2[j * d + n];
      a[j] = s;
      u[j] = s3;
      dh[j] = sg;
      if (swiglu) {
        h[j] = s3 * swish(s);
        da[j] = sg * s3 * swish_grad(s);
      } else {
        h[j] = act_value(act, s);
        da[j] = sg * act_grad(act, s);
      }
    }
    for (int64_t n = 0; n < d; ++n) {
      double y = 0.0, dx = 0.0;
      for (int64_t j = 0; j < dff; ++j) {
        y += h[j] * W2[j * d + n];
        dx += da[j] * W1[n * dff + j];
        if (swiglu) dx += dh[j] * swish(a[j]) * W3[n * dff + j];
      }
      Y_rows[q * d + n] = y + (b2 ? b2[n] : 0.0);
      dX_rows[q * d + n] = dx;
    }
    for (int64_t j = 0; j < dff; ++j) {
      if (A_rows) A_rows[q * dff + j] = a[j];
      if (H_rows) H_rows[q * dff + j] = h[j];
      if (dA_rows) dA_rows[q * dff + j] = da[j];
      if (swiglu && U_rows) U_rows[q * dff + j] = u[j];
      if (swiglu && dU_rows) dU_rows[q * dff + j] = dh[j] * swish(a[j]);
    }
    free(a);
  }
  return err ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* oracle_wgrad_units: for the listed hidden units j (columns of W1/W3, rows
 * of W2), dW1[:, j], dW3[:, j] (SwiGLU) and dW2[j, :], each a sum over all T
 * tokens of its definition.  Outputs are [nunits x d]: dW1_cols[q*d + k] =
 * dW1[k][j_q], dW2_rows[q*d + n] = dW2[j_q][n].                              */
int oracle_wgrad_units(int64_t T, int64_t d, int64_t dff, int act, const double* X, const double* W1,
                       const double* W3, const double* W2, const double* b1, const double* b3,
                       const double* dY, int64_t nunits, const int64_t* units, double* dW1_cols,
                       double* dW3_cols, double* dW2_rows, double* db1_units, double* db3_units) {
  if (T < 0 || d < 1 || dff < 1 || !valid_act(act) || nunits < 0 || !units || !X || !W1 || !W2 ||
      !dY || !dW1_cols || !dW2_rows)
    return ORACLE_ERR_ARG;
  int swiglu = act == ORACLE_ACT_SWIGLU;
  if (swiglu && (!W3 || !dW3_cols)) return ORACLE_ERR_ARG;
  for (int64_t q = 0; q < nunits; ++q)
    if (units[q] < 0 || units[q] >= dff) return ORACLE_ERR_ARG;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t q = 0; q < nunits; ++q) {
    int64_t j = units[q];
    size_t nt = (size_t)(T ? T : 1);
    double* h = (double*)malloc(nt * 3 * sizeof(double));
    if (!h) { err = 1; continue; }
    double* da = h + nt;
    double* du = h + 2 * nt;
    for (int64_t r = 0; r < T; ++r) {
      double a = 0.0, u = 0.0, dh = 0.0;
      for (int64_t k = 0; k < d; ++k) {
        a += X[r * d + k] * W1[k * dff + j];
        if (swiglu) u += X[r * d + k] * W3[k * dff + j];
      }
      if (b1) a += b1[j];
      if (swiglu && b3) u += b3[j];
      for (int64_t n = 0; n < d; ++n) dh += dY[r * d + n] * W2[j * d + n];
      if (swiglu) {
        h[r] = u * swish(a);
        da[r] = dh * u * swish_grad(a);
        du[r] = dh * swish(a);
      } else {
        h[r] = act_value(act, a);
        da[r] = dh * act_grad(act, a);
        du[r] = 0.0;
      }
    }
    for (int64_t k = 0; k < d; ++k) {
      double s1 = 0.0, s3 = 0.0, s2 = 0.0;
      for (int64_t r = 0; r < T; ++r) {
        s1 += X[r * d + k] * da[r];
        if (swiglu) s3 += X[r * d + k] * du[r];
        s2 += h[r] * dY[r * d + k];
      }
      dW1_cols[q * d + k] = s1;
      if (swiglu) dW3_cols[q * d + k] = s3;
      dW2_rows[q * d + k] = s2;
    }
    if (db1_units) {
      double s = 0.0;
      for (int64_t r = 0; r < T; ++r) s += da[r];
      db1_units[q] = s;
    }
    if (db3_units && swiglu) {
      double s = 0.0;
      for (int64_t r = 0; r < T; ++r) s += du[r];
      db3_units[q] = s;
    }
    free(h);
  }
  return err ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* ---- sequence-parallel layout ----------------------------------------------
 * "AI Training Network Primer" ch. 3, section 3.4, Fig. 3.7 (sequence
 * parallelism with TP = t): every rank keeps a stripe of the tokens; an
 * all-gather rebuilds the full X before the block, and a reduce-scatter after
 * it sums the shards' partial outputs and gives every rank the rows of its
 * own stripe; the backward pass mirrors it (all-gather of the dY stripes,
 * reduce-scatter of the partial dX).  Here the stripes are arrays of
 * nstripes pointers with stripe_rows[j] rows each (their sum is T), in token
 * order.  The activations H_i and the weight gradients are full per shard.  */
static int gather_rows(int64_t d, int32_t nstripes, const int64_t* stripe_rows, const double* const* src,
                       double* dst) {
  int64_t r = 0;
  for (int32_t j = 0; j < nstripes; ++j) {
    if (stripe_rows[j] < 0 || (stripe_rows[j] > 0 && !src[j])) return ORACLE_ERR_ARG;
    if (stripe_rows[j]) memcpy(dst + r * d, src[j], (size_t)(stripe_rows[j] * d) * sizeof(double));
    r += stripe_rows[j];
  }
  return ORACLE_OK;
}

static int64_t stripes_total(int32_t nstripes, const int64_t* stripe_rows) {
  int64_t r = 0;
  for (int32_t j = 0; j < nstripes; ++j) r += stripe_rows[j];
  return r;
}

/* Y_j = sum over shards i of the rows of stripe j of Z_i (+ b2, once). */
int oracle_forward_sp(int64_t T, int64_t d, int32_t t, const int64_t* d_i, int act, int32_t nstripes,
                      const int64_t* stripe_rows, const double* const* X_j, const double* const* W1_i,
                      const double* const* W3_i, const double* const* W2_i, const double* const* b1_i,
                      const double* const* b3_i, const double* b2, double* const* Y_j, double* const* H_i) {
  if (T < 0 || d < 1 || t < 1 || nstripes < 1 || !stripe_rows || !X_j || !Y_j || !d_i || !valid_act(act) ||
      !W1_i || !W2_i || stripes_total(nstripes, stripe_rows) != T)
    return ORACLE_ERR_ARG;
  int swiglu = act == ORACLE_ACT_SWIGLU;
  if (swiglu && !W3_i) return ORACLE_ERR_ARG;
  size_t nx = (size_t)(T * d ? T * d : 1);
  double* X = (double*)malloc(nx * sizeof(double));       /* all-gather */
  double* Z = (double*)malloc((size_t)t * nx * sizeof(double)); /* partial outputs Z_i */
  if (!X || !Z) { free(X); free(Z); return ORACLE_ERR_NOMEM; }
  int rc = gather_rows(d, nstripes, stripe_rows, X_j, X);
  for (int32_t s = 0; rc == ORACLE_OK && s < t; ++s) {
    int64_t di = d_i[s];
    if (di < 1) { rc = ORACLE_ERR_ARG; break; }
    size_t n = (size_t)(T * di ? T * di : 1);
    double* A = (double*)malloc(n * sizeof(double));
    double* U = swiglu ? (double*)malloc(n * sizeof(double)) : NULL;
    double* H = (double*)malloc(n * sizeof(double));
    if (!A || !H || (swiglu && !U)) { free(A); free(U); free(H); rc = ORACLE_ERR_NOMEM; break; }
    matmul(T, di, d, X, d, 1, W1_i[s], di, 1, A, di);
    add_row_bias(T, di, A, b1_i ? b1_i[s] : NULL);
    if (swiglu) {
      matmul(T, di, d, X, d, 1, W3_i[s], di, 1, U, di);
      add_row_bias(T, di, U, b3_i ? b3_i[s] : NULL);
      for (int64_t i = 0; i < T * di; ++i) H[i] = U[i] * swish(A[i]);
    } else {
      for (int64_t i = 0; i < T * di; ++i) H[i] = act_value(act, A[i]);
    }
    matmul(T, d, di, H, di, 1, W2_i[s], d, 1, Z + (size_t)s * nx, d);
    if (H_i && H_i[s]) memcpy(H_i[s], H, (size_t)(T * di) * sizeof(double));
    free(A); free(U); free(H);
  }
  /* reduce-scatter: stripe j receives the shard sum of its own rows */
  int64_t r0 = 0;
  for (int32_t j = 0; rc == ORACLE_OK && j < nstripes; ++j) {
    for (int64_t r = 0; r < stripe_rows[j]; ++r)
      for (int64_t c = 0; c < d; ++c) {
        double v = 0.0;
        for (int32_t s = 0; s < t; ++s) v += Z[(size_t)s * nx + (size_t)((r0 + r) * d + c)];
        Y_j[j][r * d + c] = v + (b2 ? b2[c] : 0.0);
      }
    r0 += stripe_rows[j];
  }
  free(X); free(Z);
  return rc;
}

/* dX_j = sum over shards of the rows of stripe j of dX_i; weight and bias
 * gradients from the gathered X and dY.                                      */
int oracle_backward_sp(int64_t T, int64_t d, int32_t t, const int64_t* d_i, int act, int32_t nstripes,
                       const int64_t* stripe_rows, const double* const* X_j, const double* const* W1_i,
                       const double* const* W3_i, const double* const* W2_i, const double* const* b1_i,
                       const double* const* b3_i, const double* const* dY_j, double* const* dX_j,
                       double* const* dW1_i, double* const* dW3_i, double* const* dW2_i, double* const* db1_i,
                       double* const* db3_i, double* db2) {
  if (T < 0 || d < 1 || t < 1 || nstripes < 1 || !stripe_rows || !X_j || !dY_j || !dX_j ||
      stripes_total(nstripes, stripe_rows) != T)
    return ORACLE_ERR_ARG;
  size_t nx = (size_t)(T * d ? T * d : 1);
  double* X = (double*)malloc(nx * sizeof(double));
  double* dY = (double*)malloc(nx * sizeof(double));
  double* dX = (double*)malloc(nx * sizeof(double));
  if (!X || !dY || !dX) { free(X); free(dY); free(dX); return ORACLE_ERR_NOMEM; }
  int rc = gather_rows(d, nstripes, stripe_rows, X_j, X);        /* all-gather of X */
  if (rc == ORACLE_OK) rc = gather_rows(d, nstripes, stripe_rows, dY_j, dY); /* all-gather of dY */
  if (rc == ORACLE_OK)
    rc = oracle_backward_sharded(T, d, t, d_i, act, X, W1_i, W3_i, W2_i, b1_i, b3_i, dY, dX, dW1_i, dW3_i, dW2_i,
                                 db1_i, db3_i, db2);
  int64_t r0 = 0;  /* the f-sum of the partial dX_i, scattered by stripe */
  for (int32_t j = 0; rc == ORACLE_OK && j < nstripes; ++j) {
    if (stripe_rows[j]) memcpy(dX_j[j], dX + r0 * d, (size_t)(stripe_rows[j] * d) * sizeof(double));
    r0 += stripe_rows[j];
  }
  free(X); free(dY); free(dX);
  return rc;
}

/* ---- tensor-parallel attention projections -------------------------------
 * The attention core (softmax) is a different operation and is not part of
 * this library; O (the attention output per token) is an input here.
 *   Q = X WQ, K = X WK, V = X WV      (WQ [d x dq]; WK, WV [d x dkv])
 *   Z = O WO                          (O [T x dq], WO [dq x d])
 * dq = query heads x head size, dkv = key/value heads x head size (equal
 * to dq without grouped-query attention).
 * Backward, given dZ and the attention core's dQ, dK, dV:
 *   dO = dZ WO^T, dWO = O^T dZ, dX = dQ WQ^T + dK WK^T + dV WV^T,
 *   dWQ = X^T dQ, dWK = X^T dK, dWV = X^T dV.
 * Sharded by heads ("Parallelism" tag page of Jiang Yi's homepage, post
 * "megatron-lm", Method / Attention: W_Q = [W_Q1 ... W_Qh] by heads,
 * O = [o_1 ... o_h] W_O; "Tensor parallelism" (brunomaga.github.io),
 * Megatron_MHA: column-parallel QKV, row-parallel output projection, f on the
 * input, g on the output; "AI Training Network Primer" ch. 3, Fig. 3.5: with
 * grouped-query attention a shard owns 16 query heads and one key/value head,
 * so its W_Q slice is wider than its W_K and W_V slices).  Shard i owns
 * wq_i columns of WQ (and rows of WO) and wkv_i columns of WK and WV;
 * Z = sum_i O_i WO_i (g) and dX = sum_i of the shard's three products (f).   */
int oracle_attn_forward(int64_t T, int64_t d, int64_t dq, int64_t dkv, const double* X, const double* WQ,
                        const double* WK, const double* WV, const double* O, const double* WO, double* Q, double* K,
                        double* V, double* Z) {
  if (T < 0 || d < 1 || dq < 1 || dkv < 1 || !X || !WQ || !WK || !WV || !O || !WO || !Q || !K || !V || !Z)
    return ORACLE_ERR_ARG;
  matmul(T, dq, d, X, d, 1, WQ, dq, 1, Q, dq);
  matmul(T, dkv, d, X, d, 1, WK, dkv, 1, K, dkv);
  matmul(T, dkv, d, X, d, 1, WV, dkv, 1, V, dkv);
  matmul(T, d, dq, O, dq, 1, WO, d, 1, Z, d);
  return ORACLE_OK;
}

int oracle_attn_backward(int64_t T, int64_t d, int64_t dq, int64_t dkv, const double* X, const double* WQ,
                         const double* WK, const double* WV, const double* O, const double* WO, const double* dZ,
                         const double* dQ, const double* dK, const double* dV, double* dO, double* dWO, double* dX,
                         double* dWQ, double* dWK, double* dWV) {
  if (T < 0 || d < 1 || dq < 1 || dkv < 1 || !X || !WQ || !WK || !WV || !O || !WO || !dZ || !dQ || !dK || !dV ||
      !dO || !dWO || !dX || !dWQ || !dWK || !dWV)
    return ORACLE_ERR_ARG;
  double* tmp = (double*)malloc((size_t)(T * d ? T * d : 1) * sizeof(double));
  if (!tmp) return ORACLE_ERR_NOMEM;
  matmul(T, dq, d, dZ, d, 1, WO, 1, d, dO, dq);      /* dO = dZ WO^T */
  matmul(dq, d, T, O, 1, dq, dZ, d, 1, dWO, d);      /* dWO = O^T dZ */
  matmul(T, d, dq, dQ, dq, 1, WQ, 1, dq, dX, d);     /* dX = dQ WQ^T ... */
  matmul(T, d, dkv, dK, dkv, 1, WK, 1, dkv, tmp, d);
  for (int64_t i = 0; i < T * d; ++i) dX[i] += tmp[i];
  matmul(T, d, dkv, dV, dkv, 1, WV, 1, dkv, tmp, d);
  for (int64_t i = 0; i < T * d; ++i) dX[i] += tmp[i];
  matmul(d, dq, T, X, 1, d, dQ, dq, 1, dWQ, dq);     /* dWQ = X^T dQ */
  matmul(d, dkv, T, X, 1, d, dK, dkv, 1, dWK, dkv);
  matmul(d, dkv, T, X, 1, d, dV, dkv, 1, dWV, dkv);
  free(tmp);
  return ORACLE_OK;
}

/* Per-shard form: arrays of t shard pointers; the g-sum gives Z, the f-sum dX;
 * every weight gradient is per shard.                                         */
int oracle_attn_sharded(int64_t T, int64_t d, int32_t t, const int64_t* wq_i, const int64_t* wkv_i,
                        const double* X, const double* const* WQ_i, const double* const* WK_i,
                        const double* const* WV_i, const double* const* O_i, const double* const* WO_i,
                        const double* dZ, const double* const* dQ_i, const double* const* dK_i,
                        const double* const* dV_i, double* Z, double* dX, double* const* dWO_i, double* const* dWQ_i,
                        double* const* dWK_i, double* const* dWV_i) {
  if (T < 0 || d < 1 || t < 1 || !wq_i || !wkv_i || !X || !WQ_i || !WK_i || !WV_i || !O_i || !WO_i || !dZ ||
      !dQ_i || !dK_i || !dV_i || !Z || !dX || !dWO_i || !dWQ_i || !dWK_i || !dWV_i)
    return ORACLE_ERR_ARG;
  size_t nx = (size_t)(T * d ? T * d : 1);
  double* part = (double*)malloc(nx * sizeof(double));
  if (!part) return ORACLE_ERR_NOMEM;
  for (int64_t i = 0; i < T * d; ++i) Z[i] = dX[i] = 0.0;
  for (int32_t s = 0; s < t; ++s) {
    const int64_t wq = wq_i[s], wkv = wkv_i[s];
    matmul(T, d, wq, O_i[s], wq, 1, WO_i[s], d, 1, part, d);
    for (int64_t i = 0; i < T * d; ++i) Z[i] += part[i]; /* g */
    matmul(wq, d, T, O_i[s], 1, wq, dZ, d, 1, dWO_i[s], d);
    matmul(d, wq, T, X, 1, d, dQ_i[s], wq, 1, dWQ_i[s], wq);
    matmul(d, wkv, T, X, 1, d, dK_i[s], wkv, 1, dWK_i[s], wkv);
    matmul(d, wkv, T, X, 1, d, dV_i[s], wkv, 1, dWV_i[s], wkv);
    matmul(T, d, wq, dQ_i[s], wq, 1, WQ_i[s], 1, wq, part, d);
    for (int64_t i = 0; i < T * d; ++i) dX[i] += part[i]; /* f */
    matmul(T, d, wkv, dK_i[s], wkv, 1, WK_i[s], 1, wkv, part, d);
    for (int64_t i = 0; i < T * d; ++i) dX[i] += part[i];
    matmul(T, d, wkv, dV_i[s], wkv, 1, WV_i[s], 1, wkv, part, d);
    for (int64_t i = 0; i < T * d; ++i) dX[i] += part[i];
  }
  free(part);
  return ORACLE_OK;
}

/* db2 = sum over the T tokens of dY[r, :] -- the gradient of the bias added
 * once after the g-sum (g backward is the identity).  db2 is [d].           */
int oracle_db2(int64_t T, int64_t d, const double* dY, double* db2) {
  if (T < 0 || d < 1 || !dY || !db2) return ORACLE_ERR_ARG;
  col_sums(T, d, dY, db2);
  return ORACLE_OK;
}

/* Scalar access for the closed-form pins (value of the activation, its
 * derivative, for act in {GeLU, Swish-as-SwiGLU-gate, identity, ReLU}).      */
double oracle_act_value(int act, double a) { return act == ORACLE_ACT_SWIGLU ? swish(a) : act_value(act, a); }
double oracle_act_grad(int act, double a) { return act == ORACLE_ACT_SWIGLU ? swish_grad(a) : act_grad(act, a); }

int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
