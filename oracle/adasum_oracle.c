/*
 * adasum_oracle.c -- plain, slow, single-threaded fp64 CPU oracle for the Adasum
 * gradient combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path loads, links or calls this
 * file.  Only the tests, the smoke check and the benchmark's CPU-baseline leg use it,
 * through the ctypes loader in oracle/__init__.py.  It shares no code, header, table
 * or helper with the CUDA library.
 *
 * Source: "Scaling Distributed Training with Adaptive Summation" (Maleki et al.,
 * arXiv 2006.02924), Section 3.
 *   - Pair operator (Section 3, Equations 1-2 and the average of the two emulated
 *     sequential SGD orders that defines the operator):
 *         Adasum(a, b) = (1 - a.b / (2 |a|^2)) a + (1 - a.b / (2 |b|^2)) b
 *     This is the form the derivation yields: Hessian estimated as g g^T (Appendix
 *     A.1), step 1/|g|^2 (Appendix A.2), the two processing orders averaged.
 *   - Recursive application over many workers as a binary tree (Section 3, the
 *     recursive application used in practice because it moves fewer bytes): level 0
 *     pairs (2i, 2i+1), the next level pairs the level-0 results the same way, log2(K)
 *     levels in all.
 *   - The linear recursion the same section states first: g[0,n+1] = Adasum(g[0,n],
 *     g_{n+1}), i.e. a chain folding the workers in from left to right
 *     (oracle_adasum_chain).
 *   - Per-layer application (Section 3, after Figure 1): every segment of the flat
 *     gradient is combined on its own, with its own dot products and norms.
 *   - Special cases (Section 3, discussion after the tree): orthogonal inputs sum,
 *     parallel inputs average.
 *   - Orthogonality metric (Section 3, Figure 1): |Adasum(g_1..g_n)|^2 / sum_i |g_i|^2.
 *
 * Readings where the text is silent (each is listed in the design notes):
 *   - A zero-norm operand: its 0/0 quotient is taken as 0, so its coefficient is 1 and
 *     the pair reduces to a plain sum.  The test is exact (== 0.0), with no epsilon.
 *   - bf16 storage: inputs are decoded exactly, every intermediate stays in fp64, and
 *     the final result is rounded once, to nearest with ties to even.
 *   - Sums are taken in plain sequential order.
 *   - A worker count that is not a power of two: at every level pairs (2i, 2i+1) are
 *     combined and an unpaired last vector passes to the next level unchanged.  (This
 *     equals padding with zero gradients, because Adasum(x, 0) = x.)
 *   - Fused Momentum-SGD (heavy ball): v' = mu v + A, w' = w - lr v', evaluated in fp64
 *     from the unrounded Adasum result A and rounded to fp32 at the end.
 *   - Adasum after the optimizer (Section 3, Figure 3): every worker k first takes its own
 *     heavy-ball step on its own momentum, v_k' = mu v_k + g_k (stored in fp32, its state),
 *     proposes the update -lr v_k', and the proposals are combined by Adasum and applied:
 *     w' = w + Adasum(-lr v_0', ..., -lr v_{K-1}').
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (no fast-math, no FMA contraction, so
 * x86-64 and aarch64 hosts give the same bits).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

enum {
  ORACLE_OK = 0,
  ORACLE_ERR_ARG = 1,     /* bad K, bad offsets, null pointer */
  ORACLE_ERR_NOMEM = 2
};

/* ---- bf16 storage format: 1 sign, 8 exponent, 7 stored fraction bits; the upper
 *      half of an IEEE binary32 word. ------------------------------------------- */

double oracle_bf16_decode(uint16_t h) {
  uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* Round an fp64 value straight to bf16, to nearest, ties to even, in one step (no
 * intermediate fp32 rounding).  bf16 keeps 8 significant bits; below the smallest
 * normal (2^-126) the spacing is fixed at 2^-133; results at or above 2^128 are Inf. */
uint16_t oracle_bf16_encode(double x) {
  if (isnan(x)) return (uint16_t)0x7FC0;
  uint16_t sign = signbit(x) ? (uint16_t)0x8000 : (uint16_t)0;
  double ax = fabs(x);
  if (isinf(ax)) return (uint16_t)(sign | 0x7F80);
  if (ax == 0.0) return sign;
  int e;
  frexp(ax, &e);           /* ax in [2^(e-1), 2^e) */
  int q = e - 8;           /* spacing of 8-significant-bit numbers in that binade */
  if (q < -133) q = -133;  /* subnormal bf16 spacing */
  double r = nearbyint(ldexp(ax, -q)); /* default rounding mode: nearest, ties to even */
  double y = ldexp(r, q);
  if (y >= 0x1p128) return (uint16_t)(sign | 0x7F80);
  float f = (float)y;      /* exact: y has at most 8 significant bits and fits binary32 */
  uint32_t bits;
  memcpy(&bits, &f, sizeof bits);
  return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

static double load_elem(const void *base, int dtype, int64_t i) {
  if (dtype == ORACLE_F32) return (double)((const float *)base)[i];
  return oracle_bf16_decode(((const uint16_t *)base)[i]);
}

static void store_elem(void *base, int dtype, int64_t i, double v) {
  if (dtype == ORACLE_F32)
    ((float *)base)[i] = (float)v; /* IEEE conversion, round to nearest even */
  else
    ((uint16_t *)base)[i] = oracle_bf16_encode(v);
}


/* One Adasum pair on fp64 vectors of length n, written to dst.  dst may equal a.
 * When mdst is given, it also carries the magnitude bound m = |alpha| m_a + |beta| m_b
 * that the tests use to size the fp32-arithmetic floor of the bf16 tolerance. */
static void adasum_pair_f64(double *dst, const double *a, const double *b, int64_t n,
                            double *mdst, const double *ma, const double *mb) {
  double d = 0.0, p = 0.0, q = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    d += a[j] * b[j];
    p += a[j] * a[j];
    q += b[j] * b[j];
  }
  double alpha = 1.0 - (p == 0.0 ? 0.0 : d / (2.0 * p));
  double beta = 1.0 - (q == 0.0 ? 0.0 : d / (2.0 * q));
  for (int64_t j = 0; j < n; ++j) {
    double v = alpha * a[j] + beta * b[j];
    if (mdst) mdst[j] = fabs(alpha) * ma[j] + fabs(beta) * mb[j];
    dst[j] = v;
  }
}

/* Shared by the tree and the chain: validates arguments and, per segment, loads the K
 * inputs into level[] (and their magnitudes), calls `combine` to reduce them into
 * level[0], then writes the outputs. */
typedef void (*combine_fn)(double *level, double *mlevel, int K, int64_t n);

static void tree_levels(double *level, double *mlevel, int K, int64_t n);
static void chain_levels(double *level, double *mlevel, int K, int64_t n);

static int run_segments(const void *const *grads, int K, const int64_t *offs, int L, int dtype,
                        void *out, double *out64, double *mag, double *ortho, combine_fn combine) {
  if (!grads || !offs || K < 1 || L < 0) return ORACLE_ERR_ARG;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return ORACLE_ERR_ARG;
  if (offs[0] < 0) return ORACLE_ERR_ARG;
  for (int s = 0; s < L; ++s)
    if (offs[s + 1] < offs[s]) return ORACLE_ERR_ARG;
  for (int k = 0; k < K; ++k)
    if (!grads[k] && offs[L] > 0) return ORACLE_ERR_ARG;

  for (int s = 0; s < L; ++s) {
    const int64_t base = offs[s];
    const int64_t n = offs[s + 1] - offs[s];
    if (n == 0) {
      if (ortho) ortho[s] = NAN;
      continue;
    }
    /* level[k] holds the k-th vector of the current tree level (fp64). */
    double *level = (double *)malloc((size_t)K * (size_t)n * sizeof(double));
    double *mlevel = mag ? (double *)malloc((size_t)K * (size_t)n * sizeof(double)) : NULL;
    if (!level || (mag && !mlevel)) {
      free(level);
      free(mlevel);
      return ORACLE_ERR_NOMEM;
    }
    double sumsq = 0.0;
    for (int k = 0; k < K; ++k) {
      double *v = level + (size_t)k * (size_t)n;
      for (int64_t j = 0; j < n; ++j) {
        v[j] = load_elem(grads[k], dtype, base + j);
        sumsq += v[j] * v[j];
        if (mlevel) mlevel[(size_t)k * (size_t)n + j] = fabs(v[j]);
      }
    }
    combine(level, mlevel, K, n);
    double rsq = 0.0;
    for (int64_t j = 0; j < n; ++j) {
      rsq += level[j] * level[j];
      if (out) store_elem(out, dtype, base + j, level[j]);
      if (out64) out64[base + j] = level[j];
      if (mag) mag[base + j] = mlevel[j];
    }
    if (ortho) ortho[s] = (sumsq == 0.0) ? NAN : rsq / sumsq;
    free(level);
    free(mlevel);
  }
  return ORACLE_OK;
}

/* Binary tree: the pair (2i, 2i+1) of one level becomes vector i of the next; with an odd
 * count the last vector moves on unchanged.  Writing result i into slot i is safe: slots
 * 2i and 2i+1 are read first, and slots below 2i were already consumed by earlier pairs
 * of the same level (the carried vector's new slot width/2 likewise). */
static void tree_levels(double *level, double *mlevel, int K, int64_t n) {
  for (int width = K; width > 1; width = (width + 1) / 2) {
    for (int i = 0; i < width / 2; ++i) {
        double *dst = level + (size_t)i * (size_t)n;
        const double *a = level + (size_t)(2 * i) * (size_t)n;
        const double *b = level + (size_t)(2 * i + 1) * (size_t)n;
        double *mdst = mlevel ? mlevel + (size_t)i * (size_t)n : NULL;
        const double *ma = mlevel ? mlevel + (size_t)(2 * i) * (size_t)n : NULL;
        const double *mb = mlevel ? mlevel + (size_t)(2 * i + 1) * (size_t)n : NULL;
        adasum_pair_f64(dst, a, b, n, mdst, ma, mb);
    }
    if (width % 2 == 1) {
      const size_t from = (size_t)(width - 1) * (size_t)n, to = (size_t)(width / 2) * (size_t)n;
      memmove(level + to, level + from, (size_t)n * sizeof(double));
      if (mlevel) memmove(mlevel + to, mlevel + from, (size_t)n * sizeof(double));
    }
  }
}

/* Linear chain: g[0,k] = Adasum(g[0,k-1], g_k), accumulated in slot 0. */
static void chain_levels(double *level, double *mlevel, int K, int64_t n) {
  for (int k = 1; k < K; ++k) {
    const double *b = level + (size_t)k * (size_t)n;
    adasum_pair_f64(level, level, b, n, mlevel, mlevel, mlevel ? mlevel + (size_t)k * (size_t)n : NULL);
  }
}

/* Adasum over K workers (any K >= 1) as a binary tree, for every segment
 * [offs[s], offs[s+1]).
 *   grads  : K host pointers, each to offs[L] elements of `dtype`.
 *   out    : optional, offs[L] elements of `dtype`, the rounded result.
 *   out64  : optional, offs[L] doubles, the unrounded fp64 result.
 *   mag    : optional, offs[L] doubles, the magnitude bound m per element.
 *   ortho  : optional, L doubles, |A|^2 / sum_k |g_k|^2 per segment (NaN for 0/0).
 * Returns ORACLE_OK, ORACLE_ERR_ARG or ORACLE_ERR_NOMEM. */
int oracle_adasum_reduce(const void *const *grads, int K, const int64_t *offs, int L,
                         int dtype, void *out, double *out64, double *mag, double *ortho) {
  return run_segments(grads, K, offs, L, dtype, out, out64, mag, ortho, tree_levels);
}

/* The same outputs for the linear chain g[0,n+1] = Adasum(g[0,n], g_{n+1}). */
int oracle_adasum_chain(const void *const *grads, int K, const int64_t *offs, int L,
                        int dtype, void *out, double *out64, double *mag, double *ortho) {
  return run_segments(grads, K, offs, L, dtype, out, out64, mag, ortho, chain_levels);
}

/* The two-worker case: one segment of n elements. */
int oracle_adasum_pair(const void *a, const void *b, int64_t n, int dtype, void *out,
                       double *out64) {
  if (n < 0) return ORACLE_ERR_ARG;
  const void *g[2] = {a, b};
  int64_t offs[2] = {0, n};
  return oracle_adasum_reduce(g, 2, offs, 1, dtype, out, out64, NULL, NULL);
}

/* Adasum after the optimizer: per-worker heavy-ball steps, then the workers' proposed
 * updates combined by the Adasum tree and applied.
 *   grads : K host pointers to N elements of `dtype`;  v : K host fp32 arrays (updated);
 *   w     : fp32 weights (updated).
 * v_k' = fp32(mu v_k + g_k) (evaluated in fp64, rounded once: the stored state);
 * A = Adasum over the updates -lr v_k' (fp64, from the stored fp32 v_k');  w' = fp32(w + A). */
int oracle_local_momentum_adasum(const void *const *grads, int K, const int64_t *offs, int L,
                                 int dtype, float *const *v, float *w, double lr, double mu) {
  if (!grads || !v || !w || K < 1 || L < 0 || !offs) return ORACLE_ERR_ARG;
  const int64_t N = offs[L];
  for (int k = 0; k < K; ++k)
    for (int64_t j = 0; j < N; ++j)
      v[k][j] = (float)(mu * (double)v[k][j] + load_elem(grads[k], dtype, j));
  /* the proposed updates -lr v_k', exactly as fp64 values, stored as fp64 arrays */
  double **upd = (double **)malloc((size_t)K * sizeof(double *));
  if (!upd) return ORACLE_ERR_NOMEM;
  for (int k = 0; k < K; ++k) upd[k] = NULL;
  int rc = ORACLE_OK;
  for (int k = 0; k < K && rc == ORACLE_OK; ++k) {
    upd[k] = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    if (!upd[k]) rc = ORACLE_ERR_NOMEM;
    else
      for (int64_t j = 0; j < N; ++j) upd[k][j] = -lr * (double)v[k][j];
  }
  if (rc == ORACLE_OK) {
    double *A = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    if (!A) {
      rc = ORACLE_ERR_NOMEM;
    } else {
      /* per segment, the tree over the fp64 updates */
      for (int s = 0; s < L && rc == ORACLE_OK; ++s) {
        const int64_t base = offs[s], n = offs[s + 1] - offs[s];
        if (n == 0) continue;
        double *level = (double *)malloc((size_t)K * (size_t)n * sizeof(double));
        if (!level) {
          rc = ORACLE_ERR_NOMEM;
          break;
        }
        for (int k = 0; k < K; ++k) memcpy(level + (size_t)k * (size_t)n, upd[k] + base, (size_t)n * sizeof(double));
        tree_levels(level, NULL, K, n);
        memcpy(A + base, level, (size_t)n * sizeof(double));
        free(level);
      }
      if (rc == ORACLE_OK)
        for (int64_t j = 0; j < N; ++j) w[j] = (float)((double)w[j] + A[j]);
      free(A);
    }
  }
  for (int k = 0; k < K; ++k) free(upd[k]);
  free(upd);
  return rc;
}

/* Heavy-ball Momentum-SGD step applied to the Adasum result A (fp64, unrounded):
 *   v' = mu * v + A,   w' = w - lr * v'
 * evaluated in fp64 and rounded to fp32 once at the end.  lr and mu are passed as the
 * doubles of the fp32 values the GPU receives. */
int oracle_momentum_sgd(const double *A, int64_t n, const float *w, const float *v,
                        double lr, double mu, float *w_out, float *v_out) {
  if (n < 0 || (n > 0 && (!A || !w || !v || !w_out || !v_out))) return ORACLE_ERR_ARG;
  for (int64_t j = 0; j < n; ++j) {
    double vn = mu * (double)v[j] + A[j];
    double wn = (double)w[j] - lr * vn;
    v_out[j] = (float)vn;
    w_out[j] = (float)wn;
  }
  return ORACLE_OK;
}
