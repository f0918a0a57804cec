/*
 * tpffn_oracle.c -- plain, slow, float64 CPU oracle for the Megatron
 * tensor-parallel feed-forward sublayer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes (all in float64, row-major, weights stored [out][in]):
 *
 *   Dense form -- "7.9 Tensor and pipeline parallelism (TP, PP)", §2.1
 *   "The FFN, sharded", first display:  y = W2 sigma(W1 x), applied to each
 *   token row x of an [N, d] activation (so y_n = W2 sigma(W1 x_n)).
 *     GELU : z = W1 x + b1,  h = gelu_tanh(z)
 *     SwiGLU ("S17 Tensor & Pipeline Parallelism", listing "the megatron
 *     pattern"):  a = W1 x, g = W3 x, h = silu(a) * g
 *     NONE : h = x (a row-parallel linear alone, e.g. the attention output
 *     projection of §2.2 "Attention, sharded")
 *     IDENTITY (oracle-only, for the linear special-case pin): h = W1 x + b1
 *   then y = W2 h + b2.
 *
 *   Sharded form -- same §2.1: rows [t*s, (t+1)*s) of W1 (and W3, b1) form
 *   shard t ("column-shard W1 along its output dimension"), columns
 *   [t*s, (t+1)*s) of W2 form shard t ("row-shard W2 along its input
 *   dimension"); h^(t) = sigma(W1^(t) x), y^(t) = W2^(t) h^(t), and the
 *   g-operator sums y = sum_t y^(t), taken here in the order t = 0..T_p-1.
 *   b2 is added once after the sum (the page says only that biases "shard
 *   analogously"; adding b2 per shard would add it T_p times).
 *
 *   Backward -- not written out on the pages; §2.1 fixes only where the sums
 *   go (g: all-reduce forward / identity backward, f: identity forward /
 *   all-reduce backward).  The oracle applies the ordinary chain rule:
 *     dh = W2^T dy,  dz = dh * sigma'(z)  (SwiGLU: da = dh*g*silu'(a),
 *     dg = dh*silu(a)),  dW2 = dy h^T, dW1 = dz x^T, dW3 = dg x^T,
 *     db1 = sum_n dz, db2 = sum_n dy,  dx = sum_t (W1^(t)T dz^(t) [+ W3^(t)T dg^(t)])
 *   with the dx shard-sum (the f operator) again in the order t = 0..T_p-1.
 *
 * Precision modes.  round_bf16 == 0: every intermediate is float64.
 * round_bf16 == 1: the activations that the configuration stores in bf16
 * ("bf16 weights/activations, fp32 accumulate") are rounded to bf16
 * (round-to-nearest-even) at the points where they are stored: z (saved),
 * h, a and g (saved), dz / da / dg.  Sums stay in float64.
 *
 * Activation functions: gelu_tanh is the tanh approximation of Hendrycks &
 * Gimpel (2016), 0.5 u (1 + tanh(sqrt(2/pi) (u + 0.044715 u^3))); silu(u) =
 * u / (1 + exp(-u)).  libm tanh/exp in double precision.
 *
 * Parallelism: OpenMP over independent outputs only (token rows, hidden
 * units).  Every sum runs in one thread, in index order, so results do not
 * depend on the thread count.
 */
#define _DEFAULT_SOURCE 1
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_ACT_NONE 0
#define ORC_ACT_GELU_TANH 1
#define ORC_ACT_SWIGLU 2
#define ORC_ACT_IDENTITY 3

/* ---------------------------------------------------------------- scalars */

/* gelu_tanh(u) = 0.5 u (1 + tanh(c (u + 0.044715 u^3))), c = sqrt(2/pi). */
double orc_gelu_tanh(double u) {
  const double c = sqrt(2.0 / M_PI);
  return 0.5 * u * (1.0 + tanh(c * (u + 0.044715 * u * u * u)));
}

/* d/du of the expression above (product rule, tanh' = 1 - tanh^2). */
double orc_gelu_tanh_grad(double u) {
  const double c = sqrt(2.0 / M_PI);
  double inner = c * (u + 0.044715 * u * u * u);
  double th = tanh(inner);
  double dinner = c * (1.0 + 3.0 * 0.044715 * u * u);
  return 0.5 * (1.0 + th) + 0.5 * u * (1.0 - th * th) * dinner;
}

double orc_sigmoid(double u) { return 1.0 / (1.0 + exp(-u)); }

double orc_silu(double u) { return u * orc_sigmoid(u); }

/* silu'(u) = sg (1 + u (1 - sg)),  sg = sigmoid(u). */
double orc_silu_grad(double u) {
  double sg = orc_sigmoid(u);
  return sg * (1.0 + u * (1.0 - sg));
}

/* Round a double to the nearest bfloat16 value (8 significand bits incl. the
 * implicit one, exponent range of float32), ties to even.  Written from the
 * format's definition: find the two neighbouring bf16 values and pick. */
double orc_round_bf16(double v) {
  if (v == 0.0 || isnan(v) || isinf(v)) return v;
  double a = fabs(v);
  int e;
  frexp(a, &e);              /* a = m * 2^e, m in [0.5, 1) */
  int unit_exp = e - 8;      /* spacing of 8-bit significands at this binade */
  if (e - 1 < -126) unit_exp = -126 - 7;   /* subnormal bf16 spacing */
  double ulp = ldexp(1.0, unit_exp);
  double q = a / ulp;        /* exact: power-of-two scaling */
  double lo = floor(q);
  double rem = q - lo;
  double r;
  if (rem > 0.5) r = lo + 1.0;
  else if (rem < 0.5) r = lo;
  else r = (fmod(lo, 2.0) == 0.0) ? lo : lo + 1.0;
  double out = r * ulp;
  if (out > 3.3895313892515355e38) out = INFINITY;   /* beyond bf16 max */
  return v < 0 ? -out : out;
}

static inline double RND(int on, double v) { return on ? orc_round_bf16(v) : v; }

static double act_fwd(int act, double u) {
  switch (act) {
    case ORC_ACT_GELU_TANH: return orc_gelu_tanh(u);
    case ORC_ACT_IDENTITY: return u;
    default: return u;
  }
}
static double act_grad(int act, double u) {
  switch (act) {
    case ORC_ACT_GELU_TANH: return orc_gelu_tanh_grad(u);
    default: return 1.0;
  }
}

/* ------------------------------------------------------------ the problem */

typedef struct {
  int64_t N, d, d_ff;
  int T_p, act, round_bf16;
  const double* x;   /* [N][d]   (act NONE: [N][d_ff], the concatenated heads) */
  const double* W1;  /* [d_ff][d] (unused for NONE) */
  const double* W3;  /* [d_ff][d] (SwiGLU only) */
  const double* b1;  /* [d_ff] or NULL */
  const double* W2;  /* [d][d_ff] */
  const double* b2;  /* [d] or NULL */
} orc_ffn;

/* Hidden pre-activations of token n, hidden unit j.  Dot products in index
 * order over the input width. */
static double dot_row(const double* a, const double* b, int64_t len) {
  double acc = 0.0;
  for (int64_t k = 0; k < len; ++k) acc += a[k] * b[k];
  return acc;
}

/* Forward quantities of one (token n, hidden j) pair.
 * out: h (the stored hidden activation), z_saved / a_saved / g_saved (the
 * saved values), and optionally the values before bf16 rounding:
 * pre[0] = sigma(z) (or silu(a) g), pre[1] = z (or a), pre[2] = g. */
static void hidden_unit_ex(const orc_ffn* P, int64_t n, int64_t j, double* h,
                           double* z_saved, double* a_saved, double* g_saved, double* pre) {
  const int R = P->round_bf16;
  if (P->act == ORC_ACT_NONE) {
    *h = P->x[n * P->d_ff + j];
    if (pre) { pre[0] = *h; pre[1] = 0.0; pre[2] = 0.0; }
    return;
  }
  const double* xn = P->x + n * P->d;
  if (P->act == ORC_ACT_SWIGLU) {
    double a = dot_row(xn, P->W1 + j * P->d, P->d);
    double g = dot_row(xn, P->W3 + j * P->d, P->d);
    double hv = orc_silu(a) * g;
    *h = RND(R, hv);
    if (a_saved) *a_saved = RND(R, a);
    if (g_saved) *g_saved = RND(R, g);
    if (pre) { pre[0] = hv; pre[1] = a; pre[2] = g; }
    return;
  }
  double z = dot_row(xn, P->W1 + j * P->d, P->d);
  if (P->b1) z += P->b1[j];
  double hv = act_fwd(P->act, z);
  *h = RND(R, hv);
  if (z_saved) *z_saved = RND(R, z);
  if (pre) { pre[0] = hv; pre[1] = z; pre[2] = 0.0; }
}

static void hidden_unit(const orc_ffn* P, int64_t n, int64_t j, double* h,
                        double* z_saved, double* a_saved, double* g_saved) {
  hidden_unit_ex(P, n, j, h, z_saved, a_saved, g_saved, NULL);
}

static int64_t shard_width(const orc_ffn* P) { return P->d_ff / P->T_p; }

/* ------------------------------------------------------------- forward */

/* Dense form over a subset of token rows (rows == NULL: all N rows).
 * y: [n_rows][d].  h (optional): [n_rows][d_ff]. */
void orc_ffn_forward_dense(const orc_ffn* P, int64_t n_rows, const int64_t* rows,
                           double* y, double* h) {
  const int64_t d = P->d, dff = P->d_ff;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n_rows; ++r) {
    int64_t n = rows ? rows[r] : r;
    double* hrow = (double*)malloc(sizeof(double) * dff);
    for (int64_t j = 0; j < dff; ++j) hidden_unit(P, n, j, &hrow[j], NULL, NULL, NULL);
    for (int64_t c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int64_t j = 0; j < dff; ++j) acc += P->W2[c * dff + j] * hrow[j];
      if (P->b2) acc += P->b2[c];
      y[r * d + c] = acc;
    }
    if (h) memcpy(h + r * dff, hrow, sizeof(double) * dff);
    free(hrow);
  }
}

/* Explicitly sharded form over a subset of token rows.
 * partials: [T_p][n_rows][d] (optional), y: [n_rows][d],
 * h: [n_rows][d_ff] (optional), z_saved: [n_rows][d_ff] (optional, GELU),
 * ag_saved: [n_rows][2][d_ff] (optional, SwiGLU: a then g). */
void orc_ffn_forward_sharded(const orc_ffn* P, int64_t n_rows, const int64_t* rows,
                             double* partials, double* y, double* h,
                             double* z_saved, double* ag_saved) {
  const int64_t d = P->d, dff = P->d_ff, s = shard_width(P);
  const int T = P->T_p;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n_rows; ++r) {
    int64_t n = rows ? rows[r] : r;
    double* part = (double*)malloc(sizeof(double) * (size_t)T * d);
    double* ht = (double*)malloc(sizeof(double) * s);
    for (int t = 0; t < T; ++t) {
      /* shard t: hidden units [t*s, (t+1)*s) -- no data from other shards */
      for (int64_t jj = 0; jj < s; ++jj) {
        int64_t j = t * s + jj;
        double zs = 0, as = 0, gs = 0;
        hidden_unit(P, n, j, &ht[jj], &zs, &as, &gs);
        if (h) h[r * dff + j] = ht[jj];
        if (z_saved) z_saved[r * dff + j] = zs;
        if (ag_saved) { ag_saved[(r * 2 + 0) * dff + j] = as; ag_saved[(r * 2 + 1) * dff + j] = gs; }
      }
      /* y^(t) = W2^(t) h^(t): columns [t*s, (t+1)*s) of W2 */
      for (int64_t c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int64_t jj = 0; jj < s; ++jj) acc += P->W2[c * dff + t * s + jj] * ht[jj];
        part[(int64_t)t * d + c] = acc;
      }
    }
    /* g operator: y = sum_t y^(t), t ascending, then b2 once */
    for (int64_t c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int t = 0; t < T; ++t) acc += part[(int64_t)t * d + c];
      if (P->b2) acc += P->b2[c];
      y[r * d + c] = acc;
      if (partials)
        for (int t = 0; t < T; ++t) partials[((int64_t)t * n_rows + r) * d + c] = part[(int64_t)t * d + c];
    }
    free(ht);
    free(part);
  }
}

/* Counter-example the pages warn about ("the bad option" of splitting the
 * first matrix by rows, i.e. along the input dimension): each shard applies
 * the activation to its partial product, and the results are summed:
 * h_bad = sum_t sigma(W1[:, t-th input slice] x[t-th slice] + b1/T_p).
 * Used only to show that it does NOT reproduce the dense output. */
void orc_ffn_forward_rowsplit_bad(const orc_ffn* P, double* y) {
  const int64_t d = P->d, dff = P->d_ff;
  const int T = P->T_p;
  const int64_t kw = d / T;
  for (int64_t n = 0; n < P->N; ++n) {
    const double* xn = P->x + n * d;
    for (int64_t c = 0; c < d; ++c) y[n * d + c] = P->b2 ? P->b2[c] : 0.0;
    for (int64_t j = 0; j < dff; ++j) {
      double hj = 0.0;
      for (int t = 0; t < T; ++t) {
        double zt = 0.0;
        for (int64_t k = t * kw; k < (t + 1) * kw; ++k) zt += P->W1[j * d + k] * xn[k];
        if (P->b1) zt += P->b1[j] / T;
        hj += act_fwd(P->act, zt);
      }
      for (int64_t c = 0; c < d; ++c) y[n * d + c] += P->W2[c * dff + j] * hj;
    }
  }
}

/* ------------------------------------------------------------ backward */

/* Backward quantities of one (token n, hidden j): dh (exact), then the
 * stored gradient(s): dz (GELU / IDENTITY), or da, dg (SwiGLU), or dc = dh
 * (NONE).  h is also returned (for dW2).  pre (optional): the values of dz
 * (da) and dg before bf16 rounding. */
static void hidden_unit_bwd_ex(const orc_ffn* P, const double* dy, int64_t n, int64_t j,
                               double* h, double* dz, double* dg, double* pre) {
  const int R = P->round_bf16;
  const int64_t d = P->d, dff = P->d_ff;
  double dh = 0.0;
  for (int64_t c = 0; c < d; ++c) dh += dy[n * d + c] * P->W2[c * dff + j];
  double zs = 0, as = 0, gs = 0;
  hidden_unit(P, n, j, h, &zs, &as, &gs);
  double v0 = dh, v1 = 0.0;
  if (P->act == ORC_ACT_SWIGLU) {
    /* as, gs are the saved (possibly bf16) a and g */
    v0 = dh * gs * orc_silu_grad(as);
    v1 = dh * orc_silu(as);
  } else if (P->act != ORC_ACT_NONE) {
    v0 = dh * act_grad(P->act, zs);
  }
  if (pre) { pre[0] = v0; pre[1] = v1; }
  if (P->act == ORC_ACT_NONE) { *dz = dh; if (dg) *dg = 0.0; return; }
  *dz = RND(R, v0);
  if (dg) *dg = RND(R, v1);
}

static void hidden_unit_bwd(const orc_ffn* P, const double* dy, int64_t n, int64_t j,
                            double* h, double* dz, double* dg) {
  hidden_unit_bwd_ex(P, dy, n, j, h, dz, dg, NULL);
}

/* Stored hidden quantities at selected (token row, hidden unit) positions,
 * with their values before bf16 rounding and the magnitudes of the dot
 * products that produce them.  rows == NULL: all tokens; cols == NULL: all
 * hidden units.  out holds 9 planes of [n_rows][n_cols]:
 *   0 h_pre  : sigma(z) or silu(a) g            1 z_pre : z (GELU) or a
 *   2 g_pre  : g (SwiGLU)                       3 dh    : W2^T dy (exact)
 *   4 dz_pre : dh sigma'(z_saved), or da        5 dg_pre: dg (SwiGLU)
 *   6 nz     : sqrt(sum_k (x_k W1_jk)^2)        7 ng    : same for W3
 *   8 ndh    : sqrt(sum_c (dy_c W2_cj)^2)
 * The tests use them to find rounding decisions that lie within the GPU's
 * accumulation error of a bf16 midpoint.  dy may be NULL (planes 3-5, 8 = 0). */
void orc_ffn_hidden_dump(const orc_ffn* P, const double* dy, int64_t n_rows, const int64_t* rows,
                         int64_t n_cols, const int64_t* cols, double* out) {
  const int64_t d = P->d, dff = P->d_ff;
  const int64_t plane = n_rows * n_cols;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n_rows; ++r) {
    int64_t n = rows ? rows[r] : r;
    for (int64_t q = 0; q < n_cols; ++q) {
      int64_t j = cols ? cols[q] : q;
      double h, zs, as, gs, pre[3], bpre[2] = {0.0, 0.0}, dz, dg;
      hidden_unit_ex(P, n, j, &h, &zs, &as, &gs, pre);
      double dh = 0.0, ndh = 0.0, nz = 0.0, ng = 0.0;
      if (dy) {
        hidden_unit_bwd_ex(P, dy, n, j, &h, &dz, &dg, bpre);
        for (int64_t c = 0; c < d; ++c) {
          double t = dy[n * d + c] * P->W2[c * dff + j];
          dh += t;
          ndh += t * t;
        }
      }
      if (P->act != ORC_ACT_NONE) {
        const double* xn = P->x + n * d;
        for (int64_t k = 0; k < d; ++k) {
          double t = xn[k] * P->W1[j * d + k];
          nz += t * t;
          if (P->act == ORC_ACT_SWIGLU) {
            double u = xn[k] * P->W3[j * d + k];
            ng += u * u;
          }
        }
      }
      const int64_t o = r * n_cols + q;
      out[0 * plane + o] = pre[0];
      out[1 * plane + o] = pre[1];
      out[2 * plane + o] = pre[2];
      out[3 * plane + o] = dh;
      out[4 * plane + o] = bpre[0];
      out[5 * plane + o] = bpre[1];
      out[6 * plane + o] = sqrt(nz);
      out[7 * plane + o] = sqrt(ng);
      out[8 * plane + o] = sqrt(ndh);
    }
  }
}

/* dx for a subset of token rows, with the per-shard partials.
 * dx: [n_rows][d_in]  with d_in = d (d_ff for NONE, where shard t owns the
 * input columns [t*s, (t+1)*s) and no sum is taken).
 * dx_partials: [T_p][n_rows][d] (optional; not for NONE). */
void orc_ffn_backward_rows(const orc_ffn* P, const double* dy, int64_t n_rows,
                           const int64_t* rows, double* dx_partials, double* dx) {
  const int64_t d = P->d, dff = P->d_ff, s = shard_width(P);
  const int T = P->T_p;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n_rows; ++r) {
    int64_t n = rows ? rows[r] : r;
    double* dz = (double*)malloc(sizeof(double) * dff);
    double* dg = (double*)malloc(sizeof(double) * dff);
    for (int64_t j = 0; j < dff; ++j) {
      double hj;
      hidden_unit_bwd(P, dy, n, j, &hj, &dz[j], &dg[j]);
    }
    if (P->act == ORC_ACT_NONE) {
      for (int64_t j = 0; j < dff; ++j) dx[r * dff + j] = dz[j];
    } else {
      double* part = (double*)malloc(sizeof(double) * (size_t)T * d);
      for (int t = 0; t < T; ++t)
        for (int64_t k = 0; k < d; ++k) {
          double acc = 0.0;
          for (int64_t jj = 0; jj < s; ++jj) {
            int64_t j = t * s + jj;
            acc += dz[j] * P->W1[j * d + k];
            if (P->act == ORC_ACT_SWIGLU) acc += dg[j] * P->W3[j * d + k];
          }
          part[(int64_t)t * d + k] = acc;
        }
      /* f operator in backward: dx = sum_t dx^(t), t ascending */
      for (int64_t k = 0; k < d; ++k) {
        double acc = 0.0;
        for (int t = 0; t < T; ++t) acc += part[(int64_t)t * d + k];
        dx[r * d + k] = acc;
        if (dx_partials)
          for (int t = 0; t < T; ++t) dx_partials[((int64_t)t * n_rows + r) * d + k] = part[(int64_t)t * d + k];
      }
      free(part);
    }
    free(dg);
    free(dz);
  }
}

/* Dense-form dx (no shards): dx = W1^T dz (+ W3^T dg) summed over all hidden
 * units in index order.  Used for the shard-sum invariant of the backward. */
void orc_ffn_backward_dense_dx(const orc_ffn* P, const double* dy, double* dx) {
  const int64_t d = P->d, dff = P->d_ff;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t n = 0; n < P->N; ++n) {
    double* dz = (double*)malloc(sizeof(double) * dff);
    double* dg = (double*)malloc(sizeof(double) * dff);
    for (int64_t j = 0; j < dff; ++j) { double hj; hidden_unit_bwd(P, dy, n, j, &hj, &dz[j], &dg[j]); }
    for (int64_t k = 0; k < d; ++k) {
      double acc = 0.0;
      for (int64_t j = 0; j < dff; ++j) {
        acc += dz[j] * P->W1[j * d + k];
        if (P->act == ORC_ACT_SWIGLU) acc += dg[j] * P->W3[j * d + k];
      }
      dx[n * d + k] = acc;
    }
    free(dg);
    free(dz);
  }
}

/* Weight and bias gradients at selected entries.  Each shard owns its own
 * weights, so there is no cross-shard sum here.
 *   js [n_j]: hidden units;  ks [n_k]: input features (d; unused for NONE);
 *   cs [n_c]: output features.
 *   dW1 [n_j][n_k] = sum_n dz[n][j] x[n][k]      (GELU/IDENTITY/SwiGLU's da)
 *   dW3 [n_j][n_k] = sum_n dg[n][j] x[n][k]      (SwiGLU)
 *   dW2 [n_c][n_j] = sum_n dy[n][c] h[n][j]
 *   db1 [n_j]      = sum_n dz[n][j]
 *   db2 [n_c]      = sum_n dy[n][c]
 * Any output pointer may be NULL. */
void orc_ffn_wgrad_entries(const orc_ffn* P, const double* dy,
                           int64_t n_j, const int64_t* js, int64_t n_k, const int64_t* ks,
                           int64_t n_c, const int64_t* cs,
                           double* dW1, double* dW3, double* dW2, double* db1, double* db2) {
  const int64_t N = P->N, d = P->d;
  const int64_t d_in = (P->act == ORC_ACT_NONE) ? P->d_ff : P->d;
  (void)d_in;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t a = 0; a < n_j; ++a) {
    int64_t j = js[a];
    double* hcol = (double*)malloc(sizeof(double) * N);
    double* dzcol = (double*)malloc(sizeof(double) * N);
    double* dgcol = (double*)malloc(sizeof(double) * N);
    for (int64_t n = 0; n < N; ++n) hidden_unit_bwd(P, dy, n, j, &hcol[n], &dzcol[n], &dgcol[n]);
    if (P->act != ORC_ACT_NONE) {
      for (int64_t b = 0; b < n_k; ++b) {
        int64_t k = ks[b];
        double acc1 = 0.0, acc3 = 0.0;
        for (int64_t n = 0; n < N; ++n) {
          acc1 += dzcol[n] * P->x[n * d + k];
          acc3 += dgcol[n] * P->x[n * d + k];
        }
        if (dW1) dW1[a * n_k + b] = acc1;
        if (dW3) dW3[a * n_k + b] = acc3;
      }
    }
    for (int64_t b = 0; b < n_c; ++b) {
      int64_t c = cs[b];
      double acc = 0.0;
      for (int64_t n = 0; n < N; ++n) acc += dy[n * d + c] * hcol[n];
      if (dW2) dW2[b * n_j + a] = acc;
    }
    if (db1) {
      double acc = 0.0;
      for (int64_t n = 0; n < N; ++n) acc += dzcol[n];
      db1[a] = acc;
    }
    free(dgcol);
    free(dzcol);
    free(hcol);
  }
  if (db2) {
    for (int64_t b = 0; b < n_c; ++b) {
      double acc = 0.0;
      for (int64_t n = 0; n < N; ++n) acc += dy[n * d + cs[b]];
      db2[b] = acc;
    }
  }
}

/* Number of OpenMP threads the oracle will use (for reporting). */
int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ================================================================ attention
 *
 * Head-sharded self-attention sublayer -- "7.9 Tensor and pipeline
 * parallelism (TP, PP)", §2.2 "Attention, sharded": shard t owns the query
 * heads [t*H/T_p, (t+1)*H/T_p) and the key/value heads [t*Hkv/T_p, ...) (the
 * divisibility rule of "S17 Tensor & Pipeline Parallelism", "Attention shards
 * by head, and GQA caps the degree"); it computes Q, K, V for its heads, the
 * scaled dot-product attention of each head (query head h reads key/value
 * head h / (H/Hkv)), and the row-sharded output projection
 * y^(t) = c^(t) W_O^(t)T of its heads' outputs c^(t); y = sum_t y^(t) in the
 * order t = 0..T_p-1.  Per head: s_ij = (q_i . k_j) / sqrt(hd) (j <= i when
 * causal), p_i = softmax_j(s_i), o_i = sum_j p_ij v_j.
 *
 * Layouts (row-major, tokens of sequence b are rows b*S .. b*S+S-1):
 *   q, o, dq, dO [B*S][H*hd]     k, v, dk, dv [B*S][Hkv*hd]
 *   weights [out][in]: Wq [H*hd][d], Wk, Wv [Hkv*hd][d], Wo [d][H*hd].
 * round_bf16: q, k, v and the head outputs o are rounded to bf16 where the
 * sublayer stores them, and so are dO, dq, dk, dv in the backward; the
 * probabilities p and the score gradients dS are transient (never stored)
 * and stay exact, and the key/value gradients of a GQA group are summed over
 * its query heads before their one rounding. */

typedef struct {
  int64_t B, S, H, Hkv, hd;
  int causal, round_bf16;
} orc_attn_core;

/* Softmax probabilities of query i (global row r = b*S + i) of head h;
 * p[0..S-1], zero where masked.  Returns the log-sum-exp of the scaled
 * scores. */
static double attn_probs(const orc_attn_core* C, const double* q, const double* k, int64_t b, int64_t h,
                         int64_t i, double* p) {
  const int64_t S = C->S, hd = C->hd, nq = C->H * hd, nk = C->Hkv * hd;
  const int64_t hk = h / (C->H / C->Hkv);
  const double scale = 1.0 / sqrt((double)hd);
  const int64_t jmax = C->causal ? i : S - 1;
  const double* qi = q + (b * S + i) * nq + h * hd;
  double m = -INFINITY;
  for (int64_t j = 0; j <= jmax; ++j) {
    p[j] = dot_row(qi, k + (b * S + j) * nk + hk * hd, hd) * scale;
    if (p[j] > m) m = p[j];
  }
  double sum = 0.0;
  for (int64_t j = 0; j <= jmax; ++j) {
    p[j] = exp(p[j] - m);
    sum += p[j];
  }
  for (int64_t j = 0; j < S; ++j) p[j] = (j <= jmax) ? p[j] / sum : 0.0;
  return m + log(sum);
}

/* Attention core forward: o = softmax(q k^T / sqrt(hd)) v per head;
 * lse [B][H][S] (may be NULL) receives the log-sum-exp of each row. */
void orc_attn_core_fwd(const orc_attn_core* C, const double* q, const double* k, const double* v, double* o,
                       double* lse) {
  const int64_t B = C->B, S = C->S, H = C->H, hd = C->hd, nq = H * hd, nk = C->Hkv * hd;
  const int64_t G = H / C->Hkv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bhi = 0; bhi < B * H * S; ++bhi) {
    const int64_t b = bhi / (H * S), h = (bhi / S) % H, i = bhi % S;
    double* p = (double*)malloc(sizeof(double) * S);
    const double l = attn_probs(C, q, k, b, h, i, p);
    if (lse) lse[(b * H + h) * S + i] = l;
    for (int64_t jd = 0; jd < hd; ++jd) {
      double acc = 0.0;
      for (int64_t j = 0; j < S; ++j) acc += p[j] * v[(b * S + j) * nk + (h / G) * hd + jd];
      o[(b * S + i) * nq + h * hd + jd] = RND(C->round_bf16, acc);
    }
    free(p);
  }
}

/* Attention core backward: given dO, dq = dS k, dk = dS^T q, dv = P^T dO
 * with dS_ij = p_ij (dO_i . v_j - sum_l p_il dO_i . v_l) / sqrt(hd). */
void orc_attn_core_bwd(const orc_attn_core* C, const double* q, const double* k, const double* v,
                       const double* dO, double* dq, double* dk, double* dv) {
  const int R = C->round_bf16;
  const int64_t B = C->B, S = C->S, H = C->H, Hkv = C->Hkv, hd = C->hd, nq = H * hd, nk = Hkv * hd;
  const int64_t G = H / Hkv;
  const double scale = 1.0 / sqrt((double)hd);
  double* P = (double*)malloc(sizeof(double) * B * H * S * S);
  double* dS = (double*)malloc(sizeof(double) * B * H * S * S);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bhi = 0; bhi < B * H * S; ++bhi) {
    const int64_t b = bhi / (H * S), h = (bhi / S) % H, i = bhi % S, hk = h / G;
    double* p = P + bhi * S;
    double* ds = dS + bhi * S;
    attn_probs(C, q, k, b, h, i, p);
    const double* dOi = dO + (b * S + i) * nq + h * hd;
    double rowdot = 0.0;
    for (int64_t j = 0; j < S; ++j) {
      ds[j] = dot_row(dOi, v + (b * S + j) * nk + hk * hd, hd);
      rowdot += p[j] * ds[j];
    }
    for (int64_t j = 0; j < S; ++j) ds[j] = p[j] * (ds[j] - rowdot) * scale;
  }
  /* dq */
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bhi = 0; bhi < B * H * S; ++bhi) {
    const int64_t b = bhi / (H * S), h = (bhi / S) % H, i = bhi % S, hk = h / G;
    for (int64_t jd = 0; jd < hd; ++jd) {
      double acc = 0.0;
      for (int64_t j = 0; j < S; ++j) acc += dS[bhi * S + j] * k[(b * S + j) * nk + hk * hd + jd];
      dq[(b * S + i) * nq + h * hd + jd] = RND(R, acc);
    }
  }
  /* dk, dv: key/value head hk collects the G query heads of its group */
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bki = 0; bki < B * Hkv * S; ++bki) {
    const int64_t b = bki / (Hkv * S), hk = (bki / S) % Hkv, j = bki % S;
    for (int64_t jd = 0; jd < hd; ++jd) {
      double ak = 0.0, av = 0.0;
      for (int64_t g = 0; g < G; ++g) {
        const int64_t h = hk * G + g;
        for (int64_t i = 0; i < S; ++i) {
          const int64_t row = (b * H + h) * S + i;
          ak += dS[row * S + j] * q[(b * S + i) * nq + h * hd + jd];
          av += P[row * S + j] * dO[(b * S + i) * nq + h * hd + jd];
        }
      }
      dk[(b * S + j) * nk + hk * hd + jd] = RND(R, ak);
      dv[(b * S + j) * nk + hk * hd + jd] = RND(R, av);
    }
  }
  free(dS);
  free(P);
}

typedef struct {
  orc_attn_core core;
  int64_t d;
  int T_p;
  const double* x;   /* [B*S][d] */
  const double* Wq;  /* [H*hd][d] */
  const double* Wk;  /* [Hkv*hd][d] */
  const double* Wv;  /* [Hkv*hd][d] */
  const double* Wo;  /* [d][H*hd] */
} orc_attn;

/* q, k, v of every token (rounded where stored). */
static void attn_project(const orc_attn* A, double* q, double* k, double* v) {
  const orc_attn_core* C = &A->core;
  const int R = C->round_bf16;
  const int64_t n = C->B * C->S, d = A->d, nq = C->H * C->hd, nk = C->Hkv * C->hd;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    const double* xr = A->x + r * d;
    for (int64_t c = 0; c < nq; ++c) q[r * nq + c] = RND(R, dot_row(xr, A->Wq + c * d, d));
    for (int64_t c = 0; c < nk; ++c) {
      k[r * nk + c] = RND(R, dot_row(xr, A->Wk + c * d, d));
      v[r * nk + c] = RND(R, dot_row(xr, A->Wv + c * d, d));
    }
  }
}

/* Sublayer forward: c [B*S][H*hd] (head outputs), y [B*S][d] = sum over
 * shards t = 0..T_p-1 of c^(t) Wo^(t)T, Wo^(t) = columns [t*nq/T_p, ...). */
void orc_attn_forward(const orc_attn* A, double* c_out, double* y_out) {
  const orc_attn_core* C = &A->core;
  const int64_t n = C->B * C->S, d = A->d, nq = C->H * C->hd, nk = C->Hkv * C->hd;
  double* q = (double*)malloc(sizeof(double) * n * nq);
  double* k = (double*)malloc(sizeof(double) * n * nk);
  double* v = (double*)malloc(sizeof(double) * n * nk);
  attn_project(A, q, k, v);
  orc_attn_core_fwd(C, q, k, v, c_out, NULL);
  const int T = A->T_p;
  const int64_t s = nq / T;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r)
    for (int64_t o = 0; o < d; ++o) {
      double acc = 0.0;
      for (int t = 0; t < T; ++t) {
        double part = 0.0;
        for (int64_t jj = t * s; jj < (t + 1) * s; ++jj) part += A->Wo[o * nq + jj] * c_out[r * nq + jj];
        acc += part;
      }
      y_out[r * d + o] = acc;
    }
  free(v);
  free(k);
  free(q);
}

/* Sublayer backward given dy [B*S][d]: dx [B*S][d] = sum over shards
 * t = 0..T_p-1 of (dq^(t) Wq^(t) + dk^(t) Wk^(t) + dv^(t) Wv^(t)), and the
 * weight gradients dWq [H*hd][d], dWk, dWv [Hkv*hd][d], dWo [d][H*hd]
 * (each may be NULL), summed over all tokens. */
void orc_attn_backward(const orc_attn* A, const double* dy, double* dx, double* dWq, double* dWk, double* dWv,
                       double* dWo) {
  const orc_attn_core* C = &A->core;
  const int R = C->round_bf16;
  const int64_t n = C->B * C->S, d = A->d, nq = C->H * C->hd, nk = C->Hkv * C->hd;
  double* q = (double*)malloc(sizeof(double) * n * nq);
  double* k = (double*)malloc(sizeof(double) * n * nk);
  double* v = (double*)malloc(sizeof(double) * n * nk);
  double* c = (double*)malloc(sizeof(double) * n * nq);
  double* dO = (double*)malloc(sizeof(double) * n * nq);
  double* dq = (double*)malloc(sizeof(double) * n * nq);
  double* dk = (double*)malloc(sizeof(double) * n * nk);
  double* dv = (double*)malloc(sizeof(double) * n * nk);
  attn_project(A, q, k, v);
  orc_attn_core_fwd(C, q, k, v, c, NULL);
  /* dO = dy Wo: shard t's head columns only need its own Wo^(t) -- no sum */
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r)
    for (int64_t col = 0; col < nq; ++col) {
      double acc = 0.0;
      for (int64_t o = 0; o < d; ++o) acc += dy[r * d + o] * A->Wo[o * nq + col];
      dO[r * nq + col] = RND(R, acc);
    }
  orc_attn_core_bwd(C, q, k, v, dO, dq, dk, dv);
  const int T = A->T_p;
  const int64_t sq = nq / T, sk = nk / T;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r)
    for (int64_t kk = 0; kk < d; ++kk) {
      double acc = 0.0;
      for (int t = 0; t < T; ++t) {
        double part = 0.0;
        for (int64_t c2 = t * sq; c2 < (t + 1) * sq; ++c2) part += dq[r * nq + c2] * A->Wq[c2 * d + kk];
        for (int64_t c2 = t * sk; c2 < (t + 1) * sk; ++c2) {
          part += dk[r * nk + c2] * A->Wk[c2 * d + kk];
          part += dv[r * nk + c2] * A->Wv[c2 * d + kk];
        }
        acc += part;
      }
      dx[r * d + kk] = acc;
    }
#pragma omp parallel for schedule(static)
  for (int64_t kk = 0; kk < d; ++kk) {
    for (int64_t c2 = 0; c2 < nq; ++c2) {
      double acc = 0.0;
      for (int64_t r = 0; r < n; ++r) acc += dq[r * nq + c2] * A->x[r * d + kk];
      if (dWq) dWq[c2 * d + kk] = acc;
    }
    for (int64_t c2 = 0; c2 < nk; ++c2) {
      double ak = 0.0, av = 0.0;
      for (int64_t r = 0; r < n; ++r) {
        ak += dk[r * nk + c2] * A->x[r * d + kk];
        av += dv[r * nk + c2] * A->x[r * d + kk];
      }
      if (dWk) dWk[c2 * d + kk] = ak;
      if (dWv) dWv[c2 * d + kk] = av;
    }
  }
  if (dWo) {
#pragma omp parallel for schedule(static)
    for (int64_t o = 0; o < d; ++o)
      for (int64_t col = 0; col < nq; ++col) {
        double acc = 0.0;
        for (int64_t r = 0; r < n; ++r) acc += dy[r * d + o] * c[r * nq + col];
        dWo[o * nq + col] = acc;
      }
  }
  free(dv); free(dk); free(dq); free(dO); free(c); free(v); free(k); free(q);
}

/* Rounding allowances of a bf16 attention core (test infrastructure, not a
 * result).  A computation that stores q, k, v, o, dq, dk, dv in bf16, feeds
 * the probabilities p and the score gradients dS to its products in bf16, and
 * forms D_i = dO_i . o_i from the stored o strays from the exact values by
 * rounding alone.  With u one bf16 unit (relative) this returns, per output
 * element, the root-sum-square of the rounding of every term of its sum plus
 * the coherent error that the error of D_i adds to every dS_ij of a row:
 *   a_o  = u (rss_j p_ij v_jd + |o_id|)
 *   dD_i = u sum_d |dO_id| (|o_id| + rss_j p_ij v_jd)
 *   a_dq = rss_j (u dS_ij k_jd) + dD_i |sum_j p_ij k_jd| / sqrt(hd) + u |dq_id|
 *   a_dk = rss_(h in group, i) ((u |dS_ij| + p_ij dD_i / sqrt(hd)) q_id) + u |dk_jd|
 *   a_dv = rss_(h in group, i) (u p_ij dO_id) + u |dv_jd|
 * (dS includes the 1/sqrt(hd) of the scores).  Layouts as the core. */
void orc_attn_core_allowance(const orc_attn_core* C, const double* q, const double* k, const double* v,
                             const double* dO, double u, double* a_o, double* a_dq, double* a_dk, double* a_dv) {
  const int64_t B = C->B, S = C->S, H = C->H, Hkv = C->Hkv, hd = C->hd, nq = H * hd, nk = Hkv * hd;
  const int64_t G = H / Hkv;
  const double scale = 1.0 / sqrt((double)hd);
  double* P = (double*)malloc(sizeof(double) * B * H * S * S);
  double* dS = (double*)malloc(sizeof(double) * B * H * S * S);
  double* dD = (double*)malloc(sizeof(double) * B * H * S);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bhi = 0; bhi < B * H * S; ++bhi) {
    const int64_t b = bhi / (H * S), h = (bhi / S) % H, i = bhi % S, hk = h / G;
    double* p = P + bhi * S;
    double* ds = dS + bhi * S;
    attn_probs(C, q, k, b, h, i, p);
    const double* dOi = dO + (b * S + i) * nq + h * hd;
    double rowdot = 0.0, dd = 0.0;
    for (int64_t j = 0; j < S; ++j) {
      ds[j] = dot_row(dOi, v + (b * S + j) * nk + hk * hd, hd);
      rowdot += p[j] * ds[j];
    }
    for (int64_t jd = 0; jd < hd; ++jd) {
      double o = 0.0, r2 = 0.0;
      for (int64_t j = 0; j < S; ++j) {
        const double t = p[j] * v[(b * S + j) * nk + hk * hd + jd];
        o += t;
        r2 += t * t;
      }
      a_o[(b * S + i) * nq + h * hd + jd] = u * (sqrt(r2) + fabs(o));
      dd += fabs(dOi[jd]) * (fabs(o) + sqrt(r2));
    }
    dD[bhi] = u * dd;
    for (int64_t j = 0; j < S; ++j) ds[j] = p[j] * (ds[j] - rowdot) * scale;
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bhi = 0; bhi < B * H * S; ++bhi) {
    const int64_t b = bhi / (H * S), h = (bhi / S) % H, i = bhi % S, hk = h / G;
    for (int64_t jd = 0; jd < hd; ++jd) {
      double r2 = 0.0, pk = 0.0, dq = 0.0;
      for (int64_t j = 0; j < S; ++j) {
        const double kk = k[(b * S + j) * nk + hk * hd + jd];
        const double t = u * dS[bhi * S + j] * kk;
        r2 += t * t;
        pk += P[bhi * S + j] * kk;
        dq += dS[bhi * S + j] * kk;
      }
      a_dq[(b * S + i) * nq + h * hd + jd] = sqrt(r2) + dD[bhi] * scale * fabs(pk) + u * fabs(dq);
    }
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bki = 0; bki < B * Hkv * S; ++bki) {
    const int64_t b = bki / (Hkv * S), hk = (bki / S) % Hkv, j = bki % S;
    for (int64_t jd = 0; jd < hd; ++jd) {
      double rk = 0.0, rv = 0.0, dk = 0.0, dv = 0.0;
      for (int64_t g = 0; g < G; ++g) {
        const int64_t h = hk * G + g;
        for (int64_t i = 0; i < S; ++i) {
          const int64_t row = (b * H + h) * S + i;
          const double pij = P[row * S + j], dsij = dS[row * S + j];
          const double qq = q[(b * S + i) * nq + h * hd + jd], gg = dO[(b * S + i) * nq + h * hd + jd];
          const double tk = (u * fabs(dsij) + pij * dD[row] * scale) * qq;
          const double tv = u * pij * gg;
          rk += tk * tk;
          rv += tv * tv;
          dk += dsij * qq;
          dv += pij * gg;
        }
      }
      a_dk[(b * S + j) * nk + hk * hd + jd] = sqrt(rk) + u * fabs(dk);
      a_dv[(b * S + j) * nk + hk * hd + jd] = sqrt(rv) + u * fabs(dv);
    }
  }
  free(dD);
  free(dS);
  free(P);
}

/* The sublayer's stored intermediates: q, k, v (rounded as stored), the head
 * outputs c, and dO = dy Wo (rounded as stored). */
void orc_attn_intermediates(const orc_attn* A, const double* dy, double* q, double* k, double* v, double* c,
                            double* dO) {
  const orc_attn_core* C = &A->core;
  const int64_t n = C->B * C->S, d = A->d, nq = C->H * C->hd;
  attn_project(A, q, k, v);
  orc_attn_core_fwd(C, q, k, v, c, NULL);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r)
    for (int64_t col = 0; col < nq; ++col) {
      double acc = 0.0;
      for (int64_t o = 0; o < d; ++o) acc += dy[r * d + o] * A->Wo[o * nq + col];
      dO[r * nq + col] = RND(C->round_bf16, acc);
    }
}

/* Sampled rows of the attention core with their rounding allowances (test
 * infrastructure for full-size shapes, where the whole core is too slow).
 * Query samples (rb, rh, ri): o row, lse (natural log) and dq row of query ri
 * of head rh in sequence rb.  Key samples (kb, khk, kj): dk and dv rows of key
 * kj of key/value head khk in sequence kb.  Values and allowances are those
 * of orc_attn_core_fwd / orc_attn_core_bwd / orc_attn_core_allowance at the
 * same positions (D_i is taken as dO_i . o_i, equal to sum_j p_ij dO_i . v_j).
 * Row statistics are computed per (sequence, head, query) in parallel and
 * accumulated in a fixed order, so results do not depend on the thread count. */
typedef struct {
  double lse, D, dD;
} attn_rowstat;

static void attn_row_stats(const orc_attn_core* C, const double* q, const double* k, const double* v,
                           const double* dO, double u, int64_t b, int64_t h, int64_t i, double* p, double* o,
                           double* rss_o, attn_rowstat* st) {
  const int64_t S = C->S, hd = C->hd, nq = C->H * hd, nk = C->Hkv * hd;
  const int64_t hk = h / (C->H / C->Hkv);
  st->lse = attn_probs(C, q, k, b, h, i, p);
  const double* dOi = dO + (b * S + i) * nq + h * hd;
  double D = 0.0, dd = 0.0;
  for (int64_t jd = 0; jd < hd; ++jd) {
    double acc = 0.0, r2 = 0.0;
    for (int64_t j = 0; j < S; ++j) {
      const double t = p[j] * v[(b * S + j) * nk + hk * hd + jd];
      acc += t;
      r2 += t * t;
    }
    o[jd] = acc;
    rss_o[jd] = sqrt(r2);
    D += dOi[jd] * acc;
    dd += fabs(dOi[jd]) * (fabs(acc) + sqrt(r2));
  }
  st->D = D;
  st->dD = u * dd;
}

void orc_attn_core_sample(const orc_attn_core* C, const double* q, const double* k, const double* v,
                          const double* dO, double u, int64_t nr, const int64_t* rb, const int64_t* rh,
                          const int64_t* ri, double* o_out, double* lse_out, double* dq_out, double* a_o,
                          double* a_dq, int64_t nkv, const int64_t* kb, const int64_t* khk, const int64_t* kj,
                          double* dk_out, double* dv_out, double* a_dk, double* a_dv) {
  const int64_t S = C->S, hd = C->hd, H = C->H, Hkv = C->Hkv, nq = H * hd, nk = Hkv * hd;
  const int64_t G = H / Hkv;
  const double scale = 1.0 / sqrt((double)hd);
  /* query samples */
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t s = 0; s < nr; ++s) {
    const int64_t b = rb[s], h = rh[s], i = ri[s], hk = h / G;
    double* p = (double*)malloc(sizeof(double) * S);
    double* o = o_out + s * hd;
    double* rss = (double*)malloc(sizeof(double) * hd);
    attn_rowstat st;
    attn_row_stats(C, q, k, v, dO, u, b, h, i, p, o, rss, &st);
    lse_out[s] = st.lse;
    const double* dOi = dO + (b * S + i) * nq + h * hd;
    double* ds = (double*)malloc(sizeof(double) * S);
    for (int64_t j = 0; j < S; ++j)
      ds[j] = p[j] * (dot_row(dOi, v + (b * S + j) * nk + hk * hd, hd) - st.D) * scale;
    for (int64_t jd = 0; jd < hd; ++jd) {
      double dq = 0.0, r2 = 0.0, pk = 0.0;
      for (int64_t j = 0; j < S; ++j) {
        const double kk = k[(b * S + j) * nk + hk * hd + jd];
        dq += ds[j] * kk;
        r2 += (u * ds[j] * kk) * (u * ds[j] * kk);
        pk += p[j] * kk;
      }
      dq_out[s * hd + jd] = dq;
      a_dq[s * hd + jd] = sqrt(r2) + st.dD * scale * fabs(pk) + u * fabs(dq);
      a_o[s * hd + jd] = u * (rss[jd] + fabs(o[jd]));
    }
    free(ds);
    free(rss);
    free(p);
  }
  /* key samples: each needs p_ij, dS_ij and dD_i of every visible query i of
   * every query head of the group */
  for (int64_t s = 0; s < nkv; ++s) {
    const int64_t b = kb[s], hk = khk[s], j = kj[s];
    const int64_t i0 = C->causal ? j : 0;
    const int64_t ni = S - i0;
    double* pij = (double*)malloc(sizeof(double) * G * ni);
    double* dsij = (double*)malloc(sizeof(double) * G * ni);
    double* ddi = (double*)malloc(sizeof(double) * G * ni);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t gi = 0; gi < G * ni; ++gi) {
      const int64_t g = gi / ni, i = i0 + gi % ni, h = hk * G + g;
      double* p = (double*)malloc(sizeof(double) * S);
      double* o = (double*)malloc(sizeof(double) * hd);
      double* rss = (double*)malloc(sizeof(double) * hd);
      attn_rowstat st;
      attn_row_stats(C, q, k, v, dO, u, b, h, i, p, o, rss, &st);
      const double dp = dot_row(dO + (b * S + i) * nq + h * hd, v + (b * S + j) * nk + hk * hd, hd);
      pij[gi] = p[j];
      dsij[gi] = p[j] * (dp - st.D) * scale;
      ddi[gi] = st.dD;
      free(rss);
      free(o);
      free(p);
    }
    for (int64_t jd = 0; jd < hd; ++jd) {
      double dk = 0.0, dv = 0.0, rk = 0.0, rv = 0.0;
      for (int64_t gi = 0; gi < G * ni; ++gi) {
        const int64_t g = gi / ni, i = i0 + gi % ni, h = hk * G + g;
        const double qq = q[(b * S + i) * nq + h * hd + jd], gg = dO[(b * S + i) * nq + h * hd + jd];
        dk += dsij[gi] * qq;
        dv += pij[gi] * gg;
        const double tk = (u * fabs(dsij[gi]) + pij[gi] * ddi[gi] * scale) * qq;
        const double tv = u * pij[gi] * gg;
        rk += tk * tk;
        rv += tv * tv;
      }
      dk_out[s * hd + jd] = dk;
      dv_out[s * hd + jd] = dv;
      a_dk[s * hd + jd] = sqrt(rk) + u * fabs(dk);
      a_dv[s * hd + jd] = sqrt(rv) + u * fabs(dv);
    }
    free(ddi);
    free(dsij);
    free(pij);
  }
}
