/*
 * GBLA oracle — plain, slow, fp64 CPU statement of what the GBLA layer computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the CPU
 * baseline leg of the benchmark load this library.  It shares no code, header,
 * table or helper with the CUDA path, and the CUDA path never calls it.
 *
 * Source of every step: "Gated Bidirectional Linear Attention for Generative
 * Retrieval" (close-reading notes), section "Core method":
 *   Eq. 2  single-query BLA form            Eq. 3  matrix form, computation order
 *   Eq. 4  X~ = Conv1d(X), Q,K,V = X~ W      Eq. 5  key gate g_j inside both sums
 *   Eq. 6  K~ = g (.) phi(K)                 Eq. 7  RmsNorm(O) (.) SiLU(X~ W_R)
 *   "Multi-head" paragraph: every head h owns W_Q^h, W_K^h, W_V^h, w_g^h, W_R^h.
 * Second, independent forms used only to pin this file against itself:
 *   - the O(L^2) explicit sum of Eq. 5 (oracle_core_explicit);
 *   - the bidirectional RNN with the -1/2 k_i v_i^T diagonal correction and an
 *     all-ones mask, from "Linear Attention for Efficient Bidirectional
 *     Sequence Modeling" (LION notes), "Bidirectional RNN" (Theorem 3.1)
 *     (oracle_core_lion_rnn).
 * The core under LION's decay masks (Lion-d, Lion-s; LION notes, mask
 * construction and instantiated models) is stated the same two ways:
 * oracle_decay_core_explicit (the definition) and oracle_decay_core_rnn.
 * The bidirectional softmax attention of the SA blocks of the hybrid
 * [SA, LA, LA] encoder (GBLA notes, "Core method" 1, Eq. 1, and the hybrid
 * encoder paragraph) is oracle_sa_forward, Eq. 1 written out per query, and
 * oracle_sa_rows the same at chosen (query, head) pairs of long sequences.
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *   phi(x) = elu(x) + 1 with alpha = 1, no 1/sqrt(d_h) scale;
 *   Conv1d is depthwise over the d channels, causal, kernel 4, zero left pad of
 *   3 at every sequence start, optional bias, no activation; tap t multiplies
 *   x[l - 3 + t] (PyTorch cross-correlation order);
 *   gate: sigmoid(x~ . w_g + b_g) per token and head (gate_mode 0), or the
 *   pages' softmax of x~ . w_g over the valid tokens of the sequence (mode 1);
 *   RmsNorm over the d_h features of one head and token, eps given, scale
 *   gamma[d_h] shared by all heads (NULL = ones); SiLU gate reads X~ (post conv);
 *   no epsilon in the division (den > 0 since phi > 0 and g > 0);
 *   tokens that belong to no sequence (padding) give y = 0 and dx = 0.
 *
 * Layouts (all row-major, doubles): x, x~ [T, d]; W_* [d, H*d_h] (column block
 * h*d_h .. h*d_h+d_h-1 is head h); w_g [d, H]; q, k, v, r, o [T, H*d_h];
 * s, g, den [T, H]; state [n_seq, H, d_h, d_h+1] with z as column d_h.
 * A sequence is (start, len): rows start .. start+len-1 of the [T, *] arrays.
 *
 * The backward is the hand-derived chain rule of the forward, step by step in
 * reverse; it is pinned by central finite differences and by PyTorch autograd
 * through library routines in the tests.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- scalars */

/* phi(x) = elu(x) + 1: x + 1 for x > 0, e^x otherwise (elu with alpha = 1). */
static double phi(double x) { return x > 0.0 ? x + 1.0 : exp(x); }
/* d phi / dx: 1 for x > 0, e^x otherwise. */
static double dphi(double x) { return x > 0.0 ? 1.0 : exp(x); }
static double sigm(double x) { return 1.0 / (1.0 + exp(-x)); }
static double silu(double x) { return x * sigm(x); }
/* d/dx [x sigma(x)] = sigma(x) (1 + x (1 - sigma(x))). */
static double dsilu(double x) {
  double s = sigm(x);
  return s * (1.0 + x * (1.0 - s));
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ------------------------------------------------------------------ core */

/*
 * BLA core with key gate, Eq. 5 / Eq. 6, state form (Eq. 3 computation order):
 *   S = sum_j g_j phi(k_j) v_j^T,  z = sum_j g_j phi(k_j)      (per seq, head)
 *   o_i = phi(q_i)^T S / phi(q_i)^T z.
 * q, k, v: [T, H*dh] with row stride ld (>= H*dh); g: [T, H] (gate VALUES, >= 0).
 * Outputs o [T, ld] (only sequence rows written), den [T, H] (may be NULL),
 * state [n_seq, H, dh, dh+1] (may be NULL).
 */
void oracle_core_forward(int64_t T, int H, int dh, int n_seq,
                         const int64_t* start, const int64_t* len,
                         const double* q, const double* k, const double* v,
                         const double* g, double* o, double* den,
                         double* state) {
  (void)T;
  const int64_t ld = (int64_t)H * dh;
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int b = 0; b < n_seq; ++b) {
    for (int h = 0; h < H; ++h) {
      double* S = (double*)calloc((size_t)dh * (dh + 1), sizeof(double));
      for (int64_t j = start[b]; j < start[b] + len[b]; ++j) {
        const double gj = g[j * H + h];
        for (int e = 0; e < dh; ++e) {
          const double kt = gj * phi(k[j * ld + h * dh + e]); /* K~ = g phi(K) */
          for (int f = 0; f < dh; ++f)
            S[e * (dh + 1) + f] += kt * v[j * ld + h * dh + f];
          S[e * (dh + 1) + dh] += kt; /* z */
        }
      }
      for (int64_t i = start[b]; i < start[b] + len[b]; ++i) {
        double dn = 0.0;
        for (int e = 0; e < dh; ++e) dn += phi(q[i * ld + h * dh + e]) * S[e * (dh + 1) + dh];
        for (int f = 0; f < dh; ++f) {
          double n = 0.0;
          for (int e = 0; e < dh; ++e) n += phi(q[i * ld + h * dh + e]) * S[e * (dh + 1) + f];
          o[i * ld + h * dh + f] = n / dn;
        }
        if (den) den[i * H + h] = dn;
      }
      if (state)
        memcpy(state + ((size_t)b * H + h) * dh * (dh + 1), S,
               sizeof(double) * dh * (dh + 1));
      free(S);
    }
  }
}

/*
 * The same output from the O(L^2) single-query form of Eq. 5, never forming S:
 *   o_i = sum_j g_j (phi(q_i) . phi(k_j)) v_j / sum_j g_j (phi(q_i) . phi(k_j)).
 */
void oracle_core_explicit(int64_t T, int H, int dh, int n_seq,
                          const int64_t* start, const int64_t* len,
                          const double* q, const double* k, const double* v,
                          const double* g, double* o) {
  (void)T;
  const int64_t ld = (int64_t)H * dh;
  for (int b = 0; b < n_seq; ++b)
    for (int h = 0; h < H; ++h)
      for (int64_t i = start[b]; i < start[b] + len[b]; ++i) {
        double num[1024];
        double dsum = 0.0;
        for (int f = 0; f < dh; ++f) num[f] = 0.0;
        for (int64_t j = start[b]; j < start[b] + len[b]; ++j) {
          double sim = 0.0;
          for (int e = 0; e < dh; ++e)
            sim += phi(q[i * ld + h * dh + e]) * phi(k[j * ld + h * dh + e]);
          const double w = g[j * H + h] * sim;
          for (int f = 0; f < dh; ++f) num[f] += w * v[j * ld + h * dh + f];
          dsum += w;
        }
        for (int f = 0; f < dh; ++f) o[i * ld + h * dh + f] = num[f] / dsum;
      }
}

/*
 * The same output from LION's bidirectional RNN (Theorem 3.1) with an all-ones
 * mask (Lambda_i = 1) and keys k~_j = g_j phi(k_j):
 *   forward scan  S^F_i = S^F_{i-1} + k~_i v_i^T,  y^F_i = q~_i^T (S^F_i - 1/2 k~_i v_i^T)
 *   backward scan S^B_i = S^B_{i+1} + k~_i v_i^T,  y^B_i = q~_i^T (S^B_i - 1/2 k~_i v_i^T)
 *   y_i = y^F_i + y^B_i.  The halves remove the diagonal that both scans count
 *   (mask M = M^F + M^B - I).  The combining formula is lost in the page text;
 *   the sum is the reading that the mask identity gives.  The numerator uses v,
 *   the denominator the same recurrence with v == 1, and o_i = num_i / den_i.
 */
void oracle_core_lion_rnn(int64_t T, int H, int dh, int n_seq,
                          const int64_t* start, const int64_t* len,
                          const double* q, const double* k, const double* v,
                          const double* g, double* o) {
  (void)T;
  const int64_t ld = (int64_t)H * dh;
  const int W = dh + 1; /* column dh carries the v == 1 recurrence */
  for (int b = 0; b < n_seq; ++b)
    for (int h = 0; h < H; ++h) {
      const int64_t n = len[b], s0 = start[b];
      double* S = (double*)calloc((size_t)dh * W, sizeof(double));
      double* yF = (double*)calloc((size_t)(n > 0 ? n : 1) * W, sizeof(double));
      /* forward direction */
      for (int64_t t = 0; t < n; ++t) {
        const int64_t i = s0 + t;
        for (int e = 0; e < dh; ++e) {
          const double kt = g[i * H + h] * phi(k[i * ld + h * dh + e]);
          for (int f = 0; f < W; ++f)
            S[e * W + f] += kt * (f < dh ? v[i * ld + h * dh + f] : 1.0);
        }
        for (int f = 0; f < W; ++f) {
          double acc = 0.0;
          for (int e = 0; e < dh; ++e) {
            const double kt = g[i * H + h] * phi(k[i * ld + h * dh + e]);
            const double vf = f < dh ? v[i * ld + h * dh + f] : 1.0;
            acc += phi(q[i * ld + h * dh + e]) * (S[e * W + f] - 0.5 * kt * vf);
          }
          yF[t * W + f] = acc;
        }
      }
      /* backward direction */
      memset(S, 0, sizeof(double) * dh * W);
      for (int64_t t = n - 1; t >= 0; --t) {
        const int64_t i = s0 + t;
        for (int e = 0; e < dh; ++e) {
          const double kt = g[i * H + h] * phi(k[i * ld + h * dh + e]);
          for (int f = 0; f < W; ++f)
            S[e * W + f] += kt * (f < dh ? v[i * ld + h * dh + f] : 1.0);
        }
        double y[1025];
        for (int f = 0; f < W; ++f) {
          double acc = 0.0;
          for (int e = 0; e < dh; ++e) {
            const double kt = g[i * H + h] * phi(k[i * ld + h * dh + e]);
            const double vf = f < dh ? v[i * ld + h * dh + f] : 1.0;
            acc += phi(q[i * ld + h * dh + e]) * (S[e * W + f] - 0.5 * kt * vf);
          }
          y[f] = yF[t * W + f] + acc;
        }
        for (int f = 0; f < dh; ++f) o[i * ld + h * dh + f] = y[f] / y[dh];
      }
      free(yF);
      free(S);
    }
}

/*
 * The gated core under LION's decay masks ("Linear Attention for Efficient
 * Bidirectional Sequence Modeling" notes, "Bidirectional mask construction"
 * and the table of instantiated models): with a decay lambda_t in [0, 1] per
 * token t (and head),
 *   M^F_ij = prod_{t=j+1..i} lambda_t (j <= i),  M^B_ij = prod_{t=i+1..j} lambda_t (j >= i),
 *   M = M^F + M^B - I  (so M_ii = 1),
 *   o_i = sum_j M_ij g_j (phi(q_i) . phi(k_j)) v_j / sum_j M_ij g_j (phi(q_i) . phi(k_j)),
 * the row scaling of Y = Scale(Q K^T (.) M) V with this layer's feature map and
 * key gate.  Lion-d is a constant lambda_t = lambda (M_ij = lambda^|i-j|),
 * Lion-s a per-token lambda_t = sigmoid(W x_t + b); lambda == 1 gives the
 * all-ones mask of Eq. 5.  Written as the O(L^2) definition; den_i is the
 * denominator.
 */
void oracle_decay_core_explicit(int64_t T, int H, int dh, int n_seq,
                                const int64_t* start, const int64_t* len,
                                const double* q, const double* k, const double* v,
                                const double* g, const double* lam, double* o, double* den) {
  const int64_t ld = (int64_t)H * dh;
  /* phi(q) and phi(k), once */
  double* pq = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * ld);
  double* pk = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * ld);
  for (int64_t i = 0; i < T * ld; ++i) {
    pq[i] = phi(q[i]);
    pk[i] = phi(k[i]);
  }
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int b = 0; b < n_seq; ++b)
    for (int h = 0; h < H; ++h)
      for (int64_t i = start[b]; i < start[b] + len[b]; ++i) {
        double num[1024];
        double dsum = 0.0;
        for (int f = 0; f < dh; ++f) num[f] = 0.0;
        /* M_ij for j = i, then outward: going down, M_ij = M_i(j+1) lambda_{j+1};
         * going up, M_ij = M_i(j-1) lambda_j (the decays strictly after
         * min(i, j) and up to max(i, j)) */
        for (int dir = 0; dir < 2; ++dir) {
          double m = 1.0;
          for (int64_t j = dir == 0 ? i : i + 1; dir == 0 ? j >= start[b] : j < start[b] + len[b]; j += dir == 0 ? -1 : 1) {
            if (dir == 0 && j < i) m *= lam[(j + 1) * H + h];
            if (dir == 1) m *= lam[j * H + h];
            double sim = 0.0;
            for (int e = 0; e < dh; ++e) sim += pq[i * ld + h * dh + e] * pk[j * ld + h * dh + e];
            const double w = m * g[j * H + h] * sim;
            for (int f = 0; f < dh; ++f) num[f] += w * v[j * ld + h * dh + f];
            dsum += w;
          }
        }
        for (int f = 0; f < dh; ++f) o[i * ld + h * dh + f] = num[f] / dsum;
        if (den) den[i * H + h] = dsum;
      }
  free(pq);
  free(pk);
}

/*
 * Bidirectional softmax attention, Eq. 1 of the GBLA notes ("Core method" 1):
 *   o_i = sum_j exp(q_i . k_j / sqrt(d_h)) v_j / sum_j exp(q_i . k_j / sqrt(d_h))
 * over every key j of query i's sequence (no mask: both directions), per head.
 * The largest score of the row is subtracted inside the exponentials (it
 * cancels between numerator and denominator); lse_i = m_i + log of the
 * denominator (the log-sum-exp of the scaled scores) is returned when lse is
 * not NULL.  Rows in no sequence are left untouched.
 */
void oracle_sa_forward(int64_t T, int H, int dh, int n_seq,
                       const int64_t* start, const int64_t* len,
                       const double* q, const double* k, const double* v, double* o, double* lse) {
  const int64_t ld = (int64_t)H * dh;
  const double scale = 1.0 / sqrt((double)dh);
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int b = 0; b < n_seq; ++b)
    for (int h = 0; h < H; ++h) {
      double* sc = (double*)malloc(sizeof(double) * (size_t)(len[b] > 0 ? len[b] : 1));
      for (int64_t i = start[b]; i < start[b] + len[b]; ++i) {
        double m = -INFINITY;
        for (int64_t j = start[b]; j < start[b] + len[b]; ++j) {
          double s = 0.0;
          for (int e = 0; e < dh; ++e) s += q[i * ld + h * dh + e] * k[j * ld + h * dh + e];
          s *= scale;
          sc[j - start[b]] = s;
          if (s > m) m = s;
        }
        double num[1024];
        double den = 0.0;
        for (int f = 0; f < dh; ++f) num[f] = 0.0;
        for (int64_t j = start[b]; j < start[b] + len[b]; ++j) {
          const double w = exp(sc[j - start[b]] - m);
          for (int f = 0; f < dh; ++f) num[f] += w * v[j * ld + h * dh + f];
          den += w;
        }
        for (int f = 0; f < dh; ++f) o[i * ld + h * dh + f] = num[f] / den;
        if (lse) lse[i * H + h] = m + log(den);
      }
      free(sc);
    }
}

/*
 * Eq. 1 at chosen (query row, head) pairs only, for sequences too long to
 * compute every row: the same sum as oracle_sa_forward, one query at a time.
 * Pair p is row rows[p] of head heads[p]; its d_h outputs go to o[p*dh ..];
 * a row in no sequence gives zeros.
 */
void oracle_sa_rows(int64_t T, int H, int dh, int n_seq, const int64_t* start, const int64_t* len,
                    const double* q, const double* k, const double* v, int n, const int64_t* rows,
                    const int* heads, double* o) {
  const int64_t ld = (int64_t)H * dh;
  const double scale = 1.0 / sqrt((double)dh);
#pragma omp parallel for schedule(dynamic)
  for (int p = 0; p < n; ++p) {
    const int64_t i = rows[p];
    const int h = heads[p];
    double* out = o + (int64_t)p * dh;
    for (int f = 0; f < dh; ++f) out[f] = 0.0;
    int b = -1;
    for (int s = 0; s < n_seq && b < 0; ++s)
      if (i >= start[s] && i < start[s] + len[s]) b = s;
    if (b < 0 || i < 0 || i >= T || h < 0 || h >= H) continue;
    double* sc = (double*)malloc(sizeof(double) * (size_t)len[b]);
    double m = -INFINITY;
    for (int64_t j = start[b]; j < start[b] + len[b]; ++j) {
      double s = 0.0;
      for (int e = 0; e < dh; ++e) s += q[i * ld + h * dh + e] * k[j * ld + h * dh + e];
      s *= scale;
      sc[j - start[b]] = s;
      if (s > m) m = s;
    }
    double den = 0.0;
    for (int64_t j = start[b]; j < start[b] + len[b]; ++j) {
      const double w = exp(sc[j - start[b]] - m);
      for (int f = 0; f < dh; ++f) out[f] += w * v[j * ld + h * dh + f];
      den += w;
    }
    for (int f = 0; f < dh; ++f) out[f] /= den;
    free(sc);
  }
}

/*
 * The same output from LION's bidirectional RNN (Theorem 3.1) with the decays
 * as the state transitions, keys k~_j = g_j phi(k_j):
 *   S^F_i = lambda_i S^F_{i-1} + k~_i v_i^T,      y^F_i = q~_i^T (S^F_i - 1/2 k~_i v_i^T)
 *   S^B_i = lambda_{i+1} S^B_{i+1} + k~_i v_i^T,  y^B_i = q~_i^T (S^B_i - 1/2 k~_i v_i^T)
 *   y_i = y^F_i + y^B_i  (numerator with v, denominator with v == 1),
 * which unrolls to the M^F and M^B of oracle_decay_core_explicit.
 */
void oracle_decay_core_rnn(int64_t T, int H, int dh, int n_seq,
                           const int64_t* start, const int64_t* len,
                           const double* q, const double* k, const double* v,
                           const double* g, const double* lam, double* o) {
  (void)T;
  const int64_t ld = (int64_t)H * dh;
  const int W = dh + 1;
  for (int b = 0; b < n_seq; ++b)
    for (int h = 0; h < H; ++h) {
      const int64_t n = len[b], s0 = start[b];
      double* S = (double*)calloc((size_t)dh * W, sizeof(double));
      double* yF = (double*)calloc((size_t)(n > 0 ? n : 1) * W, sizeof(double));
      for (int64_t t = 0; t < n; ++t) {  /* forward */
        const int64_t i = s0 + t;
        const double a = t > 0 ? lam[i * H + h] : 0.0;  /* S^F_{-1} = 0 */
        for (int e = 0; e < dh; ++e) {
          const double kt = g[i * H + h] * phi(k[i * ld + h * dh + e]);
          for (int f = 0; f < W; ++f) S[e * W + f] = a * S[e * W + f] + kt * (f < dh ? v[i * ld + h * dh + f] : 1.0);
        }
        for (int f = 0; f < W; ++f) {
          double acc = 0.0;
          for (int e = 0; e < dh; ++e) {
            const double kt = g[i * H + h] * phi(k[i * ld + h * dh + e]);
            const double vf = f < dh ? v[i * ld + h * dh + f] : 1.0;
            acc += phi(q[i * ld + h * dh + e]) * (S[e * W + f] - 0.5 * kt * vf);
          }
          yF[t * W + f] = acc;
        }
      }
      memset(S, 0, sizeof(double) * dh * W);
      for (int64_t t = n - 1; t >= 0; --t) {  /* backward */
        const int64_t i = s0 + t;
        const double a = t + 1 < n ? lam[(i + 1) * H + h] : 0.0;  /* S^B_n = 0 */
        for (int e = 0; e < dh; ++e) {
          const double kt = g[i * H + h] * phi(k[i * ld + h * dh + e]);
          for (int f = 0; f < W; ++f) S[e * W + f] = a * S[e * W + f] + kt * (f < dh ? v[i * ld + h * dh + f] : 1.0);
        }
        double y[1025];
        for (int f = 0; f < W; ++f) {
          double acc = 0.0;
          for (int e = 0; e < dh; ++e) {
            const double kt = g[i * H + h] * phi(k[i * ld + h * dh + e]);
            const double vf = f < dh ? v[i * ld + h * dh + f] : 1.0;
            acc += phi(q[i * ld + h * dh + e]) * (S[e * W + f] - 0.5 * kt * vf);
          }
          y[f] = yF[t * W + f] + acc;
        }
        for (int f = 0; f < dh; ++f) o[i * ld + h * dh + f] = y[f] / y[dh];
      }
      free(yF);
      free(S);
    }
}

/*
 * Backward of oracle_core_forward for the scalar <d_o, o>.  Chain rule of
 * n_i = S^T q~_i, den_i = q~_i . z, o_i = n_i / den_i, S = sum k~_j v_j^T,
 * z = sum k~_j, k~_j = g_j phi(k_j), q~_i = phi(q_i):
 *   dn_i = do_i / den_i;  dden_i = -(do_i . o_i) / den_i
 *   dq~_i = S dn_i + z dden_i;               dq_i = dq~_i (.) phi'(q_i)
 *   dS = sum_i q~_i dn_i^T;  dz = sum_i q~_i dden_i
 *   dk~_j = dS v_j + dz;  dv_j = dS^T k~_j
 *   dg_j = phi(k_j) . dk~_j;  dk_j = g_j dk~_j (.) phi'(k_j)
 * Any of dq, dk, dv, dg may be NULL.
 */
void oracle_core_backward(int64_t T, int H, int dh, int n_seq,
                          const int64_t* start, const int64_t* len,
                          const double* q, const double* k, const double* v,
                          const double* g, const double* d_o, double* dq,
                          double* dk, double* dv, double* dg) {
  (void)T;
  const int64_t ld = (int64_t)H * dh;
  const int W = dh + 1;
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int b = 0; b < n_seq; ++b) {
    for (int h = 0; h < H; ++h) {
      double* S = (double*)calloc((size_t)dh * W, sizeof(double));
      double* dS = (double*)calloc((size_t)dh * W, sizeof(double));
      double o[1024], dn[1024];
      for (int64_t j = start[b]; j < start[b] + len[b]; ++j)
        for (int e = 0; e < dh; ++e) {
          const double kt = g[j * H + h] * phi(k[j * ld + h * dh + e]);
          for (int f = 0; f < dh; ++f) S[e * W + f] += kt * v[j * ld + h * dh + f];
          S[e * W + dh] += kt;
        }
      for (int64_t i = start[b]; i < start[b] + len[b]; ++i) {
        const double* qi = q + i * ld + h * dh;
        const double* doi = d_o + i * ld + h * dh;
        double den = 0.0;
        for (int e = 0; e < dh; ++e) den += phi(qi[e]) * S[e * W + dh];
        double dot = 0.0;
        for (int f = 0; f < dh; ++f) {
          double n = 0.0;
          for (int e = 0; e < dh; ++e) n += phi(qi[e]) * S[e * W + f];
          o[f] = n / den;
          dot += doi[f] * o[f];
        }
        const double dden = -dot / den;
        for (int f = 0; f < dh; ++f) dn[f] = doi[f] / den;
        for (int e = 0; e < dh; ++e) {
          double dqt = S[e * W + dh] * dden;
          for (int f = 0; f < dh; ++f) dqt += S[e * W + f] * dn[f];
          if (dq) dq[i * ld + h * dh + e] = dqt * dphi(qi[e]);
          for (int f = 0; f < dh; ++f) dS[e * W + f] += phi(qi[e]) * dn[f];
          dS[e * W + dh] += phi(qi[e]) * dden;
        }
      }
      for (int64_t j = start[b]; j < start[b] + len[b]; ++j) {
        const double* kj = k + j * ld + h * dh;
        const double* vj = v + j * ld + h * dh;
        const double gj = g[j * H + h];
        double dgj = 0.0;
        for (int e = 0; e < dh; ++e) {
          double dkt = dS[e * W + dh];
          for (int f = 0; f < dh; ++f) dkt += dS[e * W + f] * vj[f];
          dgj += phi(kj[e]) * dkt;
          if (dk) dk[j * ld + h * dh + e] = gj * dkt * dphi(kj[e]);
        }
        if (dv)
          for (int f = 0; f < dh; ++f) {
            double acc = 0.0;
            for (int e = 0; e < dh; ++e) acc += dS[e * W + f] * gj * phi(kj[e]);
            dv[j * ld + h * dh + f] = acc;
          }
        if (dg) dg[j * H + h] = dgj;
      }
      free(S);
      free(dS);
    }
  }
}

/* ------------------------------------------------------------ GBLA layer */

/* Eq. 4, Conv1d: x~[l, c] = b[c] + sum_{t=0..3} w[c, t] x[l - 3 + t, c] within
 * the sequence (positions before its first token read zero). */
void oracle_conv1d(int64_t T, int d, int n_seq, const int64_t* start,
                   const int64_t* len, const double* x, const double* w,
                   const double* bias, double* xt) {
  (void)T;
  for (int b = 0; b < n_seq; ++b)
    for (int64_t l = 0; l < len[b]; ++l)
      for (int c = 0; c < d; ++c) {
        double acc = bias ? bias[c] : 0.0;
        for (int t = 0; t < 4; ++t) {
          const int64_t src = l - 3 + t;
          if (src >= 0) acc += w[c * 4 + t] * x[(start[b] + src) * d + c];
        }
        xt[(start[b] + l) * d + c] = acc;
      }
}

/* out[t, :] = x~[t, :] W for every token t of every sequence (W is [d, n]). */
static void project(int d, int n, int n_seq, const int64_t* start,
                    const int64_t* len, const double* xt, const double* W,
                    double* out) {
  for (int b = 0; b < n_seq; ++b)
#pragma omp parallel for schedule(static)
    for (int64_t t = start[b]; t < start[b] + len[b]; ++t)
      for (int j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += xt[t * d + c] * W[(int64_t)c * n + j];
        out[t * n + j] = acc;
      }
}

/* The key gate, Eq. 5.  s = x~ w_g (+ b_g).  Mode 0: g = sigmoid(s) per token
 * and head.  Mode 1: g = softmax of s over the valid tokens of the sequence,
 * per head (the pages' definition; b_g then cancels). */
static void gate(int H, int n_seq, const int64_t* start, const int64_t* len,
                 int gate_mode, const double* s, double* g) {
  for (int b = 0; b < n_seq; ++b)
    for (int h = 0; h < H; ++h) {
      if (gate_mode == 0) {
        for (int64_t t = start[b]; t < start[b] + len[b]; ++t)
          g[t * H + h] = sigm(s[t * H + h]);
      } else {
        double m = -INFINITY, sum = 0.0;
        for (int64_t t = start[b]; t < start[b] + len[b]; ++t)
          if (s[t * H + h] > m) m = s[t * H + h];
        for (int64_t t = start[b]; t < start[b] + len[b]; ++t)
          sum += exp(s[t * H + h] - m);
        for (int64_t t = start[b]; t < start[b] + len[b]; ++t)
          g[t * H + h] = exp(s[t * H + h] - m) / sum;
      }
    }
}

/* Everything the forward computes, kept for the backward and for the tests. */
typedef struct {
  double *xt, *q, *k, *v, *r, *s, *g, *o, *den, *rstd;
} fwd_buffers;

static void forward_into(int64_t T, int d, int H, int dh, int n_seq,
                         const int64_t* start, const int64_t* len,
                         const double* x, const double* conv_w,
                         const double* conv_b, const double* Wq,
                         const double* Wk, const double* Wv, const double* Wr,
                         const double* wg, const double* bg,
                         const double* gamma, int gate_mode, double eps,
                         fwd_buffers* fb, double* y, double* state) {
  const int64_t ld = (int64_t)H * dh;
  /* Eq. 4: conv, then the projections from x~ */
  oracle_conv1d(T, d, n_seq, start, len, x, conv_w, conv_b, fb->xt);
  project(d, (int)ld, n_seq, start, len, fb->xt, Wq, fb->q);
  project(d, (int)ld, n_seq, start, len, fb->xt, Wk, fb->k);
  project(d, (int)ld, n_seq, start, len, fb->xt, Wv, fb->v);
  project(d, (int)ld, n_seq, start, len, fb->xt, Wr, fb->r); /* Eq. 7 gate input */
  project(d, H, n_seq, start, len, fb->xt, wg, fb->s);
  for (int b = 0; b < n_seq; ++b)
    for (int64_t t = start[b]; t < start[b] + len[b]; ++t)
      for (int h = 0; h < H; ++h) fb->s[t * H + h] += bg ? bg[h] : 0.0;
  /* Eq. 5: gate */
  gate(H, n_seq, start, len, gate_mode, fb->s, fb->g);
  /* Eq. 5 / 6: the gated core */
  oracle_core_forward(T, H, dh, n_seq, start, len, fb->q, fb->k, fb->v, fb->g,
                      fb->o, fb->den, state);
  /* Eq. 7: RmsNorm over d_h, times gamma, times SiLU(x~ W_R) */
  memset(y, 0, sizeof(double) * (size_t)T * ld);
  for (int b = 0; b < n_seq; ++b)
    for (int64_t t = start[b]; t < start[b] + len[b]; ++t)
      for (int h = 0; h < H; ++h) {
        const double* ot = fb->o + t * ld + h * dh;
        double ms = 0.0;
        for (int f = 0; f < dh; ++f) ms += ot[f] * ot[f];
        ms /= dh;
        const double rs = 1.0 / sqrt(ms + eps);
        fb->rstd[t * H + h] = rs;
        for (int f = 0; f < dh; ++f)
          y[t * ld + h * dh + f] = ot[f] * rs * (gamma ? gamma[f] : 1.0) *
                                   silu(fb->r[t * ld + h * dh + f]);
      }
}

static int alloc_fwd(fwd_buffers* fb, int64_t T, int d, int H, int dh) {
  const size_t td = (size_t)T * d, tl = (size_t)T * H * dh, th = (size_t)T * H;
  fb->xt = (double*)calloc(td ? td : 1, sizeof(double));
  fb->q = (double*)calloc(tl ? tl : 1, sizeof(double));
  fb->k = (double*)calloc(tl ? tl : 1, sizeof(double));
  fb->v = (double*)calloc(tl ? tl : 1, sizeof(double));
  fb->r = (double*)calloc(tl ? tl : 1, sizeof(double));
  fb->o = (double*)calloc(tl ? tl : 1, sizeof(double));
  fb->s = (double*)calloc(th ? th : 1, sizeof(double));
  fb->g = (double*)calloc(th ? th : 1, sizeof(double));
  fb->den = (double*)calloc(th ? th : 1, sizeof(double));
  fb->rstd = (double*)calloc(th ? th : 1, sizeof(double));
  return fb->xt && fb->q && fb->k && fb->v && fb->r && fb->o && fb->s &&
         fb->g && fb->den && fb->rstd;
}

static void free_fwd(fwd_buffers* fb) {
  free(fb->xt); free(fb->q); free(fb->k); free(fb->v); free(fb->r);
  free(fb->o); free(fb->s); free(fb->g); free(fb->den); free(fb->rstd);
}

/*
 * GBLA layer forward.  y [T, H*dh].  Every intermediate pointer (xt, q, k, v,
 * r, s, g, o, den, state) may be NULL; when given it receives that tensor.
 * Returns 0, or -1 when memory runs out.
 */
int oracle_gbla_forward(int64_t T, int d, int H, int dh, int n_seq,
                        const int64_t* start, const int64_t* len,
                        const double* x, const double* conv_w,
                        const double* conv_b, const double* Wq,
                        const double* Wk, const double* Wv, const double* Wr,
                        const double* wg, const double* bg,
                        const double* gamma, int gate_mode, double eps,
                        double* y, double* xt, double* q, double* k, double* v,
                        double* r, double* s, double* g, double* o,
                        double* den, double* state) {
  fwd_buffers fb;
  if (!alloc_fwd(&fb, T, d, H, dh)) { free_fwd(&fb); return -1; }
  forward_into(T, d, H, dh, n_seq, start, len, x, conv_w, conv_b, Wq, Wk, Wv,
               Wr, wg, bg, gamma, gate_mode, eps, &fb, y, state);
  const size_t td = (size_t)T * d, tl = (size_t)T * H * dh, th = (size_t)T * H;
  if (xt) memcpy(xt, fb.xt, td * sizeof(double));
  if (q) memcpy(q, fb.q, tl * sizeof(double));
  if (k) memcpy(k, fb.k, tl * sizeof(double));
  if (v) memcpy(v, fb.v, tl * sizeof(double));
  if (r) memcpy(r, fb.r, tl * sizeof(double));
  if (o) memcpy(o, fb.o, tl * sizeof(double));
  if (s) memcpy(s, fb.s, th * sizeof(double));
  if (g) memcpy(g, fb.g, th * sizeof(double));
  if (den) memcpy(den, fb.den, th * sizeof(double));
  free_fwd(&fb);
  return 0;
}

/*
 * GBLA layer backward for the scalar <dy, y>.  Recomputes the forward, then
 * walks it in reverse:
 *   Eq. 7   u = o rstd, a = SiLU(r), y = u gamma a
 *           dgamma += dy u a;  dr = dy u gamma SiLU'(r);  du = dy gamma a
 *           do = rstd (du - u mean(du u))                       (RmsNorm)
 *   Eq. 5/6 the core backward (oracle_core_backward) -> dq, dk, dv, dg
 *   Eq. 5   sigmoid: ds = dg g (1 - g);  softmax: ds_j = g_j (dg_j - sum_l g_l dg_l)
 *           db_g = sum over tokens of ds
 *   Eq. 4   dx~ = dq W_Q^T + dk W_K^T + dv W_V^T + dr W_R^T + ds w_g^T
 *           dW_* = x~^T d*;  dw_g = x~^T ds
 *           conv: dx[l - 3 + t] += w[c, t] dx~[l];  dw[c, t] += x[l - 3 + t] dx~[l];
 *           db = sum dx~
 * Outputs may be NULL.  Returns 0, or -1 when memory runs out.
 */
int oracle_gbla_backward(int64_t T, int d, int H, int dh, int n_seq,
                         const int64_t* start, const int64_t* len,
                         const double* x, const double* conv_w,
                         const double* conv_b, const double* Wq,
                         const double* Wk, const double* Wv, const double* Wr,
                         const double* wg, const double* bg,
                         const double* gamma, int gate_mode, double eps,
                         const double* dy, double* dx, double* dconv_w,
                         double* dconv_b, double* dWq, double* dWk,
                         double* dWv, double* dWr, double* dwg, double* dbg,
                         double* dgamma) {
  const int64_t ld = (int64_t)H * dh;
  const size_t td = (size_t)T * d, tl = (size_t)T * ld, th = (size_t)T * H;
  fwd_buffers fb;
  double* y = (double*)calloc(tl ? tl : 1, sizeof(double));
  double* dO = (double*)calloc(tl ? tl : 1, sizeof(double));
  double* dq = (double*)calloc(tl ? tl : 1, sizeof(double));
  double* dk = (double*)calloc(tl ? tl : 1, sizeof(double));
  double* dv = (double*)calloc(tl ? tl : 1, sizeof(double));
  double* dr = (double*)calloc(tl ? tl : 1, sizeof(double));
  double* dg = (double*)calloc(th ? th : 1, sizeof(double));
  double* ds = (double*)calloc(th ? th : 1, sizeof(double));
  double* dxt = (double*)calloc(td ? td : 1, sizeof(double));
  double* dgam = (double*)calloc((size_t)dh, sizeof(double));
  int ok = alloc_fwd(&fb, T, d, H, dh) && y && dO && dq && dk && dv && dr &&
           dg && ds && dxt && dgam;
  if (ok) {
    forward_into(T, d, H, dh, n_seq, start, len, x, conv_w, conv_b, Wq, Wk, Wv,
                 Wr, wg, bg, gamma, gate_mode, eps, &fb, y, NULL);
    /* Eq. 7 backward */
    for (int b = 0; b < n_seq; ++b)
      for (int64_t t = start[b]; t < start[b] + len[b]; ++t)
        for (int h = 0; h < H; ++h) {
          const int64_t base = t * ld + h * dh;
          const double rs = fb.rstd[t * H + h];
          double du[1024], u[1024], mean = 0.0;
          for (int f = 0; f < dh; ++f) {
            const double gm = gamma ? gamma[f] : 1.0;
            const double a = silu(fb.r[base + f]);
            u[f] = fb.o[base + f] * rs;
            dgam[f] += dy[base + f] * u[f] * a;
            dr[base + f] = dy[base + f] * u[f] * gm * dsilu(fb.r[base + f]);
            du[f] = dy[base + f] * gm * a;
            mean += du[f] * u[f];
          }
          mean /= dh;
          for (int f = 0; f < dh; ++f) dO[base + f] = rs * (du[f] - u[f] * mean);
        }
    /* Eq. 5 / 6 backward */
    oracle_core_backward(T, H, dh, n_seq, start, len, fb.q, fb.k, fb.v, fb.g,
                         dO, dq, dk, dv, dg);
    /* Eq. 5 gate backward */
    for (int b = 0; b < n_seq; ++b)
      for (int h = 0; h < H; ++h) {
        double gdg = 0.0;
        for (int64_t t = start[b]; t < start[b] + len[b]; ++t)
          gdg += fb.g[t * H + h] * dg[t * H + h];
        for (int64_t t = start[b]; t < start[b] + len[b]; ++t) {
          const double gt = fb.g[t * H + h];
          ds[t * H + h] = gate_mode == 0 ? dg[t * H + h] * gt * (1.0 - gt)
                                         : gt * (dg[t * H + h] - gdg);
        }
      }
    /* Eq. 4 backward: projections */
    const double* Ws[4] = {Wq, Wk, Wv, Wr};
    const double* dPs[4] = {dq, dk, dv, dr};
    double* dWs[4] = {dWq, dWk, dWv, dWr};
    for (int b = 0; b < n_seq; ++b)
#pragma omp parallel for schedule(static)
      for (int64_t t = start[b]; t < start[b] + len[b]; ++t)
        for (int c = 0; c < d; ++c) {
          double acc = 0.0;
          for (int m = 0; m < 4; ++m)
            for (int j = 0; j < ld; ++j) acc += dPs[m][t * ld + j] * Ws[m][c * ld + j];
          for (int h = 0; h < H; ++h) acc += ds[t * H + h] * wg[c * H + h];
          dxt[t * d + c] = acc;
        }
    for (int m = 0; m < 4; ++m) {
      if (!dWs[m]) continue;
#pragma omp parallel for schedule(dynamic)
      for (int c = 0; c < d; ++c)
        for (int j = 0; j < ld; ++j) {
          double acc = 0.0;
          for (int b = 0; b < n_seq; ++b)
            for (int64_t t = start[b]; t < start[b] + len[b]; ++t)
              acc += fb.xt[t * d + c] * dPs[m][t * ld + j];
          dWs[m][c * ld + j] = acc;
        }
    }
    if (dwg)
      for (int c = 0; c < d; ++c)
        for (int h = 0; h < H; ++h) {
          double acc = 0.0;
          for (int b = 0; b < n_seq; ++b)
            for (int64_t t = start[b]; t < start[b] + len[b]; ++t)
              acc += fb.xt[t * d + c] * ds[t * H + h];
          dwg[c * H + h] = acc;
        }
    if (dbg)
      for (int h = 0; h < H; ++h) {
        double acc = 0.0;
        for (int b = 0; b < n_seq; ++b)
          for (int64_t t = start[b]; t < start[b] + len[b]; ++t) acc += ds[t * H + h];
        dbg[h] = acc;
      }
    if (dgamma) memcpy(dgamma, dgam, sizeof(double) * dh);
    /* Eq. 4 backward: conv */
    if (dx) memset(dx, 0, td * sizeof(double));
    if (dconv_w) memset(dconv_w, 0, sizeof(double) * d * 4);
    if (dconv_b) memset(dconv_b, 0, sizeof(double) * d);
    for (int b = 0; b < n_seq; ++b)
      for (int64_t l = 0; l < len[b]; ++l)
        for (int c = 0; c < d; ++c) {
          const double gl = dxt[(start[b] + l) * d + c];
          if (dconv_b) dconv_b[c] += gl;
          for (int t = 0; t < 4; ++t) {
            const int64_t src = l - 3 + t;
            if (src < 0) continue;
            if (dx) dx[(start[b] + src) * d + c] += conv_w[c * 4 + t] * gl;
            if (dconv_w) dconv_w[c * 4 + t] += x[(start[b] + src) * d + c] * gl;
          }
        }
  }
  free_fwd(&fb);
  free(y); free(dO); free(dq); free(dk); free(dv); free(dr); free(dg);
  free(ds); free(dxt); free(dgam);
  return ok ? 0 : -1;
}
