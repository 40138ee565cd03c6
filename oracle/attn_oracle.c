/*
 * attn_oracle.c -- float64 CPU oracle for multi-head scaled dot-product
 * attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path
 * (the CUDA library) shares no code with it and never calls it.
 *
 * What it computes, per batch b, head h and query row i (0-based), is the
 * plain definition, with the whole row of scores materialised:
 *
 *   s_j  = scale * sum_t q[b,h,i,t] * k[b,h,j,t]       (eq. (1) of "Attention
 *          Is All You Need", section 3.2.1: the compatibility of the query
 *          with key j is their dot product, divided by sqrt(d_k); the caller
 *          passes scale = 1/sqrt(d_k))
 *   s_j  = -inf for every connection the mask forbids  (section 3.2.3 as read
 *          on "Lire << Attention Is All You Need >>": a forbidden connection
 *          is set to -inf before the softmax, so its weight is exactly 0)
 *            causal:       j > i            (a decoder position sees the
 *                                            positions up to and including
 *                                            itself, section 3.1 / 3.2.3)
 *            key padding:  j >= key_lens[b] (keys past each sequence's length)
 *   m    = max_j s_j
 *   w_j  = exp(s_j - m)                     (row softmax, each row sums to 1)
 *   Z    = sum_j w_j
 *   o[b,h,i,:] = sum_j w_j * v[b,h,j,:] / Z (weighted sum of the values,
 *                                            section 3.2)
 *   lse[b,h,i] = m + ln Z                   (natural log of the softmax
 *                                            normaliser of the scaled scores)
 *
 * A row in which every key is masked has no softmax; this oracle returns
 * o = 0 and lse = -inf for it.
 *
 * Inputs are float32 (bf16 values widen exactly into float32), the
 * arithmetic is float64 throughout.  Layout: q [B,H,n_q,d_k], k [B,H,n_k,d_k],
 * v [B,H,n_k,d_v], o [B,H,n_q,d_v], lse [B,H,n_q], all contiguous.
 *
 * Parity status: pinned (see tests/test_oracle.py): the worked sentence
 * example and the two-key softmax example printed on "Lire << Attention Is
 * All You Need >>" (section 3.2.1), closed forms, invariants and a
 * NumPy float64 cross-check.
 */
#include <math.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MASK_NONE 0
#define ORACLE_MASK_CAUSAL 1
#define ORACLE_MASK_KEY_PADDING 2
#define ORACLE_MASK_BAND 3 /* query i sees keys i - left .. i + right (restricted attention) */

/* One query row: scores, mask, softmax, weighted sum.  `s` is n_k doubles of
 * scratch owned by the calling thread. */
static void oracle_row(const float* q, const float* k, const float* v,
                       double* oi, double* lse_i, long H, long n_q,
                       long n_k, long d_k, long d_v, double scale,
                       int mask_kind, const int* key_lens, long row,
                       double* s) {
  long i = row % n_q;
  long bh = row / n_q;
  long b = bh / H;
  const float* qi = q + row * d_k;
  const float* kb = k + bh * n_k * d_k;
  const float* vb = v + bh * n_k * d_v;

  long limit = n_k;
  if (mask_kind == ORACLE_MASK_KEY_PADDING) {
    limit = key_lens[b];
    if (limit > n_k) limit = n_k;
    if (limit < 0) limit = 0;
  }

  double m = -INFINITY;
  for (long j = 0; j < n_k; ++j) {
    int forbidden = (j >= limit) || (mask_kind == ORACLE_MASK_CAUSAL && j > i);
    if (forbidden) {
      s[j] = -INFINITY;
      continue;
    }
    double dot = 0.0;
    for (long t = 0; t < d_k; ++t) dot += (double)qi[t] * (double)kb[j * d_k + t];
    s[j] = scale * dot;
    if (s[j] > m) m = s[j];
  }

  if (m == -INFINITY) { /* every key masked: no softmax for this row */
    for (long c = 0; c < d_v; ++c) oi[c] = 0.0;
    *lse_i = -INFINITY;
    return;
  }

  double Z = 0.0;
  for (long j = 0; j < n_k; ++j) {
    double w = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
    s[j] = w;
    Z += w;
  }
  for (long c = 0; c < d_v; ++c) {
    double acc = 0.0;
    for (long j = 0; j < n_k; ++j) acc += s[j] * (double)vb[j * d_v + c];
    oi[c] = acc / Z;
  }
  *lse_i = m + log(Z);
}

static int oracle_check(long B, long H, long n_q, long n_k, long d_k, long d_v,
                        int mask_kind, const int* key_lens) {
  if (B < 0 || H < 0 || n_q < 0 || n_k < 0 || d_k < 1 || d_v < 1) return -1;
  if (mask_kind < 0 || mask_kind > 2) return -1;
  if (mask_kind == ORACLE_MASK_KEY_PADDING && key_lens == NULL && B > 0) return -1;
  return 0;
}

/* Every row of every (b, h).  Returns 0, or -1 on bad arguments, -2 when
 * scratch cannot be allocated. */
int oracle_attn_fwd_f64(const float* q, const float* k, const float* v,
                        double* o, double* lse, long B, long H, long n_q,
                        long n_k, long d_k, long d_v, double scale,
                        int mask_kind, const int* key_lens, int n_threads) {
  if (oracle_check(B, H, n_q, n_k, d_k, d_v, mask_kind, key_lens)) return -1;
  long rows = B * H * n_q;
  int failed = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
#endif
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(n_k > 0 ? n_k : 1));
    if (s == NULL) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      failed = 1;
    }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 16)
#endif
    for (long r = 0; r < rows; ++r) {
      if (s != NULL)
        oracle_row(q, k, v, o + r * d_v, lse + r, H, n_q, n_k, d_k, d_v, scale,
                   mask_kind, key_lens, r, s);
    }
    free(s);
  }
  (void)n_threads;
  return failed ? -2 : 0;
}

/* Only the listed rows (flat index (b*H + h)*n_q + i); o_rows is
 * [n_rows, d_v], lse_rows [n_rows].  For sampled checks at sizes where the
 * full oracle would take too long. */
int oracle_attn_rows_f64(const float* q, const float* k, const float* v,
                         double* o_rows, double* lse_rows, long B, long H,
                         long n_q, long n_k, long d_k, long d_v, double scale,
                         int mask_kind, const int* key_lens, const long* rows,
                         long n_rows, int n_threads) {
  if (oracle_check(B, H, n_q, n_k, d_k, d_v, mask_kind, key_lens)) return -1;
  long total = B * H * n_q;
  for (long r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= total) return -1;
  int failed = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
#endif
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(n_k > 0 ? n_k : 1));
    if (s == NULL) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      failed = 1;
    }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
    for (long r = 0; r < n_rows; ++r) {
      if (s == NULL) continue;
      oracle_row(q, k, v, o_rows + r * d_v, lse_rows + r, H, n_q, n_k, d_k,
                 d_v, scale, mask_kind, key_lens, rows[r], s);
    }
    free(s);
  }
  (void)n_threads;
  return failed ? -2 : 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Backward of the same operation: the gradients of a scalar loss through
 * O = softmax(scale * Q K^T + M) V, given dO = dLoss/dO.  For each (b, h),
 * with P the row-softmax matrix recomputed here from q, k (float64):
 *
 *   dV = P^T dO
 *   dP = dO V^T
 *   D_i = sum_c dO[i,c] * O[i,c]      (= sum_j P[i,j] dP[i,j])
 *   dS = P (elementwise) (dP - D_i)   (the softmax Jacobian, row by row)
 *   dQ = scale * dS K,   dK = scale * dS^T Q
 *
 * Forbidden connections have P = 0, hence dS = 0 there; a row with no
 * visible key contributes nothing.  Inputs float32, arithmetic float64;
 * layout as the forward, dO [B,H,n_q,d_v], dq/dk/dv like q/k/v.
 * Returns 0, -1 on bad arguments, -2 when scratch cannot be allocated.
 */
static int bwd_core(const float* q, const float* k, const float* v, const float* dout,
                    double* dq, double* dk, double* dv, long B, long H, long n_q, long n_k,
                    long d_k, long d_v, double scale, int mask_kind, const int* key_lens,
                    long left, long right, int n_threads) {
  if (mask_kind == ORACLE_MASK_BAND) {
    if (B < 0 || H < 0 || n_q < 0 || n_k < 0 || d_k < 1 || d_v < 1 || left < 0 || right < 0)
      return -1;
  } else if (oracle_check(B, H, n_q, n_k, d_k, d_v, mask_kind, key_lens)) {
    return -1;
  }
  int failed = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (long bh = 0; bh < B * H; ++bh) {
    const long b = bh / H;
    const float* qb = q + bh * n_q * d_k;
    const float* kb = k + bh * n_k * d_k;
    const float* vb = v + bh * n_k * d_v;
    const float* gb = dout + bh * n_q * d_v;
    double* dqb = dq + bh * n_q * d_k;
    double* dkb = dk + bh * n_k * d_k;
    double* dvb = dv + bh * n_k * d_v;
    double* P = (double*)malloc(sizeof(double) * (size_t)(n_q * n_k > 0 ? n_q * n_k : 1));
    double* dS = (double*)malloc(sizeof(double) * (size_t)(n_q * n_k > 0 ? n_q * n_k : 1));
    if (P == NULL || dS == NULL) {
      free(P);
      free(dS);
#ifdef _OPENMP
#pragma omp atomic write
#endif
      failed = 1;
      continue;
    }
    long limit = n_k;
    if (mask_kind == ORACLE_MASK_KEY_PADDING) {
      limit = key_lens[b];
      if (limit > n_k) limit = n_k;
      if (limit < 0) limit = 0;
    }
    /* P: the row softmax of the masked, scaled scores */
    for (long i = 0; i < n_q; ++i) {
      double m = -INFINITY;
      for (long j = 0; j < n_k; ++j) {
        int forbidden = (j >= limit) || (mask_kind == ORACLE_MASK_CAUSAL && j > i) ||
                        (mask_kind == ORACLE_MASK_BAND && (j < i - left || j > i + right));
        double s = -INFINITY;
        if (!forbidden) {
          double dot = 0.0;
          for (long t = 0; t < d_k; ++t) dot += (double)qb[i * d_k + t] * (double)kb[j * d_k + t];
          s = scale * dot;
        }
        P[i * n_k + j] = s;
        if (s > m) m = s;
      }
      double Z = 0.0;
      for (long j = 0; j < n_k; ++j) {
        double w = (m == -INFINITY || P[i * n_k + j] == -INFINITY) ? 0.0 : exp(P[i * n_k + j] - m);
        P[i * n_k + j] = w;
        Z += w;
      }
      for (long j = 0; j < n_k; ++j) P[i * n_k + j] = Z > 0.0 ? P[i * n_k + j] / Z : 0.0;
    }
    /* dV = P^T dO */
    for (long j = 0; j < n_k; ++j)
      for (long c = 0; c < d_v; ++c) {
        double acc = 0.0;
        for (long i = 0; i < n_q; ++i) acc += P[i * n_k + j] * (double)gb[i * d_v + c];
        dvb[j * d_v + c] = acc;
      }
    /* dS = P * (dP - D), dP = dO V^T, D_i = sum_j P_ij dP_ij */
    for (long i = 0; i < n_q; ++i) {
      double D = 0.0;
      for (long j = 0; j < n_k; ++j) {
        double dp = 0.0;
        for (long c = 0; c < d_v; ++c) dp += (double)gb[i * d_v + c] * (double)vb[j * d_v + c];
        dS[i * n_k + j] = dp;
        D += P[i * n_k + j] * dp;
      }
      for (long j = 0; j < n_k; ++j) dS[i * n_k + j] = P[i * n_k + j] * (dS[i * n_k + j] - D);
    }
    /* dQ = scale dS K ; dK = scale dS^T Q */
    for (long i = 0; i < n_q; ++i)
      for (long t = 0; t < d_k; ++t) {
        double acc = 0.0;
        for (long j = 0; j < n_k; ++j) acc += dS[i * n_k + j] * (double)kb[j * d_k + t];
        dqb[i * d_k + t] = scale * acc;
      }
    for (long j = 0; j < n_k; ++j)
      for (long t = 0; t < d_k; ++t) {
        double acc = 0.0;
        for (long i = 0; i < n_q; ++i) acc += dS[i * n_k + j] * (double)qb[i * d_k + t];
        dkb[j * d_k + t] = scale * acc;
      }
    free(P);
    free(dS);
  }
  (void)n_threads;
  return failed ? -2 : 0;
}

/*
 * Restricted self-attention ("Lire << Attention Is All You Need >>", section
 * 4 and Table 1; the slide deck "Attention Is All You Need", Table 1: each
 * output position attends only to a neighbourhood of the input positions
 * around it).  Query i sees the keys j with  i - left <= j <= i + right
 * (left = right = w: a window of 2w + 1 positions centred on i; right = 0: a
 * causal window of the left + 1 most recent positions); every other
 * connection is -inf before the softmax.  Same definition otherwise as
 * oracle_row; a row with no key in its window gets o = 0, lse = -inf.
 */
static void oracle_band_row(const float* q, const float* k, const float* v, double* oi,
                            double* lse_i, long H, long n_q, long n_k, long d_k, long d_v,
                            double scale, long left, long right, long row, double* s) {
  long i = row % n_q;
  long bh = row / n_q;
  (void)H;
  const float* qi = q + (bh * n_q + i) * d_k;
  const float* kb = k + bh * n_k * d_k;
  const float* vb = v + bh * n_k * d_v;
  double m = -INFINITY;
  for (long j = 0; j < n_k; ++j) {
    int forbidden = (j < i - left) || (j > i + right);
    if (forbidden) {
      s[j] = -INFINITY;
      continue;
    }
    double dot = 0.0;
    for (long t = 0; t < d_k; ++t) dot += (double)qi[t] * (double)kb[j * d_k + t];
    s[j] = scale * dot;
    if (s[j] > m) m = s[j];
  }
  for (long c = 0; c < d_v; ++c) oi[c] = 0.0;
  if (m == -INFINITY) {
    *lse_i = -INFINITY;
    return;
  }
  double Z = 0.0;
  for (long j = 0; j < n_k; ++j) {
    if (s[j] == -INFINITY) continue;
    double w = exp(s[j] - m);
    Z += w;
    for (long c = 0; c < d_v; ++c) oi[c] += w * (double)vb[j * d_v + c];
  }
  for (long c = 0; c < d_v; ++c) oi[c] /= Z;
  *lse_i = m + log(Z);
}

/* Every row, or (rows != NULL) only the listed flat rows (b*H + h)*n_q + i.
 * left, right >= 0.  Returns 0, -1 on bad arguments, -2 when scratch cannot
 * be allocated. */
int oracle_attn_band_f64(const float* q, const float* k, const float* v, double* o, double* lse,
                         long B, long H, long n_q, long n_k, long d_k, long d_v, double scale,
                         long left, long right, const long* rows, long n_rows, int n_threads) {
  if (B < 0 || H < 0 || n_q < 1 || n_k < 1 || d_k < 1 || d_v < 1 || left < 0 || right < 0)
    return -1;
  const long total = rows ? n_rows : B * H * n_q;
  int failed = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
#endif
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)n_k);
    if (s == NULL) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      failed = 1;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 64)
#endif
      for (long x = 0; x < total; ++x) {
        long row = rows ? rows[x] : x;
        oracle_band_row(q, k, v, o + x * d_v, lse + x, H, n_q, n_k, d_k, d_v, scale, left, right,
                        row, s);
      }
      free(s);
    }
  }
  (void)n_threads;
  return failed ? -2 : 0;
}

/* The backward of the forward above (masks none, causal, key padding). */
int oracle_attn_bwd_f64(const float* q, const float* k, const float* v, const float* dout,
                        double* dq, double* dk, double* dv, long B, long H, long n_q,
                        long n_k, long d_k, long d_v, double scale, int mask_kind,
                        const int* key_lens, int n_threads) {
  if (mask_kind == ORACLE_MASK_BAND) return -1;
  return bwd_core(q, k, v, dout, dq, dk, dv, B, H, n_q, n_k, d_k, d_v, scale, mask_kind,
                  key_lens, 0, 0, n_threads);
}

/* The backward of restricted self-attention (oracle_attn_band_f64): the same
 * gradient with the window i - left <= j <= i + right as the mask. */
int oracle_attn_bwd_band_f64(const float* q, const float* k, const float* v, const float* dout,
                             double* dq, double* dk, double* dv, long B, long H, long n_q,
                             long n_k, long d_k, long d_v, double scale, long left, long right,
                             int n_threads) {
  return bwd_core(q, k, v, dout, dq, dk, dv, B, H, n_q, n_k, d_k, d_v, scale, ORACLE_MASK_BAND,
                  NULL, left, right, n_threads);
}
