/*
 * attn_oracle.c -- plain fp64 CPU attention: the correctness oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA path and must never be used as a
 * fallback for it.
 *
 * What it computes is the plain definition of scaled dot-product attention,
 * written out with no tiling, no online softmax and no reordering:
 *
 *   "Bloque C -- implementar la referencia" (lab 02 page, lynx-cortex
 *   phase-27 "Forward de flash attention en Triton"): S = Q K^T * sm_scale,
 *   masked entries set to -inf, P = softmax(S) row by row, O = P V;
 *   and the "standard attention" half of the worked example in
 *   "FlashAttention: Nunca materializar la matriz de atencion" (cruxr.ai,
 *   "Optimizaciones de Atencion"): the full score row, its maximum, the
 *   exponentials shifted by that maximum, their sum, the normalised weights
 *   and the weighted sum of V rows.
 *
 * Per query row i of head h in batch b (Q,O: B x Hq x Nq x d; K,V: B x Hkv x
 * Nk x d; all row-major):
 *   1. kvh = h / (Hq / Hkv)                       (consecutive GQA grouping)
 *   2. p   = Nk - Nq + i                           (bottom-right alignment)
 *   3. key j is live iff (!causal || j <= p) && (window <= 0 || p - j < window)
 *      (causal keeps j <= i, "position i attends to itself", lab 02 "Errores
 *       tipicos"; the sliding window keeps the last `window` tokens, motivation
 *       page "Otras tres variantes de attention")
 *   4. s_j = sm_scale * sum_k Q[b,h,i,k] K[b,kvh,j,k] for live j, -inf else
 *   5. M = max_j s_j, w_j = exp(s_j - M), l = sum_j w_j  (batch softmax)
 *   6. O[b,h,i,:] = sum_j (w_j / l) V[b,kvh,j,:]
 *   7. LSE[b,h,i] = M + ln(l)   (natural log of the sum of exp of the scaled,
 *      masked scores; lab 02 kernel skeleton stores m + log(l))
 * A row with no live key has no defined softmax; the oracle returns NaN for
 * its O and -inf for its LSE so that any comparison against it fails.
 *
 * Arithmetic is IEEE fp64 with the host libm's exp/log, compiled without
 * -ffast-math; rows run in parallel with OpenMP, each row sequentially.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ENOMEM -2

static int key_is_live(long p, long j, int causal, int window) {
  if (causal && j > p) return 0;
  if (window > 0 && p - j >= window) return 0;
  return 1;
}

/* One query row: q (d), Kh/Vh (Nk x d) of its kv head, scratch s (Nk). */
static void attend_one_row(const double *q, const double *Kh, const double *Vh,
                           long Nq, long Nk, long d, long i, int causal,
                           int window, double sm_scale, double *s, double *o,
                           double *lse) {
  const long p = Nk - Nq + i;
  double M = -INFINITY;
  for (long j = 0; j < Nk; ++j) {
    if (!key_is_live(p, j, causal, window)) {
      s[j] = -INFINITY;
      continue;
    }
    const double *k = Kh + j * d;
    double dot = 0.0;
    for (long c = 0; c < d; ++c) dot += q[c] * k[c];
    s[j] = sm_scale * dot;
    if (s[j] > M) M = s[j];
  }
  if (M == -INFINITY) { /* empty live set */
    for (long c = 0; c < d; ++c) o[c] = NAN;
    *lse = -INFINITY;
    return;
  }
  double l = 0.0;
  for (long j = 0; j < Nk; ++j) {
    const double w = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - M);
    s[j] = w;
    l += w;
  }
  for (long c = 0; c < d; ++c) o[c] = 0.0;
  for (long j = 0; j < Nk; ++j) {
    if (s[j] == 0.0) continue;
    const double pj = s[j] / l;
    const double *v = Vh + j * d;
    for (long c = 0; c < d; ++c) o[c] += pj * v[c];
  }
  *lse = M + log(l);
}

static int check_args(int B, int Hq, int Hkv, int Nq, int Nk, int d,
                      double sm_scale) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || d <= 0)
    return ORACLE_EINVAL;
  if (Hq % Hkv != 0) return ORACLE_EINVAL;
  if (!(sm_scale > 0.0) || isinf(sm_scale)) return ORACLE_EINVAL;
  return ORACLE_OK;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Full attention: every (b, h, i).  LSE may be NULL.  nthreads <= 0 uses the
 * OpenMP default.  Returns 0, or a negative code on bad arguments / no memory. */
int oracle_attn_fwd(const double *Q, const double *K, const double *V,
                    double *O, double *LSE, int B, int Hq, int Hkv, int Nq,
                    int Nk, int d, int causal, int window, double sm_scale,
                    int nthreads) {
  int rc = check_args(B, Hq, Hkv, Nq, Nk, d, sm_scale);
  if (rc) return rc;
  if (!Q || !K || !V || !O) return ORACLE_EINVAL;
  const long rows = (long)B * Hq * Nq;
  const int g = Hq / Hkv;
  int failed = 0;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(| : failed)
#endif
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)Nk);
    if (!s) {
      failed = 1;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 16)
#endif
      for (long r = 0; r < rows; ++r) {
        const long i = r % Nq;
        const long bh = r / Nq;
        const long h = bh % Hq;
        const long b = bh / Hq;
        const long kvh = h / g;
        const double *Kh = K + ((b * Hkv + kvh) * (long)Nk) * d;
        const double *Vh = V + ((b * Hkv + kvh) * (long)Nk) * d;
        double lse;
        attend_one_row(Q + r * d, Kh, Vh, Nq, Nk, d, i, causal, window,
                       sm_scale, s, O + r * d, &lse);
        if (LSE) LSE[r] = lse;
      }
      free(s);
    }
  }
  return failed ? ORACLE_ENOMEM : ORACLE_OK;
}

/* Selected rows only.  row_ids[n] is the flat index (b*Hq + h)*Nq + i of a
 * query row; Qrows holds those rows' Q vectors (n x d), in the same order.
 * O (n x d) and LSE (n) receive the results. */
int oracle_attn_rows(const double *Qrows, const int64_t *row_ids, long n,
                     const double *K, const double *V, double *O, double *LSE,
                     int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                     int window, double sm_scale, int nthreads) {
  int rc = check_args(B, Hq, Hkv, Nq, Nk, d, sm_scale);
  if (rc) return rc;
  if (!Qrows || !row_ids || !K || !V || !O || n < 0) return ORACLE_EINVAL;
  const long rows = (long)B * Hq * Nq;
  for (long t = 0; t < n; ++t)
    if (row_ids[t] < 0 || row_ids[t] >= rows) return ORACLE_EINVAL;
  const int g = Hq / Hkv;
  int failed = 0;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(| : failed)
#endif
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)Nk);
    if (!s) {
      failed = 1;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
      for (long t = 0; t < n; ++t) {
        const long r = (long)row_ids[t];
        const long i = r % Nq;
        const long bh = r / Nq;
        const long h = bh % Hq;
        const long b = bh / Hq;
        const long kvh = h / g;
        const double *Kh = K + ((b * Hkv + kvh) * (long)Nk) * d;
        const double *Vh = V + ((b * Hkv + kvh) * (long)Nk) * d;
        double lse;
        attend_one_row(Qrows + t * d, Kh, Vh, Nq, Nk, d, i, causal, window,
                       sm_scale, s, O + t * d, &lse);
        if (LSE) LSE[t] = lse;
      }
      free(s);
    }
  }
  return failed ? ORACLE_ENOMEM : ORACLE_OK;
}

/* Paged K/V cache (motivation page, "PagedAttention es un problema
 * distinto": the cache is a pool of fixed-size pages and each request has a
 * page table naming, in order, the pages that hold its tokens).  The
 * request's keys are first gathered through its table into a flat array,
 * then each row is the plain definition above with that request's own key
 * count n_b = seq_lens[b]:
 *   token t of request b = pool page table[b * max_pages + t / page_size],
 *   slot t % page_size;   pool layout (num_pages, Hkv, page_size, d).
 * Query row i of request b sits at position n_b - Nq + i (step 2 with Nk =
 * n_b).  Only the first ceil(n_b / page_size) table entries and the first
 * n_b slots are read.  Returns ORACLE_EINVAL when a length is outside [1,
 * max_pages * page_size] or a table entry that is read lies outside the
 * pool. */
int oracle_attn_paged(const double *Q, const double *Kpool, const double *Vpool,
                      const int32_t *table, const int32_t *seq_lens, double *O,
                      double *LSE, int B, int Hq, int Hkv, int Nq, int d,
                      int page_size, int num_pages, int max_pages, int causal,
                      int window, double sm_scale, int nthreads) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || d <= 0 || Hq % Hkv != 0)
    return ORACLE_EINVAL;
  if (page_size <= 0 || num_pages <= 0 || max_pages <= 0) return ORACLE_EINVAL;
  if (!(sm_scale > 0.0) || isinf(sm_scale)) return ORACLE_EINVAL;
  if (!Q || !Kpool || !Vpool || !table || !seq_lens || !O) return ORACLE_EINVAL;
  long max_len = 0;
  for (int b = 0; b < B; ++b) {
    const long n = seq_lens[b];
    if (n < 1 || n > (long)max_pages * page_size) return ORACLE_EINVAL;
    for (long j = 0; j < (n + page_size - 1) / page_size; ++j) {
      const int32_t pg = table[(long)b * max_pages + j];
      if (pg < 0 || pg >= num_pages) return ORACLE_EINVAL;
    }
    if (n > max_len) max_len = n;
  }
  const int g = Hq / Hkv;
  int failed = 0;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(| : failed)
#endif
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)max_len);
    double *Kh = (double *)malloc(sizeof(double) * (size_t)max_len * d);
    double *Vh = (double *)malloc(sizeof(double) * (size_t)max_len * d);
    if (!s || !Kh || !Vh) {
      failed = 1;
    } else {
      /* one (request, query head) per iteration: gather its kv head's keys
       * and values in token order, then attend each of its Nq rows */
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
      for (long bh = 0; bh < (long)B * Hq; ++bh) {
        const long b = bh / Hq, h = bh % Hq, kvh = h / g;
        const long n = seq_lens[b];
        for (long t = 0; t < n; ++t) {
          const long pg = table[b * max_pages + t / page_size];
          const long src = ((pg * Hkv + kvh) * page_size + t % page_size) * (long)d;
          for (long c = 0; c < d; ++c) {
            Kh[t * d + c] = Kpool[src + c];
            Vh[t * d + c] = Vpool[src + c];
          }
        }
        for (long i = 0; i < Nq; ++i) {
          const long r = bh * Nq + i;
          double lse;
          attend_one_row(Q + r * d, Kh, Vh, Nq, n, d, i, causal, window, sm_scale,
                         s, O + r * d, &lse);
          if (LSE) LSE[r] = lse;
        }
      }
    }
    free(s);
    free(Kh);
    free(Vh);
  }
  return failed ? ORACLE_ENOMEM : ORACLE_OK;
}

/* Gradients of the forward definition above (the pages keep the LSE "for
 * the backward pass" and leave the backward itself for later; what it
 * computes is fixed by the forward: the chain rule through steps 4-6).  For
 * a loss with dO = dL/dO, per query row i of head h (kv head kvh), with the
 * row's normalised weights P_ij (0 for masked keys) from steps 4-5:
 *   dV[kvh,j]  += P_ij dO_i                       (step 6 is linear in V)
 *   dP_ij       = dO_i . V[kvh,j]
 *   dS_ij       = P_ij (dP_ij - sum_k P_ik dP_ik)  (softmax Jacobian)
 *   dQ_i        = sm_scale sum_j dS_ij K[kvh,j]    (step 4)
 *   dK[kvh,j]  += sm_scale dS_ij Q_i
 * dK and dV of a kv head sum over the query heads of its group.  Q, dO, dQ:
 * B x Hq x Nq x d; K, V, dK, dV: B x Hkv x Nk x d.  Every row must have a
 * live key (the forward's R4 reading); rows without one return
 * ORACLE_EINVAL.  Serial over heads (dK/dV accumulate across a group). */
int oracle_attn_bwd(const double *Q, const double *K, const double *V,
                    const double *dO, double *dQ, double *dK, double *dV,
                    int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                    int window, double sm_scale) {
  int rc = check_args(B, Hq, Hkv, Nq, Nk, d, sm_scale);
  if (rc) return rc;
  if (!Q || !K || !V || !dO || !dQ || !dK || !dV) return ORACLE_EINVAL;
  const int g = Hq / Hkv;
  double *p = (double *)malloc(sizeof(double) * (size_t)Nk);
  double *dp = (double *)malloc(sizeof(double) * (size_t)Nk);
  if (!p || !dp) {
    free(p);
    free(dp);
    return ORACLE_ENOMEM;
  }
  for (long x = 0; x < (long)B * Hkv * Nk * d; ++x) dK[x] = dV[x] = 0.0;
  rc = ORACLE_OK;
  for (long b = 0; b < B && rc == ORACLE_OK; ++b) {
    for (long h = 0; h < Hq && rc == ORACLE_OK; ++h) {
      const long kvh = h / g;
      const double *Kh = K + ((b * Hkv + kvh) * (long)Nk) * d;
      const double *Vh = V + ((b * Hkv + kvh) * (long)Nk) * d;
      double *dKh = dK + ((b * Hkv + kvh) * (long)Nk) * d;
      double *dVh = dV + ((b * Hkv + kvh) * (long)Nk) * d;
      for (long i = 0; i < Nq; ++i) {
        const long r = (b * Hq + h) * (long)Nq + i;
        const double *q = Q + r * d, *go = dO + r * d;
        double *gq = dQ + r * d;
        const long pos = Nk - Nq + i;
        /* steps 4-5: the row's weights */
        double M = -INFINITY;
        for (long j = 0; j < Nk; ++j) {
          if (!key_is_live(pos, j, causal, window)) {
            p[j] = -INFINITY;
            continue;
          }
          double dot = 0.0;
          for (long c = 0; c < d; ++c) dot += q[c] * Kh[j * d + c];
          p[j] = sm_scale * dot;
          if (p[j] > M) M = p[j];
        }
        if (M == -INFINITY) {
          rc = ORACLE_EINVAL;
          break;
        }
        double l = 0.0;
        for (long j = 0; j < Nk; ++j) {
          p[j] = (p[j] == -INFINITY) ? 0.0 : exp(p[j] - M);
          l += p[j];
        }
        for (long j = 0; j < Nk; ++j) p[j] /= l;
        /* dP and its P-weighted row sum */
        double Dsum = 0.0;
        for (long j = 0; j < Nk; ++j) {
          if (p[j] == 0.0) {
            dp[j] = 0.0;
            continue;
          }
          double dot = 0.0;
          for (long c = 0; c < d; ++c) dot += go[c] * Vh[j * d + c];
          dp[j] = dot;
          Dsum += p[j] * dot;
        }
        for (long c = 0; c < d; ++c) gq[c] = 0.0;
        for (long j = 0; j < Nk; ++j) {
          if (p[j] == 0.0) continue;
          const double ds = p[j] * (dp[j] - Dsum);
          for (long c = 0; c < d; ++c) {
            dVh[j * d + c] += p[j] * go[c];
            gq[c] += sm_scale * ds * Kh[j * d + c];
            dKh[j * d + c] += sm_scale * ds * q[c];
          }
        }
      }
    }
  }
  free(p);
  free(dp);
  return rc;
}
