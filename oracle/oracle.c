/*
 * oracle.c -- plain, slow CPU reference for masked attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load this file; the library's GPU path never
 * does, and this file includes nothing from it.
 *
 * What it computes (the forward pass that all three pages speed up, and that
 * each of them keeps exact):
 *
 *     O = softmax(Q K^T / sqrt(d) + M) V,   M[i][j] = 0 if (i, j) allowed, else -inf
 *
 *   - Tessera abstract (arXiv 2609.25869): block-sparse attention computes only
 *     the blocks a logical mask selects, and the runtime changes how tiles run
 *     without dropping or adding any interaction the mask names, so the result
 *     is the masked softmax above.
 *   - Sparse VideoGen / Splash digest, "Splash Attention" section: empty tiles
 *     are skipped and exact coordinate masking is applied on boundary tiles, so
 *     the element-level mask is what is computed.
 *   - FG-Attn abstract: skipping happens at M x 1 slices (a block of M = 64
 *     queries times one key); a query attends exactly to the keys of its block's
 *     slice list.
 *
 * Every value is computed in fp64 from bf16 inputs widened exactly.  A row with
 * no allowed key returns O = 0 and lse = -inf.  Each row is done in two passes
 * over its allowed keys (maximum first, then the exponentials), which is the
 * textbook definition and not the streaming (online) form the GPU uses.
 *
 * The mask forms (readings of the pages, where they are silent):
 *   UNIFORM : allowed(i, j) = L[b][h][i / bq][j / bk]; the last logical block
 *             row / column is truncated at N, not padded.
 *   SEGMENTS: allowed(i, j) = L[b][h][seg_q(i)][seg_k(j)] for ascending bounds.
 *   SVG     : spatial head  -> frame(i) == frame(j) or frame(j) == 0
 *             temporal head -> |i mod S - j mod S| <= r (spatial index within
 *                              radius r of the query's; r = 0: the same index)
 *             with frame(t) = t / S, tokens in frame-major order (t = f*S + s).
 *             The oracle never permutes tokens.
 *   KEYLIST : allowed(i, j) = j is in the sorted key list of query block i / M.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#include "oracle_mask.h"

static int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

static double bf16_to_double(uint16_t x) {
  uint32_t bits = ((uint32_t)x) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* index of the segment [bounds[s], bounds[s+1]) holding t (bounds ascending) */
static int32_t find_segment(const int32_t *bounds, int32_t nseg, int32_t t) {
  int32_t lo = 0, hi = nseg - 1;
  while (lo < hi) {
    int32_t mid = (lo + hi + 1) / 2;
    if (bounds[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

/*
 * Write the allowed keys of row i of head (b, h) into keys[] in ascending
 * order and return how many there are.
 */
static int64_t allowed_keys(const oracle_mask *m, int32_t b, int32_t h, int32_t i,
                            int32_t *keys) {
  const int32_t N = m->N;
  int64_t n = 0;
  switch (m->kind) {
  case OR_UNIFORM: {
    const int64_t nqb = cdiv64(N, m->bq), nkb = cdiv64(N, m->bk);
    const uint8_t *row = m->blocks + (((int64_t)b * m->H + h) * nqb + i / m->bq) * nkb;
    for (int32_t j = 0; j < N; ++j)
      if (row[j / m->bk]) keys[n++] = j;
    break;
  }
  case OR_SEGMENTS: {
    const int32_t sq = find_segment(m->q_bounds, m->n_qseg, i);
    const uint8_t *row = m->blocks + (((int64_t)b * m->H + h) * m->n_qseg + sq) * m->n_kseg;
    for (int32_t j = 0; j < N; ++j)
      if (row[find_segment(m->k_bounds, m->n_kseg, j)]) keys[n++] = j;
    break;
  }
  case OR_SVG: {
    const int32_t S = m->frame_size;
    if (m->head_kind[h] == 0) {            /* spatial: same frame, or frame 0 */
      const int32_t fi = i / S;
      for (int32_t j = 0; j < N; ++j)
        if (j / S == fi || j / S == 0) keys[n++] = j;
    } else {                               /* temporal: spatial index within r */
      const int32_t si = i % S, r = m->temporal_radius;
      const int32_t lo = si - r < 0 ? 0 : si - r, hi = si + r > S - 1 ? S - 1 : si + r;
      for (int32_t f = 0; f * S < N; ++f)
        for (int32_t sj = lo; sj <= hi; ++sj) keys[n++] = f * S + sj;
    }
    break;
  }
  case OR_KEYLIST: {
    const int64_t nqb = cdiv64(N, m->slice_m);
    const int64_t r = ((int64_t)b * m->H + h) * nqb + i / m->slice_m;
    for (int64_t p = m->indptr[r]; p < m->indptr[r + 1]; ++p) {
      const int32_t j = m->indices[p];
      /* a list is a set of keys: ascending, no repeats, inside [0, N) */
      if (j < 0 || j >= N || (n > 0 && j <= keys[n - 1])) return -1;
      keys[n++] = j;
    }
    break;
  }
  default:
    return -1;
  }
  return n;
}

/*
 * One output row by the definition: two passes over the allowed keys.
 * probs (optional) receives the normalised probabilities in key order.
 */
static int attend_row(const oracle_mask *m, const uint16_t *q, const uint16_t *k,
                       const uint16_t *v, int32_t b, int32_t h, int32_t i,
                       double *out, double *lse, int32_t *keys, double *s,
                       double *qd, double *probs, int64_t *n_out) {
  const int32_t N = m->N, d = m->d;
  const int64_t head = ((int64_t)b * m->H + h) * N;
  const int64_t n = allowed_keys(m, b, h, i, keys);
  if (n_out) *n_out = n;
  for (int32_t c = 0; c < d; ++c) out[c] = 0.0;
  if (n < 0) return -1;
  if (n == 0) {
    *lse = -INFINITY;
    return 0;
  }
  for (int32_t c = 0; c < d; ++c) qd[c] = bf16_to_double(q[(head + i) * d + c]);
  const double scale = 1.0 / sqrt((double)d);
  double mx = -INFINITY;
  for (int64_t t = 0; t < n; ++t) {
    const uint16_t *kr = k + (head + keys[t]) * d;
    double dot = 0.0;
    for (int32_t c = 0; c < d; ++c) dot += qd[c] * bf16_to_double(kr[c]);
    s[t] = dot * scale;
    if (s[t] > mx) mx = s[t];
  }
  double l = 0.0;
  for (int64_t t = 0; t < n; ++t) {
    s[t] = exp(s[t] - mx);
    l += s[t];
  }
  for (int64_t t = 0; t < n; ++t) {
    const uint16_t *vr = v + (head + keys[t]) * d;
    const double p = s[t] / l;
    if (probs) probs[t] = p;
    for (int32_t c = 0; c < d; ++c) out[c] += p * bf16_to_double(vr[c]);
  }
  *lse = mx + log(l);
  return 0;
}

static int check_mask(const oracle_mask *m) {
  if (m->B <= 0 || m->H <= 0 || m->N < 0 || m->d <= 0) return -1;
  switch (m->kind) {
  case OR_UNIFORM: return (m->bq > 0 && m->bk > 0 && m->blocks) ? 0 : -1;
  case OR_SEGMENTS: return (m->n_qseg > 0 && m->n_kseg > 0 && m->q_bounds && m->k_bounds && m->blocks) ? 0 : -1;
  case OR_SVG: return (m->frame_size > 0 && m->n_frames > 0 && m->head_kind &&
                       m->temporal_radius >= 0 &&
                       (int64_t)m->frame_size * m->n_frames == m->N) ? 0 : -1;
  case OR_KEYLIST: return (m->slice_m > 0 && m->indptr && m->indices) ? 0 : -1;
  default: return -1;
  }
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Selected rows.  rows[r] = (b * H + h) * N + i.  out: [nrows][d], lse: [nrows],
 * counts (optional): [nrows] number of allowed keys.  Returns 0, or -1 on a bad
 * mask description or row id.
 */
int oracle_attention_rows(const oracle_mask *m, const uint16_t *q, const uint16_t *k,
                          const uint16_t *v, const int64_t *rows, int64_t nrows,
                          double *out, double *lse, int64_t *counts, int nthreads) {
  if (check_mask(m)) return -1;
  const int64_t total = (int64_t)m->B * m->H * m->N;
  for (int64_t r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= total) return -1;
  set_threads(nthreads);
  int bad = 0;
#pragma omp parallel
  {
    int32_t *keys = (int32_t *)malloc(sizeof(int32_t) * (size_t)(m->N > 0 ? m->N : 1));
    double *s = (double *)malloc(sizeof(double) * (size_t)(m->N > 0 ? m->N : 1));
    double *qd = (double *)malloc(sizeof(double) * (size_t)m->d);
    const int ok = keys && s && qd;
#pragma omp for schedule(dynamic, 16)
    for (int64_t r = 0; r < nrows; ++r) {
      const int64_t bh = rows[r] / m->N;
      const int32_t i = (int32_t)(rows[r] % m->N);
      if (!ok || attend_row(m, q, k, v, (int32_t)(bh / m->H), (int32_t)(bh % m->H), i,
                            out + r * m->d, lse + r, keys, s, qd, NULL,
                            counts ? counts + r : NULL)) {
#pragma omp atomic write
        bad = 1;
      }
    }
    free(keys);
    free(s);
    free(qd);
  }
  return bad ? -1 : 0;
}

/* Every row of every head.  out: [B][H][N][d], lse: [B][H][N]. */
int oracle_attention(const oracle_mask *m, const uint16_t *q, const uint16_t *k,
                     const uint16_t *v, double *out, double *lse, int nthreads) {
  if (check_mask(m)) return -1;
  const int64_t total = (int64_t)m->B * m->H * m->N;
  int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(total > 0 ? total : 1));
  if (!rows) return -1;
  for (int64_t r = 0; r < total; ++r) rows[r] = r;
  const int rc = oracle_attention_rows(m, q, k, v, rows, total, out, lse, NULL, nthreads);
  free(rows);
  return rc;
}

/* Probabilities of one row in ascending key order; returns the key count. */
int64_t oracle_probs_row(const oracle_mask *m, const uint16_t *q, const uint16_t *k,
                         const uint16_t *v, int32_t b, int32_t h, int32_t i,
                         int32_t *keys, double *probs, double *out, double *lse) {
  if (check_mask(m)) return -1;
  double *s = (double *)malloc(sizeof(double) * (size_t)(m->N > 0 ? m->N : 1));
  double *qd = (double *)malloc(sizeof(double) * (size_t)m->d);
  int64_t n = -1;
  if (s && qd && attend_row(m, q, k, v, b, h, i, out, lse, keys, s, qd, probs, &n)) n = -1;
  free(s);
  free(qd);
  return n;
}

/* Allowed keys of one row (ascending); returns the count, or -1. */
int64_t oracle_row_keys(const oracle_mask *m, int32_t b, int32_t h, int32_t i, int32_t *keys) {
  if (check_mask(m)) return -1;
  return allowed_keys(m, b, h, i, keys);
}

/*
 * |E| per (b, h): the number of allowed (query, key) pairs; per_bh: [B*H].
 * Returns the total, or -1.
 */
int64_t oracle_count_allowed(const oracle_mask *m, int64_t *per_bh, int nthreads) {
  if (check_mask(m)) return -1;
  set_threads(nthreads);
  const int64_t nbh = (int64_t)m->B * m->H;
  int64_t total = 0;
  for (int64_t bh = 0; bh < nbh; ++bh) per_bh[bh] = 0;
  int bad = 0;
#pragma omp parallel
  {
    int32_t *keys = (int32_t *)malloc(sizeof(int32_t) * (size_t)(m->N > 0 ? m->N : 1));
    for (int64_t bh = 0; bh < nbh; ++bh) {
      int64_t acc = 0;
#pragma omp for schedule(dynamic, 64)
      for (int32_t i = 0; i < m->N; ++i) {
        const int64_t n = keys ? allowed_keys(m, (int32_t)(bh / m->H), (int32_t)(bh % m->H), i, keys) : -1;
        if (n < 0) {
#pragma omp atomic write
          bad = 1;
        } else {
          acc += n;
        }
      }
#pragma omp atomic
      per_bh[bh] += acc;
    }
    free(keys);
  }
  if (bad) return -1;
  for (int64_t bh = 0; bh < nbh; ++bh) total += per_bh[bh];
  return total;
}
