/*
 * coverage.c -- checks an exported tile plan against the oracle's allowed set.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.c).  The export layout is decoded here
 * from its written description in the library's public header; no header or
 * code of the library is included.
 *
 * What is checked (Tessera abstract: the runtime keeps every interaction the
 * logical mask names; Splash digest, "Splash Attention": empty tiles are
 * skipped, exact masking only on boundary tiles):
 *   code 1  an allowed (query, key) pair that no tile computes
 *   code 2  a computed pair that the mask does not allow
 *   code 3  a pair computed more than once
 *   code 4  a "full" tile holding a pair that is not allowed or out of range
 *   code 5  a "boundary" tile whose every element is allowed and in range
 *           (it should have been marked full)
 *   code 6  a tile that computes nothing (an empty tile was kept)
 *   code 7  a query tile with no work item, or with more than one
 *   code 8  a malformed item or entry (index out of range)
 * Temporal-major heads (layout 1) are mapped back to caller order with
 * t = (t' mod F) * S + t' / F before comparison, i.e. the inverse of
 * t' = s * F + f for t = f * S + s.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#include "oracle_mask.h"

int64_t oracle_row_keys(const oracle_mask *m, int32_t b, int32_t h, int32_t i, int32_t *keys);

typedef struct {
  char magic[4];
  int32_t version;
  int32_t B, H, N, d;
  int32_t bm, bn;
  int32_t gathered;
  int32_t n_frames, frame_size;
  int32_t slice_m;
  int64_t n_items, n_entries, n_desc, n_gidx;
} exp_header;

typedef struct { int32_t bh, q_tile, begin, end, layout, r0, r1, r2; } exp_item;
typedef struct { int32_t kv, desc; } exp_entry;
typedef struct {
  uint8_t n_r, n_c;
  uint8_t r_start[8];
  uint8_t c_start[9];
  uint8_t pad[5];
  uint64_t bits;
} exp_desc_grid;
typedef struct { uint32_t colmask[2][4]; } exp_desc_list;

typedef struct {
  const exp_header *h;
  const exp_item *items;
  const exp_entry *entries;
  const uint8_t *descs;
  const int32_t *gidx;
  const int8_t *head_layout;
} plan_view;

static int32_t unpermute(int32_t tp, int32_t F, int32_t S) { return (tp % F) * S + tp / F; }

/* Is element (row r, column c) of a tile selected by the tile itself?  q0 is
   the item's first row in the head's layout. */
static int tile_allows(const plan_view *p, const exp_entry *e, int32_t q0, int32_t r, int32_t c) {
  if (e->desc < 0) return 1;
  if (p->h->gathered) {
    const exp_desc_list *d = (const exp_desc_list *)(p->descs + (size_t)e->desc * 32);
    const int seg = r / p->h->slice_m;
    return (d->colmask[seg][c >> 5] >> (c & 31)) & 1u;
  }
  const exp_desc_grid *d = (const exp_desc_grid *)(p->descs + (size_t)e->desc * 32);
  if (d->n_r == 0) {
    /* band form: segments of F tokens in the head's layout, |t / F - k / F| <= R */
    const int64_t F = (int64_t)(d->bits >> 32), R = (int64_t)(uint32_t)d->bits;
    const int64_t t = (int64_t)q0 + r, k = (int64_t)e->kv + c;
    if (F <= 0 || t >= p->h->N || k >= p->h->N) return 0;
    const int64_t dist = t / F - k / F;
    return (dist <= R && -dist <= R) ? 1 : 0;
  }
  if (c >= d->c_start[d->n_c]) return 0;
  int rs = 0, cs = 0;
  while (rs + 1 < d->n_r && d->r_start[rs + 1] <= r) ++rs;
  while (cs + 1 < d->n_c && d->c_start[cs + 1] <= c) ++cs;
  return (int)((d->bits >> (rs * 8 + cs)) & 1u);
}

static void report_add(int64_t *rep, int64_t max_report, int64_t *n_err, int64_t code,
                       int64_t b, int64_t h, int64_t i, int64_t j) {
  int64_t slot;
#pragma omp atomic capture
  slot = (*n_err)++;
  if (slot < max_report) {
    rep[slot * 5 + 0] = code;
    rep[slot * 5 + 1] = b;
    rep[slot * 5 + 2] = h;
    rep[slot * 5 + 3] = i;
    rep[slot * 5 + 4] = j;
  }
}

/*
 * Returns the number of failures (0 = plan is exact), or a negative code for a
 * malformed export.  stats (optional, 8 x int64): tiles, full tiles, boundary
 * tiles, computed elements (tile area over valid rows), covered elements,
 * allowed elements (oracle), items, 0.
 */
int64_t coverage_check(const oracle_mask *m, const uint8_t *buf, size_t len, int64_t *rep,
                       int64_t max_report, int64_t *stats, int nthreads) {
  if (len < sizeof(exp_header)) return -1;
  plan_view p;
  p.h = (const exp_header *)buf;
  const exp_header *h = p.h;
  if (memcmp(h->magic, "TSRP", 4) != 0 || h->version != 1) return -2;
  if (h->B != m->B || h->H != m->H || h->N != m->N) return -3;
  if (h->bm <= 0 || h->bn <= 0 || h->bn > 128 || h->bm > 128) return -4;
  const size_t need = sizeof(exp_header) + (size_t)h->n_items * sizeof(exp_item) +
                      (size_t)h->n_entries * sizeof(exp_entry) + (size_t)h->n_desc * 32 +
                      (size_t)h->n_gidx * 4 + (size_t)h->H;
  if (len < need) return -5;
  size_t off = sizeof(exp_header);
  p.items = (const exp_item *)(buf + off);
  off += (size_t)h->n_items * sizeof(exp_item);
  p.entries = (const exp_entry *)(buf + off);
  off += (size_t)h->n_entries * sizeof(exp_entry);
  p.descs = buf + off;
  off += (size_t)h->n_desc * 32;
  p.gidx = (const int32_t *)(buf + off);
  off += (size_t)h->n_gidx * 4;
  p.head_layout = (const int8_t *)(buf + off);
  if (h->gathered && (h->slice_m <= 0 || h->bm / h->slice_m > 2)) return -6;

#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  const int32_t N = h->N, BM = h->bm, BN = h->bn;
  const int32_t F = h->n_frames, S = h->frame_size;
  const int64_t nqt = (N + BM - 1) / BM, nbh = (int64_t)h->B * h->H;
  int64_t n_err = 0;
  int64_t st[8] = {0, 0, 0, 0, 0, 0, h->n_items, 0};

  /* every query tile exactly once */
  int32_t *seen = (int32_t *)calloc((size_t)(nbh * nqt > 0 ? nbh * nqt : 1), sizeof(int32_t));
  if (!seen) return -7;
  for (int64_t it = 0; it < h->n_items; ++it) {
    const exp_item *I = &p.items[it];
    if (I->bh < 0 || I->bh >= nbh || I->q_tile < 0 || I->q_tile >= nqt || I->begin < 0 ||
        I->end < I->begin || I->end > h->n_entries || (I->layout != 0 && I->layout != 1) ||
        (I->layout == 1 && (F <= 0 || S <= 0 || p.head_layout[I->bh % h->H] != 1))) {
      report_add(rep, max_report, &n_err, 8, it, 0, 0, 0);
      continue;
    }
    seen[I->bh * nqt + I->q_tile]++;
  }
  for (int64_t t = 0; t < nbh * nqt; ++t)
    if (seen[t] != 1) report_add(rep, max_report, &n_err, 7, t / nqt / h->H, (t / nqt) % h->H, (t % nqt) * BM, seen[t]);
  free(seen);
  if (n_err) {
    if (stats) memcpy(stats, st, sizeof st);
    return n_err;
  }

#pragma omp parallel
  {
    /* per item: allowed[r][j] from the oracle and cnt[r][j] from the tiles, both
       indexed by the caller-order key j */
    uint8_t *cnt = (uint8_t *)malloc((size_t)BM * (size_t)(N > 0 ? N : 1));
    uint8_t *allowed = (uint8_t *)malloc((size_t)BM * (size_t)(N > 0 ? N : 1));
    int32_t *keys = (int32_t *)malloc(sizeof(int32_t) * (size_t)(N > 0 ? N : 1));
    int64_t lst[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma omp for schedule(dynamic, 4)
    for (int64_t it = 0; it < h->n_items; ++it) {
      if (!cnt || !allowed || !keys) {
        report_add(rep, max_report, &n_err, 8, -1, 0, 0, 0);
        continue;
      }
      const exp_item *I = &p.items[it];
      const int32_t b = (int32_t)(I->bh / h->H), hh = (int32_t)(I->bh % h->H);
      const int32_t q0 = I->q_tile * BM;
      const int32_t R = (N - q0 < BM) ? N - q0 : BM;
      const int lay = I->layout;
      memset(cnt, 0, (size_t)R * (size_t)N);
      memset(allowed, 0, (size_t)R * (size_t)N);
      int bad_row = 0;
      for (int32_t r = 0; r < R; ++r) {
        const int32_t row_o = lay ? unpermute(q0 + r, F, S) : q0 + r;
        const int64_t nk = oracle_row_keys(m, b, hh, row_o, keys);
        if (nk < 0) { bad_row = 1; break; }
        lst[5] += nk;
        for (int64_t t = 0; t < nk; ++t) allowed[(size_t)r * N + keys[t]] = 1;
      }
      if (bad_row) {
        report_add(rep, max_report, &n_err, 8, b, hh, q0, -1);
        continue;
      }
      for (int32_t e = I->begin; e < I->end; ++e) {
        const exp_entry *E = &p.entries[e];
        if ((E->desc >= 0 && E->desc >= h->n_desc) ||
            (h->gathered && (E->kv < 0 || (int64_t)E->kv + BN > h->n_gidx)) ||
            (!h->gathered && (E->kv < 0 || E->kv >= N))) {
          report_add(rep, max_report, &n_err, 8, b, hh, q0, e);
          continue;
        }
        lst[0]++;
        if (E->desc < 0) lst[1]++; else lst[2]++;
        lst[3] += (int64_t)R * BN;
        int64_t sel = 0, valid_sel = 0;
        int full_bad = 0;
        for (int32_t r = 0; r < R; ++r) {
          const int32_t row_o = lay ? unpermute(q0 + r, F, S) : q0 + r;
          for (int32_t c = 0; c < BN; ++c) {
            const int64_t key = h->gathered ? (int64_t)p.gidx[E->kv + c] : (int64_t)E->kv + c;
            if (!tile_allows(&p, E, q0, r, c)) continue;
            ++sel;
            if (key < 0 || key >= N) {
              if (E->desc < 0) full_bad = 1;
              else report_add(rep, max_report, &n_err, 2, b, hh, row_o, key);
              continue;
            }
            ++valid_sel;
            const int32_t ko = lay ? unpermute((int32_t)key, F, S) : (int32_t)key;
            if (E->desc < 0 && !allowed[(size_t)r * N + ko]) full_bad = 1;
            uint8_t *cc = &cnt[(size_t)r * N + ko];
            if (*cc < 2) ++*cc;
          }
        }
        if (E->desc < 0 && full_bad) report_add(rep, max_report, &n_err, 4, b, hh, q0, e);
        if (E->desc >= 0 && valid_sel == 0) report_add(rep, max_report, &n_err, 6, b, hh, q0, e);
        if (E->desc >= 0 && sel == (int64_t)R * BN && valid_sel == sel)
          report_add(rep, max_report, &n_err, 5, b, hh, q0, e);
      }
      for (int32_t r = 0; r < R; ++r) {
        const int32_t row_o = lay ? unpermute(q0 + r, F, S) : q0 + r;
        const uint8_t *cr = cnt + (size_t)r * N, *ar = allowed + (size_t)r * N;
        for (int32_t j = 0; j < N; ++j) {
          const uint8_t c = cr[j];
          if (c) lst[4] += 1;
          if (ar[j] && c == 0) report_add(rep, max_report, &n_err, 1, b, hh, row_o, j);
          else if (!ar[j] && c) report_add(rep, max_report, &n_err, 2, b, hh, row_o, j);
          else if (c > 1) report_add(rep, max_report, &n_err, 3, b, hh, row_o, j);
        }
      }
    }
#pragma omp critical
    for (int q = 0; q < 6; ++q) st[q] += lst[q];
    free(cnt);
    free(allowed);
    free(keys);
  }
  if (stats) memcpy(stats, st, sizeof st);
  return n_err;
}
