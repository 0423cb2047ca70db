/*
 * oracle_mask.h -- the oracle's description of a mask (TEST INFRASTRUCTURE ONLY).
 *
 * Shared by oracle.c (attention by the definition) and coverage.c (the plan
 * checker); nothing of the GPU library is included.  Field order and types
 * match the oracle's ctypes binding in __init__.py.
 */
#ifndef ORACLE_MASK_H
#define ORACLE_MASK_H
#include <stdint.h>

#define OR_UNIFORM 0
#define OR_SEGMENTS 1
#define OR_SVG 2
#define OR_KEYLIST 3

typedef struct {
  int32_t kind;
  int32_t B, H, N, d;
  /* UNIFORM */
  int32_t bq, bk;
  /* SEGMENTS */
  int32_t n_qseg, n_kseg;
  const int32_t *q_bounds, *k_bounds;
  /* UNIFORM and SEGMENTS: [B][H][rows][cols] of 0/1 */
  const uint8_t *blocks;
  /* SVG */
  int32_t n_frames, frame_size;
  const int8_t *head_kind;
  /* KEYLIST: CSR over (b, h, query block) */
  int32_t slice_m;
  const int64_t *indptr;
  const int32_t *indices;
  /* SVG temporal heads: spatial radius r >= 0 */
  int32_t temporal_radius;
} oracle_mask;

#endif
