/*
 * tsr.h -- C ABI of the GB300 block-sparse attention forward library
 *          (libtsr_gb300.so).
 *
 * The library computes, on one GPU,
 *
 *     O = softmax(Q K^T / sqrt(d) + M) V,      lse = log(sum_j exp(q.k_j / sqrt(d)))
 *
 * where M is 0 on the allowed (query, key) pairs of a mask and -inf elsewhere,
 * with the sum in lse running over the allowed keys only.  The mask comes in
 * one of four forms:
 *
 *   TSR_MASK_UNIFORM  a logical block mask over bq x bk blocks.  "Decoupling
 *                     Logical Masks from GPU Execution for Dynamic Block-Sparse
 *                     Attention" (Tessera), abstract: block-sparse attention
 *                     computes only the blocks that a logical mask selects.
 *   TSR_MASK_SEGMENTS the same with variable block boundaries (Tessera abstract:
 *                     logical block geometry differs from mask to mask).
 *   TSR_MASK_SVG      per-head spatial / temporal patterns ("Accelerating
 *                     Spatio-Temporal Attention for Video Diffusion on TPUs",
 *                     sections "Sparse VideoGen" and "Splash Attention").
 *   TSR_MASK_KEYLIST  M x 1 key slices: one sorted key list per block of M
 *                     queries ("FG-Attn: Leveraging Fine-Grained Sparsity In
 *                     Diffusion Transformers", abstract).
 *
 * Work is split in two calls, as in Tessera's runtime (abstract: a physical
 * mapping layer, a task organisation layer and profile-guided regime selection):
 *
 *   tsr_plan()         maps the logical mask onto 128-row physical tiles on the
 *                      GPU (retain / combine / subdivide), marks each tile full or
 *                      boundary, drops empty tiles, builds the per-query-tile work
 *                      lists in longest-first order and picks the regime from the
 *                      offline-profiled lookup table;
 *   tsr_bsa_forward()  runs the attention over the plan.
 *
 * Conventions for every entry point
 *   - All tensor and mask pointers are DEVICE pointers unless a comment says
 *     HOST.  The caller owns them; the library never frees them.
 *   - Q, K, V and O are bf16 [B][H][N][d] row-major (d contiguous) with
 *     d in {64, 128}; lse is fp32 [B][H][N].  Every base pointer must be
 *     16-byte aligned.  N = number of queries = number of keys.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is queued
 *     on it; inputs must stay valid until that work completes.
 *   - Functions return a tsr_status.  Nothing throws across the ABI.  On failure
 *     tsr_last_error() returns a message for the calling thread.
 *   - Argument errors are found on the host before anything is launched.
 */
#ifndef TSR_GB300_H
#define TSR_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TSR_ABI_VERSION 3

typedef enum {
  TSR_OK = 0,
  TSR_ERR_INVALID_ARG = 1,   /* bad shape, pointer, alignment or mask content      */
  TSR_ERR_UNSUPPORTED = 2,   /* valid, but outside what this build implements       */
  TSR_ERR_CUDA = 3,          /* a CUDA runtime / driver call failed                 */
  TSR_ERR_OOM = 4,           /* device or host allocation failed                    */
  TSR_ERR_TIMEOUT = 5,       /* a device-side wait gave up (kernel returned early)  */
  TSR_ERR_INTERNAL = 6       /* a device-side consistency check failed              */
} tsr_status;

typedef enum {
  TSR_MASK_UNIFORM = 0,
  TSR_MASK_SEGMENTS = 1,
  TSR_MASK_SVG = 2,
  TSR_MASK_KEYLIST = 3
} tsr_mask_kind;

typedef enum { TSR_HEAD_SPATIAL = 0, TSR_HEAD_TEMPORAL = 1 } tsr_head_kind;

/*
 * Logical mask and geometry.
 *
 * UNIFORM : blocks = uint8 [B][H][ceil(N/bq)][ceil(N/bk)], nonzero = allowed.
 *           allowed(i, j) = blocks[b][h][i / bq][j / bk].  The last block row and
 *           column are truncated at N.  bq, bk >= 16.
 * SEGMENTS: q_bounds = int32 [n_qseg + 1] ascending, q_bounds[0] = 0,
 *           q_bounds[n_qseg] = N (k_bounds likewise), each segment >= 16 tokens;
 *           blocks = uint8 [B][H][n_qseg][n_kseg];
 *           allowed(i, j) = blocks[b][h][seg_q(i)][seg_k(j)].
 * SVG     : head_kind = int8 [H] (tsr_head_kind), N = n_frames * frame_size,
 *           tokens frame-major (t = f * frame_size + s).
 *             spatial  head: allowed(i, j) = frame(i) == frame(j) || frame(j) == 0
 *             temporal head: allowed(i, j) = |i mod frame_size - j mod frame_size|
 *                                            <= temporal_radius
 *           (temporal_radius = 0: the same spatial index in every frame).
 *           Temporal heads run in temporal-major order (t' = s * n_frames + f):
 *           the attention kernel reads their Q/K/V rows through the inverse
 *           permutation and writes O and lse back in the caller's order; nothing
 *           is copied.  With temporal_radius = 0, n_frames <= 32 and no
 *           TSR_PLAN_TEMPORAL_TILES / TSR_PLAN_DEBUG_CHECKS, a temporal head is
 *           instead computed as frame_size independent n_frames x n_frames
 *           blocks (one per spatial index) by a kernel of its own (P rounded
 *           to bf16 for the P V product there too).  It runs on a stream the
 *           plan owns, forked from the call's stream before the attention
 *           launch and joined back into it after: work queued on the call's
 *           stream afterwards sees both kernels' results.
 *           Any n_frames >= 1; frame_size >= 16 when a head is
 *           spatial (a 128-token tile may hold at most 8 frames; smaller frames
 *           give TSR_ERR_UNSUPPORTED); temporal_radius >= 0.
 * KEYLIST : slice_m in {64, 128}.  indptr = int64 [B*H*ceil(N/slice_m) + 1] (CSR
 *           over (b, h, query block), indptr[0] = 0), indices = int32 keys, each
 *           list ascending, unique, in [0, N).  allowed(i, j) = j in the list of
 *           (b, h, i / slice_m).  Violations give TSR_ERR_INVALID_ARG.  indices
 *           may be NULL when every list is empty.
 *
 * The device arrays must stay valid until the work tsr_plan() queues completes.
 */
typedef struct {
  int32_t kind;              /* tsr_mask_kind */
  int32_t B, H, N, d;
  /* UNIFORM */
  int32_t bq, bk;
  /* SEGMENTS */
  int32_t n_qseg, n_kseg;
  const int32_t *q_bounds, *k_bounds;
  /* UNIFORM and SEGMENTS */
  const uint8_t *blocks;
  /* SVG */
  int32_t n_frames, frame_size;
  const int8_t *head_kind;
  /* KEYLIST */
  int32_t slice_m;
  const int64_t *indptr;
  const int32_t *indices;
  /* SVG temporal heads: spatial radius (ABI version 2) */
  int32_t temporal_radius;
} tsr_mask;

/* Plan options (pass NULL for defaults; zero fields mean "from the table"). */
typedef struct {
  int32_t bn;        /* 0 = from the regime table; 64 or 128 = force KV tile width   */
  int32_t stages;    /* 0 = from the regime table; else K/V pipeline depth (2..6)    */
  int32_t ctas_per_sm; /* 0 = from the regime table; 1 or 2                           */
  int32_t flags;     /* TSR_PLAN_* bits                                              */
  int32_t orient;    /* tile orientation (ABI version 3): 0 = from the regime table
                        (128-row tiles when stages or ctas_per_sm is set: those
                        are parameters of 128-row tiles), TSR_ORIENT_ROWS or
                        TSR_ORIENT_KEYS                                         */
  int32_t kv_split;  /* split-KV (ABI version 3): each work item's key tiles cut
                        into parts whose partial results the attention kernel
                        merges.  0 = automatic (a 128-row plan with fewer work
                        items than CTA slots is cut into 2 or 4 parts, until
                        every slot has one), 1 = never, 2 or 4 = that many parts.
                        tsr_attention_host and tsr_attention_noalloc split only
                        when asked (noalloc: never).  A split plan holds
                        n_items * kv_split * bm * d * 4 bytes of partial
                        results (fp32) in device memory             */
} tsr_plan_opts;

/* Physical tile orientations.
 *   TSR_ORIENT_ROWS  128 query rows x bn keys per tile: S = Q K^T with the
 *                    queries on the tensor core's M = 128 side.
 *   TSR_ORIENT_KEYS  64 query rows x 64 keys per tile, two tiles of a query
 *                    block's list computed together as S^T = K Q^T with 128 keys
 *                    on the M side and the 64 queries on the N side (d = 128).
 *                    A 64-row query block is never widened to 128 rows, so a
 *                    key block is computed only for the query blocks that need it. */
#define TSR_ORIENT_ROWS 1
#define TSR_ORIENT_KEYS 2

#define TSR_PLAN_SYNC_CHECK 1  /* tsr_bsa_forward synchronises and reads the device
                                  error word (slower; for debugging)               */
#define TSR_PLAN_NO_LPT     2  /* keep work items in (b, h, q-tile) order          */
#define TSR_PLAN_TEST_STALL 4  /* TEST ONLY: the attention kernel waits on a barrier
                                  that is never signalled, so its bounded-wait path
                                  runs: after 0.1 s it gives up, frees its resources
                                  and tsr_plan_device_status() returns
                                  TSR_ERR_TIMEOUT; the context stays usable      */
#define TSR_PLAN_DEBUG_CHECKS 8  /* after every tsr_plan / tsr_plan_update, a device
                                  pass checks every index of the plan (items,
                                  entries, descriptors, gathered keys; each query
                                  tile exactly once) and the call returns
                                  TSR_ERR_INTERNAL on a violation; every
                                  tsr_bsa_forward(_batch) also counts the tiles
                                  the kernel computed and compares them with the
                                  plan.  Both synchronise `stream`.  SVG temporal
                                  heads then run on the attention tiles.        */
#define TSR_PLAN_TEMPORAL_TILES 16  /* SVG temporal heads run on the attention tiles
                                  (temporal-major order) even where the
                                  per-position kernel could take them           */

typedef struct tsr_plan_s *tsr_plan_t;   /* opaque, library-owned */

/* Statistics of a plan (host copy). */
typedef struct {
  int32_t bm, bn, stages, ctas_per_sm;  /* chosen regime                           */
  int32_t gathered;                     /* 1 = KEYLIST gathered tiles              */
  int32_t n_temporal_heads;
  int64_t n_items;                      /* work items (one per 128-row query tile) */
  int64_t n_entries;                    /* physical K/V tiles over all items       */
  int64_t n_boundary;                   /* of which boundary (masked) tiles        */
  int64_t n_logical_on;                 /* allowed logical blocks / slices         */
  int64_t n_logical_total;
  int64_t max_item_len;
  int32_t regime_id;                    /* row of the regime table used (-1: opts) */
  int32_t orient;                       /* TSR_ORIENT_ROWS or TSR_ORIENT_KEYS       */
  int32_t kv_split;                     /* parts per work item (1 = not split)     */
  int32_t temporal_band;                /* 1: SVG temporal heads run one F x F block
                                           per spatial position, outside the
                                           attention tiles (their items stay in
                                           the plan and its export)              */
} tsr_plan_stats;

/*
 * tsr_plan -- physical mapping + task organisation + regime selection.
 *
 * Tessera abstract: a mapping layer turns logical blocks into physical tiles by
 * keeping them, merging several into one tile or cutting one into several; a
 * task layer groups tiles into GPU tasks for data reuse, parallelism and
 * copy/compute overlap; a table filled by offline profiling picks the execution
 * plan cheaply.  Splash digest, "Splash Attention": tiles with nothing to compute
 * are never loaded, and element-exact masking is applied on boundary tiles only.
 *
 * Runs as CUDA kernels on `stream`; synchronises `stream` to size the plan
 * (twice: for the mask's density, then for the tile counts; a re-plan whose
 * tile height is unchanged, once).  On success *out receives a new plan that
 * the caller must release with tsr_plan_destroy().  The plan owns device memory
 * (tiles, descriptors, work items, its work counter and, for SVG plans whose
 * temporal heads run by spatial position, a stream and two events) and may be
 * used by any number of tsr_bsa_forward() calls on the same device with
 * matching B, H, N, d, one after another (calls on different streams must be
 * ordered by the caller: they share the plan's work counter).
 */
tsr_status tsr_plan(const tsr_mask *mask, const tsr_plan_opts *opts, tsr_plan_t *out,
                    void *stream);

/*
 * tsr_plan_update -- rebuild an existing plan for a new mask with the same B, H,
 * N and d (any mask kind), reusing the plan's device storage; it grows only when
 * the new mask needs more tiles than any mask planned before.  Tessera abstract:
 * masks change from request to request, so planning cost is part of every call.
 * Same synchronisation and errors as tsr_plan(); on failure the plan must not be
 * used for tsr_bsa_forward until a later update succeeds.  The plan must not be
 * in use by queued tsr_bsa_forward work on another stream.
 */
tsr_status tsr_plan_update(tsr_plan_t plan, const tsr_mask *mask, void *stream);

/*
 * tsr_bsa_forward -- the attention over a plan.
 *
 * q, k, v: bf16 [B][H][N][d] (device).  out: bf16 [B][H][N][d] (device), lse:
 * fp32 [B][H][N] (device).  Every row of out and lse is written: rows with no
 * allowed key get O = 0 and lse = -inf.  out must not alias q, k or v.
 * Asynchronous on `stream` unless the plan was made with TSR_PLAN_SYNC_CHECK.
 * Device-side failures (a bounded wait that gave up) are reported by
 * tsr_plan_device_status().
 */
tsr_status tsr_bsa_forward(const void *q, const void *k, const void *v, tsr_plan_t plan,
                           void *out, float *lse, void *stream);

/*
 * tsr_bsa_forward_batch -- several BSA requests of possibly different shapes
 * (B, H, N, mask) in ONE persistent launch (Tessera abstract: speedups are
 * counted per BSA request; a serving step holds several).  Each request is
 * what tsr_bsa_forward takes: device q, k, v, out (bf16 [B][H][N][d]), lse
 * (fp32 [B][H][N]) and its own plan; the work items of all requests share one
 * scheduler, request after request, each request's longest first.
 * Requirements: 1 <= n <= 16; every plan on the current device, with the same
 * d, the same regime (bn, stages, ctas_per_sm -- plan the batch's masks with the
 * same tsr_plan_opts) and the same mask family (all KEYLIST or none); a plan
 * at most once per batch.  Otherwise TSR_ERR_INVALID_ARG / TSR_ERR_UNSUPPORTED
 * before any launch.  Device-side failures (a wait that timed out) go to the
 * error word of the first request's plan; tsr_plan_device_status on that plan
 * reports them.  The plans' storage must not be re-planned until the launch
 * has completed.
 */
typedef struct {
  const void *q, *k, *v;
  tsr_plan_t plan;
  void *out;
  float *lse;
} tsr_request;

tsr_status tsr_bsa_forward_batch(const tsr_request *reqs, int32_t n, void *stream);

/* Synchronise `stream` and return the plan's device error word as a status
   (TSR_OK, TSR_ERR_TIMEOUT or TSR_ERR_INTERNAL); clears it. */
tsr_status tsr_plan_device_status(tsr_plan_t plan, void *stream);

tsr_status tsr_plan_destroy(tsr_plan_t plan);

tsr_status tsr_plan_get_stats(tsr_plan_t plan, tsr_plan_stats *stats /* HOST */);

/*
 * tsr_plan_export -- copy the plan to HOST memory for inspection.
 * With host_buf == NULL sets *bytes to the size needed.  Otherwise *bytes must
 * hold the buffer size; it receives the bytes written.  Synchronises the plan's
 * stream.  Layout (little-endian):
 *
 *   tsr_export_header                              (80 bytes)
 *   tsr_plan_item   items[n_items]                 (32 bytes each)
 *   tsr_plan_entry  entries[n_entries]             (8 bytes each)
 *   tsr_tile_desc   descs[n_desc]                  (32 bytes each)
 *   int32_t         gidx[n_gidx]                   (gathered key indices)
 *   int8_t          head_layout[H]                 (0 caller order, 1 temporal-major)
 */
tsr_status tsr_plan_export(tsr_plan_t plan, void *host_buf, size_t *bytes);

typedef struct {
  char magic[4];              /* "TSRP" */
  int32_t version;            /* 1 */
  int32_t B, H, N, d;
  int32_t bm, bn;             /* query rows and key columns per physical tile      */
  int32_t gathered;           /* 0: entries are contiguous key ranges; 1: gathered */
  int32_t n_frames, frame_size;   /* temporal-major permutation (SVG), else 0      */
  int32_t slice_m;            /* KEYLIST query block size, else 0                  */
  int64_t n_items, n_entries, n_desc, n_gidx;
} tsr_export_header;          /* 80 bytes */

/*
 * A work item: all physical tiles of one 128-row query tile.
 *   q_tile  : rows [q_tile*bm, min(N, q_tile*bm + bm)) of head bh = b*H + h, in the
 *             head's layout (temporal-major for temporal SVG heads)
 *   begin/end: its entries are entries[begin .. end)
 *   layout  : 0 caller order, 1 temporal-major
 */
typedef struct {
  int32_t bh, q_tile, begin, end;
  int32_t layout, reserved0, reserved1, reserved2;
} tsr_plan_item;

/*
 * A physical K/V tile.  kv: first key of bn contiguous keys (gathered = 0), or the
 * offset into gidx of bn key indices (gathered = 1).  desc: -1 = full tile (all
 * bm x bn elements allowed and in range), else index of its boundary descriptor.
 */
typedef struct {
  int32_t kv, desc;
} tsr_plan_entry;

/*
 * Boundary descriptor (32 bytes).
 * Contiguous plans (grid form): rows [r_start[r], r_start[r+1]) of the tile form
 * row segment r (r < n_r, the last one ends at bm), columns [c_start[c],
 * c_start[c+1]) form column segment c (c < n_c); columns >= c_start[n_c] are out
 * of range.  Element (row, col) is allowed iff bit (r*8 + c) of `bits` is set.
 * Gathered plans (list form): n_r = bm / slice_m row segments of slice_m rows;
 * column c is allowed for row segment r iff bit c of colmask[r] is set.
 * Band form (temporal SVG heads; n_r = 0, n_c = 0, bits = F << 32 | R): with
 * row token t = q_tile * bm + row and key token k = entry key start + col, both
 * in temporal-major order, the element is allowed iff t < N, k < N and
 * |t / F - k / F| <= R (integer division).
 */
typedef struct {
  uint8_t n_r, n_c;
  uint8_t r_start[8];
  uint8_t c_start[9];
  uint8_t pad[5];
  uint64_t bits;
} tsr_tile_desc;

typedef struct {
  uint32_t colmask[2][4];
} tsr_tile_desc_list;

/*
 * tsr_temporal_permute -- the temporal-major token permutation on its own
 * (Splash digest, "Splash Attention": token memory permuted into temporal-major
 * order so the temporal pattern is contiguous).
 *
 * For every head h with head_kind[h] == TSR_HEAD_TEMPORAL (head_kind: HOST int8
 * [H]; NULL = all heads):
 *   inverse == 0: dst[b][h][s*F + f][:] = src[b][h][f*S + s][:]
 *   inverse != 0: dst[b][h][f*S + s][:] = src[b][h][s*F + f][:]
 * with F = n_frames, S = frame_size.  Rows of other heads are not touched.
 * src, dst: [B][H][F*S][row_bytes] (device, 16-byte aligned, row_bytes % 16 == 0),
 * must not overlap.
 */
tsr_status tsr_temporal_permute(const void *src, void *dst, int32_t B, int32_t H,
                                int32_t n_frames, int32_t frame_size, int32_t row_bytes,
                                const int8_t *head_kind, int32_t inverse, void *stream);

/*
 * tsr_svg_route -- route each head to the spatial or the temporal SVG pattern
 * from sampled queries (Sparse VideoGen digest, "Sparse VideoGen": heads are
 * assigned to a spatial or a temporal sparse pattern on the fly; the pages give
 * no criterion, this is the reading taken).
 *
 * For every (b, h) and every sampled query row i = samples[s] (tokens
 * frame-major, t = f * frame_size + s), the head's attention output is
 * computed under dense attention, the spatial pattern and the temporal pattern
 * (with temporal_radius), and
 *   stats[b][h][0] = sum_s |O_spatial(i)  - O_dense(i)|^2
 *   stats[b][h][1] = sum_s |O_temporal(i) - O_dense(i)|^2
 *   stats[b][h][2] = sum_s |O_dense(i)|^2
 * head_kind[h] = TSR_HEAD_TEMPORAL iff sum_b stats[b][h][1] < sum_b stats[b][h][0],
 * else TSR_HEAD_SPATIAL: usable as the head_kind of an SVG tsr_mask.
 *
 * q, k, v: device bf16 [B][H][n_frames * frame_size][d], d in {64, 128},
 * 16-byte aligned.  samples: HOST int32 [n_samples], 1 <= n_samples <= 1024,
 * each in [0, N) (the caller draws them; the same rows for every head).
 * stats: device fp32 [B][H][3], 16-byte aligned; head_kind: device int8 [H].
 * Both are written on `stream`.  fp32 arithmetic on CUDA cores; the sums are
 * accumulated with atomics, so their last bits vary from run to run.
 * Errors: TSR_ERR_INVALID_ARG for bad shapes, pointers or sample rows,
 * TSR_ERR_UNSUPPORTED for more than 1024 samples or N above 2^24.
 */
tsr_status tsr_svg_route(const void *q, const void *k, const void *v, int32_t B, int32_t H,
                         int32_t n_frames, int32_t frame_size, int32_t d, int32_t temporal_radius,
                         const int32_t *samples, int32_t n_samples, float *stats,
                         int8_t *head_kind, void *stream);

/*
 * tsr_attention_host -- one whole call from HOST memory: copies the mask arrays
 * and Q, K, V to the device, plans, runs the forward and copies O and lse back,
 * then synchronises.  Every pointer in `mask` and q, k, v, out, lse are HOST
 * pointers with the layouts above.  Device buffers are cached per thread between
 * calls (released by tsr_release_host_buffers()).  Heads are processed in
 * groups so that copy-in, attention and copy-out overlap; host buffers in
 * page-locked memory (cudaMallocHost, or pinned tensors) copy asynchronously,
 * pageable ones are staged by the driver and copy much more slowly.
 */
tsr_status tsr_attention_host(const tsr_mask *mask, const tsr_plan_opts *opts,
                              const void *q, const void *k, const void *v, void *out,
                              float *lse);

void tsr_release_host_buffers(void);

/*
 * tsr_attention_noalloc -- plan and attention in one call, with no device
 * allocation.  (The pages have no counterpart; this is a deployment aid.)
 *
 * For callers that cannot call cudaMalloc: code that must take every byte of
 * device memory from its own pool or budget (a server that reserved the GPU up
 * front, a framework whose allocator forbids raw cudaMalloc), and code on a
 * latency-critical path where cudaMalloc / cudaFree and the device-wide wait of
 * cudaFree are not acceptable.  The call plans into, and runs over, one scratch
 * array compiled into the library; the caller still passes q, k, v, out and lse
 * (device pointers, layouts as for tsr_bsa_forward) and the mask (device arrays,
 * UNIFORM or SEGMENTS only; other kinds give TSR_ERR_UNSUPPORTED).
 *
 *   - The scratch array is 32 MiB, held on every GPU that loads the library until
 *     the process exits.  A plan that does not fit (about 512 B + 56 B per
 *     128-row query tile + 8 B per kept tile + 32 B per boundary tile) is rejected
 *     with TSR_ERR_UNSUPPORTED before the attention runs; use tsr_plan() then.
 *   - All calls share the array and it keeps the last call's contents (the call
 *     clears what must start at zero).  Calls whose GPU work overlaps -- from two
 *     host threads or on two streams -- race on it and must be serialised.
 *   - The first call on a device looks up the array's device address, and does
 *     again whenever the calling thread's CUDA context has changed since (e.g.
 *     after cudaDeviceReset).
 *   - Every call synchronises `stream` (to size the plan, and at the end to read
 *     the device error word, returned as TSR_ERR_TIMEOUT / TSR_ERR_INTERNAL).
 *   - Plans 128-row tiles (TSR_ORIENT_ROWS) whatever the regime table picks, and
 *     never splits work items (kv_split 1).
 */
tsr_status tsr_attention_noalloc(const tsr_mask *mask, const void *q, const void *k,
                                 const void *v, void *out, float *lse, void *stream);

/*
 * Regime table (profile-guided regime selection, Tessera abstract).
 * tsr_regime_load reads a table file (text, one regime per line: kind bq bk
 * n_min n_max dens_min dens_max d bn stages ctas [orient], "*" = any; see the
 * file shipped next to the library); NULL reloads the built-in default.  A row
 * without the orient field names 128-row tiles (TSR_ORIENT_ROWS); a key-major
 * row (TSR_ORIENT_KEYS) must read d = 128, bn 64, stages 2, ctas 1, the one
 * key-major kernel.  A table naming a kernel variant that does not exist is
 * refused (TSR_ERR_INVALID_ARG) and the loaded table is kept.
 * tsr_regime_lookup returns the regime chosen for a mask class (d = 128).
 */
tsr_status tsr_regime_load(const char *path /* HOST, NULL = built-in */);

typedef struct {
  int32_t bn, stages, ctas_per_sm, id;
  int32_t orient;               /* TSR_ORIENT_ROWS or TSR_ORIENT_KEYS */
} tsr_regime;

tsr_status tsr_regime_lookup(int32_t kind, int32_t bq, int32_t bk, int32_t N,
                             double density, tsr_regime *out /* HOST */);

const char *tsr_status_string(tsr_status s);
const char *tsr_last_error(void);        /* thread-local; "" when none */
int32_t tsr_abi_version(void);           /* TSR_ABI_VERSION            */

#ifdef __cplusplus
}
#endif
#endif /* TSR_GB300_H */
