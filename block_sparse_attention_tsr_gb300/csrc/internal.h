// internal.h -- library-private declarations shared by the .cu files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <string>
#include <vector>

#include "../../include/tsr.h"

namespace tsr {

constexpr int kBM = 128;  // query rows per physical tile (the tcgen05 M = 128 datapath)

void set_error(const std::string& msg);
const char* last_error_cstr();
tsr_status fail(tsr_status s, const std::string& msg);
tsr_status cuda_fail(cudaError_t e, const char* what);

#define TSR_CUDA(expr)                                  \
  do {                                                  \
    cudaError_t e_ = (expr);                            \
    if (e_ != cudaSuccess) return cuda_fail(e_, #expr); \
  } while (0)

// Logical mask as the planner kernels see it (device pointers).
struct MaskDev {
  int32_t kind, B, H, N;
  int32_t bq, bk;
  int32_t n_qseg, n_kseg;
  const int32_t* q_bounds;
  const int32_t* k_bounds;
  const uint8_t* blocks;
  int32_t F, S;
  int32_t R;                 // SVG temporal radius
  const int8_t* head_kind;   // device copy, [H]
  int32_t slice_m;
  const int64_t* indptr;
  const int32_t* indices;
};

struct Regime {
  int32_t bn, stages, ctas, id;
  int32_t orient = TSR_ORIENT_ROWS;   // TSR_ORIENT_ROWS or TSR_ORIENT_KEYS
};

// Query rows per physical tile of an orientation.
constexpr int32_t bm_of(int32_t orient) { return orient == TSR_ORIENT_KEYS ? 64 : kBM; }

// A grow-only device buffer owned by a plan.
struct DevBuf {
  void* p = nullptr;
  size_t cap = 0;
};

struct tsr_plan_impl {
  int device = 0;
  int32_t B = 0, H = 0, N = 0, d = 0;
  int32_t kind = 0;
  int32_t bn = 128, stages = 3, ctas = 1, regime_id = -1;
  int32_t orient = TSR_ORIENT_ROWS, bm = kBM;   // tile orientation and query rows per tile
  int32_t gathered = 0, slice_m = 0;
  int32_t F = 0, S = 0, R = 0;
  int32_t flags = 0;
  int64_t n_items = 0, n_entries = 0, n_desc = 0, n_gidx = 0;
  int64_t n_logical_on = 0, n_logical_total = 0, max_item_len = 0;
  std::vector<int8_t> head_layout;  // host copy: 1 = temporal-major
  int32_t n_temporal = 0;
  int32_t group_heads = 0;    // > 0: heads per longest-first scheduling group (else sized for L2)
  // split-KV: each work item's tile list cut into kv_split parts (1 = off); the
  // parts are the launch's work units, written to `units` in item order
  int32_t kv_split = 1;
  void* units = nullptr;      // tsr_plan_item [n_launch * kv_split] (kv_split > 1)
  // SVG temporal heads of radius 0 with at most 32 frames run as one F x F block
  // per spatial position (svg_temporal.cu); the attention kernels then take the
  // spatial heads' items only: `launch`, the items without the temporal heads'
  // in their scheduled order.  Otherwise launch = items, n_launch = n_items.
  int32_t temporal_band = 0;
  void* launch = nullptr;
  int64_t n_launch = 0;
  std::vector<int64_t> spatial_before;   // [B*H + 1]: spatial heads among bh < i
  // the per-position kernel's stream, forked from the caller's stream before
  // the attention launch and joined after it (created with the first such plan)
  cudaStream_t band_stream = nullptr;
  cudaEvent_t band_fork = nullptr, band_join = nullptr;
  // device buffers (owned)
  void* items = nullptr;     // tsr_plan_item [n_items]
  void* entries = nullptr;   // tsr_plan_entry [n_entries]
  void* descs = nullptr;     // 32 B [n_desc]
  int32_t* gidx = nullptr;   // [n_gidx]
  int32_t* counter = nullptr;
  uint32_t* err = nullptr;
  int8_t* head_kind_dev = nullptr;
  // storage reused when the plan is rebuilt for a new mask (tsr_plan_update)
  DevBuf b_items, b_entries, b_descs, b_cnt, b_tot, b_ebegin, b_dbegin, b_hist, b_gidx;
  // split-KV storage: units, each unit's partial O (fp32 [bm][d]) and lse (base 2,
  // [bm]), one arrival counter per work item
  DevBuf b_units, b_part_o, b_part_lse, b_part_cnt;
  DevBuf b_launch;
  unsigned long long* host_tot = nullptr;   // pinned: 8 totals + the error word
  int8_t* host_kinds = nullptr;             // pinned: SVG head kinds, read after the count sync
  bool has_opts = false;
  tsr_plan_opts opts{};
};

// Make `b` hold at least `bytes` (contents are not preserved when it grows).
tsr_status devbuf_reserve(DevBuf& b, size_t bytes);
void devbuf_free(DevBuf& b);

// planner (plan.cu)
tsr_status plan_build(const tsr_mask* mask, const tsr_plan_opts* opts, tsr_plan_impl* P,
                      cudaStream_t stream);

tsr_status plan_build_keylist(const tsr_mask* mask, const tsr_plan_opts* opts, tsr_plan_impl* P,
                              cudaStream_t stream);
tsr_status plan_schedule_into(const int32_t* cnt_e, const int32_t* cnt_b, int64_t n_items,
                              int32_t nqt, int32_t H, int32_t lpt, int32_t max_len,
                              int32_t group_heads, int32_t* ebegin, int32_t* dbegin,
                              int32_t* hist, void* items, cudaStream_t stream);
// Heads per longest-first scheduling group: as many (b, h) as keep their K and
// V (plus extra_per_head bytes that stream through L2 with them, e.g. gathered
// key indices) within ~96 MB of the L2.
int32_t heads_per_group(int32_t N, int32_t d, int64_t n_heads, double extra_per_head = 0.0);
tsr_status plan_count_into(const MaskDev& m, int32_t nqt, int32_t* cnt, unsigned long long* tot,
                           uint32_t* err, int64_t n_grid, cudaStream_t stream);
tsr_status plan_finish_into(const MaskDev& m, int32_t nqt, int32_t bn, const int32_t* cnt_e,
                            const int32_t* cnt_b, int32_t max_len, int32_t* ebegin,
                            int32_t* dbegin, int32_t* hist, void* items, void* entries,
                            void* descs, cudaStream_t stream);

// The attention launch list (plan.cu): the spatial heads' items when the SVG
// temporal heads go to the per-position kernel, else the items themselves.
tsr_status plan_launch_list(tsr_plan_impl* P, cudaStream_t stream);

// split-KV (plan.cu): the number of parts per work item (the caller's
// opts->kv_split, else enough parts for about eight work units per CTA slot,
// at most 4), and the units and partial-result storage of a split plan
tsr_status plan_split(tsr_plan_impl* P, const tsr_plan_opts* opts, cudaStream_t stream);

// device-side plan consistency checks (check.cu)
tsr_status plan_check(const tsr_plan_impl* P, cudaStream_t stream);

// forward kernels (fwd.cu)
struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* lse;
  const tsr_plan_impl* plan;
  // Work items [item_lo, item_hi) of the plan (item_hi < 0: all of them), and
  // the launch's own work counter (null: the plan's).  Launches of one plan
  // that may run at the same time need disjoint item ranges and their own
  // counters, and no debug tile counting.
  int64_t item_lo = 0, item_hi = -1;
  int32_t* counter = nullptr;
};
tsr_status launch_forward(const FwdArgs& a, cudaStream_t stream);
// Up to 16 requests in one launch (same d, regime and mask family).
tsr_status launch_forward_batch(const FwdArgs* reqs, int n_req, cudaStream_t stream);
bool variant_exists(int d, int bn, int stages, int ctas, bool gathered);
bool variant_pick(int d, bool gathered, int bn, int stages, int ctas, int* out_bn, int* out_st,
                  int* out_ct);
// The regime for a plan: the table's choice, with the caller's overrides (opts
// fields that are nonzero) taking precedence; completed to a compiled variant.
tsr_status resolve_regime(Regime table, const tsr_plan_opts* opts, int d, bool gathered,
                          Regime* out);

// SVG head routing (route.cu)
tsr_status launch_route(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                        int32_t F, int32_t S, int32_t d, int32_t R, const int32_t* samples,
                        int32_t n_samples, float* stats, int8_t* head_kind, cudaStream_t stream);

// SVG temporal heads, one F x F block per spatial position (svg_temporal.cu):
// radius 0, 1 <= F <= 32, d in {64, 128}.  Heads bh in [bh_lo, bh_hi) whose kind
// is temporal; the others are left alone.
bool svg_temporal_eligible(int32_t F, int32_t R, int32_t d);
tsr_status launch_svg_temporal(const void* q, const void* k, const void* v, void* out, float* lse,
                               int32_t H, int32_t N, int32_t d, int32_t F, int32_t S,
                               const int8_t* head_kind, int64_t bh_lo, int64_t bh_hi,
                               cudaStream_t stream);

// permutation (permute.cu)
tsr_status launch_permute(const void* src, void* dst, int32_t B, int32_t H, int32_t F, int32_t S,
                          int32_t row_bytes, const int8_t* head_kind_host, int32_t inverse,
                          cudaStream_t stream);

// regime table (api.cu)
Regime regime_lookup(int32_t kind, int32_t bq, int32_t bk, int32_t N, double density, int32_t d);

// tensor maps (fwd.cu)
bool encode_tmap_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                    uint64_t outer, uint32_t box_inner, uint32_t box_rows);

int num_sms(int device);

}  // namespace tsr

struct tsr_plan_s : tsr::tsr_plan_impl {};
