// api.cu -- the C ABI declared in include/tsr.h: argument checks, plan
// lifetime, forward dispatch, plan export, the host-memory entry point and the
// regime table (Tessera abstract: profile-guided regime selection through a
// lookup table filled by offline profiling).
#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <array>
#include <cmath>
#include <cstring>
#include <fstream>
#include <mutex>
#include <new>
#include <sstream>
#include <string>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace tsr {

namespace {
thread_local std::string g_last_error;
}

void set_error(const std::string& msg) { g_last_error = msg; }
const char* last_error_cstr() { return g_last_error.c_str(); }

tsr_status fail(tsr_status s, const std::string& msg) {
  set_error(msg);
  return s;
}

tsr_status cuda_fail(cudaError_t e, const char* what) {
  set_error(std::string(what) + ": " + cudaGetErrorString(e));
  return e == cudaErrorMemoryAllocation ? TSR_ERR_OOM : TSR_ERR_CUDA;
}

int num_sms(int device) {
  static int cache[64] = {0};
  if (device >= 0 && device < 64 && cache[device]) return cache[device];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0)
    n = 1;
  if (device >= 0 && device < 64) cache[device] = n;
  return n;
}

// ----------------------------------------------------------- regime table
//
// One row per line: kind bq bk n_min n_max dens_min dens_max d  bn stages ctas
// [orient] ("*" = any; a row without the orientation field, or with "*" there,
// names 128-row tiles).  The first matching row wins.  A key-major row
// (orient 2) names the one key-major kernel: d = 128, bn 64, stages 2, ctas 1.  The rows shipped with the
// library come from timing every kernel variant on this GPU over synthetic
// masks of each class (the table file next to the library); the built-in rows
// below are the fallback when no file is loaded.
namespace {

struct RegimeRow {
  int kind, bq, bk;
  int64_t n_min, n_max;
  double d_min, d_max;
  int d, bn, stages, ctas, orient;
};

const char* kBuiltinTable =
    "# kind bq bk n_min n_max dens_min dens_max d bn stages ctas\n"
    "* * * * * * * 128 128 3 1\n"
    "* * * * * * * 64 128 4 1\n";

std::mutex g_table_mu;
std::vector<RegimeRow> g_table;
bool g_table_loaded = false;

bool parse_field_i(const std::string& s, int64_t* v) {
  if (s == "*") {
    *v = -1;
    return true;
  }
  char* end = nullptr;
  *v = std::strtoll(s.c_str(), &end, 10);
  return end && *end == 0;
}
bool parse_field_d(const std::string& s, double* v) {
  if (s == "*") {
    *v = -1.0;
    return true;
  }
  char* end = nullptr;
  *v = std::strtod(s.c_str(), &end);
  return end && *end == 0;
}

bool parse_table(const std::string& text, std::vector<RegimeRow>* out, std::string* why) {
  std::istringstream in(text);
  std::string line;
  int lineno = 0;
  std::vector<RegimeRow> rows;
  while (std::getline(in, line)) {
    ++lineno;
    const size_t hash = line.find('#');
    if (hash != std::string::npos) line = line.substr(0, hash);
    std::istringstream ls(line);
    std::vector<std::string> f;
    std::string tok;
    while (ls >> tok) f.push_back(tok);
    if (f.empty()) continue;
    if (f.size() != 11 && f.size() != 12) {
      *why = "line " + std::to_string(lineno) + ": expected 11 or 12 fields";
      return false;
    }
    int64_t kind, bq, bk, nmin, nmax, d, bn, st, ct, orient = TSR_ORIENT_ROWS;
    double dmin, dmax;
    if (!parse_field_i(f[0], &kind) || !parse_field_i(f[1], &bq) || !parse_field_i(f[2], &bk) ||
        !parse_field_i(f[3], &nmin) || !parse_field_i(f[4], &nmax) ||
        !parse_field_d(f[5], &dmin) || !parse_field_d(f[6], &dmax) || !parse_field_i(f[7], &d) ||
        !parse_field_i(f[8], &bn) || !parse_field_i(f[9], &st) || !parse_field_i(f[10], &ct) ||
        bn < 0 || st < 0 || ct < 0 || (f.size() == 12 && !parse_field_i(f[11], &orient))) {
      *why = "line " + std::to_string(lineno) + ": bad field";
      return false;
    }
    if (orient < 0) orient = TSR_ORIENT_ROWS;
    if (orient != TSR_ORIENT_ROWS && orient != TSR_ORIENT_KEYS) {
      *why = "line " + std::to_string(lineno) + ": orientation must be 1 or 2";
      return false;
    }
    rows.push_back(RegimeRow{static_cast<int>(kind), static_cast<int>(bq), static_cast<int>(bk),
                             nmin, nmax, dmin, dmax, static_cast<int>(d), static_cast<int>(bn),
                             static_cast<int>(st), static_cast<int>(ct), static_cast<int>(orient)});
  }
  *out = rows;
  return true;
}

bool rows_valid(const std::vector<RegimeRow>& rows) {
  for (const RegimeRow& r : rows) {
    if (r.orient == TSR_ORIENT_KEYS) {
      if (r.d != 128 || r.bn != 64 || r.stages != 2 || r.ctas != 1) return false;
      continue;
    }
    if ((r.bn != 64 && r.bn != 128) || (r.d != 64 && r.d != 128) ||
        !variant_exists(r.d, r.bn, r.stages, r.ctas, r.kind == TSR_MASK_KEYLIST))
      return false;
  }
  return true;
}

void ensure_table() {
  if (g_table_loaded) return;
  std::string why;
  const char* env = std::getenv("TSR_REGIME_TABLE");
  if (env && *env) {
    std::ifstream f(env);
    std::stringstream ss;
    ss << f.rdbuf();
    std::vector<RegimeRow> rows;
    if (f && parse_table(ss.str(), &rows, &why) && rows_valid(rows)) {
      g_table = rows;
      g_table_loaded = true;
      return;
    }
  }
  parse_table(kBuiltinTable, &g_table, &why);
  g_table_loaded = true;
}

}  // namespace

Regime regime_lookup(int32_t kind, int32_t bq, int32_t bk, int32_t N, double density, int32_t d) {
  std::lock_guard<std::mutex> lk(g_table_mu);
  ensure_table();
  for (size_t i = 0; i < g_table.size(); ++i) {
    const RegimeRow& r = g_table[i];
    if (r.kind >= 0 && r.kind != kind) continue;
    if (r.bq >= 0 && r.bq != bq) continue;
    if (r.bk >= 0 && r.bk != bk) continue;
    if (r.n_min >= 0 && N < r.n_min) continue;
    if (r.n_max >= 0 && N > r.n_max) continue;
    if (r.d_min >= 0 && density < r.d_min) continue;
    if (r.d_max >= 0 && density >= r.d_max) continue;
    if (r.d >= 0 && r.d != d) continue;
    return Regime{r.bn, r.stages, r.ctas, static_cast<int32_t>(i), r.orient};
  }
  return Regime{128, d == 64 ? 4 : 3, 1, -1, TSR_ORIENT_ROWS};
}

}  // namespace tsr

using namespace tsr;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

tsr_status check_mask(const tsr_mask* m) {
  if (!m) return fail(TSR_ERR_INVALID_ARG, "mask is NULL");
  if (m->B <= 0 || m->H <= 0 || m->N <= 0) return fail(TSR_ERR_INVALID_ARG, "B, H, N must be > 0");
  if (m->d != 64 && m->d != 128) return fail(TSR_ERR_INVALID_ARG, "d must be 64 or 128");
  if (m->N > (1 << 24)) return fail(TSR_ERR_UNSUPPORTED, "N above 2^24");
  if (static_cast<int64_t>(m->B) * m->H > (1 << 20)) return fail(TSR_ERR_UNSUPPORTED, "B*H above 2^20");
  switch (m->kind) {
    case TSR_MASK_UNIFORM:
      if (m->bq < 16 || m->bk < 16) return fail(TSR_ERR_INVALID_ARG, "bq, bk must be >= 16");
      if (!m->blocks) return fail(TSR_ERR_INVALID_ARG, "blocks is NULL");
      return TSR_OK;
    case TSR_MASK_SEGMENTS:
      if (m->n_qseg <= 0 || m->n_kseg <= 0 || !m->q_bounds || !m->k_bounds || !m->blocks)
        return fail(TSR_ERR_INVALID_ARG, "segment bounds / blocks missing");
      return TSR_OK;
    case TSR_MASK_SVG:
      if (m->n_frames <= 0 || m->frame_size <= 0 ||
          static_cast<int64_t>(m->n_frames) * m->frame_size != m->N || !m->head_kind)
        return fail(TSR_ERR_INVALID_ARG, "SVG needs N = n_frames * frame_size and head_kind");
      if (m->temporal_radius < 0) return fail(TSR_ERR_INVALID_ARG, "temporal_radius must be >= 0");
      return TSR_OK;
    case TSR_MASK_KEYLIST:
      if (m->slice_m != 64 && m->slice_m != 128)
        return fail(TSR_ERR_UNSUPPORTED, "KEYLIST slice_m must be 64 or 128");
      // indices may be NULL when every list is empty (checked against indptr
      // before anything reads a list)
      if (!m->indptr) return fail(TSR_ERR_INVALID_ARG, "indptr missing");
      return TSR_OK;
    default:
      return fail(TSR_ERR_INVALID_ARG, "unknown mask kind");
  }
}

tsr_status check_bounds(const int32_t* dev, int32_t n, int32_t N, cudaStream_t st) {
  std::vector<int32_t> h(static_cast<size_t>(n) + 1);
  TSR_CUDA(cudaMemcpyAsync(h.data(), dev, sizeof(int32_t) * (n + 1), cudaMemcpyDeviceToHost, st));
  TSR_CUDA(cudaStreamSynchronize(st));
  if (h[0] != 0 || h[n] != N) return fail(TSR_ERR_INVALID_ARG, "segment bounds must run 0 .. N");
  for (int32_t i = 0; i < n; ++i)
    if (h[i + 1] <= h[i]) return fail(TSR_ERR_INVALID_ARG, "segment bounds must ascend");
  return TSR_OK;
}

void free_plan(tsr_plan_s* P) {
  if (!P) return;
  for (DevBuf* b : {&P->b_items, &P->b_entries, &P->b_descs, &P->b_cnt, &P->b_tot, &P->b_ebegin,
                    &P->b_dbegin, &P->b_hist, &P->b_gidx, &P->b_units, &P->b_part_o, &P->b_part_lse,
                    &P->b_part_cnt, &P->b_launch})
    devbuf_free(*b);
  cudaFree(P->counter);
  cudaFree(P->err);
  cudaFree(P->head_kind_dev);
  if (P->band_stream) cudaStreamDestroy(P->band_stream);
  if (P->band_fork) cudaEventDestroy(P->band_fork);
  if (P->band_join) cudaEventDestroy(P->band_join);
  if (P->host_tot) cudaFreeHost(P->host_tot);
  if (P->host_kinds) cudaFreeHost(P->host_kinds);
  delete P;
}

// Mask-dependent part of planning, shared by tsr_plan and tsr_plan_update.
tsr_status plan_fill(tsr_plan_s* P, const tsr_mask* mask, cudaStream_t st) {
  P->kind = mask->kind;
  P->n_temporal = 0;
  P->head_layout.assign(mask->H, 0);
  if (mask->kind == TSR_MASK_SEGMENTS) {
    if (tsr_status s = check_bounds(mask->q_bounds, mask->n_qseg, mask->N, st)) return s;
    if (tsr_status s = check_bounds(mask->k_bounds, mask->n_kseg, mask->N, st)) return s;
  }
  if (mask->kind == TSR_MASK_SVG) {
    // The head kinds, copied on the stream without a synchronisation of their
    // own: the device copy feeds the planner kernels (which only compare a
    // kind with TSR_HEAD_TEMPORAL, so an invalid value cannot misaddress), the
    // pinned host copy is checked after the planner's count synchronisation.
    P->F = mask->n_frames;
    P->S = mask->frame_size;
    P->R = mask->temporal_radius;
    if (!P->head_kind_dev) TSR_CUDA(cudaMalloc(&P->head_kind_dev, mask->H));
    if (!P->host_kinds) TSR_CUDA(cudaMallocHost(&P->host_kinds, mask->H));
    TSR_CUDA(cudaMemcpyAsync(P->head_kind_dev, mask->head_kind, mask->H, cudaMemcpyDeviceToDevice,
                             st));
    TSR_CUDA(cudaMemcpyAsync(P->host_kinds, mask->head_kind, mask->H, cudaMemcpyDeviceToHost, st));
  }
  P->gathered = 0;
  P->slice_m = 0;
  P->n_gidx = 0;
  if (mask->kind == TSR_MASK_KEYLIST) {
    if (tsr_status s = plan_build_keylist(mask, P->has_opts ? &P->opts : nullptr, P, st)) return s;
  } else if (tsr_status s = plan_build(mask, P->has_opts ? &P->opts : nullptr, P, st)) {
    return s;
  }
  if (tsr_status s = plan_launch_list(P, st)) return s;
  if (tsr_status s = plan_split(P, P->has_opts ? &P->opts : nullptr, st)) return s;
  if (P->flags & TSR_PLAN_DEBUG_CHECKS) {
    if (tsr_status s = plan_check(P, st)) return s;
    uint32_t e = 0;
    TSR_CUDA(cudaMemcpyAsync(&e, P->err, sizeof e, cudaMemcpyDeviceToHost, st));
    TSR_CUDA(cudaStreamSynchronize(st));
    if (e) return fail(TSR_ERR_INTERNAL, "plan check failed (error word " + std::to_string(e) + ")");
  }
  return TSR_OK;
}

// Debug checks after a launch: the tiles the kernel computed against the plans.
tsr_status check_tiles_done(const tsr_plan_s* const* plans, int n, cudaStream_t st) {
  unsigned long long done = 0;
  TSR_CUDA(cudaMemcpyAsync(&done, static_cast<unsigned long long*>(plans[0]->b_tot.p) + 7,
                           sizeof done, cudaMemcpyDeviceToHost, st));
  TSR_CUDA(cudaStreamSynchronize(st));
  unsigned long long want = 0;
  for (int i = 0; i < n; ++i) want += static_cast<unsigned long long>(plans[i]->n_entries);
  if (done != want)
    return fail(TSR_ERR_INTERNAL, "the kernel computed " + std::to_string(done) + " tiles, the plan has " +
                                      std::to_string(want));
  return TSR_OK;
}

// Device buffers, streams, events and per-head-group plans of
// tsr_attention_host, kept per thread and grown on demand.
struct HostCache {
  void* buf[8] = {nullptr};
  size_t cap[8] = {0};
  cudaStream_t stream = nullptr, stream2 = nullptr;   // attention, alternating by group
  cudaStream_t s_in = nullptr, s_out = nullptr, s_plan = nullptr;
  uint32_t* host_err = nullptr;                // pinned: one error word per head group
  size_t host_err_cap = 0;
  int64_t* stage = nullptr;                    // pinned: rebased key-list indptr slices
  size_t stage_cap = 0;
  std::vector<cudaEvent_t> ev;                 // 3 per head group: inputs, plan, attention
  std::vector<tsr_plan_t> plans;               // one per head group
  std::vector<std::array<int64_t, 11>> plan_key;
  tsr_plan_t full_plan = nullptr;              // one plan over every head (one-plan mode)
  std::array<int64_t, 12> full_key{};
  int32_t* counters = nullptr;                 // one work counter per head group (one-plan mode)
  size_t counters_cap = 0;
  int device = -1;
  void release() {
    for (tsr_plan_t pl : plans) tsr_plan_destroy(pl);
    plans.clear();
    plan_key.clear();
    if (full_plan) tsr_plan_destroy(full_plan);
    full_plan = nullptr;
    cudaFree(counters);
    counters = nullptr;
    counters_cap = 0;
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
    ev.clear();
    for (int i = 0; i < 8; ++i) {
      cudaFree(buf[i]);
      buf[i] = nullptr;
      cap[i] = 0;
    }
    for (cudaStream_t* s : {&stream, &stream2, &s_in, &s_out, &s_plan}) {
      if (*s) cudaStreamDestroy(*s);
      *s = nullptr;
    }
    if (host_err) cudaFreeHost(host_err);
    host_err = nullptr;
    host_err_cap = 0;
    if (stage) cudaFreeHost(stage);
    stage = nullptr;
    stage_cap = 0;
    device = -1;
  }
  ~HostCache() { release(); }
  tsr_status get(int slot, size_t bytes, void** p) {
    if (bytes == 0) bytes = 16;
    if (cap[slot] < bytes) {
      cudaFree(buf[slot]);
      buf[slot] = nullptr;
      cap[slot] = 0;
      const cudaError_t e = cudaMalloc(&buf[slot], bytes);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(TSR_ERR_OOM, "device buffer for host call");
      }
      cap[slot] = bytes;
    }
    *p = buf[slot];
    return TSR_OK;
  }
};
thread_local HostCache g_host_cache;

// tsr_plan with the heads per longest-first scheduling group fixed
// (group_heads > 0; 0 = sized for L2).
tsr_status plan_new(const tsr_mask* mask, const tsr_plan_opts* opts, int32_t group_heads,
                    cudaStream_t st, tsr_plan_t* out) {
  *out = nullptr;
  if (tsr_status s = check_mask(mask)) return s;
  if (opts && opts->bn && opts->bn != 64 && opts->bn != 128)
    return fail(TSR_ERR_INVALID_ARG, "opts->bn must be 0, 64 or 128");
  if (opts && (opts->orient < 0 || opts->orient > TSR_ORIENT_KEYS))
    return fail(TSR_ERR_INVALID_ARG, "opts->orient must be 0, 1 or 2");
  if (opts && opts->kv_split != 0 && opts->kv_split != 1 && opts->kv_split != 2 && opts->kv_split != 4)
    return fail(TSR_ERR_INVALID_ARG, "opts->kv_split must be 0, 1, 2 or 4");
  tsr_plan_s* P = new (std::nothrow) tsr_plan_s();
  if (!P) return fail(TSR_ERR_OOM, "host allocation failed");
  struct Guard {
    tsr_plan_s* p;
    ~Guard() { free_plan(p); }
  } guard{P};
  TSR_CUDA(cudaGetDevice(&P->device));
  P->B = mask->B;
  P->H = mask->H;
  P->N = mask->N;
  P->d = mask->d;
  P->group_heads = group_heads;
  P->flags = opts ? opts->flags : 0;
  if (opts) {
    P->has_opts = true;
    P->opts = *opts;
  }
  TSR_CUDA(cudaMalloc(&P->counter, sizeof(int32_t)));
  TSR_CUDA(cudaMalloc(&P->err, sizeof(uint32_t)));
  TSR_CUDA(cudaMemsetAsync(P->err, 0, sizeof(uint32_t), st));
  if (tsr_status s = plan_fill(P, mask, st)) return s;
  guard.p = nullptr;
  *out = P;
  return TSR_OK;
}

}  // namespace

extern "C" {

int32_t tsr_abi_version(void) { return TSR_ABI_VERSION; }

const char* tsr_status_string(tsr_status s) {
  switch (s) {
    case TSR_OK: return "ok";
    case TSR_ERR_INVALID_ARG: return "invalid argument";
    case TSR_ERR_UNSUPPORTED: return "unsupported";
    case TSR_ERR_CUDA: return "CUDA error";
    case TSR_ERR_OOM: return "out of memory";
    case TSR_ERR_TIMEOUT: return "device wait timed out";
    case TSR_ERR_INTERNAL: return "internal error";
  }
  return "unknown status";
}

const char* tsr_last_error(void) { return last_error_cstr(); }

tsr_status tsr_plan(const tsr_mask* mask, const tsr_plan_opts* opts, tsr_plan_t* out,
                    void* stream) {
  set_error("");
  if (!out) return fail(TSR_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  return plan_new(mask, opts, 0, static_cast<cudaStream_t>(stream), out);
}

tsr_status tsr_plan_update(tsr_plan_t plan, const tsr_mask* mask, void* stream) {
  set_error("");
  if (!plan) return fail(TSR_ERR_INVALID_ARG, "plan is NULL");
  if (tsr_status s = check_mask(mask)) return s;
  if (mask->B != plan->B || mask->H != plan->H || mask->N != plan->N || mask->d != plan->d)
    return fail(TSR_ERR_INVALID_ARG, "tsr_plan_update needs the plan's B, H, N and d");
  int dev = 0;
  TSR_CUDA(cudaGetDevice(&dev));
  if (dev != plan->device) return fail(TSR_ERR_INVALID_ARG, "plan was made on another device");
  return plan_fill(plan, mask, static_cast<cudaStream_t>(stream));
}

tsr_status tsr_plan_destroy(tsr_plan_t plan) {
  free_plan(plan);
  return TSR_OK;
}

tsr_status tsr_plan_device_status(tsr_plan_t plan, void* stream) {
  if (!plan) return fail(TSR_ERR_INVALID_ARG, "plan is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t e = 0;
  TSR_CUDA(cudaMemcpyAsync(&e, plan->err, sizeof e, cudaMemcpyDeviceToHost, st));
  TSR_CUDA(cudaMemsetAsync(plan->err, 0, sizeof(uint32_t), st));
  TSR_CUDA(cudaStreamSynchronize(st));
  if (e & DEV_ERR_TIMEOUT)
    return fail(TSR_ERR_TIMEOUT, "a device-side wait timed out (error word " + std::to_string(e) + ")");
  if (e) return fail(TSR_ERR_INTERNAL, "device error word " + std::to_string(e));
  return TSR_OK;
}

tsr_status tsr_bsa_forward(const void* q, const void* k, const void* v, tsr_plan_t plan, void* out,
                           float* lse, void* stream) {
  if (!plan) return fail(TSR_ERR_INVALID_ARG, "plan is NULL");
  if (!q || !k || !v || !out || !lse) return fail(TSR_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return fail(TSR_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (out == q || out == k || out == v) return fail(TSR_ERR_INVALID_ARG, "out aliases an input");
  int dev = 0;
  TSR_CUDA(cudaGetDevice(&dev));
  if (dev != plan->device) return fail(TSR_ERR_INVALID_ARG, "plan was made on another device");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  FwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.plan = plan;
  if (tsr_status e = launch_forward(a, st)) return e;
  if (plan->flags & TSR_PLAN_DEBUG_CHECKS) {
    if (tsr_status e = tsr_plan_device_status(plan, stream)) return e;
    const tsr_plan_s* one[1] = {plan};
    return check_tiles_done(one, 1, st);
  }
  if (plan->flags & TSR_PLAN_SYNC_CHECK) return tsr_plan_device_status(plan, stream);
  return TSR_OK;
}

tsr_status tsr_bsa_forward_batch(const tsr_request* reqs, int32_t n, void* stream) {
  set_error("");
  if (!reqs || n < 1 || n > 16) return fail(TSR_ERR_INVALID_ARG, "1 to 16 requests per call");
  int dev = 0;
  TSR_CUDA(cudaGetDevice(&dev));
  FwdArgs a[16];
  for (int32_t r = 0; r < n; ++r) {
    const tsr_request& q = reqs[r];
    const std::string at = "request " + std::to_string(r) + ": ";
    if (!q.plan) return fail(TSR_ERR_INVALID_ARG, at + "plan is NULL");
    if (!q.q || !q.k || !q.v || !q.out || !q.lse)
      return fail(TSR_ERR_INVALID_ARG, at + "NULL tensor pointer");
    if (!aligned16(q.q) || !aligned16(q.k) || !aligned16(q.v) || !aligned16(q.out) ||
        !aligned16(q.lse))
      return fail(TSR_ERR_INVALID_ARG, at + "tensor pointers must be 16-byte aligned");
    if (q.out == q.q || q.out == q.k || q.out == q.v)
      return fail(TSR_ERR_INVALID_ARG, at + "out aliases an input");
    if (dev != q.plan->device) return fail(TSR_ERR_INVALID_ARG, at + "plan was made on another device");
    for (int32_t s2 = 0; s2 < r; ++s2)
      if (reqs[s2].plan == q.plan)
        return fail(TSR_ERR_INVALID_ARG, at + "a plan may appear once per batch");
    a[r] = FwdArgs{q.q, q.k, q.v, q.out, q.lse, q.plan};
  }
  if (tsr_status e = launch_forward_batch(a, n, static_cast<cudaStream_t>(stream))) return e;
  if (reqs[0].plan->flags & TSR_PLAN_DEBUG_CHECKS) {
    if (tsr_status e = tsr_plan_device_status(reqs[0].plan, stream)) return e;
    const tsr_plan_s* plans[16];
    for (int32_t r = 0; r < n; ++r) plans[r] = reqs[r].plan;
    return check_tiles_done(plans, n, static_cast<cudaStream_t>(stream));
  }
  if (reqs[0].plan->flags & TSR_PLAN_SYNC_CHECK) return tsr_plan_device_status(reqs[0].plan, stream);
  return TSR_OK;
}

tsr_status tsr_plan_get_stats(tsr_plan_t plan, tsr_plan_stats* s) {
  if (!plan || !s) return fail(TSR_ERR_INVALID_ARG, "NULL argument");
  memset(s, 0, sizeof *s);
  s->bm = plan->bm;
  s->bn = plan->bn;
  s->stages = plan->stages;
  s->ctas_per_sm = plan->ctas;
  s->gathered = plan->gathered;
  s->n_temporal_heads = plan->n_temporal;
  s->n_items = plan->n_items;
  s->n_entries = plan->n_entries;
  s->n_boundary = plan->n_desc;
  s->n_logical_on = plan->n_logical_on;
  s->n_logical_total = plan->n_logical_total;
  s->max_item_len = plan->max_item_len;
  s->regime_id = plan->regime_id;
  s->orient = plan->orient;
  s->kv_split = plan->kv_split;
  s->temporal_band = plan->temporal_band;
  return TSR_OK;
}

tsr_status tsr_plan_export(tsr_plan_t plan, void* host_buf, size_t* bytes) {
  if (!plan || !bytes) return fail(TSR_ERR_INVALID_ARG, "NULL argument");
  const size_t need = sizeof(tsr_export_header) + sizeof(tsr_plan_item) * plan->n_items +
                      sizeof(tsr_plan_entry) * plan->n_entries +
                      sizeof(tsr_tile_desc) * plan->n_desc + 4 * plan->n_gidx + plan->H;
  if (!host_buf) {
    *bytes = need;
    return TSR_OK;
  }
  if (*bytes < need) return fail(TSR_ERR_INVALID_ARG, "export buffer too small");
  TSR_CUDA(cudaDeviceSynchronize());
  uint8_t* o = static_cast<uint8_t*>(host_buf);
  tsr_export_header h;
  memset(&h, 0, sizeof h);
  memcpy(h.magic, "TSRP", 4);
  h.version = 1;
  h.B = plan->B;
  h.H = plan->H;
  h.N = plan->N;
  h.d = plan->d;
  h.bm = plan->bm;
  h.bn = plan->bn;
  h.gathered = plan->gathered;
  h.n_frames = plan->n_temporal ? plan->F : 0;
  h.frame_size = plan->n_temporal ? plan->S : 0;
  h.slice_m = plan->slice_m;
  h.n_items = plan->n_items;
  h.n_entries = plan->n_entries;
  h.n_desc = plan->n_desc;
  h.n_gidx = plan->n_gidx;
  memcpy(o, &h, sizeof h);
  size_t off = sizeof h;
  auto pull = [&](const void* src, size_t n) -> cudaError_t {
    cudaError_t e = cudaSuccess;
    if (n) e = cudaMemcpy(o + off, src, n, cudaMemcpyDeviceToHost);
    off += n;
    return e;
  };
  TSR_CUDA(pull(plan->items, sizeof(tsr_plan_item) * plan->n_items));
  TSR_CUDA(pull(plan->entries, sizeof(tsr_plan_entry) * plan->n_entries));
  TSR_CUDA(pull(plan->descs, sizeof(tsr_tile_desc) * plan->n_desc));
  TSR_CUDA(pull(plan->gidx, 4 * plan->n_gidx));
  memcpy(o + off, plan->head_layout.data(), plan->H);
  off += plan->H;
  *bytes = off;
  return TSR_OK;
}

tsr_status tsr_temporal_permute(const void* src, void* dst, int32_t B, int32_t H,
                                int32_t n_frames, int32_t frame_size, int32_t row_bytes,
                                const int8_t* head_kind, int32_t inverse, void* stream) {
  if (!src || !dst) return fail(TSR_ERR_INVALID_ARG, "NULL pointer");
  if (B <= 0 || H <= 0 || n_frames <= 0 || frame_size <= 0 || row_bytes <= 0 || row_bytes % 16)
    return fail(TSR_ERR_INVALID_ARG, "bad shape (row_bytes must be a positive multiple of 16)");
  if (static_cast<int64_t>(n_frames) * frame_size > (1 << 30))
    return fail(TSR_ERR_UNSUPPORTED, "too many tokens");
  if (!aligned16(src) || !aligned16(dst))
    return fail(TSR_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  const size_t bytes = static_cast<size_t>(B) * H * n_frames * frame_size * row_bytes;
  const uint8_t* a = static_cast<const uint8_t*>(src);
  const uint8_t* b = static_cast<const uint8_t*>(dst);
  if (a < b + bytes && b < a + bytes) return fail(TSR_ERR_INVALID_ARG, "src and dst overlap");
  return launch_permute(src, dst, B, H, n_frames, frame_size, row_bytes, head_kind, inverse,
                        static_cast<cudaStream_t>(stream));
}

tsr_status tsr_svg_route(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                         int32_t n_frames, int32_t frame_size, int32_t d, int32_t temporal_radius,
                         const int32_t* samples, int32_t n_samples, float* stats,
                         int8_t* head_kind, void* stream) {
  set_error("");
  if (!q || !k || !v || !samples || !stats || !head_kind)
    return fail(TSR_ERR_INVALID_ARG, "NULL pointer");
  if (B <= 0 || H <= 0 || n_frames <= 0 || frame_size <= 0 || n_samples <= 0 ||
      temporal_radius < 0)
    return fail(TSR_ERR_INVALID_ARG, "B, H, n_frames, frame_size, n_samples must be > 0, "
                                     "temporal_radius >= 0");
  if (d != 64 && d != 128) return fail(TSR_ERR_INVALID_ARG, "d must be 64 or 128");
  const int64_t N = static_cast<int64_t>(n_frames) * frame_size;
  if (N > (1 << 24)) return fail(TSR_ERR_UNSUPPORTED, "N above 2^24");
  if (static_cast<int64_t>(B) * H > (1 << 20)) return fail(TSR_ERR_UNSUPPORTED, "B*H above 2^20");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(stats))
    return fail(TSR_ERR_INVALID_ARG, "q, k, v and stats must be 16-byte aligned");
  for (int32_t s = 0; s < n_samples; ++s)
    if (samples[s] < 0 || samples[s] >= N)
      return fail(TSR_ERR_INVALID_ARG, "sampled row " + std::to_string(s) + " outside [0, N)");
  return launch_route(q, k, v, B, H, n_frames, frame_size, d, temporal_radius, samples, n_samples,
                      stats, head_kind, static_cast<cudaStream_t>(stream));
}

tsr_status tsr_attention_host(const tsr_mask* mask, const tsr_plan_opts* opts, const void* q,
                              const void* k, const void* v, void* out, float* lse) {
  set_error("");
  if (tsr_status s = check_mask(mask)) return s;
  if (!q || !k || !v || !out || !lse) return fail(TSR_ERR_INVALID_ARG, "NULL tensor pointer");
  HostCache& hc = g_host_cache;
  int dev = 0;
  TSR_CUDA(cudaGetDevice(&dev));
  if (hc.device != dev) {
    hc.release();
    hc.device = dev;
  }
  for (cudaStream_t* st : {&hc.stream, &hc.stream2, &hc.s_in, &hc.s_out, &hc.s_plan})
    if (!*st) TSR_CUDA(cudaStreamCreateWithFlags(st, cudaStreamNonBlocking));
  const int64_t BH = static_cast<int64_t>(mask->B) * mask->H;
  const size_t row_b = static_cast<size_t>(mask->N) * mask->d * 2;   // one head of Q, K, V or O
  const size_t tb = BH * row_b;
  const size_t lb = static_cast<size_t>(BH) * mask->N * 4;
  // Heads are processed in groups: the inputs of group g + 1 are copied in while
  // group g is attended and group g - 1 is copied out (copy engines and SMs
  // overlap).  Only the first group's copy-in and the last group's copy-out are
  // exposed, so the groups grow from one head by a factor of 1.2 (attention of
  // a group then covers the copy-in of the next whenever attending a head takes
  // at least 1.2x as long as copying it in; a 480p head of the block-mask
  // workload is attended in ~0.146 ms and copied in over a ~208 GB/s host link
  // in ~0.121 ms, so faster growth leaves the SMs waiting for inputs) up to about
  // 160 MB of Q, K and V, and the last two groups are two heads and one.
  std::vector<int64_t> gs{0};
  {
    const int64_t cap = std::max<int64_t>(1, static_cast<int64_t>((160u << 20) / (3 * row_b)));
    const int64_t tail = BH >= 8 ? 3 : 0;
    int64_t left = BH - tail;
    double r = 1.0;
    while (left > 0) {
      const int64_t sz = std::min<int64_t>({cap, static_cast<int64_t>(std::ceil(r)), left});
      gs.push_back(gs.back() + sz);
      left -= sz;
      r *= 1.2;
    }
    if (tail) {
      gs.push_back(gs.back() + 2);
      gs.push_back(gs.back() + 1);
    }
  }
  const int64_t G = static_cast<int64_t>(gs.size()) - 1;
  void *dq, *dk, *dv, *dout, *dlse;
  if (tsr_status s = hc.get(0, tb, &dq)) return s;
  if (tsr_status s = hc.get(1, tb, &dk)) return s;
  if (tsr_status s = hc.get(2, tb, &dv)) return s;
  if (tsr_status s = hc.get(3, tb, &dout)) return s;
  if (tsr_status s = hc.get(4, lb, &dlse)) return s;
  while (static_cast<int64_t>(hc.ev.size()) < 4 * G) {
    cudaEvent_t e;
    TSR_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    hc.ev.push_back(e);
  }
  // Steps 1 to 3 run in one function so that every failure, once a copy that
  // reads or writes the caller's buffers may be queued, still reaches the
  // synchronisation below.
  cudaStream_t sp = hc.s_plan;
  int64_t n_err = G;
  const tsr_status s_run = [&]() -> tsr_status {
    // 1. the mask to the device, and one mask view per head group
    std::vector<int64_t> kl_start, kl_base;      // key lists: per-group slices
    void* kl_dp = nullptr;
    void* kl_di = nullptr;
    std::vector<tsr_mask> views(G, *mask);
    const int64_t nqb = (mask->kind == TSR_MASK_KEYLIST) ? (mask->N + mask->slice_m - 1) / mask->slice_m : 0;
    if (mask->kind == TSR_MASK_UNIFORM || mask->kind == TSR_MASK_SEGMENTS) {
      const int64_t per_head = (mask->kind == TSR_MASK_UNIFORM)
                                   ? static_cast<int64_t>((mask->N + mask->bq - 1) / mask->bq) *
                                         ((mask->N + mask->bk - 1) / mask->bk)
                                   : static_cast<int64_t>(mask->n_qseg) * mask->n_kseg;
      void* db;
      if (tsr_status s = hc.get(5, BH * per_head, &db)) return s;
      TSR_CUDA(cudaMemcpyAsync(db, mask->blocks, BH * per_head, cudaMemcpyHostToDevice, sp));
      const int32_t* qb = nullptr;
      const int32_t* kb = nullptr;
      if (mask->kind == TSR_MASK_SEGMENTS) {
        void* dbnd;
        const size_t nq = mask->n_qseg + 1, nk = mask->n_kseg + 1;
        if (tsr_status s = hc.get(6, 4 * (nq + nk), &dbnd)) return s;
        int32_t* pb = static_cast<int32_t*>(dbnd);
        TSR_CUDA(cudaMemcpyAsync(pb, mask->q_bounds, 4 * nq, cudaMemcpyHostToDevice, sp));
        TSR_CUDA(cudaMemcpyAsync(pb + nq, mask->k_bounds, 4 * nk, cudaMemcpyHostToDevice, sp));
        qb = pb;
        kb = pb + nq;
      }
      for (int64_t g = 0; g < G; ++g) {
        views[g].blocks = static_cast<const uint8_t*>(db) + gs[g] * per_head;
        views[g].q_bounds = qb;
        views[g].k_bounds = kb;
      }
    } else if (mask->kind == TSR_MASK_KEYLIST) {
      const int64_t n_lists = BH * nqb;
      const int64_t n_idx = mask->indptr[n_lists];   // HOST arrays here
      if (n_idx < 0 || mask->indptr[0] != 0)
        return fail(TSR_ERR_INVALID_ARG, "indptr must run upward from 0");
      // each group's slice of indptr, rebased to start at 0, staged in pinned
      // memory; the slices and their keys are copied per group in step 2
      const size_t n_stage = static_cast<size_t>(n_lists + G);
      if (hc.stage_cap < n_stage) {
        if (hc.stage) cudaFreeHost(hc.stage);
        hc.stage = nullptr;
        hc.stage_cap = 0;
        TSR_CUDA(cudaMallocHost(&hc.stage, sizeof(int64_t) * n_stage));
        hc.stage_cap = n_stage;
      }
      kl_start.resize(G);
      kl_base.resize(G + 1);
      int64_t pos = 0;
      for (int64_t g = 0; g < G; ++g) {
        const int64_t l0 = gs[g] * nqb, l1 = gs[g + 1] * nqb;
        kl_start[g] = pos;
        kl_base[g] = mask->indptr[l0];
        for (int64_t l = l0; l <= l1; ++l) hc.stage[pos++] = mask->indptr[l] - kl_base[g];
      }
      kl_base[G] = n_idx;
      if (tsr_status s = hc.get(5, sizeof(int64_t) * n_stage, &kl_dp)) return s;
      if (tsr_status s = hc.get(6, sizeof(int32_t) * static_cast<size_t>(n_idx), &kl_di)) return s;
      for (int64_t g = 0; g < G; ++g) {
        views[g].indptr = static_cast<const int64_t*>(kl_dp) + kl_start[g];
        views[g].indices = static_cast<const int32_t*>(kl_di) + kl_base[g];
      }
    } else if (mask->kind == TSR_MASK_SVG) {
      // head kinds of the flattened (b, h) order
      std::vector<int8_t> kinds(BH);
      for (int64_t i = 0; i < BH; ++i) kinds[i] = mask->head_kind[i % mask->H];
      void* dh;
      if (tsr_status s = hc.get(7, BH, &dh)) return s;
      TSR_CUDA(cudaMemcpyAsync(dh, kinds.data(), BH, cudaMemcpyHostToDevice, sp));
      TSR_CUDA(cudaStreamSynchronize(sp));
      for (int64_t g = 0; g < G; ++g) views[g].head_kind = static_cast<const int8_t*>(dh) + gs[g];
    }
    // 2. inputs, group by group (queued after the mask, which the copy engine
    // would otherwise move only after every input); key lists go group by group
    // too, each group's slice just ahead of its inputs, and its plan waits only
    // for that slice
    const char* hq = static_cast<const char*>(q);
    const char* hk = static_cast<const char*>(k);
    const char* hv = static_cast<const char*>(v);
    for (int64_t g = 0; g < G; ++g) {
      const int64_t b0 = gs[g], cnt = gs[g + 1] - gs[g];
      const size_t off = b0 * row_b, n = cnt * row_b;
      if (mask->kind == TSR_MASK_KEYLIST) {
        const int64_t n_ptr = cnt * nqb + 1, k0 = kl_base[g], k1 = kl_base[g + 1];
        TSR_CUDA(cudaMemcpyAsync(static_cast<int64_t*>(kl_dp) + kl_start[g], hc.stage + kl_start[g],
                                 sizeof(int64_t) * n_ptr, cudaMemcpyHostToDevice, hc.s_in));
        if (k1 > k0)
          TSR_CUDA(cudaMemcpyAsync(static_cast<int32_t*>(kl_di) + k0, mask->indices + k0,
                                   sizeof(int32_t) * (k1 - k0), cudaMemcpyHostToDevice, hc.s_in));
        TSR_CUDA(cudaEventRecord(hc.ev[3 * G + g], hc.s_in));
      }
      TSR_CUDA(cudaMemcpyAsync(static_cast<char*>(dq) + off, hq + off, n, cudaMemcpyHostToDevice, hc.s_in));
      TSR_CUDA(cudaMemcpyAsync(static_cast<char*>(dk) + off, hk + off, n, cudaMemcpyHostToDevice, hc.s_in));
      TSR_CUDA(cudaMemcpyAsync(static_cast<char*>(dv) + off, hv + off, n, cudaMemcpyHostToDevice, hc.s_in));
      TSR_CUDA(cudaEventRecord(hc.ev[3 * g], hc.s_in));
    }
    // 3. per head group: its plan (kept from call to call while the grouping and
    // options are unchanged, re-planned for the new mask), its attention once its
    // inputs and plan are ready, and its outputs back.  Planning group g + 1 (one
    // host synchronisation on the plan stream) overlaps attention g.  (Planning
    // two groups ahead measured slower: a key-list plan then waits for a slice
    // queued behind the next group's inputs.)  Consecutive groups alternate
    // between two attention streams, so one persistent launch's last CTAs
    // overlap the next one's first.
    // The head-group launches overlap one another (two attention streams), so
    // a launch's tail is covered by the next one: no automatic split-KV here
    // (an explicit opts->kv_split is honoured).
    tsr_plan_opts host_opts = opts ? *opts : tsr_plan_opts{};
    if (host_opts.kv_split == 0) host_opts.kv_split = 1;
    // Key lists are planned group by group; each group takes the regime of the
    // whole request (looked up from its total list length), so the result is
    // the one a single plan over every head gives.
    if (mask->kind == TSR_MASK_KEYLIST && !host_opts.orient && !host_opts.bn && !host_opts.stages &&
        !host_opts.ctas_per_sm) {
      const double n_lists = static_cast<double>(BH) * static_cast<double>(nqb);
      const double density = n_lists > 0 ? static_cast<double>(mask->indptr[BH * nqb]) / n_lists / mask->N
                                         : 0.0;
      Regime rg;
      if (tsr_status st = resolve_regime(regime_lookup(TSR_MASK_KEYLIST, mask->slice_m, 1, mask->N,
                                                       density, mask->d),
                                         nullptr, mask->d, true, &rg))
        return st;
      host_opts.orient = rg.orient;
      if (rg.orient != TSR_ORIENT_KEYS) {
        host_opts.bn = rg.bn;
        host_opts.stages = rg.stages;
        host_opts.ctas_per_sm = rg.ctas;
      }
    }
    const tsr_plan_opts& o = host_opts;
    if (static_cast<int64_t>(hc.plans.size()) != G) {
      for (tsr_plan_t pl : hc.plans) tsr_plan_destroy(pl);
      hc.plans.assign(G, nullptr);
      hc.plan_key.assign(G, {});
    }
    if (hc.host_err_cap < static_cast<size_t>(G)) {
      if (hc.host_err) cudaFreeHost(hc.host_err);
      hc.host_err = nullptr;
      hc.host_err_cap = 0;
      TSR_CUDA(cudaMallocHost(&hc.host_err, sizeof(uint32_t) * G));
      hc.host_err_cap = G;
    }
    auto plan_group = [&](int64_t g) -> tsr_status {
      tsr_mask& vw = views[g];
      vw.B = 1;
      vw.H = static_cast<int32_t>(gs[g + 1] - gs[g]);
      const std::array<int64_t, 11> key = {vw.kind, vw.H, vw.N, vw.d, o.bn, o.stages, o.ctas_per_sm,
                                            o.flags, o.orient, o.kv_split, opts ? 1 : 0};
      if (mask->kind == TSR_MASK_KEYLIST) TSR_CUDA(cudaStreamWaitEvent(sp, hc.ev[3 * G + g], 0));
      tsr_status st;
      if (hc.plans[g] && hc.plan_key[g] == key) {
        st = tsr_plan_update(hc.plans[g], &vw, sp);
      } else {
        if (hc.plans[g]) tsr_plan_destroy(hc.plans[g]);
        hc.plans[g] = nullptr;
        st = tsr_plan(&vw, &host_opts, &hc.plans[g], sp);
        hc.plan_key[g] = key;
      }
      if (st != TSR_OK) return st;
      TSR_CUDA(cudaEventRecord(hc.ev[3 * g + 1], sp));
      return TSR_OK;
    };
    auto launch_group = [&](int64_t g) -> tsr_status {
      cudaStream_t sa = (g & 1) ? hc.stream2 : hc.stream;
      const int64_t b0 = gs[g];
      const size_t off = b0 * row_b, n = (gs[g + 1] - gs[g]) * row_b;
      TSR_CUDA(cudaStreamWaitEvent(sa, hc.ev[3 * g], 0));
      TSR_CUDA(cudaStreamWaitEvent(sa, hc.ev[3 * g + 1], 0));
      if (tsr_status st = tsr_bsa_forward(static_cast<char*>(dq) + off, static_cast<char*>(dk) + off,
                                          static_cast<char*>(dv) + off, hc.plans[g],
                                          static_cast<char*>(dout) + off,
                                          static_cast<float*>(dlse) + b0 * mask->N, sa))
        return st;
      TSR_CUDA(cudaEventRecord(hc.ev[3 * g + 2], sa));
      TSR_CUDA(cudaStreamWaitEvent(hc.s_out, hc.ev[3 * g + 2], 0));
      TSR_CUDA(cudaMemcpyAsync(static_cast<char*>(out) + off, static_cast<char*>(dout) + off, n,
                               cudaMemcpyDeviceToHost, hc.s_out));
      TSR_CUDA(cudaMemcpyAsync(lse + b0 * mask->N, static_cast<float*>(dlse) + b0 * mask->N,
                               static_cast<size_t>(n / row_b) * mask->N * 4, cudaMemcpyDeviceToHost,
                               hc.s_out));
      // the group's device error word (its kernels have run once s_out gets here)
      TSR_CUDA(cudaMemcpyAsync(hc.host_err + g, hc.plans[g]->err, sizeof(uint32_t),
                               cudaMemcpyDeviceToHost, hc.s_out));
      TSR_CUDA(cudaMemsetAsync(hc.plans[g]->err, 0, sizeof(uint32_t), hc.s_out));
      return TSR_OK;
    };
    // One-plan mode (every mask form but key lists, whose slices arrive group by
    // group, and without the debug / synchronous-check / test flags, which check
    // each launch): one plan over every head with one head per longest-first
    // group, so head group g's work items are the contiguous range
    // [gs[g] * nqt, gs[g + 1] * nqt); each group's launch takes its range and its
    // own work counter.  Planning happens once, while the first inputs copy in.
    const bool one_plan =
        mask->kind != TSR_MASK_KEYLIST &&
        !(o.flags & (TSR_PLAN_DEBUG_CHECKS | TSR_PLAN_SYNC_CHECK | TSR_PLAN_TEST_STALL));
    tsr_status s = TSR_OK;
    if (one_plan) {
      n_err = 1;
      tsr_mask full = views[0];                  // device arrays from their start
      full.B = mask->B;
      full.H = mask->H;
      const std::array<int64_t, 12> key = {full.kind, full.B, full.H, full.N, full.d, o.bn, o.stages,
                                            o.ctas_per_sm, o.flags, o.orient, o.kv_split, opts ? 1 : 0};
      if (hc.full_plan && hc.full_key == key) {
        s = tsr_plan_update(hc.full_plan, &full, sp);
      } else {
        if (hc.full_plan) tsr_plan_destroy(hc.full_plan);
        hc.full_plan = nullptr;
        s = plan_new(&full, &host_opts, 1, sp, &hc.full_plan);
        hc.full_key = key;
      }
      if (s == TSR_OK && hc.counters_cap < static_cast<size_t>(G)) {
        cudaFree(hc.counters);
        hc.counters = nullptr;
        hc.counters_cap = 0;
        const cudaError_t e = cudaMalloc(&hc.counters, sizeof(int32_t) * G);
        if (e != cudaSuccess) s = cuda_fail(e, "work counters");
        else hc.counters_cap = G;
      }
      if (s == TSR_OK) TSR_CUDA(cudaEventRecord(hc.ev[1], sp));
      const int64_t nqt = hc.full_plan ? (mask->N + hc.full_plan->bm - 1) / hc.full_plan->bm : 0;
      for (int64_t g = 0; g < G && s == TSR_OK; ++g) {
        cudaStream_t sa = (g & 1) ? hc.stream2 : hc.stream;
        const int64_t b0 = gs[g];
        const size_t off = b0 * row_b, n = (gs[g + 1] - gs[g]) * row_b;
        TSR_CUDA(cudaStreamWaitEvent(sa, hc.ev[3 * g], 0));
        TSR_CUDA(cudaStreamWaitEvent(sa, hc.ev[1], 0));
        FwdArgs a;
        a.q = dq;
        a.k = dk;
        a.v = dv;
        a.out = dout;
        a.lse = static_cast<float*>(dlse);
        a.plan = hc.full_plan;
        a.item_lo = gs[g] * nqt;
        a.item_hi = gs[g + 1] * nqt;
        a.counter = hc.counters + g;
        s = launch_forward(a, sa);
        if (s != TSR_OK) break;
        TSR_CUDA(cudaEventRecord(hc.ev[3 * g + 2], sa));
        TSR_CUDA(cudaStreamWaitEvent(hc.s_out, hc.ev[3 * g + 2], 0));
        TSR_CUDA(cudaMemcpyAsync(static_cast<char*>(out) + off, static_cast<char*>(dout) + off, n,
                                 cudaMemcpyDeviceToHost, hc.s_out));
        TSR_CUDA(cudaMemcpyAsync(lse + b0 * mask->N, static_cast<float*>(dlse) + b0 * mask->N,
                                 static_cast<size_t>(n / row_b) * mask->N * 4,
                                 cudaMemcpyDeviceToHost, hc.s_out));
      }
      if (s == TSR_OK) {
        TSR_CUDA(cudaMemcpyAsync(hc.host_err, hc.full_plan->err, sizeof(uint32_t),
                                 cudaMemcpyDeviceToHost, hc.s_out));
        TSR_CUDA(cudaMemsetAsync(hc.full_plan->err, 0, sizeof(uint32_t), hc.s_out));
      }
    } else {
      for (int64_t g = 0; g < G && s == TSR_OK; ++g) {
        s = plan_group(g);
        if (s == TSR_OK) s = launch_group(g);
      }
    }
    return s;
  }();
  tsr_status s = s_run;
  // no copy may still read or write the caller's buffers after the return
  const cudaError_t e1 = cudaStreamSynchronize(hc.s_out);
  const cudaError_t e2 = cudaStreamSynchronize(hc.stream);
  const cudaError_t e4 = cudaStreamSynchronize(hc.stream2);
  const cudaError_t e3 = cudaStreamSynchronize(hc.s_in);
  const cudaError_t e5 = cudaStreamSynchronize(sp);
  if (s == TSR_OK && e1 != cudaSuccess) s = cuda_fail(e1, "copy of the outputs to host");
  if (s == TSR_OK && (e2 != cudaSuccess || e4 != cudaSuccess))
    s = cuda_fail(e2 != cudaSuccess ? e2 : e4, "attention stream");
  if (s == TSR_OK && e3 != cudaSuccess) s = cuda_fail(e3, "copy of the inputs");
  if (s == TSR_OK && e5 != cudaSuccess) s = cuda_fail(e5, "plan stream");
  for (int64_t g = 0; g < n_err && s == TSR_OK; ++g) {
    const uint32_t e = hc.host_err[g];
    if (e & DEV_ERR_TIMEOUT) s = fail(TSR_ERR_TIMEOUT, "a device-side wait timed out");
    else if (e) s = fail(TSR_ERR_INTERNAL, "device error word " + std::to_string(e));
  }
  return s;
}

void tsr_release_host_buffers(void) { g_host_cache.release(); }

tsr_status tsr_regime_load(const char* path) {
  std::lock_guard<std::mutex> lk(g_table_mu);
  std::string why;
  if (!path) {
    parse_table(kBuiltinTable, &g_table, &why);
    g_table_loaded = true;
    return TSR_OK;
  }
  std::ifstream f(path);
  if (!f) return fail(TSR_ERR_INVALID_ARG, std::string("cannot open regime table ") + path);
  std::stringstream ss;
  ss << f.rdbuf();
  std::vector<RegimeRow> rows;
  if (!parse_table(ss.str(), &rows, &why)) return fail(TSR_ERR_INVALID_ARG, "regime table: " + why);
  if (!rows_valid(rows))
    return fail(TSR_ERR_INVALID_ARG, "regime table names a kernel variant that does not exist");
  g_table = rows;
  g_table_loaded = true;
  return TSR_OK;
}

tsr_status tsr_regime_lookup(int32_t kind, int32_t bq, int32_t bk, int32_t N, double density,
                             tsr_regime* out) {
  if (!out) return fail(TSR_ERR_INVALID_ARG, "out is NULL");
  const Regime r = regime_lookup(kind, bq, bk, N, density, 128);
  out->bn = r.bn;
  out->stages = r.stages;
  out->ctas_per_sm = r.ctas;
  out->id = r.id;
  out->orient = r.orient;
  return TSR_OK;
}

}  // extern "C"
