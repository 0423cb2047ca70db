// noalloc.cu -- block-sparse attention that allocates no device memory.
//
// tsr_plan() allocates the plan (tile lists, descriptors, counters) with
// cudaMalloc, and frees its temporaries with cudaFree, which also waits for the
// whole device.  Some callers cannot do that: code that must take all device
// memory from its own pool or budget (an inference server that reserved the GPU
// up front, a framework allocator that forbids raw cudaMalloc), and code on a
// latency-critical path where cudaMalloc / cudaFree and their implicit device
// synchronisation are not acceptable.  tsr_attention_noalloc() serves them: it
// plans into, and runs the attention over, one fixed scratch array compiled into
// the library (a file-scope __device__ array), so it makes no allocation of its
// own.  The caller still owns and passes Q, K, V, O and lse.
//
// Limits and rules (also stated in include/tsr.h):
//   * the scratch array holds kStaticScratchBytes (32 MiB) on every GPU that
//     loads the library, until the process exits;
//   * a call whose plan does not fit is rejected with TSR_ERR_UNSUPPORTED before
//     the attention runs;
//   * every call shares the array, and calls whose GPU work overlaps (two host
//     threads, or two streams) race on it; serialise them;
//   * the first call on a device (and the first in each new CUDA context on it)
//     looks up the array's device address (cudaGetSymbolAddress); make that
//     first call before any stream capture begins;
//   * every call synchronises its stream (to size the plan and to read the
//     device error word).
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#include <string>

#include "internal.h"
#include "ptx.cuh"

// The scratch array itself.  In host code this name is only a host-side handle
// for the symbol, not a device address: the device address comes from
// cudaGetSymbolAddress below.
static constexpr size_t kStaticScratchBytes = size_t{32} << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace tsr {

namespace {

std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {nullptr};
CUcontext g_scratch_ctx[64] = {nullptr};   // the context each address belongs to

// The calling thread's current CUDA context (the driver entry point is looked
// up through the runtime, so the library needs no link against libcuda).
CUcontext current_context() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        p == nullptr || q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  }
  CUcontext c = nullptr;
  return fn(&c) == CUDA_SUCCESS ? c : nullptr;
}

// Device address of the scratch array on `device` (which must be current):
// looked up on the first call on the device, and again whenever the current
// context is not the one the cached address was taken in (after
// cudaDeviceReset, or under another context), so a stale address is never used.
tsr_status scratch_address(int device, unsigned char** out) {
  if (device < 0 || device >= 64) return fail(TSR_ERR_UNSUPPORTED, "device index above 63");
  const CUcontext ctx = current_context();   // null before the runtime has set one up
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[device] || ctx == nullptr || g_scratch_ctx[device] != ctx) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      g_scratch_addr[device] = nullptr;
      return cuda_fail(e == cudaSuccess ? cudaErrorInvalidSymbol : e,
                       "cudaGetSymbolAddress of the static scratch array");
    }
    g_scratch_addr[device] = p;
    g_scratch_ctx[device] = current_context();   // the context the lookup ran in
  }
  *out = static_cast<unsigned char*>(g_scratch_addr[device]);
  return TSR_OK;
}

size_t round256(size_t x) { return (x + 255) & ~size_t{255}; }

// Segment bounds must run 0 .. N and ascend; read back in fixed-size chunks.
tsr_status check_bounds_chunked(const int32_t* dev, int32_t n, int32_t N, cudaStream_t st) {
  int32_t buf[1024];
  int32_t prev = -1;
  for (int32_t base = 0; base <= n; base += 1024) {
    const int32_t cnt = std::min<int32_t>(1024, n + 1 - base);
    TSR_CUDA(cudaMemcpyAsync(buf, dev + base, sizeof(int32_t) * cnt, cudaMemcpyDeviceToHost, st));
    TSR_CUDA(cudaStreamSynchronize(st));
    for (int32_t i = 0; i < cnt; ++i) {
      const int32_t v = buf[i];
      if ((base + i == 0 && v != 0) || (base + i == n && v != N) || v <= prev)
        return fail(TSR_ERR_INVALID_ARG, "segment bounds must ascend from 0 to N");
      prev = v;
    }
  }
  return TSR_OK;
}

}  // namespace

}  // namespace tsr

using namespace tsr;

extern "C" tsr_status tsr_attention_noalloc(const tsr_mask* mask, const void* q, const void* k,
                                            const void* v, void* out, float* lse, void* stream) {
  set_error("");
  if (!mask) return fail(TSR_ERR_INVALID_ARG, "mask is NULL");
  if (mask->kind != TSR_MASK_UNIFORM && mask->kind != TSR_MASK_SEGMENTS)
    return fail(TSR_ERR_UNSUPPORTED,
                "tsr_attention_noalloc plans UNIFORM and SEGMENTS masks only; use tsr_plan for "
                "SVG and KEYLIST masks");
  if (mask->B <= 0 || mask->H <= 0 || mask->N <= 0 || (mask->d != 64 && mask->d != 128))
    return fail(TSR_ERR_INVALID_ARG, "B, H, N must be > 0 and d 64 or 128");
  if (mask->N > (1 << 24)) return fail(TSR_ERR_UNSUPPORTED, "N above 2^24");
  if (mask->kind == TSR_MASK_UNIFORM && (mask->bq < 16 || mask->bk < 16 || !mask->blocks))
    return fail(TSR_ERR_INVALID_ARG, "UNIFORM needs bq, bk >= 16 and blocks");
  if (mask->kind == TSR_MASK_SEGMENTS &&
      (mask->n_qseg <= 0 || mask->n_kseg <= 0 || !mask->q_bounds || !mask->k_bounds || !mask->blocks))
    return fail(TSR_ERR_INVALID_ARG, "segment bounds / blocks missing");
  if (!q || !k || !v || !out || !lse) return fail(TSR_ERR_INVALID_ARG, "NULL tensor pointer");
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out) || misaligned(lse))
    return fail(TSR_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (out == q || out == k || out == v) return fail(TSR_ERR_INVALID_ARG, "out aliases an input");

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0;
  TSR_CUDA(cudaGetDevice(&dev));
  unsigned char* base = nullptr;
  if (tsr_status s = scratch_address(dev, &base)) return s;
  if (mask->kind == TSR_MASK_SEGMENTS) {
    if (tsr_status s = check_bounds_chunked(mask->q_bounds, mask->n_qseg, mask->N, st)) return s;
    if (tsr_status s = check_bounds_chunked(mask->k_bounds, mask->n_kseg, mask->N, st)) return s;
  }

  const int32_t B = mask->B, H = mask->H, N = mask->N;
  const int32_t nqt = (N + kBM - 1) / kBM;
  const int64_t n_items = static_cast<int64_t>(B) * H * nqt;
  // layout: [err, counter | totals | per-tile counts (4 x n_items) | ... rest after counting]
  uint32_t* err = reinterpret_cast<uint32_t*>(base);
  int32_t* counter = reinterpret_cast<int32_t*>(base + 4);
  unsigned long long* tot = reinterpret_cast<unsigned long long*>(base + 256);
  size_t off = 512;
  int32_t* cnt = reinterpret_cast<int32_t*>(base + off);
  off += round256(sizeof(int32_t) * 4 * static_cast<size_t>(n_items));
  if (off > kStaticScratchBytes)
    return fail(TSR_ERR_UNSUPPORTED, "problem too large for the 32 MiB static scratch (" +
                                         std::to_string(n_items) + " query tiles)");
  // the array keeps the previous call's contents: clear the error word, the
  // work counter and the totals, which are accumulated with atomics
  TSR_CUDA(cudaMemsetAsync(base, 0, 512, st));

  MaskDev m;
  memset(&m, 0, sizeof m);
  m.kind = mask->kind;
  m.B = B;
  m.H = H;
  m.N = N;
  m.bq = mask->bq;
  m.bk = mask->bk;
  m.n_qseg = mask->n_qseg;
  m.n_kseg = mask->n_kseg;
  m.q_bounds = mask->q_bounds;
  m.k_bounds = mask->k_bounds;
  m.blocks = mask->blocks;
  const int64_t n_grid =
      (m.kind == TSR_MASK_UNIFORM)
          ? static_cast<int64_t>(B) * H * ((N + m.bq - 1) / m.bq) * ((N + m.bk - 1) / m.bk)
          : static_cast<int64_t>(B) * H * m.n_qseg * m.n_kseg;
  if (tsr_status s = plan_count_into(m, nqt, cnt, tot, err, n_grid, st)) return s;
  unsigned long long host_tot[8];
  uint32_t host_err = 0;
  TSR_CUDA(cudaMemcpyAsync(host_tot, tot, sizeof host_tot, cudaMemcpyDeviceToHost, st));
  TSR_CUDA(cudaMemcpyAsync(&host_err, err, sizeof host_err, cudaMemcpyDeviceToHost, st));
  TSR_CUDA(cudaStreamSynchronize(st));
  if (host_err & DEV_ERR_UNSUPPORTED)
    return fail(TSR_ERR_UNSUPPORTED, "a 128-token tile overlaps more than 8 logical segments");
  if (host_err) return fail(TSR_ERR_INTERNAL, "planner error word " + std::to_string(host_err));

  const double density = static_cast<double>(host_tot[6]) / static_cast<double>(n_grid);
  // the table's regime, completed to a compiled variant of the 128-row tiles
  // this planner builds
  tsr_plan_opts rows_only{};
  rows_only.orient = TSR_ORIENT_ROWS;
  Regime rg;
  if (tsr_status s = resolve_regime(regime_lookup(m.kind, m.bq, m.bk, N, density, mask->d),
                                    &rows_only, mask->d, false, &rg))
    return s;
  const int which = (rg.bn == 64) ? 0 : 1;
  const int64_t n_entries = static_cast<int64_t>(host_tot[2 * which]);
  const int64_t n_desc = static_cast<int64_t>(host_tot[2 * which + 1]);
  const int64_t max_len = static_cast<int64_t>(host_tot[4 + which]);

  int32_t* ebegin = reinterpret_cast<int32_t*>(base + off);
  off += round256(sizeof(int32_t) * static_cast<size_t>(n_items));
  int32_t* dbegin = reinterpret_cast<int32_t*>(base + off);
  off += round256(sizeof(int32_t) * static_cast<size_t>(n_items));
  int32_t* hist = reinterpret_cast<int32_t*>(base + off);
  off += round256(sizeof(int32_t) * static_cast<size_t>(max_len + 2));
  void* items = base + off;
  off += round256(sizeof(tsr_plan_item) * static_cast<size_t>(n_items));
  void* entries = base + off;
  off += round256(sizeof(tsr_plan_entry) * static_cast<size_t>(n_entries));
  void* descs = base + off;
  off += round256(sizeof(tsr_tile_desc) * static_cast<size_t>(n_desc));
  if (off > kStaticScratchBytes)
    return fail(TSR_ERR_UNSUPPORTED,
                "plan needs " + std::to_string(off) + " bytes of scratch; the static scratch "
                "holds " + std::to_string(kStaticScratchBytes) + " (32 MiB): use tsr_plan");

  if (tsr_status s = plan_finish_into(m, nqt, rg.bn, cnt + (2 * which) * n_items,
                                      cnt + (2 * which + 1) * n_items,
                                      static_cast<int32_t>(max_len), ebegin, dbegin, hist, items,
                                      entries, descs, st))
    return s;

  tsr_plan_impl P;
  P.device = dev;
  P.B = B;
  P.H = H;
  P.N = N;
  P.d = mask->d;
  P.kind = mask->kind;
  P.bn = rg.bn;
  P.stages = rg.stages;
  P.ctas = rg.ctas;
  P.regime_id = rg.id;
  P.n_items = n_items;
  P.n_entries = n_entries;
  P.n_desc = n_desc;
  P.items = items;
  P.entries = entries;
  P.descs = descs;
  P.counter = counter;
  P.err = err;
  FwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.plan = &P;
  if (tsr_status s = launch_forward(a, st)) return s;
  TSR_CUDA(cudaMemcpyAsync(&host_err, err, sizeof host_err, cudaMemcpyDeviceToHost, st));
  TSR_CUDA(cudaStreamSynchronize(st));
  if (host_err & DEV_ERR_TIMEOUT) return fail(TSR_ERR_TIMEOUT, "a device-side wait timed out");
  if (host_err) return fail(TSR_ERR_INTERNAL, "device error word " + std::to_string(host_err));
  return TSR_OK;
}
