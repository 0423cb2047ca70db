// fwd.cu -- host side of the forward pass: tensor maps, kernel parameters,
// the compiled-variant registry and the dispatch to the per-mode translation
// units (the kernel itself is in fwd_kernel.cuh).
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <memory>
#include <new>
#include <string>

#include "fwd_kernel.cuh"
#include "fwd_t_kernel.cuh"
#include "internal.h"

namespace tsr {

using fwd::FwdParams;
using fwd::vkey;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool get_encode() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      fn == nullptr || q != cudaDriverEntryPointSuccess)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

}  // namespace

bool encode_tmap_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                    uint64_t outer, uint32_t box_inner, uint32_t box_rows) {
  if (!get_encode()) return false;
  cuuint64_t dims[3] = {inner, rows, outer};
  cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool variant_exists(int d, int bn, int stages, int ctas, bool gathered) {
  const int key = vkey(d, bn, stages, ctas);
#define TSR_CHECK(D_, BN_, S_, C_) if (key == vkey(D_, BN_, S_, C_)) return true;
  if (gathered) {
    TSR_VARIANTS_GATHERED(TSR_CHECK)
  } else {
    TSR_VARIANTS_CONTIGUOUS(TSR_CHECK)
  }
#undef TSR_CHECK
  return false;
}

// Complete a partly specified regime: fields given as 0 are free; the first
// compiled variant that matches every given field is taken.
bool variant_pick(int d, bool gathered, int bn, int stages, int ctas, int* out_bn, int* out_st,
                  int* out_ct) {
#define TSR_PICK(D_, BN_, S_, C_)                                                         \
  if (D_ == d && (!bn || bn == BN_) && (!stages || stages == S_) && (!ctas || ctas == C_)) { \
    *out_bn = BN_;                                                                        \
    *out_st = S_;                                                                         \
    *out_ct = C_;                                                                         \
    return true;                                                                          \
  }
  if (gathered) {
    TSR_VARIANTS_GATHERED(TSR_PICK)
  } else {
    TSR_VARIANTS_CONTIGUOUS(TSR_PICK)
  }
#undef TSR_PICK
  return false;
}

tsr_status launch_forward(const FwdArgs& a, cudaStream_t stream) {
  return launch_forward_batch(&a, 1, stream);
}

tsr_status launch_forward_batch(const FwdArgs* reqs, int n_req, cudaStream_t stream) {
  if (n_req < 1 || n_req > fwd::kMaxBatch)
    return fail(TSR_ERR_INVALID_ARG, "1 to " + std::to_string(fwd::kMaxBatch) + " requests per call");
  const tsr_plan_impl* P0 = reqs[0].plan;
  // one launch needs one kernel variant: the same head dimension, regime and
  // gather mode for every request; temporal heads anywhere select the variant
  // that may gather through the permutation, unless the per-position kernel
  // takes them
  bool temporal = false;
  // each request's range in its launch list, and the heads whose temporal
  // blocks the per-position kernel computes
  int64_t lo_of[fwd::kMaxBatch], hi_of[fwd::kMaxBatch], bh_lo[fwd::kMaxBatch], bh_hi[fwd::kMaxBatch];
  for (int r = 0; r < n_req; ++r) {
    const tsr_plan_impl* P = reqs[r].plan;
    if (P->device != P0->device || P->d != P0->d || P->bn != P0->bn || P->stages != P0->stages ||
        P->ctas != P0->ctas || P->gathered != P0->gathered || P->orient != P0->orient)
      return fail(TSR_ERR_UNSUPPORTED,
                  "requests of one batch need the same d, regime (orientation, bn, stages, ctas) "
                  "and mask family (key lists or not); plan them with the same tsr_plan_opts");
    temporal = temporal || (P->n_temporal > 0 && !P->temporal_band);
    const int64_t ilo = reqs[r].item_lo, ihi = reqs[r].item_hi < 0 ? P->n_items : reqs[r].item_hi;
    if (ilo < 0 || ihi > P->n_items || ilo > ihi) return fail(TSR_ERR_INTERNAL, "bad item range");
    lo_of[r] = ilo;
    hi_of[r] = ihi;
    bh_lo[r] = bh_hi[r] = 0;
    if (P->temporal_band) {
      // whole heads: the plan's items are in head order (one head per
      // scheduling group), nqt of them per head, unless the range is all items
      const int64_t BH = static_cast<int64_t>(P->B) * P->H, nqt = (P->N + P->bm - 1) / P->bm;
      if (ilo == 0 && ihi == P->n_items) {
        bh_hi[r] = BH;
      } else {
        if (P->group_heads != 1 || ilo % nqt || ihi % nqt)
          return fail(TSR_ERR_INTERNAL, "item range of a plan with separate temporal heads");
        bh_lo[r] = ilo / nqt;
        bh_hi[r] = ihi / nqt;
      }
      lo_of[r] = nqt * P->spatial_before[bh_lo[r]];
      hi_of[r] = nqt * P->spatial_before[bh_hi[r]];
    }
  }
  // SVG temporal heads by spatial position run on a plan's own stream, forked
  // from `stream` here (after everything queued before this call) and joined
  // after the attention launch: launched after the persistent attention grid,
  // their CTAs take the SMs that grid leaves idle in its tail
  const tsr_plan_impl* Pb = nullptr;
  for (int r = 0; r < n_req && !Pb; ++r)
    if (reqs[r].plan->temporal_band) Pb = reqs[r].plan;
  if (Pb) TSR_CUDA(cudaEventRecord(Pb->band_fork, stream));
  const int key = vkey(P0->d, P0->bn, P0->stages, P0->ctas);
  auto fill = [&](auto& prm) -> tsr_status {
    memset(&prm, 0, sizeof prm);
    int64_t total = 0;
    for (int r = 0; r < n_req; ++r) {
      const FwdArgs& a = reqs[r];
      const tsr_plan_impl* P = a.plan;
      fwd::ReqParams& q = prm.req[r];
      const uint64_t D = P->d, N = P->N, BH = static_cast<uint64_t>(P->B) * P->H;
      // key-major plans load 64-row boxes everywhere (a query block, and each
      // 64-key tile of a step)
      const uint32_t qrows = P->orient == TSR_ORIENT_KEYS ? 64 : kBM;
      const uint32_t krows = P->orient == TSR_ORIENT_KEYS ? 64 : P->bn;
      const bool ok = encode_tmap_3d(&q.tq, a.q, D, N, BH, 64, qrows) &&
                      encode_tmap_3d(&q.tk, a.k, D, N, BH, 64, krows) &&
                      encode_tmap_3d(&q.tv, a.v, D, N, BH, 64, krows);
      if (!ok)
        return fail(TSR_ERR_CUDA, "cuTensorMapEncodeTiled failed (pointer alignment or shape)");
      // the range is in launch-list items; a split plan launches their units
      const int64_t ilo = lo_of[r], ihi = hi_of[r];
      const bool split = P->kv_split > 1;
      const int64_t lo = ilo * P->kv_split, hi = ihi * P->kv_split;
      q.items = static_cast<const int4*>(split ? P->units : P->temporal_band ? P->launch : P->items) +
                2 * lo;
      if (split) {
        q.part_o = static_cast<float*>(P->b_part_o.p);
        q.part_lse = static_cast<float*>(P->b_part_lse.p);
        q.part_cnt = static_cast<int32_t*>(P->b_part_cnt.p);
        if (ihi > ilo)
          TSR_CUDA(cudaMemsetAsync(q.part_cnt + ilo, 0, sizeof(int32_t) * (ihi - ilo), stream));
      }
      q.entries = static_cast<const int2*>(P->entries);
      q.descs = static_cast<const uint4*>(P->descs);
      q.out = static_cast<__nv_bfloat16*>(a.out);
      q.lse = a.lse;
      q.qg = static_cast<const __nv_bfloat16*>(a.q);
      q.kg = static_cast<const __nv_bfloat16*>(a.k);
      q.vg = static_cast<const __nv_bfloat16*>(a.v);
      q.gidx = P->gidx;
      q.item_begin = static_cast<int32_t>(total);
      q.N = P->N;
      q.F = P->F;
      q.S = P->S;
      q.slice_m = P->slice_m;
      total += hi - lo;
    }
    if (total >= (int64_t{1} << 31)) return fail(TSR_ERR_UNSUPPORTED, "more than 2^31 work items");
    prm.n_req = n_req;
    prm.n_items = static_cast<int32_t>(total);
    prm.counter = reqs[0].counter ? reqs[0].counter : P0->counter;
    prm.err = P0->err;
    prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(P0->d)));
    prm.tiles_done = ((P0->flags & TSR_PLAN_DEBUG_CHECKS) && P0->b_tot.p)
                         ? static_cast<unsigned long long*>(P0->b_tot.p) + 7
                         : nullptr;
    prm.test_stall = (P0->flags & TSR_PLAN_TEST_STALL) ? 1 : 0;
    prm.timeout_ns = prm.test_stall ? 100000000ull : kWaitTimeoutNs;
    return TSR_OK;
  };
  // KEYLIST plans gather K / V by key list; plans with temporal-major heads take
  // the variant that may gather through the permutation; the rest are TMA only.
  auto launch = [&](const auto& prm) -> tsr_status {
    if (prm.tiles_done)
      TSR_CUDA(cudaMemsetAsync(prm.tiles_done, 0, sizeof(unsigned long long), stream));
    if (prm.n_items == 0) return TSR_OK;
    TSR_CUDA(cudaMemsetAsync(prm.counter, 0, sizeof(int32_t), stream));
    const int n = prm.n_items, dev = P0->device;
    if (P0->orient == TSR_ORIENT_KEYS) {
      const int mode = P0->gathered ? fwd::kModeList : temporal ? fwd::kModePerm : fwd::kModeTma;
      return fwd_t::launch_t_mode(prm, mode, n, dev, stream);
    }
    if (P0->gathered) return fwd::launch_mode_list(prm, key, n, dev, stream);
    if (temporal) return fwd::launch_mode_perm(prm, key, n, dev, stream);
    return fwd::launch_mode_tma(prm, key, n, dev, stream);
  };
  tsr_status st;
  if (n_req == 1) {
    FwdParams prm;
    if (tsr_status e = fill(prm)) return e;
    st = launch(prm);
  } else {
    std::unique_ptr<fwd::FwdParamsBatch> prm(new (std::nothrow) fwd::FwdParamsBatch);
    if (!prm) return fail(TSR_ERR_OOM, "host allocation failed");
    if (tsr_status e = fill(*prm)) return e;
    st = launch(*prm);
  }
  if (st == TSR_OK && Pb) {
    TSR_CUDA(cudaStreamWaitEvent(Pb->band_stream, Pb->band_fork, 0));
    for (int r = 0; r < n_req; ++r) {
      const tsr_plan_impl* P = reqs[r].plan;
      if (!P->temporal_band) continue;
      if (tsr_status e = launch_svg_temporal(reqs[r].q, reqs[r].k, reqs[r].v, reqs[r].out, reqs[r].lse,
                                             P->H, P->N, P->d, P->F, P->S, P->head_kind_dev,
                                             bh_lo[r], bh_hi[r], Pb->band_stream))
        return e;
    }
    TSR_CUDA(cudaEventRecord(Pb->band_join, Pb->band_stream));
    TSR_CUDA(cudaStreamWaitEvent(stream, Pb->band_join, 0));
  }
  if (st != TSR_ERR_UNSUPPORTED) return st;
  return fail(TSR_ERR_UNSUPPORTED, "no kernel variant for d=" + std::to_string(P0->d) + " bn=" +
                                       std::to_string(P0->bn) + " stages=" +
                                       std::to_string(P0->stages) + " ctas=" +
                                       std::to_string(P0->ctas) +
                                       (P0->gathered ? " (gathered)" : "") +
                                       (n_req > 1 ? " in batched launches" : ""));
}

}  // namespace tsr
