// fwd.cu -- host side of the forward pass: tensor maps, kernel parameters,
// the compiled-variant registry and the dispatch to the per-mode translation
// units (the kernel itself is in fwd_kernel.cuh).
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <string>

#include "fwd_kernel.cuh"
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
  const tsr_plan_impl* P = a.plan;
  if (P->n_items == 0) return TSR_OK;
  FwdParams prm;
  memset(&prm, 0, sizeof prm);
  const uint64_t D = P->d, N = P->N, BH = static_cast<uint64_t>(P->B) * P->H;
  bool ok = encode_tmap_3d(&prm.tq, a.q, D, N, BH, 64, kBM) &&
            encode_tmap_3d(&prm.tk, a.k, D, N, BH, 64, P->bn) &&
            encode_tmap_3d(&prm.tv, a.v, D, N, BH, 64, P->bn);
  if (!ok) return fail(TSR_ERR_CUDA, "cuTensorMapEncodeTiled failed (pointer alignment or shape)");
  prm.items = static_cast<const int4*>(P->items);
  prm.entries = static_cast<const int2*>(P->entries);
  prm.descs = static_cast<const uint4*>(P->descs);
  prm.out = static_cast<__nv_bfloat16*>(a.out);
  prm.lse = a.lse;
  prm.counter = P->counter;
  prm.err = P->err;
  prm.n_items = static_cast<int32_t>(P->n_items);
  prm.N = P->N;
  prm.F = P->F;
  prm.S = P->S;
  prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(P->d)));
  prm.qg = static_cast<const __nv_bfloat16*>(a.q);
  prm.kg = static_cast<const __nv_bfloat16*>(a.k);
  prm.vg = static_cast<const __nv_bfloat16*>(a.v);
  prm.gidx = P->gidx;
  prm.slice_m = P->slice_m;
  prm.test_stall = (P->flags & TSR_PLAN_TEST_STALL) ? 1 : 0;
  prm.timeout_ns = prm.test_stall ? 100000000ull : kWaitTimeoutNs;
  TSR_CUDA(cudaMemsetAsync(P->counter, 0, sizeof(int32_t), stream));
  const int n = static_cast<int>(P->n_items), dev = P->device;
  const int key = vkey(P->d, P->bn, P->stages, P->ctas);
  // KEYLIST plans gather K / V by key list; plans with temporal-major heads take
  // the variant that may gather through the permutation; the rest are TMA only.
  tsr_status st;
  if (P->gathered)
    st = fwd::launch_mode_list(prm, key, n, dev, stream);
  else if (P->n_temporal > 0)
    st = fwd::launch_mode_perm(prm, key, n, dev, stream);
  else
    st = fwd::launch_mode_tma(prm, key, n, dev, stream);
  if (st != TSR_ERR_UNSUPPORTED) return st;
  return fail(TSR_ERR_UNSUPPORTED, "no kernel variant for d=" + std::to_string(P->d) + " bn=" +
                                       std::to_string(P->bn) + " stages=" +
                                       std::to_string(P->stages) + " ctas=" +
                                       std::to_string(P->ctas) +
                                       (P->gathered ? " (gathered)" : ""));
}

}  // namespace tsr
