// fwd_perm.cu -- forward kernel variants of mode kModePerm (temporal-major items gathered through the inverse permutation).
#include "fwd_kernel.cuh"

namespace tsr {
namespace fwd {

tsr_status launch_mode_perm(const FwdParams& prm, int key, int n_items, int device,
                            cudaStream_t stream) {
#define TSR_LAUNCH(D_, BN_, S_, C_) \
  if (key == vkey(D_, BN_, S_, C_)) return launch_variant<D_, BN_, S_, C_, kModePerm, 1>(prm, n_items, device, stream);
  TSR_VARIANTS_CONTIGUOUS(TSR_LAUNCH)
#undef TSR_LAUNCH
  return TSR_ERR_UNSUPPORTED;
}

tsr_status launch_mode_perm(const FwdParamsBatch& prm, int key, int n_items, int device,
                            cudaStream_t stream) {
#define TSR_LAUNCH(D_, BN_, S_, C_) \
  if (key == vkey(D_, BN_, S_, C_))                                                         \
    return launch_variant<D_, BN_, S_, C_, kModePerm, kMaxBatch>(prm, n_items, device, stream);
  TSR_VARIANTS_BATCH(TSR_LAUNCH)
#undef TSR_LAUNCH
  return TSR_ERR_UNSUPPORTED;
}

}  // namespace fwd
}  // namespace tsr
