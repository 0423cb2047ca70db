// fwd_list.cu -- forward kernel variants of mode kModeList (K / V rows gathered from key lists).
#include "fwd_kernel.cuh"

namespace tsr {
namespace fwd {

tsr_status launch_mode_list(const FwdParams& prm, int key, int n_items, int device,
                            cudaStream_t stream) {
#define TSR_LAUNCH(D_, BN_, S_, C_) \
  if (key == vkey(D_, BN_, S_, C_)) return launch_variant<D_, BN_, S_, C_, kModeList, 1>(prm, n_items, device, stream);
  TSR_VARIANTS_GATHERED(TSR_LAUNCH)
#undef TSR_LAUNCH
  return TSR_ERR_UNSUPPORTED;
}

tsr_status launch_mode_list(const FwdParamsBatch& prm, int key, int n_items, int device,
                            cudaStream_t stream) {
#define TSR_LAUNCH(D_, BN_, S_, C_) \
  if (key == vkey(D_, BN_, S_, C_))                                                         \
    return launch_variant<D_, BN_, S_, C_, kModeList, kMaxBatch>(prm, n_items, device, stream);
  TSR_VARIANTS_BATCH(TSR_LAUNCH)
#undef TSR_LAUNCH
  return TSR_ERR_UNSUPPORTED;
}

}  // namespace fwd
}  // namespace tsr
