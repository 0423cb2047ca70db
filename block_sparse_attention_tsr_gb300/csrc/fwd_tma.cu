// fwd_tma.cu -- forward kernel variants of mode kModeTma (every tile loaded by TMA).
#include "fwd_kernel.cuh"

namespace tsr {
namespace fwd {

tsr_status launch_mode_tma(const FwdParams& prm, int key, int n_items, int device,
                           cudaStream_t stream) {
#define TSR_LAUNCH(D_, BN_, S_, C_) \
  if (key == vkey(D_, BN_, S_, C_)) return launch_variant<D_, BN_, S_, C_, kModeTma, 1>(prm, n_items, device, stream);
  TSR_VARIANTS_CONTIGUOUS(TSR_LAUNCH)
#undef TSR_LAUNCH
  return TSR_ERR_UNSUPPORTED;
}

tsr_status launch_mode_tma(const FwdParamsBatch& prm, int key, int n_items, int device,
                           cudaStream_t stream) {
#define TSR_LAUNCH(D_, BN_, S_, C_) \
  if (key == vkey(D_, BN_, S_, C_))                                                         \
    return launch_variant<D_, BN_, S_, C_, kModeTma, kMaxBatch>(prm, n_items, device, stream);
  TSR_VARIANTS_BATCH(TSR_LAUNCH)
#undef TSR_LAUNCH
  return TSR_ERR_UNSUPPORTED;
}

}  // namespace fwd
}  // namespace tsr
