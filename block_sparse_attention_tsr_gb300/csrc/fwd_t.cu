// fwd_t.cu -- instantiations of the key-major (transposed) attention kernel:
// TMA mode (block masks, segments, SVG without temporal heads), permuted-gather
// mode (SVG with temporal heads) and key-list gathers.
#include "fwd_t_kernel.cuh"

namespace tsr {
namespace fwd_t {

tsr_status launch_t_mode(const fwd::FwdParams& prm, int mode, int n_items, int device,
                         cudaStream_t stream) {
  switch (mode) {
    case kModeTma: return launch_t<kModeTma, 1>(prm, n_items, device, stream);
    case kModePerm: return launch_t<kModePerm, 1>(prm, n_items, device, stream);
    case kModeList: return launch_t<kModeList, 1>(prm, n_items, device, stream);
  }
  return TSR_ERR_UNSUPPORTED;
}

tsr_status launch_t_mode(const fwd::FwdParamsBatch& prm, int mode, int n_items, int device,
                         cudaStream_t stream) {
  switch (mode) {
    case kModeTma: return launch_t<kModeTma, fwd::kMaxBatch>(prm, n_items, device, stream);
    case kModePerm: return launch_t<kModePerm, fwd::kMaxBatch>(prm, n_items, device, stream);
    case kModeList: return launch_t<kModeList, fwd::kMaxBatch>(prm, n_items, device, stream);
  }
  return TSR_ERR_UNSUPPORTED;
}

}  // namespace fwd_t
}  // namespace tsr
