// Prefill path of the HC gated residual (tensor-core kernels).
#include "hc_gr_internal.cuh"

namespace hcgr {

size_t prefill_ws_bytes(int64_t max_M, int HC, int HS, int r) {
  (void)max_M; (void)HC; (void)HS; (void)r;
  return 0;
}

cudaError_t launch_prefill(const Call& c, const Workspace& ws, const Device& dev,
                           cudaStream_t stream) {
  (void)c; (void)ws; (void)dev; (void)stream;
  return cudaErrorNotSupported;
}

}  // namespace hcgr
