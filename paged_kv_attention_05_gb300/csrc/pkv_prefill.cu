// Prefill / chunk attention (requests with more than one query token).
// Placeholder launcher: the tensor-core kernel is added next.
#include "pkv_internal.cuh"

namespace pkv {

cudaError_t launch_prefill(const AttnArgs& a, const Workspace& ws, int sms, cudaStream_t st) {
  (void)a;
  (void)ws;
  (void)sms;
  (void)st;
  return cudaSuccess;
}

}  // namespace pkv
