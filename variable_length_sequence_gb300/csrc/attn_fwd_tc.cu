// tcgen05 forward path (not yet enabled: the dispatcher falls back to the
// CUDA-core kernel).
#include "nsp_internal.cuh"

namespace nsp {

cudaError_t launch_attn_fwd_tc(const AttnProblem& p, const FwdWsLayout& L, char* ws,
                               cudaStream_t s, bool* launched) {
  (void)p; (void)L; (void)ws; (void)s;
  *launched = false;
  return cudaSuccess;
}

}  // namespace nsp
