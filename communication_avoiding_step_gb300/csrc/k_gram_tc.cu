// Step a3 on tcgen05 tensor cores (sm_103a): not built yet in this revision; the
// CUDA-core kernel serves every shape meanwhile.
#include "casgd_internal.cuh"

namespace casgd {

bool gram_tc_supported(int64_t, int64_t, int) { return false; }

cudaError_t launch_gram_tc(const uint16_t*, int64_t, int64_t, int64_t, int, int, bool, float*,
                           Ctrl*, uint32_t, Ctx&) {
  return cudaErrorNotSupported;
}

}  // namespace casgd
