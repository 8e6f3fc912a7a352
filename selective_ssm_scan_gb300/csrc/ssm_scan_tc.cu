// tcgen05 tensor-core chunked scan (placeholder until the kernel lands).
#include "common.cuh"

namespace sss {

bool ssm_scan_tc_supports(sss_dtype, sss_dtype, sss_dtype, int64_t, int, int, int, int) {
  return false;
}

cudaError_t ssm_scan_tc_launch(const void*, sss_dtype, const void*, const float*, const void*,
                               const void*, const float*, float*, void*, sss_dtype, int64_t,
                               int64_t, int, int, int, int, int*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace sss
