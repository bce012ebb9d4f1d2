// Self-test of the on-chip wait bound.  The decode kernels wait on shared-memory
// barriers (copies landing, contractions finishing) through one bounded wait:
// a wait that runs out sets GDN_DEV_TIMEOUT and the block returns instead of
// hanging.  This kernel runs that same wait on a barrier that no thread ever
// arrives on, so a caller can see the bound work without anything being stuck.
#include <string>

#include "gdn_kernels.h"

namespace {

__global__ void wait_selftest_kernel(uint32_t *status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = gdn::smem_addr(&bar);
  if (threadIdx.x == 0) {
    gdn::mbar_init(b, 1);
    gdn::fence_mbar_init();
  }
  __syncthreads();
  // phase 0 needs one arrival and gets none
  if (threadIdx.x == 0 && !gdn::mbar_wait_bounded(b, 0u, limit_ns)) gdn::set_status(status, GDN_DEV_TIMEOUT);
}

}  // namespace

extern "C" {

gdn_status_t gdn_selftest_wait_timeout(uint32_t *dev_status, uint32_t limit_us, gdn_stream_t stream) {
  if (!dev_status) {
    gdn::set_last_error("gdn_selftest_wait_timeout: dev_status is NULL");
    return GDN_ERR_INVALID_ARG;
  }
  if (limit_us < 1 || limit_us > 100000) {
    gdn::set_last_error("gdn_selftest_wait_timeout: limit_us must be in [1, 100000]");
    return GDN_ERR_INVALID_ARG;
  }
  wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(dev_status, (uint64_t)limit_us * 1000u);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    gdn::set_last_error((std::string("gdn_selftest_wait_timeout launch: ") + cudaGetErrorString(e)).c_str());
    return GDN_ERR_CUDA;
  }
  return GDN_OK;
}

}  // extern "C"
