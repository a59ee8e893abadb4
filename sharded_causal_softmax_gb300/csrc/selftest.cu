// The failure path every tensor-core kernel shares, run on its own: one
// bounded mbarrier wait that nothing completes.  After the library's wait
// limit the wait gives up, sets the CTA's abort flag and records
// SCA_ERR_TIMEOUT in the caller's status word; the kernel then returns, and
// the context stays usable.  Nothing faults, traps or hangs.
#include "common.cuh"
#include "host_common.h"
#include "ptx.cuh"

namespace sca {

__global__ void wait_timeout_kernel(int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);   // one arrival would complete phase 0; none comes
    abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort, status);
}

}  // namespace sca

extern "C" int sca_selftest_wait_timeout(int* dev_status, void* stream) {
  SCA_REQUIRE(dev_status, SCA_ERR_ARG, "sca_selftest_wait_timeout: NULL status word");
  sca::wait_timeout_kernel<<<1, 32, 0, sca::as_stream(stream)>>>(dev_status);
  return sca::cuda_status(cudaGetLastError(), "sca_selftest_wait_timeout launch");
}
