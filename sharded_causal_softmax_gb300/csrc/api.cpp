// Library-wide C-ABI entry points: error reporting, status read-back,
// version.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "host_common.h"

namespace sca {

static thread_local char g_last_error[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return SCA_OK;
  return fail(SCA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace sca

extern "C" const char* sca_last_error(void) { return sca::g_last_error; }

extern "C" int sca_version(void) { return 1 * 10000 + 0 * 100 + 0; }

extern "C" int sca_read_status(const int* dev_status, void* stream) {
  SCA_REQUIRE(dev_status != nullptr, SCA_ERR_ARG, "sca_read_status: dev_status is NULL");
  int host = 0;
  cudaStream_t st = sca::as_stream(stream);
  cudaError_t e = cudaMemcpyAsync(&host, dev_status, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return sca::cuda_status(e, "sca_read_status");
  if (host != SCA_OK) sca::fail(host, "device reported status %d", host);
  return host;
}
