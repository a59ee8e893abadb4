// Host-side helpers shared by the C-ABI entry points: thread-local error
// message, argument checks, CUDA error mapping.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sca.h"

namespace sca {

// Record a message for sca_last_error() and return `code`.
int fail(int code, const char* fmt, ...);

// Map a CUDA error (if any) to SCA_ERR_CUDA with a message.
int cuda_status(cudaError_t e, const char* what);

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace sca

#define SCA_REQUIRE(cond, code, ...)            \
  do {                                          \
    if (!(cond)) return ::sca::fail(code, __VA_ARGS__); \
  } while (0)
