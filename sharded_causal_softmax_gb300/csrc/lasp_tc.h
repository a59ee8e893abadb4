// Tensor-core launchers of the linear-attention block kernels (lasp_tc.cu):
// bf16 inputs [BH, S, 128], blocks of L rows (a multiple of kLaspTcSub),
// arguments validated by the callers in lasp.cu.  Each returns an
// sca_status.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sca {

constexpr int kLaspTcSub = 128;     // the tensor-core block size is a multiple of this
constexpr int kLaspTcMaxBlock = 4096;

int lasp_tc_states(const void* a, const void* b, float* st, int64_t BH, int64_t S, int L, int* status,
                   cudaStream_t stream);

int lasp_tc_fwd(const void* q, const void* k, const void* v, const float* st, const float* shard_in, float* o,
                int64_t BH, int64_t S, int P, int L, float scale, int* status, cudaStream_t stream);

int lasp_tc_bwd(const void* q, const void* k, const void* v, const void* dout, const float* st_f, const float* in_f,
                const float* st_b, const float* in_b, float* dq, float* dk, float* dv, int64_t BH, int64_t S, int P,
                int L, float scale, int* status, cudaStream_t stream);

}  // namespace sca
