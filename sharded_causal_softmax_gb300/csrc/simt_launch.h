// Launchers of the attention kernels, called by the C-ABI entry points after
// validation.  Each returns the CUDA launch status.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace sca {

// fp32-arithmetic kernels (fp32 or bf16 inputs), attn_simt.cu
cudaError_t simt_forward(AttnArgs& a, int dtype, cudaStream_t st);
cudaError_t simt_backward(AttnArgs& a, int dtype, cudaStream_t st);

// tcgen05 tensor-core kernels (bf16 inputs), fwd_tc.cu / bwd_tc.cu.
// Return cudaErrorNotSupported if a layout cannot be described by a TMA map.
cudaError_t tc_forward(AttnArgs& a, cudaStream_t st);
// f16_inputs: SCA_F16_Q / SCA_F16_DOUT bits of sca_attn_dims (the backward
// reads those inputs as fp16 and skips converting them).
cudaError_t tc_backward(AttnArgs& a, int f16_inputs, cudaStream_t st);

}  // namespace sca
