// Backward on the tensor cores: not built yet; attn_bwd_shard runs the
// fp32-arithmetic kernels for every dtype until it is.
#include "simt_launch.h"

namespace sca {

cudaError_t tc_backward(AttnArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace sca
