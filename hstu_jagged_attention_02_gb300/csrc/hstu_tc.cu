// Tensor-core backward entry points (the CUDA-core backward runs until the
// tcgen05 backward kernel is available).
#include "hstu_internal.h"

namespace hstu {

bool tc_bwd_supported(int, int, int) { return false; }
cudaError_t launch_tc_bwd(const AttnParams&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace hstu
