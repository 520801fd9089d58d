// Tensor-core (tcgen05 / TMEM / TMA) HSTU attention kernels for sm_103a.
#include "hstu_internal.h"

namespace hstu {

bool tc_fwd_supported(int, int, int) { return false; }
bool tc_bwd_supported(int, int, int) { return false; }
cudaError_t launch_tc_fwd(const AttnParams&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_bwd(const AttnParams&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace hstu
