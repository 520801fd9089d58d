// Norm-gate kernels (forward and backward) for u of type float and o, y, dy, du
// of type float; the kernels themselves are in hstu_norm_impl.cuh.
#include "hstu_norm_impl.cuh"

namespace hstu {

cudaError_t norm_dispatch_f32_f32(const NormParams& p, bool bwd, cudaStream_t st) { return by_width<float, float>(p, bwd, st); }

}  // namespace hstu
