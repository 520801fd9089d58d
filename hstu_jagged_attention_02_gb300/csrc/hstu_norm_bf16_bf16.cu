// Norm-gate kernels (forward and backward) for u of type __nv_bfloat16 and o, y, dy, du
// of type __nv_bfloat16; the kernels themselves are in hstu_norm_impl.cuh.
#include "hstu_norm_impl.cuh"

namespace hstu {

cudaError_t norm_dispatch_bf16_bf16(const NormParams& p, bool bwd, cudaStream_t st) { return by_width<__nv_bfloat16, __nv_bfloat16>(p, bwd, st); }

}  // namespace hstu
