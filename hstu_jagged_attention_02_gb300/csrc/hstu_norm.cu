// Pointwise transformation of HSTU (ai6s.net survey, section 2.1.2, eq. (3)):
// y = Norm(o) * u per token, over the token's H * d_v features, and its
// backward.  Norm is LayerNorm with population variance and no affine, or
// the identity.  One warp per token; HBM-bound (reads o and u, writes y).
//
// Element types: u has the input type TI; o, y, dy and du have the output
// type TO.  The backward's dO (an input of the attention backward) is FP32, or
// a BF16 hi/lo pair for the tensor-core path.
//
// Lane l of the warp owns features (r * 32 + l) * VEC + [0, VEC) for
// r < PER: with VEC = 4 every access is a 16-byte (FP32) or 8-byte (BF16)
// vector and a warp touches 512 / 256 contiguous bytes per access.
//
// Fused dropout (ai6s.net survey, section 2.1.3: dropout fused with its
// neighbouring operators): y = dropout(Norm(o) * u), and in the backward dy
// passes the same mask and scale.  Element e = t F + f is kept iff 32-bit
// word e & 7 of Philox4x64-10(counter (e >> 3, offset, 0, 0), key (seed, 0))
// is at least floor(p 2^32); no mask is stored.
//
// The kernels are in hstu_norm_impl.cuh, instantiated per element type in
// hstu_norm_f32.cu, hstu_norm_bf16.cu and hstu_norm_bf16_bf16.cu; this file
// dispatches to them and holds the FP32 -> output-type conversion.
#include "hstu_internal.h"

namespace hstu {

cudaError_t norm_dispatch_f32_f32(const NormParams& p, bool bwd, cudaStream_t st);
cudaError_t norm_dispatch_bf16_f32(const NormParams& p, bool bwd, cudaStream_t st);
cudaError_t norm_dispatch_bf16_bf16(const NormParams& p, bool bwd, cudaStream_t st);

namespace {

template <typename TO>
__global__ void convert_kernel(const float* __restrict__ src, TO* __restrict__ dst, int64_t count) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = from_f<TO>(src[i]);
}

cudaError_t dispatch(const NormParams& p, bool bwd, cudaStream_t st) {
  if (p.T <= 0) return cudaSuccess;
  if (p.dtype == HSTU_FP32) return norm_dispatch_f32_f32(p, bwd, st);
  return p.out_dtype == HSTU_FP32 ? norm_dispatch_bf16_f32(p, bwd, st)
                                  : norm_dispatch_bf16_bf16(p, bwd, st);
}

}  // namespace

cudaError_t launch_norm_gate_fwd(const NormParams& p, cudaStream_t st) { return dispatch(p, false, st); }
cudaError_t launch_norm_gate_bwd(const NormParams& p, cudaStream_t st) { return dispatch(p, true, st); }

cudaError_t launch_convert_f32(const float* src, void* dst, int64_t count, int out_dtype, cudaStream_t st) {
  if (count <= 0) return cudaSuccess;
  int64_t grid = (count / 4 + 255) / 256;
  if (grid > 152 * 16) grid = 152 * 16;
  if (grid < 1) grid = 1;
  if (out_dtype == HSTU_BF16)
    convert_kernel<__nv_bfloat16><<<(unsigned)grid, 256, 0, st>>>(src, static_cast<__nv_bfloat16*>(dst), count);
  else
    convert_kernel<float><<<(unsigned)grid, 256, 0, st>>>(src, static_cast<float*>(dst), count);
  return cudaGetLastError();
}

}  // namespace hstu
