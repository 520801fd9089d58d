// Pointwise transformation of HSTU (ai6s.net survey, section 2.1.2, eq. (3)):
// y = Norm(o) * u per token, over the token's H * d_v features, and its
// backward.  Norm is LayerNorm with population variance and no affine, or
// the identity.  One warp per token; HBM-bound (reads o and u, writes y).
//
// Element types: u has the input type TI; o, y, dy and du have the output
// type TO.  The backward's dO (an input of the attention backward) is FP32, or
// a BF16 hi/lo pair for the tensor-core path.
#include "hstu_internal.h"

namespace hstu {

namespace {

constexpr int kWarps = 8;  // tokens per CTA

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// mean and 1/sqrt(var + eps) of the PER*32-strided row held in x (lanes own
// features f = r*32 + lane, f < F)
template <int PER>
__device__ __forceinline__ void row_stats(const float* x, int F, float eps, float& mean, float& rstd) {
  const int lane = threadIdx.x & 31;
  float s = 0.f;
#pragma unroll
  for (int r = 0; r < PER; ++r) s += x[r];
  mean = warp_sum(s) / F;
  float v = 0.f;
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    const float d = (r * 32 + lane) < F ? x[r] - mean : 0.f;
    v += d * d;
  }
  rstd = rsqrtf(warp_sum(v) / F + eps);
}

template <typename TI, typename TO, int PER>
__global__ void __launch_bounds__(kWarps * 32) norm_gate_fwd_kernel(NormParams p) {
  const int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (t >= p.T) return;
  const int lane = threadIdx.x & 31;
  const int F = p.F;
  const TO* o = static_cast<const TO*>(p.o) + t * F;
  const TI* u = p.u ? static_cast<const TI*>(p.u) + t * F : nullptr;
  float x[PER];
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    const int f = r * 32 + lane;
    x[r] = f < F ? to_f(o[f]) : 0.f;
  }
  float mean = 0.f, rstd = 1.f;
  if (p.norm == HSTU_NORM_LAYERNORM) row_stats<PER>(x, F, p.eps, mean, rstd);
  if (p.y) {
    TO* y = static_cast<TO*>(p.y) + t * F;
#pragma unroll
    for (int r = 0; r < PER; ++r) {
      const int f = r * 32 + lane;
      if (f < F) {
        const float xn = (x[r] - mean) * rstd;
        y[f] = from_f<TO>(u ? xn * to_f(u[f]) : xn);
      }
    }
  }
  if (lane == 0) {
    if (p.mean) p.mean[t] = mean;
    if (p.rstd) p.rstd[t] = rstd;
  }
}

// du = xn * dy;  g = dy * u;  LayerNorm: dO = rstd * (g - mean(g) - xn * mean(g xn)); none: dO = g
template <typename TI, typename TO, int PER>
__global__ void __launch_bounds__(kWarps * 32) norm_gate_bwd_kernel(NormParams p) {
  const int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (t >= p.T) return;
  const int lane = threadIdx.x & 31;
  const int F = p.F;
  const TO* o = static_cast<const TO*>(p.o) + t * F;
  const TI* u = p.u ? static_cast<const TI*>(p.u) + t * F : nullptr;
  const TO* dy = static_cast<const TO*>(p.dy) + t * F;
  float x[PER], g[PER];
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    const int f = r * 32 + lane;
    x[r] = f < F ? to_f(o[f]) : 0.f;
  }
  float mean = 0.f, rstd = 1.f;
  const bool ln = p.norm == HSTU_NORM_LAYERNORM;
  if (ln) row_stats<PER>(x, F, p.eps, mean, rstd);
  float mg = 0.f, mgx = 0.f;
  TO* du = p.du ? static_cast<TO*>(p.du) + t * F : nullptr;
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    const int f = r * 32 + lane;
    float gg = 0.f;
    if (f < F) {
      const float xn = (x[r] - mean) * rstd;
      const float d = to_f(dy[f]);
      gg = u ? d * to_f(u[f]) : d;
      if (du) du[f] = from_f<TO>(xn * d);
      mg += gg;
      mgx += gg * xn;
      x[r] = xn;
    }
    g[r] = gg;
  }
  if (ln) {
    mg = warp_sum(mg) / F;
    mgx = warp_sum(mgx) / F;
  }
  if (p.split) {  // BF16 pair: hi = bf16(x), lo = bf16(x - hi)
    __nv_bfloat16* hi = static_cast<__nv_bfloat16*>(p.dO) + t * F;
    __nv_bfloat16* lo = static_cast<__nv_bfloat16*>(p.dO_lo) + t * F;
#pragma unroll
    for (int r = 0; r < PER; ++r) {
      const int f = r * 32 + lane;
      if (f < F) {
        const float val = ln ? rstd * (g[r] - mg - x[r] * mgx) : g[r];
        const __nv_bfloat16 h = __float2bfloat16_rn(val);
        hi[f] = h;
        lo[f] = __float2bfloat16_rn(val - __bfloat162float(h));
      }
    }
  } else {
    float* dO = static_cast<float*>(p.dO) + t * F;
#pragma unroll
    for (int r = 0; r < PER; ++r) {
      const int f = r * 32 + lane;
      if (f < F) dO[f] = ln ? rstd * (g[r] - mg - x[r] * mgx) : g[r];
    }
  }
}

template <typename TO>
__global__ void convert_kernel(const float* __restrict__ src, TO* __restrict__ dst, int64_t count) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = from_f<TO>(src[i]);
}

template <typename TI, typename TO, int PER>
cudaError_t launch_t(const NormParams& p, bool bwd, cudaStream_t st) {
  const int64_t grid = (p.T + kWarps - 1) / kWarps;
  if (bwd)
    norm_gate_bwd_kernel<TI, TO, PER><<<(unsigned)grid, kWarps * 32, 0, st>>>(p);
  else
    norm_gate_fwd_kernel<TI, TO, PER><<<(unsigned)grid, kWarps * 32, 0, st>>>(p);
  return cudaGetLastError();
}

template <typename TI, typename TO>
cudaError_t by_width(const NormParams& p, bool bwd, cudaStream_t st) {
  const int per = (p.F + 31) / 32;
  if (per <= 2) return launch_t<TI, TO, 2>(p, bwd, st);
  if (per <= 4) return launch_t<TI, TO, 4>(p, bwd, st);
  if (per <= 8) return launch_t<TI, TO, 8>(p, bwd, st);
  if (per <= 16) return launch_t<TI, TO, 16>(p, bwd, st);
  if (per <= 32) return launch_t<TI, TO, 32>(p, bwd, st);
  return launch_t<TI, TO, 64>(p, bwd, st);
}

cudaError_t dispatch(const NormParams& p, bool bwd, cudaStream_t st) {
  if (p.T <= 0) return cudaSuccess;
  if (p.dtype == HSTU_FP32) return by_width<float, float>(p, bwd, st);
  return p.out_dtype == HSTU_FP32 ? by_width<__nv_bfloat16, float>(p, bwd, st)
                                  : by_width<__nv_bfloat16, __nv_bfloat16>(p, bwd, st);
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
