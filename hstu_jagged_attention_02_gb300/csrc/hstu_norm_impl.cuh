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
// This header holds the kernels and their width dispatch; each element-type
// combination is instantiated in a translation unit of its own
// (hstu_norm_f32.cu, hstu_norm_bf16.cu, hstu_norm_bf16_bf16.cu) so that they
// compile in parallel.
#pragma once
#include "hstu_internal.h"

namespace hstu {

namespace {

constexpr int kWarps = 8;  // tokens per CTA

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int VEC> struct Vec;
template <> struct Vec<1> {
  template <typename T> __device__ static void load(const T* p, float* v) { v[0] = to_f(p[0]); }
  template <typename T> __device__ static void store(T* p, const float* v) { p[0] = from_f<T>(v[0]); }
};
template <> struct Vec<4> {
  __device__ static void load(const float* p, float* v) {
    const float4 x = *reinterpret_cast<const float4*>(p);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  }
  __device__ static void load(const __nv_bfloat16* p, float* v) {
    const uint2 x = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(x.x << 16); v[1] = __uint_as_float(x.x & 0xFFFF0000u);
    v[2] = __uint_as_float(x.y << 16); v[3] = __uint_as_float(x.y & 0xFFFF0000u);
  }
  __device__ static void store(float* p, const float* v) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
  __device__ static void store(__nv_bfloat16* p, const float* v) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
    uint2 x;
    x.x = *reinterpret_cast<const uint32_t*>(&a);
    x.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = x;
  }
};

// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC 2011): ten rounds, each multiplying counter words 0
// and 2 by the round constants (128-bit products) and crossing the halves
// with words 1, 3 and the key; the key advances by the Weyl increments
// between rounds.
__device__ __forceinline__ void philox4x64_10(uint64_t (&c)[4], uint64_t k0, uint64_t k1) {
  constexpr uint64_t kM0 = 0xD2E7470EE14C6C93ull, kM1 = 0xCA5A826395121157ull;
  constexpr uint64_t kW0 = 0x9E3779B97F4A7C15ull, kW1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += kW0;
      k1 += kW1;
    }
    const uint64_t hi0 = __umul64hi(kM0, c[0]), lo0 = kM0 * c[0];
    const uint64_t hi1 = __umul64hi(kM1, c[2]), lo1 = kM1 * c[2];
    const uint64_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
}

// Dropout factors (scale or 0) of the VEC elements at flat indices e0 ..
// e0 + VEC - 1; with VEC = 4, e0 % 4 == 0, so all four share one generator
// block and take words (e0 & 4) .. (e0 & 4) + 3.
template <int VEC>
__device__ __forceinline__ void dropout_factors(const NormParams& p, uint64_t e0, float (&m)[VEC]) {
  uint64_t c[4] = {e0 >> 3, p.drop_offset, 0ull, 0ull};
  philox4x64_10(c, p.drop_seed, 0ull);
  uint32_t w[VEC];
  if constexpr (VEC == 4) {
    const bool up = (e0 & 4) != 0;
    const uint64_t a = up ? c[2] : c[0], b = up ? c[3] : c[1];
    w[0] = (uint32_t)a;
    w[1] = (uint32_t)(a >> 32);
    w[2] = (uint32_t)b;
    w[3] = (uint32_t)(b >> 32);
  } else {
    const int k = (int)(e0 & 7);
    const uint64_t a = k < 2 ? c[0] : (k < 4 ? c[1] : (k < 6 ? c[2] : c[3]));
    w[0] = (k & 1) ? (uint32_t)(a >> 32) : (uint32_t)a;
  }
#pragma unroll
  for (int i = 0; i < VEC; ++i) m[i] = w[i] >= p.drop_thr ? p.drop_scale : 0.f;
}

// Dropout factors of every chunk of this lane's row t (the lane layout of
// feat()).  With VEC = 4 the chunks r of lanes 2i and 2i + 1 share one
// generator block (elements t F + 128 r + 8 i + [0, 8)); when PER is even,
// lane 2i computes the blocks of the even chunks and lane 2i + 1 those of
// the odd ones, and each hands its partner the partner's half: one
// generator call per lane per two chunks.
template <int VEC, int PER>
__device__ __forceinline__ void dropout_row(const NormParams& p, int64_t t, int F, float (&m)[PER][VEC]) {
  const int lane = threadIdx.x & 31;
  if constexpr (VEC == 4 && PER % 2 == 0) {
    const int q = lane & 1;
#pragma unroll
    for (int r = 0; r < PER; r += 2) {
      uint64_t c[4] = {((uint64_t)t * F + (uint64_t)(r + q) * 128 + (uint64_t)(lane >> 1) * 8) >> 3,
                       p.drop_offset, 0ull, 0ull};
      philox4x64_10(c, p.drop_seed, 0ull);
      // words 0..3 of the block serve the even lane, 4..7 the odd one
      const uint64_t mine0 = q ? c[2] : c[0], mine1 = q ? c[3] : c[1];
      const uint64_t give0 = q ? c[0] : c[2], give1 = q ? c[1] : c[3];
      const uint64_t got0 = __shfl_xor_sync(0xffffffffu, give0, 1);
      const uint64_t got1 = __shfl_xor_sync(0xffffffffu, give1, 1);
      // own block is chunk r + q; the partner's is chunk r + 1 - q
      const uint64_t w[2][2] = {{q ? got0 : mine0, q ? got1 : mine1}, {q ? mine0 : got0, q ? mine1 : got1}};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t x[4] = {(uint32_t)w[h][0], (uint32_t)(w[h][0] >> 32), (uint32_t)w[h][1],
                               (uint32_t)(w[h][1] >> 32)};
#pragma unroll
        for (int i = 0; i < 4; ++i) m[r + h][i] = x[i] >= p.drop_thr ? p.drop_scale : 0.f;
      }
    }
  } else {
#pragma unroll
    for (int r = 0; r < PER; ++r) dropout_factors<VEC>(p, (uint64_t)t * F + (uint64_t)(r * 32 + lane) * VEC, m[r]);
  }
}

// feature index of element e of chunk r of this lane
template <int VEC>
__device__ __forceinline__ int feat(int r, int lane) { return (r * 32 + lane) * VEC; }

// mean and 1/sqrt(var + eps) of the row held in x (PER chunks of VEC values)
template <int VEC, int PER>
__device__ __forceinline__ void row_stats(const float (&x)[PER][VEC], int F, float eps, float& mean, float& rstd) {
  const int lane = threadIdx.x & 31;
  float s = 0.f;
#pragma unroll
  for (int r = 0; r < PER; ++r)
#pragma unroll
    for (int e = 0; e < VEC; ++e) s += x[r][e];
  mean = warp_sum(s) / F;
  float v = 0.f;
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    if (feat<VEC>(r, lane) < F) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float d = x[r][e] - mean;
        v += d * d;
      }
    }
  }
  rstd = rsqrtf(warp_sum(v) / F + eps);
}

// Loads of a row: VEC-wide chunks r < PER of lane `lane`, zero past F.
template <int VEC, int PER, typename T>
__device__ __forceinline__ void load_row(const T* row, int F, int lane, float (&x)[PER][VEC]) {
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    const int f = feat<VEC>(r, lane);
    if (f < F) Vec<VEC>::load(row + f, x[r]);
    else
#pragma unroll
      for (int e = 0; e < VEC; ++e) x[r][e] = 0.f;
  }
}

// One warp per token, the grid one wave of CTAs walking the tokens (no
// second, partly filled wave); every load of a token is issued before any of
// its arithmetic, so a warp waits on memory once per token.
template <typename TI, typename TO, int VEC, int PER, bool DROP>
__global__ void __launch_bounds__(kWarps * 32) norm_gate_fwd_kernel(NormParams p) {
  // Launched programmatically after the attention forward that writes o: the
  // launch overlaps that kernel's tail, and every thread waits for it to
  // complete before reading.
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int F = p.F;
  const int64_t stride = (int64_t)gridDim.x * kWarps;
  for (int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); t < p.T; t += stride) {
    float x[PER][VEC], g[PER][VEC];
    load_row<VEC, PER>(static_cast<const TO*>(p.o) + t * F, F, lane, x);
    if (p.u) load_row<VEC, PER>(static_cast<const TI*>(p.u) + t * F, F, lane, g);
    float mean = 0.f, rstd = 1.f;
    if (p.norm == HSTU_NORM_LAYERNORM) row_stats<VEC, PER>(x, F, p.eps, mean, rstd);
    if (p.y) {
      TO* y = static_cast<TO*>(p.y) + t * F;
      float m[PER][VEC];
      if (DROP && p.drop) dropout_row<VEC, PER>(p, t, F, m);
#pragma unroll
      for (int r = 0; r < PER; ++r) {
        const int f = feat<VEC>(r, lane);
        if (f >= F) continue;
        float out[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) out[e] = (x[r][e] - mean) * rstd * (p.u ? g[r][e] : 1.f);
        if (DROP && p.drop)
#pragma unroll
          for (int e = 0; e < VEC; ++e) out[e] *= m[r][e];
        Vec<VEC>::store(y + f, out);
      }
    }
    if (lane == 0) {
      if (p.mean) p.mean[t] = mean;
      if (p.rstd) p.rstd[t] = rstd;
    }
  }
}

// A backward plan kept by an earlier forward (HSTU_FLAG_REUSE_PLAN), checked
// by one warp before the attention backward may use it: it must have been
// made for this call's sequence count, token count, tile edges and
// max_seq_len, from the same offsets, target and context counts and first
// timestamps of the sequences (everything the plan depends on).  A match arms
// it (its block count, the work counter at zero), so it can serve any number
// of backward calls; otherwise the attention backward gets no work and
// HSTU_ERR_DEVICE_CHECK is recorded.
__device__ __noinline__ void check_kept_plan(const NormParams& p) {
  pdl_wait();  // whatever ran before this grid is complete
  int* h = p.pc_hdr;
  const int lane = threadIdx.x & 31;
  const int64_t T = p.T;
  const bool key = h[WS_PB_VALID] == kKeptPlanValid && h[WS_PB_B] == p.pc_B && h[WS_PB_T_LO] == (int)(uint32_t)T &&
                   h[WS_PB_T_HI] == (int)(T >> 32) && h[WS_PB_TILE] == p.pc_tile && h[WS_PB_MAXN] == p.pc_max_n;
  bool ok = key;
  if (key) {  // same B and T: the kept offsets (validated when planned) index this call's arrays
    for (int b = lane; b <= p.pc_B; b += 32) {
      bool e = p.pc_off[b] == p.pc_sv_off[b];
      if (b < p.pc_B) {
        e = e && (p.pc_nt ? p.pc_nt[b] : 0) == p.pc_sv_nt[b] && (p.pc_nc ? p.pc_nc[b] : 0) == p.pc_sv_nc[b];
        const int64_t s0 = p.pc_sv_off[b];
        const int64_t t0 = (p.pc_ts && p.pc_sv_off[b + 1] > s0) ? p.pc_ts[s0] : 0;
        e = e && t0 == p.pc_sv_t0[b];
      }
      ok = ok && e;
    }
  }
  ok = __all_sync(0xffffffffu, ok);
  if (lane == 0) {
    if (ok) {
      h[WS_NBLK] = h[WS_PB_NBLK];
      h[WS_NEXT] = 0;
    } else {
      h[WS_NBLK] = 0;
      set_error(h, HSTU_ERR_DEVICE_CHECK, kPlanMismatchInfo);
    }
  }
}

// du = xn * dy;  g = dy * u;  LayerNorm: dO = rstd * (g - mean(g) - xn * mean(g xn)); none: dO = g
template <typename TI, typename TO, int VEC, int PER, bool DROP>
__global__ void __launch_bounds__(kWarps * 32) norm_gate_bwd_kernel(NormParams p) {
  // Launched programmatically after the backward's planner, with which it
  // shares no data: it runs alongside it.  One thread waits for the planner,
  // so this grid completes only after it (the attention backward, launched
  // normally after this kernel, reads the plan).  Without a planner, warp 0
  // of CTA 0 checks and arms the kept plan instead, and takes no tokens (its
  // dependent reads would otherwise delay its tokens past everyone else's).
  if (blockIdx.x == 0 && threadIdx.x == 0) pdl_wait();
  if (p.pc_hdr && blockIdx.x == 0 && threadIdx.x < 32) check_kept_plan(p);
  if (blockIdx.x == 0) {
    for (int x = threadIdx.x; x < p.zero_a_n; x += blockDim.x) p.zero_a[x] = 0.f;
    for (int x = threadIdx.x; x < p.zero_b_n; x += blockDim.x) p.zero_b[x] = 0.f;
  }
  const int lane = threadIdx.x & 31;
  const int F = p.F;
  const bool ln = p.norm == HSTU_NORM_LAYERNORM;
  const int skip = p.pc_hdr ? 1 : 0;  // warps numbered from CTA 0's warp 1 when it checks
  const int64_t stride = (int64_t)gridDim.x * kWarps - skip;
  const int64_t first = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5) - skip;
  for (int64_t t = first < 0 ? p.T : first; t < p.T; t += stride) {
    float x[PER][VEC], d[PER][VEC], g[PER][VEC];
    load_row<VEC, PER>(static_cast<const TO*>(p.o) + t * F, F, lane, x);
    load_row<VEC, PER>(static_cast<const TO*>(p.dy) + t * F, F, lane, d);
    if (p.u) load_row<VEC, PER>(static_cast<const TI*>(p.u) + t * F, F, lane, g);
    if (p.zero_rows) {  // zero_F % 4 == 0, 16-byte aligned rows
      float4* zr = reinterpret_cast<float4*>(p.zero_rows + t * p.zero_F);
      for (int f4 = lane; f4 < p.zero_F / 4; f4 += 32) zr[f4] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float mean = 0.f, rstd = 1.f;
    if (ln) row_stats<VEC, PER>(x, F, p.eps, mean, rstd);
    float m[PER][VEC];
    if (DROP && p.drop) dropout_row<VEC, PER>(p, t, F, m);
    TO* du = p.du ? static_cast<TO*>(p.du) + t * F : nullptr;
    float mg = 0.f, mgx = 0.f;
#pragma unroll
    for (int r = 0; r < PER; ++r) {
      const int f = feat<VEC>(r, lane);
      float dun[VEC];
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float dd = (DROP && p.drop) ? d[r][e] * m[r][e] : d[r][e];  // dy is the gradient of the dropped-out y
        const float xn = (x[r][e] - mean) * rstd;
        const float gg = p.u ? dd * g[r][e] : dd;   // zero past F: every input there is zero
        dun[e] = xn * dd;
        mg += gg;
        mgx += gg * xn;
        x[r][e] = xn;
        g[r][e] = gg;
      }
      if (du && f < F) Vec<VEC>::store(du + f, dun);
    }
    if (ln) {
      mg = warp_sum(mg) / F;
      mgx = warp_sum(mgx) / F;
    }
#pragma unroll
    for (int r = 0; r < PER; ++r) {
      const int f = feat<VEC>(r, lane);
      if (f >= F) continue;
      float val[VEC];
#pragma unroll
      for (int e = 0; e < VEC; ++e) val[e] = ln ? rstd * (g[r][e] - mg - x[r][e] * mgx) : g[r][e];
      if (p.split) {  // BF16 pair: hi = bf16(x), lo = bf16(x - hi)
        float hi[VEC], lo[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          hi[e] = __bfloat162float(__float2bfloat16_rn(val[e]));
          lo[e] = val[e] - hi[e];
        }
        Vec<VEC>::store(static_cast<__nv_bfloat16*>(p.dO) + t * F + f, hi);
        Vec<VEC>::store(static_cast<__nv_bfloat16*>(p.dO_lo) + t * F + f, lo);
      } else {
        Vec<VEC>::store(static_cast<float*>(p.dO) + t * F + f, val);
      }
    }
  }
}

// CTAs of one wave: the SMs times the CTAs of `kernel` one SM holds (looked
// up once per kernel and device)
template <typename K>
int64_t one_wave(K kernel) {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int sms = 0, per = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, kWarps * 32, 0) != cudaSuccess)
      return 0;
    cached[dev] = sms * (per > 0 ? per : 1);
  }
  return cached[dev];
}

template <typename TI, typename TO, int VEC, int PER, bool DROP>
cudaError_t launch_td(const NormParams& p, bool bwd, cudaStream_t st) {
  const int64_t wave = bwd ? one_wave(norm_gate_bwd_kernel<TI, TO, VEC, PER, DROP>)
                           : one_wave(norm_gate_fwd_kernel<TI, TO, VEC, PER, DROP>);
  int64_t grid = (p.T + kWarps - 1) / kWarps;
  if (wave > 0 && grid > wave) grid = wave;
  if (bwd) {
    const cudaError_t e = launch_pdl(norm_gate_bwd_kernel<TI, TO, VEC, PER, DROP>, dim3((unsigned)grid), dim3(kWarps * 32),
                                     0, st, p);
    if (e != cudaSuccess) return e;
  } else {
    const cudaError_t e = launch_pdl(norm_gate_fwd_kernel<TI, TO, VEC, PER, DROP>, dim3((unsigned)grid), dim3(kWarps * 32),
                                     0, st, p);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

// The 4-wide kernels come without and with fused dropout, so the common case
// carries no generator state in its registers; the scalar kernels (widths
// that are not a multiple of 128) test p.drop at run time.
template <typename TI, typename TO, int VEC, int PER>
cudaError_t launch_t(const NormParams& p, bool bwd, cudaStream_t st) {
  if constexpr (VEC == 4) {
    if (!p.drop) return launch_td<TI, TO, VEC, PER, false>(p, bwd, st);
  }
  return launch_td<TI, TO, VEC, PER, true>(p, bwd, st);
}

template <typename TI, typename TO>
cudaError_t by_width(const NormParams& p, bool bwd, cudaStream_t st) {
  if (p.F % 128 == 0) {  // 4-wide vectors
    const int per = p.F / 128;
    if (per <= 1) return launch_t<TI, TO, 4, 1>(p, bwd, st);
    if (per <= 2) return launch_t<TI, TO, 4, 2>(p, bwd, st);
    if (per <= 4) return launch_t<TI, TO, 4, 4>(p, bwd, st);
    if (per <= 8) return launch_t<TI, TO, 4, 8>(p, bwd, st);
    return launch_t<TI, TO, 4, 16>(p, bwd, st);
  }
  const int per = (p.F + 31) / 32;
  if (per <= 2) return launch_t<TI, TO, 1, 2>(p, bwd, st);
  if (per <= 4) return launch_t<TI, TO, 1, 4>(p, bwd, st);
  if (per <= 8) return launch_t<TI, TO, 1, 8>(p, bwd, st);
  if (per <= 16) return launch_t<TI, TO, 1, 16>(p, bwd, st);
  if (per <= 32) return launch_t<TI, TO, 1, 32>(p, bwd, st);
  return launch_t<TI, TO, 1, 64>(p, bwd, st);
}

}  // namespace

}  // namespace hstu
