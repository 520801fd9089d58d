// CUDA-core HSTU attention kernels: FP32 FMA arithmetic on 32 x 32 tiles.
//
// This is the FP32 path (true FP32 products and sums) and the fallback for
// shapes the tensor-core kernels do not cover.  Each CTA owns one work item
// of the planner (a query block of one head for the forward, a key block of
// one head for the backward) and walks the tiles the compound mask keeps.
//
// Per element (HSTU spatial aggregation, ai6s.net survey section 2.1.2):
//   z = alpha * <q_i, k_j> + rab_pos[bp] + rab_time[bt]
//   forward:  a = SiLU(z) / N,  o_i += a * v_j
//   backward: dA = <dO_i, v_j>;  dZ = dA * SiLU'(z) / N;
//             dv_j += a dO_i;  dk_j += alpha dZ q_i;  dq_i += alpha dZ k_j;
//             d_rab[bucket] += dZ
#include "hstu_internal.h"

namespace hstu {

namespace {

constexpr int TS = kSimtTile;  // 32
constexpr int NT = 256;        // threads per CTA

__device__ __forceinline__ float sigmoid_f(float z) { return 1.0f / (1.0f + expf(-z)); }

template <typename TI>
__device__ __forceinline__ float bias_of(const AttnParams& p, int h, int i, int j, int h_end,
                                         int64_t ti, int64_t tj) {
  float bias = 0.f;
  if (p.rab_pos) bias += __ldg(p.rab_pos + h * p.P + pos_bucket(i, j, h_end, p.P));
  if (p.rab_time && p.ts) bias += __ldg(p.rab_time + h * p.Tb + time_bucket(ti, tj, p.Tb));
  return bias;
}

// ------------------------------------------------------------------ forward
template <typename TI, typename TO, int D>
__global__ void __launch_bounds__(NT) simt_fwd_kernel(AttnParams p) {
  extern __shared__ __align__(16) float smem[];
  float* Qt = smem;                 // [D][TS]
  float* Kt = Qt + D * TS;          // [D][TS]
  float* Vs = Kt + D * TS;          // [TS][D]
  float* Ps = Vs + TS * D;          // [TS][TS+1]
  int64_t* tq = reinterpret_cast<int64_t*>(Ps + TS * (TS + 1) + 1);  // 8-byte aligned below
  tq = reinterpret_cast<int64_t*>((reinterpret_cast<uintptr_t>(tq) + 15) & ~uintptr_t(15));
  int64_t* tk = tq + TS;

  const int item = blockIdx.x;
  const int nblk = p.hdr[WS_NBLK];
  if (item >= nblk * p.H) return;
  const Block blk = p.blocks[item / p.H];
  const int h = item % p.H;
  const SeqInfo s = seq_info(p.off, p.nt, p.nc, blk.b);
  const int q0 = blk.blk * TS;
  const int tid = threadIdx.x;
  const TI* q = static_cast<const TI*>(p.q);
  const TI* k = static_cast<const TI*>(p.k);
  const TI* v = static_cast<const TI*>(p.v);
  const size_t ld = (size_t)p.H * D;

  for (int idx = tid; idx < TS * D; idx += NT) {
    const int i = idx / D, e = idx % D;
    const int row = q0 + i;
    Qt[e * TS + i] = row < s.n ? to_f(q[(size_t)(s.s0 + row) * ld + (size_t)h * D + e]) : 0.f;
  }
  if (tid < TS) tq[tid] = (p.ts && q0 + tid < s.n) ? p.ts[s.s0 + q0 + tid] : 0;

  constexpr int OC = D / 8;           // output columns per thread
  float acc[OC];
#pragma unroll
  for (int e = 0; e < OC; ++e) acc[e] = 0.f;
  const int ti = tid / 8;             // row of S / O
  const int tj = (tid % 8) * 4;       // 4 columns of S
  const int oe = (tid % 8) * OC;      // columns of O
  const int i = q0 + ti;

  const int nkb = fwd_kv_blocks(q0, s.n, s.c, TS, TS);
  for (int kb = 0; kb < nkb; ++kb) {
    const int k0 = kb * TS;
    if (tile_class(q0, k0, TS, TS, s.n, s.c, s.h_end) == 0) continue;
    __syncthreads();
    for (int idx = tid; idx < TS * D; idx += NT) {
      const int j = idx / D, e = idx % D;
      const int col = k0 + j;
      const bool in = col < s.n;
      const size_t g = (size_t)(s.s0 + col) * ld + (size_t)h * D + e;
      Kt[e * TS + j] = in ? to_f(k[g]) : 0.f;
      Vs[j * D + e] = in ? to_f(v[g]) : 0.f;
    }
    if (tid < TS) tk[tid] = (p.ts && k0 + tid < s.n) ? p.ts[s.s0 + k0 + tid] : 0;
    __syncthreads();

    float sv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int e = 0; e < D; ++e) {
      const float qv = Qt[e * TS + ti];
      const float4 kv = *reinterpret_cast<const float4*>(Kt + e * TS + tj);
      sv[0] = fmaf(qv, kv.x, sv[0]);
      sv[1] = fmaf(qv, kv.y, sv[1]);
      sv[2] = fmaf(qv, kv.z, sv[2]);
      sv[3] = fmaf(qv, kv.w, sv[3]);
    }
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      const int j = k0 + tj + c4;
      float a = 0.f;
      if (i < s.n && j < s.n && allowed(i, j, s.c, s.h_end)) {
        const float z = p.alpha * sv[c4] + bias_of<TI>(p, h, i, j, s.h_end, tq[ti], tk[tj + c4]);
        a = z * sigmoid_f(z) * p.inv_n;
      }
      Ps[ti * (TS + 1) + tj + c4] = a;
    }
    __syncthreads();
#pragma unroll 4
    for (int jj = 0; jj < TS; ++jj) {
      const float pv = Ps[ti * (TS + 1) + jj];
#pragma unroll
      for (int e = 0; e < OC; ++e) acc[e] = fmaf(pv, Vs[jj * D + oe + e], acc[e]);
    }
  }
  if (i < s.n) {
    TO* o = static_cast<TO*>(p.o) + (size_t)(s.s0 + i) * ld + (size_t)h * D + oe;
#pragma unroll
    for (int e = 0; e < OC; ++e) o[e] = from_f<TO>(acc[e]);
  }
}

// ----------------------------------------------------------------- backward
template <typename TI, typename TO, int D>
__global__ void __launch_bounds__(NT) simt_bwd_kernel(AttnParams p) {
  extern __shared__ __align__(16) float smem[];
  float* Kt = smem;                 // [D][TS]  key block, transposed
  float* Kr = Kt + D * TS;          // [TS][D]
  float* Vt = Kr + TS * D;          // [D][TS]
  float* Qt = Vt + D * TS;          // [D][TS]  query block
  float* Qr = Qt + D * TS;          // [TS][D]
  float* dOt = Qr + TS * D;         // [D][TS]
  float* dOr = dOt + D * TS;        // [TS][D]
  float* As = dOr + TS * D;         // [TS q][TS+1]
  float* dZt = As + TS * (TS + 1);  // [TS k][TS+1]
  float* drp = dZt + TS * (TS + 1); // [P]
  float* drt = drp + p.P;           // [Tb]
  int64_t* tk = reinterpret_cast<int64_t*>(
      (reinterpret_cast<uintptr_t>(drt + p.Tb) + 15) & ~uintptr_t(15));
  int64_t* tq = tk + TS;

  const int item = blockIdx.x;
  const int nblk = p.hdr[WS_NBLK];
  if (item >= nblk * p.H) return;
  const Block blk = p.blocks[item / p.H];
  const int h = item % p.H;
  const SeqInfo s = seq_info(p.off, p.nt, p.nc, blk.b);
  const int k0 = blk.blk * TS;
  const int tid = threadIdx.x;
  const TI* q = static_cast<const TI*>(p.q);
  const TI* k = static_cast<const TI*>(p.k);
  const TI* v = static_cast<const TI*>(p.v);
  const float* dO = static_cast<const float*>(p.dO);  // FP32: no rounding of the incoming gradient
  const size_t ld = (size_t)p.H * D;
  const bool want_rp = p.d_rab_pos && p.rab_pos;
  const bool want_rt = p.d_rab_time && p.rab_time && p.ts;

  for (int idx = tid; idx < TS * D; idx += NT) {
    const int j = idx / D, e = idx % D;
    const int col = k0 + j;
    const bool in = col < s.n;
    const size_t g = (size_t)(s.s0 + col) * ld + (size_t)h * D + e;
    const float kv = in ? to_f(k[g]) : 0.f;
    Kt[e * TS + j] = kv;
    Kr[j * D + e] = kv;
    Vt[e * TS + j] = in ? to_f(v[g]) : 0.f;
  }
  if (tid < TS) tk[tid] = (p.ts && k0 + tid < s.n) ? p.ts[s.s0 + k0 + tid] : 0;
  for (int x = tid; x < p.P + p.Tb; x += NT) drp[x] = 0.f;  // drp and drt are contiguous

  constexpr int OC = D / 8;
  float accV[OC], accK[OC];
#pragma unroll
  for (int e = 0; e < OC; ++e) accV[e] = accK[e] = 0.f;
  const int ti = tid / 8;             // S row (query) for the score phase
  const int tj = (tid % 8) * 4;       // 4 S columns (keys)
  const int rj = tid / 8;             // key row for dK/dV, query row for dQ
  const int oe = (tid % 8) * OC;

  const int nqb = (s.n + TS - 1) / TS;
  for (int qb = bwd_q_begin(k0, s.c, TS); qb < nqb; ++qb) {
    const int q0 = qb * TS;
    if (tile_class(q0, k0, TS, TS, s.n, s.c, s.h_end) == 0) continue;
    __syncthreads();
    for (int idx = tid; idx < TS * D; idx += NT) {
      const int i = idx / D, e = idx % D;
      const int row = q0 + i;
      const bool in = row < s.n;
      const size_t g = (size_t)(s.s0 + row) * ld + (size_t)h * D + e;
      const float qv = in ? to_f(q[g]) : 0.f;
      const float dv = in ? dO[g] : 0.f;
      Qt[e * TS + i] = qv;
      Qr[i * D + e] = qv;
      dOt[e * TS + i] = dv;
      dOr[i * D + e] = dv;
    }
    if (tid < TS) tq[tid] = (p.ts && q0 + tid < s.n) ? p.ts[s.s0 + q0 + tid] : 0;
    __syncthreads();

    float sv[4] = {0.f, 0.f, 0.f, 0.f}, da[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int e = 0; e < D; ++e) {
      const float qv = Qt[e * TS + ti], gv = dOt[e * TS + ti];
      const float4 kv = *reinterpret_cast<const float4*>(Kt + e * TS + tj);
      const float4 vv = *reinterpret_cast<const float4*>(Vt + e * TS + tj);
      sv[0] = fmaf(qv, kv.x, sv[0]); sv[1] = fmaf(qv, kv.y, sv[1]);
      sv[2] = fmaf(qv, kv.z, sv[2]); sv[3] = fmaf(qv, kv.w, sv[3]);
      da[0] = fmaf(gv, vv.x, da[0]); da[1] = fmaf(gv, vv.y, da[1]);
      da[2] = fmaf(gv, vv.z, da[2]); da[3] = fmaf(gv, vv.w, da[3]);
    }
    const int i = q0 + ti;
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      const int j = k0 + tj + c4;
      float a = 0.f, dz = 0.f;
      if (i < s.n && j < s.n && allowed(i, j, s.c, s.h_end)) {
        const float z = p.alpha * sv[c4] + bias_of<TI>(p, h, i, j, s.h_end, tq[ti], tk[tj + c4]);
        const float sg = sigmoid_f(z);
        a = z * sg * p.inv_n;
        dz = da[c4] * sg * (1.f + z * (1.f - sg)) * p.inv_n;
        if (want_rp) atomicAdd(drp + pos_bucket(i, j, s.h_end, p.P), dz);
        if (want_rt) atomicAdd(drt + time_bucket(tq[ti], tk[tj + c4], p.Tb), dz);
      }
      As[ti * (TS + 1) + tj + c4] = a;
      dZt[(tj + c4) * (TS + 1) + ti] = dz;
    }
    __syncthreads();
    // dV, dK for key row rj
#pragma unroll 4
    for (int ii = 0; ii < TS; ++ii) {
      const float a = As[ii * (TS + 1) + rj];
      const float dz = dZt[rj * (TS + 1) + ii];
#pragma unroll
      for (int e = 0; e < OC; ++e) {
        accV[e] = fmaf(a, dOr[ii * D + oe + e], accV[e]);
        accK[e] = fmaf(dz, Qr[ii * D + oe + e], accK[e]);
      }
    }
    // dQ for query row rj of this tile
    if (q0 + rj < s.n) {
      float dq[OC];
#pragma unroll
      for (int e = 0; e < OC; ++e) dq[e] = 0.f;
#pragma unroll 4
      for (int jj = 0; jj < TS; ++jj) {
        const float dz = dZt[jj * (TS + 1) + rj];
#pragma unroll
        for (int e = 0; e < OC; ++e) dq[e] = fmaf(dz, Kr[jj * D + oe + e], dq[e]);
      }
      float* dst = p.dq_acc + (size_t)(s.s0 + q0 + rj) * ld + (size_t)h * D + oe;
#pragma unroll
      for (int e = 0; e < OC; ++e) atomicAdd(dst + e, p.alpha * dq[e]);
    }
  }
  if (k0 + rj < s.n) {
    const size_t g = (size_t)(s.s0 + k0 + rj) * ld + (size_t)h * D + oe;
    TO* dk = static_cast<TO*>(p.dk) + g;
    TO* dv = static_cast<TO*>(p.dv) + g;
#pragma unroll
    for (int e = 0; e < OC; ++e) {
      dk[e] = from_f<TO>(p.alpha * accK[e]);
      dv[e] = from_f<TO>(accV[e]);
    }
  }
  __syncthreads();
  if (want_rp)
    for (int x = tid; x < p.P; x += NT)
      if (drp[x] != 0.f) atomicAdd(p.d_rab_pos + h * p.P + x, drp[x]);
  if (want_rt)
    for (int x = tid; x < p.Tb; x += NT)
      if (drt[x] != 0.f) atomicAdd(p.d_rab_time + h * p.Tb + x, drt[x]);
}

template <int D>
size_t fwd_smem() {
  return sizeof(float) * (3 * D * TS + TS * (TS + 1) + 1) + 16 + 2 * TS * sizeof(int64_t);
}
template <int D>
size_t bwd_smem(int P, int Tb) {
  return sizeof(float) * (7 * D * TS + 2 * TS * (TS + 1) + P + Tb) + 16 + 2 * TS * sizeof(int64_t);
}

template <typename TI, typename TO, int D>
cudaError_t fwd_launch(const AttnParams& p, int items, cudaStream_t st) {
  const size_t sm = fwd_smem<D>();
  cudaError_t e = cudaFuncSetAttribute(simt_fwd_kernel<TI, TO, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  simt_fwd_kernel<TI, TO, D><<<items, NT, sm, st>>>(p);
  return cudaGetLastError();
}

template <typename TI, typename TO, int D>
cudaError_t bwd_launch(const AttnParams& p, int items, cudaStream_t st) {
  const size_t sm = bwd_smem<D>(p.P, p.Tb);
  cudaError_t e = cudaFuncSetAttribute(simt_bwd_kernel<TI, TO, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  simt_bwd_kernel<TI, TO, D><<<items, NT, sm, st>>>(p);
  return cudaGetLastError();
}

template <typename TI, typename TO>
cudaError_t fwd_by_d(const AttnParams& p, int items, cudaStream_t st) {
  switch (p.dqk) {
    case 32: return fwd_launch<TI, TO, 32>(p, items, st);
    case 64: return fwd_launch<TI, TO, 64>(p, items, st);
    case 128: return fwd_launch<TI, TO, 128>(p, items, st);
  }
  return cudaErrorInvalidValue;
}

template <typename TI, typename TO>
cudaError_t bwd_by_d(const AttnParams& p, int items, cudaStream_t st) {
  switch (p.dqk) {
    case 32: return bwd_launch<TI, TO, 32>(p, items, st);
    case 64: return bwd_launch<TI, TO, 64>(p, items, st);
    case 128: return bwd_launch<TI, TO, 128>(p, items, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_simt_fwd(const AttnParams& p, int max_items, cudaStream_t st) {
  if (max_items <= 0) return cudaSuccess;
  if (p.dtype == HSTU_FP32) return fwd_by_d<float, float>(p, max_items, st);
  return p.out_dtype == HSTU_FP32 ? fwd_by_d<__nv_bfloat16, float>(p, max_items, st)
                                  : fwd_by_d<__nv_bfloat16, __nv_bfloat16>(p, max_items, st);
}

cudaError_t launch_simt_bwd(const AttnParams& p, int max_items, cudaStream_t st) {
  if (max_items <= 0) return cudaSuccess;
  if (p.dtype == HSTU_FP32) return bwd_by_d<float, float>(p, max_items, st);
  return p.out_dtype == HSTU_FP32 ? bwd_by_d<__nv_bfloat16, float>(p, max_items, st)
                                  : bwd_by_d<__nv_bfloat16, __nv_bfloat16>(p, max_items, st);
}

}  // namespace hstu
