// Tensor-core GEMMs of the HSTU layer with their element-wise steps fused
// into the epilogue (ai6s.net survey, section 2.1.2: pointwise projection
// eq. (1) and the output projection with the residual connection; section
// 2.1.3: two linear layers and no stored sub-layer activations beyond what
// the backward needs):
//
//   f1:  Z1 = X W1              then  z1 <- Z1,  U <- SiLU(Z1[:, 0:D])  (FP32),
//                                     V | Q | K <- SiLU(Z1[:, D:4D])    (BF16,
//                                     the attention's [T, H, d] layout)
//   f2:  acc = y_hi W2 + y_lo W2  then  out <- X + acc                  (FP32)
//
// X, y_hi, y_lo: [M, K] BF16 row-major (K-major A operands); W1 [K, 4D] and
// W2 [K, D] BF16 row-major (MN-major B operands).  Tiles of 128 rows x BN
// columns (BN = 256, or 128 for narrow outputs), k-blocks of 64 through a
// 4-stage TMA ring, tcgen05.mma (M = 128, N = BN, K = 16) into one of two
// FP32 TMEM accumulators, so the next tile's MMAs overlap this tile's
// epilogue.  Persistent CTAs walk the tiles row-block-major, so consecutive
// tiles of a CTA share their X rows in L2.
//
// Roles (320 threads): warps 0-7 epilogue (TMEM lane quarter warp % 4,
// column half warp / 4), warp 8 TMA producer, warp 9 MMA issuer and TMEM
// owner.  Every wait is bounded; a wait that runs out records HSTU_ERR_TIMEOUT
// in the layer's header word and every role exits.
#include "hstu_internal.h"
#include "tc_ptx.cuh"

namespace hstu {

namespace {

using namespace tc;

constexpr int GBM = 128, GBK = 64;
constexpr int kGStages = 4;
constexpr int kGEpiWarps = 8;
constexpr int kGProducerWarp = 8, kGMmaWarp = 9;
constexpr int kGThreads = 10 * 32;
constexpr uint32_t kGTmemCols = 512;

enum : int { GB_FULL = 0, GB_EMPTY = GB_FULL + kGStages, GB_AFULL = GB_EMPTY + kGStages, GB_AEMPTY = GB_AFULL + 2,
             GB_DRAIN = GB_AEMPTY + 2, GB_COUNT };

template <int BN>
struct GLayout {
  static constexpr int A_BYTES = GBM * GBK * 2;        // 16 KB: 128 rows x 64 k
  static constexpr int B_BOX = GBK * 64 * 2;           // 8 KB: 64 k-rows x 64 n-columns
  static constexpr int B_BYTES = (BN / 64) * B_BOX;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int BAR_OFF = kGStages * STAGE;
  static constexpr int MISC_OFF = BAR_OFF + GB_COUNT * 8;  // tmem slot, abort flag
  static constexpr int BYTES = MISC_OFF + 16;
};

__device__ __forceinline__ float sigmoid_f(float z) { return 1.0f / (1.0f + expf(-z)); }

__device__ __forceinline__ void drain_wait_g(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > 200000000ull) break;
  }
}

// MODE 0: f1 epilogue (z1, U, V|Q|K).  MODE 1: f2 epilogue (out = X + acc).
template <int MODE, int BN>
__global__ void __launch_bounds__(kGThreads, 1)
hstu_gemm_tc_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tma0,
                    const __grid_constant__ CUtensorMap tma1, const __grid_constant__ CUtensorMap tmb) {
  using L = GLayout<BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const uint32_t bar0 = base_u32 + L::BAR_OFF;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L::MISC_OFF + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(bar(GB_FULL + s), 1);
      mbar_init(bar(GB_EMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(GB_AFULL + s), 1);
      mbar_init(bar(GB_AEMPTY + s), kGEpiWarps);
    }
    mbar_init(bar(GB_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kGMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kGTmemCols);
    tmem_relinquish();
  }
  if (warp == kGProducerWarp && lane == 0) {
    tma_prefetch_desc(&tma0);
    if (p.npass > 1) tma_prefetch_desc(&tma1);
    tma_prefetch_desc(&tmb);
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  Watchdog wd;
  wd.abort = abort_flag;
  wd.err = p.err;
  wd.err_info = p.err_info;
  if (MODE == 1 && blockIdx.x == 0 && threadIdx.x == 0 && p.carry_err) {
    const int code = p.carry_err[0];
    if (code != 0 && atomicCAS(p.err, 0, code) == 0) *p.err_info = p.carry_err[1];
  }
  wd.limit_ns = 2000000000ull;
  const int mblocks = (p.M + GBM - 1) / GBM, nblocks = p.N / BN;
  const int ntiles = mblocks * nblocks;
  const int kblocks = p.K / GBK;

  if (warp == kGProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      uint32_t armed[kGStages] = {0, 0, 0, 0};
      bool ok = true;
      for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
        const int mb = t / nblocks, nb = t % nblocks;
        for (int pass = 0; ok && pass < p.npass; ++pass) {
          const CUtensorMap* ma = pass == 0 ? &tma0 : &tma1;
          for (int kb = 0; kb < kblocks; ++kb) {
            const int stage = (int)(it % kGStages);
            ok = mbar_wait(bar(GB_EMPTY + stage), ((it / kGStages) & 1) ^ 1, wd, 41);
            if (!ok) break;
            const uint32_t sA = base_u32 + stage * L::STAGE, sB = sA + L::A_BYTES;
            mbar_arrive_expect_tx(bar(GB_FULL + stage), L::STAGE);
            tma_load_2d(sA, ma, bar(GB_FULL + stage), kb * GBK, mb * GBM);
            for (int c = 0; c < BN / 64; ++c)
              tma_load_2d(sB + c * L::B_BOX, &tmb, bar(GB_FULL + stage), nb * BN + c * 64, kb * GBK);
            armed[stage] += 1;
            ++it;
          }
        }
      }
      for (int s = 0; s < kGStages; ++s)
        if (armed[s]) drain_wait_g(bar(GB_FULL + s), (armed[s] - 1) & 1);
    }
  } else if (warp == kGMmaWarp) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16(GBM, BN, false, true);
      uint32_t it = 0, tc_it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
        const uint32_t ab = tc_it & 1;
        ok = mbar_wait(bar(GB_AEMPTY + ab), ((tc_it >> 1) & 1) ^ 1, wd, 42);
        if (!ok) break;
        fence_after_sync();
        bool first = true;
        for (int pass = 0; ok && pass < p.npass; ++pass) {
          for (int kb = 0; kb < kblocks; ++kb) {
            const int stage = (int)(it % kGStages);
            ok = mbar_wait(bar(GB_FULL + stage), (it / kGStages) & 1, wd, 43);
            if (!ok) break;
            fence_after_sync();
            const uint32_t sA = base_u32 + stage * L::STAGE, sB = sA + L::A_BYTES;
#pragma unroll
            for (int kk = 0; kk < GBK / 16; ++kk)
              mma_ss(tmem + ab * 256, sdesc_sw128(sA + kk * 32, 16, 1024),
                     sdesc_sw128(sB + kk * 2048, L::B_BOX, 1024), IDESC, (first && kk == 0) ? 0u : 1u);
            first = false;
            mma_commit(bar(GB_EMPTY + stage));
            ++it;
          }
        }
        if (!ok) break;
        mma_commit(bar(GB_AFULL + ab));
        ++tc_it;
      }
      mma_commit(bar(GB_DRAIN));
      drain_wait_g(bar(GB_DRAIN), 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3, ch = warp >> 2;   // TMEM lane quarter, column half of the tile
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    uint32_t tc_it = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
      const int mb = t / nblocks, nb = t % nblocks;
      const uint32_t ab = tc_it & 1;
      ok = mbar_wait(bar(GB_AFULL + ab), (tc_it >> 1) & 1, wd, 44);
      if (!ok) break;
      fence_after_sync();
      const int row = mb * GBM + wq * 32 + lane;
      const bool row_ok = row < p.M;
#pragma unroll 1
      for (int cc = 0; cc < BN / 64; ++cc) {
        const int col = ch * (BN / 2) + cc * 32;     // within the tile
        uint32_t v[32];
        tmem_ld32(lane_base + ab * 256 + col, v);
        tmem_wait_ld();
        if (!row_ok) continue;
        const int n = nb * BN + col;                 // output column
        if (MODE == 0) {
          float4* zdst = reinterpret_cast<float4*>(p.z1 + (size_t)row * p.N + n);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            zdst[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                  __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
          const int part = n / p.D, f = n % p.D;     // 32 columns never straddle a part
          float a[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float z = __uint_as_float(v[e]);
            a[e] = z * sigmoid_f(z);
          }
          if (part == 0) {
            float4* udst = reinterpret_cast<float4*>(p.u + (size_t)row * p.D + f);
#pragma unroll
            for (int e = 0; e < 8; ++e) udst[e] = make_float4(a[4 * e], a[4 * e + 1], a[4 * e + 2], a[4 * e + 3]);
          } else {
            uint4* vdst = reinterpret_cast<uint4*>(p.vqk + (size_t)(part - 1) * p.M * p.D + (size_t)row * p.D + f);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              vdst[e] = make_uint4(pack_bf16(a[8 * e], a[8 * e + 1]), pack_bf16(a[8 * e + 2], a[8 * e + 3]),
                                   pack_bf16(a[8 * e + 4], a[8 * e + 5]), pack_bf16(a[8 * e + 6], a[8 * e + 7]));
          }
        } else {
          const uint4* xs = reinterpret_cast<const uint4*>(p.x + (size_t)row * p.N + n);
          float4* odst = reinterpret_cast<float4*>(p.out + (size_t)row * p.N + n);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint4 xv = xs[e];
            odst[2 * e] = make_float4(__uint_as_float(v[8 * e]) + bf16_lo_f(xv.x),
                                      __uint_as_float(v[8 * e + 1]) + bf16_hi_f(xv.x),
                                      __uint_as_float(v[8 * e + 2]) + bf16_lo_f(xv.y),
                                      __uint_as_float(v[8 * e + 3]) + bf16_hi_f(xv.y));
            odst[2 * e + 1] = make_float4(__uint_as_float(v[8 * e + 4]) + bf16_lo_f(xv.z),
                                          __uint_as_float(v[8 * e + 5]) + bf16_hi_f(xv.z),
                                          __uint_as_float(v[8 * e + 6]) + bf16_lo_f(xv.w),
                                          __uint_as_float(v[8 * e + 7]) + bf16_hi_f(xv.w));
          }
        }
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(GB_AEMPTY + ab));
      ++tc_it;
    }
  }

  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == kGMmaWarp) tmem_dealloc(tmem, kGTmemCols);
}

// 2-D BF16 tensor map over [rows, cols] (row-major) with a 64-column box of
// box_rows rows, 128-byte swizzle (the layer's operands).
template <int MODE, int BN>
cudaError_t launch_gemm_t(const GemmParams& p, const void* a0, const void* a1, const void* b, int num_sms,
                          cudaStream_t st) {
  CUtensorMap m0, m1, mb;
  if (!make_tmap_bf16(&m0, a0, p.M, p.K, GBM) || !make_tmap_bf16(&mb, b, p.K, p.N, GBK)) return cudaErrorInvalidValue;
  if (p.npass > 1) {
    if (!make_tmap_bf16(&m1, a1, p.M, p.K, GBM)) return cudaErrorInvalidValue;
  } else {
    m1 = m0;
  }
  const size_t smem = GLayout<BN>::BYTES + 1024;
  const void* fn = reinterpret_cast<const void*>(hstu_gemm_tc_kernel<MODE, BN>);
  cudaError_t e = cudaFuncSetAttribute(hstu_gemm_tc_kernel<MODE, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) {
    set_launch_detail(e, "hstu_gemm_tc_kernel (smem attribute)", fn, kGThreads, smem);
    return e;
  }
  const int ntiles = ((p.M + GBM - 1) / GBM) * (p.N / BN);
  const int grid = ntiles < num_sms ? ntiles : num_sms;
  if (grid <= 0) return cudaSuccess;
  hstu_gemm_tc_kernel<MODE, BN><<<grid, kGThreads, smem, st>>>(p, m0, m1, mb);
  e = cudaGetLastError();
  if (e != cudaSuccess) set_launch_detail(e, "hstu_gemm_tc_kernel", fn, kGThreads, smem);
  return e;
}

}  // namespace

bool gemm_tc_supported(int D) { return D > 0 && D % 128 == 0; }

cudaError_t launch_gemm_f1(const GemmParams& p, const void* x, const void* w1, int num_sms, cudaStream_t st) {
  return p.N % 256 == 0 ? launch_gemm_t<0, 256>(p, x, nullptr, w1, num_sms, st)
                        : launch_gemm_t<0, 128>(p, x, nullptr, w1, num_sms, st);
}

cudaError_t launch_gemm_f2(const GemmParams& p, const void* y_hi, const void* y_lo, const void* w2, int num_sms,
                           cudaStream_t st) {
  return p.N % 256 == 0 ? launch_gemm_t<1, 256>(p, y_hi, y_lo, w2, num_sms, st)
                        : launch_gemm_t<1, 128>(p, y_hi, y_lo, w2, num_sms, st);
}

}  // namespace hstu
