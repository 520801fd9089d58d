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
// 3-stage TMA ring, tcgen05.mma (M = 128, N = BN, K = 16) into one of two
// FP32 TMEM accumulators, so the next tile's MMAs overlap this tile's
// epilogue.  Persistent CTAs walk the tiles row-block-major, so the CTAs in
// flight share their X rows in L2.
//
// The epilogue is store-bound (z1 alone is 16 bytes per output column of a
// token): each warp stages its 32 x 32 chunks in 128-byte- (FP32) or
// 64-byte-swizzled (BF16) shared memory, conflict-free, and writes them with
// TMA tile stores, whole lines per row; the stores clip the ragged last row
// block.  Two staging buffers per warp, each reused once the bulk group that
// last read it is done.
//
// Roles (320 threads): warps 0-7 epilogue (TMEM lane quarter warp % 4,
// column half warp / 4), warp 8 TMA producer, warp 9 MMA issuer and TMEM
// owner.  Every wait is bounded; a wait that runs out records HSTU_ERR_TIMEOUT
// in the layer's header word and every role exits (a test-only mode makes CTA
// 0 skip its first load so that this path runs without a hang).
#include "hstu_internal.h"
#include "tc_ptx.cuh"

namespace hstu {

namespace {

using namespace tc;

constexpr int GBM = 128, GBK = 64;
constexpr int kGStages = 3;
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
  static constexpr int STG_WARP = 2 * 4096;             // two 32 x 32 FP32 staging buffers per epilogue warp
  static constexpr int STG_OFF = kGStages * STAGE;
  static constexpr int BAR_OFF = STG_OFF + kGEpiWarps * STG_WARP;
  static constexpr int MISC_OFF = BAR_OFF + GB_COUNT * 8;  // tmem slot, abort flag
  static constexpr int BYTES = MISC_OFF + 16;
};

// SiLU(z) = z / (1 + e^-z) with the fast exponential and division
// intrinsics (relative error about 1e-6; z below about -87 gives 0)
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// FP32 row `lane` (32 values) of a 32 x 32 staging buffer, 128-byte swizzle:
// 16-byte chunk c of row r at chunk c ^ (r % 8) of the row's 128 bytes
__device__ __forceinline__ void stage_f32(uint8_t* buf, int lane, const float* a) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<float4*>(buf + lane * 128 + ((c ^ (lane & 7)) << 4)) =
        make_float4(a[4 * c], a[4 * c + 1], a[4 * c + 2], a[4 * c + 3]);
}
// BF16 row `lane` (32 values, 64 bytes) of a 32 x 32 staging buffer, 64-byte
// swizzle: 16-byte chunk c of row r at chunk c ^ ((r / 2) % 4)
__device__ __forceinline__ void stage_bf16(uint8_t* buf, int lane, const float* a) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(buf + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) =
        make_uint4(pack_bf16(a[8 * c], a[8 * c + 1]), pack_bf16(a[8 * c + 2], a[8 * c + 3]),
                   pack_bf16(a[8 * c + 4], a[8 * c + 5]), pack_bf16(a[8 * c + 6], a[8 * c + 7]));
}

__device__ __forceinline__ void drain_wait_g(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > 200000000ull) break;
  }
}

// Epilogue modes.  0: f1 (z1, U, V|Q|K); 1: out = X + acc (BF16 residual);
// 2: out = acc; 3: out += acc (TMA reduce-add: split-K partial sums);
// 4: out = res + acc (FP32 residual).
enum : int { GM_F1 = 0, GM_RES_BF16 = 1, GM_STORE = 2, GM_REDUCE = 3, GM_RES_F32 = 4 };

// Operand layouts.  A_MN: A is the transpose of a row-major [K, M] array,
// loaded as two 64-column x 64-row boxes per k-block (M contiguous);
// otherwise a row-major [M, K] array, one 64 x 128 box.  B_KM: B is the
// transpose of a row-major [N, K] array, one 64-column x BN-row box
// (K contiguous); otherwise a row-major [K, N] array, BN / 64 boxes of
// 64 x 64.  Every box is 128-byte swizzled.
//
// Work items are (row block, column block, K range): the K range is all of
// K unless p.ksplit > 1, which only the reduce epilogue uses.
template <int MODE, int BN, bool A_MN, bool B_KM>
__global__ void __launch_bounds__(kGThreads, 1)
hstu_gemm_tc_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tma0,
                    const __grid_constant__ CUtensorMap tma1, const __grid_constant__ CUtensorMap tmb0,
                    const __grid_constant__ CUtensorMap tmb1, const __grid_constant__ CUtensorMap tms0,
                    const __grid_constant__ CUtensorMap tms1, const __grid_constant__ CUtensorMap tms2) {
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
    tma_prefetch_desc(&tmb0);
    if (p.npass > 1) {
      if (p.pair_b) tma_prefetch_desc(&tmb1);
      else tma_prefetch_desc(&tma1);
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  Watchdog wd;
  wd.abort = abort_flag;
  wd.err = p.err;
  wd.err_info = p.err_info;
  if (MODE != GM_F1 && blockIdx.x == 0 && threadIdx.x == 0 && p.carry_err) {
    const int code = p.carry_err[0];
    if (code != 0 && atomicCAS(p.err, 0, code) == 0) *p.err_info = p.carry_err[1];
  }
  wd.limit_ns = p.test_timeout ? 1000000ull : 2000000000ull;
  const int mblocks = (int)((p.M + GBM - 1) / GBM), nblocks = p.N / BN;
  const int ntiles = mblocks * nblocks;
  const int kbt = (int)((p.K + GBK - 1) / GBK);          // 64-blocks of K (the last one zero-filled)
  const int kper = (kbt + p.ksplit - 1) / p.ksplit;      // 64-blocks per K range
  const int nitems = ntiles * p.ksplit;
  // work item t: tile t % ntiles, K range t / ntiles, 64-blocks [kb0, kb1)
  auto item = [&](int t, int& mb, int& nb, int& kb0, int& kb1) {
    const int tile = t % ntiles, ks = t / ntiles;
    mb = tile / nblocks;
    nb = tile % nblocks;
    kb0 = ks * kper;
    kb1 = min(kbt, kb0 + kper);
  };

  if (warp == kGProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      uint32_t armed[kGStages] = {};
      bool ok = true;
      const bool withhold = p.test_timeout && blockIdx.x == 0;   // test only
      for (int t = blockIdx.x; ok && t < nitems; t += gridDim.x) {
        int mb, nb, kb0, kb1;
        item(t, mb, nb, kb0, kb1);
        for (int pass = 0; ok && pass < p.npass; ++pass) {
          const CUtensorMap* ma = (pass == 0 || p.pair_b) ? &tma0 : &tma1;
          const CUtensorMap* mbm = (pass == 0 || !p.pair_b) ? &tmb0 : &tmb1;
          for (int kb = kb0; kb < kb1; ++kb) {
            const int stage = (int)(it % kGStages);
            ok = mbar_wait(bar(GB_EMPTY + stage), ((it / kGStages) & 1) ^ 1, wd, 41);
            if (!ok) break;
            if (withhold && it == 0) {   // this stage's copy never comes: the MMA's wait runs out
              ++it;
              continue;
            }
            const uint32_t sA = base_u32 + stage * L::STAGE, sB = sA + L::A_BYTES;
            mbar_arrive_expect_tx(bar(GB_FULL + stage), L::STAGE);
            if (A_MN) {
              for (int c = 0; c < 2; ++c) tma_load_2d(sA + c * L::B_BOX, ma, bar(GB_FULL + stage), mb * GBM + c * 64, kb * GBK);
            } else {
              tma_load_2d(sA, ma, bar(GB_FULL + stage), kb * GBK, mb * GBM);
            }
            if (B_KM) {
              tma_load_2d(sB, mbm, bar(GB_FULL + stage), kb * GBK, nb * BN);
            } else {
              for (int c = 0; c < BN / 64; ++c)
                tma_load_2d(sB + c * L::B_BOX, mbm, bar(GB_FULL + stage), nb * BN + c * 64, kb * GBK);
            }
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
      constexpr uint32_t IDESC = idesc_bf16(GBM, BN, A_MN, !B_KM);
      uint32_t it = 0, tc_it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < nitems; t += gridDim.x) {
        int mb, nb, kb0, kb1;
        item(t, mb, nb, kb0, kb1);
        if (kb0 >= kb1) continue;   // an empty K range (the last split of a short K)
        const uint32_t ab = tc_it & 1;
        ok = mbar_wait(bar(GB_AEMPTY + ab), ((tc_it >> 1) & 1) ^ 1, wd, 42);
        if (!ok) break;
        fence_after_sync();
        bool first = true;
        for (int pass = 0; ok && pass < p.npass; ++pass) {
          for (int kb = kb0; kb < kb1; ++kb) {
            const int stage = (int)(it % kGStages);
            ok = mbar_wait(bar(GB_FULL + stage), (it / kGStages) & 1, wd, 43);
            if (!ok) break;
            fence_after_sync();
            const uint32_t sA = base_u32 + stage * L::STAGE, sB = sA + L::A_BYTES;
            // K-major operands step 32 bytes (16 k) along their 128-byte rows;
            // MN-major ones step 16 rows of 128 bytes, their 64-wide column
            // chunks one box (8 KB) apart
            const SDesc da = A_MN ? sdesc_w(sA, L::B_BOX, 1024) : sdesc_w(sA, 16, 1024);
            const SDesc db = B_KM ? sdesc_w(sB, 16, 1024) : sdesc_w(sB, L::B_BOX, 1024);
#pragma unroll
            for (int kk = 0; kk < GBK / 16; ++kk)
              mma_ss_w(tmem + ab * 256, da + (A_MN ? kk * 2048 : kk * 32), db + (B_KM ? kk * 32 : kk * 2048), IDESC,
                       (first && kk == 0) ? 0u : 1u);
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
    // tms0: z1 (f1) or out, FP32 [M, N]; tms1: u FP32 [M, D]; tms2: V | Q | K BF16 [3, M, D]
    const int wq = warp & 3, ch = warp >> 2;   // TMEM lane quarter, column half of the tile
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    uint8_t* stg = base + L::STG_OFF + warp * L::STG_WARP;
    const uint32_t stg_u32 = base_u32 + L::STG_OFF + warp * L::STG_WARP;
    uint32_t tc_it = 0, sc = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < nitems; t += gridDim.x) {
      int mb, nb, kb0, kb1;
      item(t, mb, nb, kb0, kb1);
      if (kb0 >= kb1) continue;   // no MMA ran for an empty K range: nothing to add
      const uint32_t ab = tc_it & 1;
      ok = mbar_wait(bar(GB_AFULL + ab), (tc_it >> 1) & 1, wd, 44);
      if (!ok) break;
      fence_after_sync();
      const int row0 = mb * GBM + wq * 32;
      const int row = row0 + lane;
      const bool in_rows = row0 < p.M;   // else the warp's 32 rows all lie past M: no store is issued
#pragma unroll 1
      for (int cc = 0; cc < BN / 64; ++cc) {
        const int col = ch * (BN / 2) + cc * 32;     // within the tile
        const int n = nb * BN + col;                 // output column
        uint32_t v[32];
        tmem_ld32(lane_base + ab * 256 + col, v);
        tmem_wait_ld();
        float a[32];
        if (MODE == GM_F1) {
#pragma unroll
          for (int e = 0; e < 32; ++e) a[e] = __uint_as_float(v[e]);
          // z1 chunk into buffer 0, once the store that last read it is done
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
          stage_f32(stg, lane, a);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (in_rows) tma_store_2d(&tms0, stg_u32, n, row0);
            bulk_commit();
          }
          // SiLU: U (FP32) or one of V, Q, K (BF16) into buffer 1; 32 columns never straddle a part
          const int part = n / p.D, f = n - part * p.D;
#pragma unroll
          for (int e = 0; e < 32; ++e) a[e] = silu_f(a[e]);
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
          if (part == 0) stage_f32(stg + 4096, lane, a);
          else stage_bf16(stg + 4096, lane, a);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (in_rows && part == 0) tma_store_2d(&tms1, stg_u32 + 4096, f, row0);
            if (in_rows && part != 0) tma_store_3d(&tms2, stg_u32 + 4096, f, row0, part - 1);
            bulk_commit();
          }
        } else {
          if (MODE == GM_RES_BF16) {
            // out = X + acc, X read as BF16 (rows past M read nothing and are not stored)
            uint4 xv[4] = {};
            if (row < p.M) {
              const uint4* xs = reinterpret_cast<const uint4*>(p.x + (size_t)row * p.N + n);
#pragma unroll
              for (int e = 0; e < 4; ++e) xv[e] = xs[e];
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              a[8 * e] = __uint_as_float(v[8 * e]) + bf16_lo_f(xv[e].x);
              a[8 * e + 1] = __uint_as_float(v[8 * e + 1]) + bf16_hi_f(xv[e].x);
              a[8 * e + 2] = __uint_as_float(v[8 * e + 2]) + bf16_lo_f(xv[e].y);
              a[8 * e + 3] = __uint_as_float(v[8 * e + 3]) + bf16_hi_f(xv[e].y);
              a[8 * e + 4] = __uint_as_float(v[8 * e + 4]) + bf16_lo_f(xv[e].z);
              a[8 * e + 5] = __uint_as_float(v[8 * e + 5]) + bf16_hi_f(xv[e].z);
              a[8 * e + 6] = __uint_as_float(v[8 * e + 6]) + bf16_lo_f(xv[e].w);
              a[8 * e + 7] = __uint_as_float(v[8 * e + 7]) + bf16_hi_f(xv[e].w);
            }
          } else if (MODE == GM_RES_F32) {
            // out = res + acc, res read as FP32 (rows past M read nothing)
            float4 rv[8] = {};
            if (row < p.M) {
              const float4* rs = reinterpret_cast<const float4*>(p.res + (size_t)row * p.N + n);
#pragma unroll
              for (int e = 0; e < 8; ++e) rv[e] = rs[e];
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              a[4 * e] = __uint_as_float(v[4 * e]) + rv[e].x;
              a[4 * e + 1] = __uint_as_float(v[4 * e + 1]) + rv[e].y;
              a[4 * e + 2] = __uint_as_float(v[4 * e + 2]) + rv[e].z;
              a[4 * e + 3] = __uint_as_float(v[4 * e + 3]) + rv[e].w;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) a[e] = __uint_as_float(v[e]);
          }
          // alternate the two buffers
          const uint32_t off = (sc & 1) * 4096;
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
          stage_f32(stg + off, lane, a);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (in_rows) {
              if (MODE == GM_REDUCE) tma_reduce_add_2d(&tms0, stg_u32 + off, n, row0);
              else tma_store_2d(&tms0, stg_u32 + off, n, row0);
            }
            bulk_commit();
          }
          ++sc;
        }
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(GB_AEMPTY + ab));
      ++tc_it;
    }
    if (lane == 0) bulk_wait_all();   // the staging buffers stay in use until every store is done
    __syncwarp();
  }

  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == kGMmaWarp) tmem_dealloc(tmem, kGTmemCols);
}

// 32 x 32 FP32 store box over a row-major [rows, cols] FP32 array, 128-byte swizzle
bool tmap_store_f32(CUtensorMap* m, const float* ptr, int64_t rows, int64_t cols) {
  const uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows}, strides[1] = {(uint64_t)cols * 4};
  const uint32_t box[2] = {32, 32};
  return make_tmap_tile(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// The kernel's seven maps.  A: 64 k-columns x 128 rows of a row-major
// [M, K] array, or 64 x 64 boxes of a row-major [K, M] array (A_MN).  B: 64
// n-columns x 64 k-rows of a row-major [K, N] array, or 64 k-columns x BN
// rows of a row-major [N, K] array (B_KM).  Every box 128-byte swizzled.
// Store maps: f1 z1, u and V | Q | K as [3, M, D] (each part clipped at row
// M); the other modes out only.
template <int MODE, int BN, bool A_MN, bool B_KM>
cudaError_t launch_gemm_t(const GemmParams& p, const void* a0, const void* a1, const void* b0, const void* b1,
                          int num_sms, cudaStream_t st) {
  CUtensorMap ma0, ma1, mb0, mb1, s0, s1, s2;
  auto map_a = [&](CUtensorMap* m, const void* a) {
    return A_MN ? make_tmap_bf16(m, a, p.K, p.M, GBK) : make_tmap_bf16(m, a, p.M, p.K, GBM);
  };
  auto map_b = [&](CUtensorMap* m, const void* b) {
    return B_KM ? make_tmap_bf16(m, b, p.N, p.K, BN) : make_tmap_bf16(m, b, p.K, p.N, GBK);
  };
  if (!map_a(&ma0, a0) || !map_b(&mb0, b0)) return cudaErrorInvalidValue;
  ma1 = ma0;
  mb1 = mb0;
  if (p.npass > 1) {
    if (p.pair_b ? !map_b(&mb1, b1) : !map_a(&ma1, a1)) return cudaErrorInvalidValue;
  }
  if (MODE == GM_F1) {
    const uint64_t dims[3] = {(uint64_t)p.D, (uint64_t)p.M, 3};
    const uint64_t strides[2] = {(uint64_t)p.D * 2, (uint64_t)p.M * p.D * 2};
    const uint32_t box[3] = {32, 32, 1};
    if (!tmap_store_f32(&s0, p.z1, p.M, p.N) || !tmap_store_f32(&s1, p.u, p.M, p.D) ||
        !make_tmap_tile(&s2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.vqk, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  } else {
    if (!tmap_store_f32(&s0, p.out, p.M, p.N)) return cudaErrorInvalidValue;
    s1 = s0;
    s2 = s0;
  }
  const size_t smem = GLayout<BN>::BYTES + 1024;
  auto kern = hstu_gemm_tc_kernel<MODE, BN, A_MN, B_KM>;
  const void* fn = reinterpret_cast<const void*>(kern);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) {
    set_launch_detail(e, "hstu_gemm_tc_kernel (smem attribute)", fn, kGThreads, smem);
    return e;
  }
  const int64_t nitems = ((p.M + GBM - 1) / GBM) * (int64_t)(p.N / BN) * p.ksplit;
  const int grid = (int)(nitems < num_sms ? nitems : num_sms);
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, kGThreads, smem, st>>>(p, ma0, ma1, mb0, mb1, s0, s1, s2);
  e = cudaGetLastError();
  if (e != cudaSuccess) set_launch_detail(e, "hstu_gemm_tc_kernel", fn, kGThreads, smem);
  return e;
}

}  // namespace

bool gemm_tc_supported(int D) { return D > 0 && D % 128 == 0; }

cudaError_t launch_gemm_f1(const GemmParams& p, const void* x, const void* w1, int num_sms, cudaStream_t st) {
  GemmParams q = p;
  q.npass = 1; q.pair_b = 0; q.ksplit = 1;
  return q.N % 256 == 0 ? launch_gemm_t<GM_F1, 256, false, false>(q, x, nullptr, w1, nullptr, num_sms, st)
                        : launch_gemm_t<GM_F1, 128, false, false>(q, x, nullptr, w1, nullptr, num_sms, st);
}

cudaError_t launch_gemm_f2(const GemmParams& p, const void* y_hi, const void* y_lo, const void* w2, int num_sms,
                           cudaStream_t st) {
  GemmParams q = p;
  q.npass = 2; q.pair_b = 0; q.ksplit = 1;
  return q.N % 256 == 0 ? launch_gemm_t<GM_RES_BF16, 256, false, false>(q, y_hi, y_lo, w2, nullptr, num_sms, st)
                        : launch_gemm_t<GM_RES_BF16, 128, false, false>(q, y_hi, y_lo, w2, nullptr, num_sms, st);
}

// out = [res +] sum over the passes of A_p W^T: A_p [M, K] row-major BF16
// (a1 the second half of a pair, or null for one pass), W [N, K] row-major
// BF16, out [M, N] FP32, res [M, N] FP32 or null
cudaError_t launch_gemm_nt(const GemmParams& p, const void* a0, const void* a1, const void* w, int num_sms,
                           cudaStream_t st) {
  GemmParams q = p;
  q.npass = a1 ? 2 : 1; q.pair_b = 0; q.ksplit = 1;
  if (q.res) {
    return q.N % 256 == 0 ? launch_gemm_t<GM_RES_F32, 256, false, true>(q, a0, a1, w, nullptr, num_sms, st)
                          : launch_gemm_t<GM_RES_F32, 128, false, true>(q, a0, a1, w, nullptr, num_sms, st);
  }
  return q.N % 256 == 0 ? launch_gemm_t<GM_STORE, 256, false, true>(q, a0, a1, w, nullptr, num_sms, st)
                        : launch_gemm_t<GM_STORE, 128, false, true>(q, a0, a1, w, nullptr, num_sms, st);
}

// out += sum over the passes of L_p^T R_p: L_p [K, M] and R_p [K, N]
// row-major BF16, out [M, N] FP32 already holding its start value (zero).
// One of l1, r1 may name the second half of a pair.  K is cut into ranges so
// that the work items about fill the GPU once; each range's partial sum is
// added into out by TMA reduce-add (FP32, in no fixed order).
cudaError_t launch_gemm_tn_reduce(const GemmParams& p, const void* l0, const void* l1, const void* r0, const void* r1,
                                  int num_sms, cudaStream_t st) {
  GemmParams q = p;
  q.npass = (l1 || r1) ? 2 : 1;
  q.pair_b = r1 ? 1 : 0;
  const bool wide = q.N % 256 == 0;
  const int64_t tiles = ((q.M + GBM - 1) / GBM) * (int64_t)(q.N / (wide ? 256 : 128));
  const int64_t kbt = (q.K + GBK - 1) / GBK;
  // the split that minimises the busiest CTA's work: waves of items x (64-blocks per
  // item + about two 64-blocks' worth for an item's start and its reduce)
  int64_t best_ks = 1, best_cost = -1;
  const int64_t sms = num_sms > 0 ? num_sms : 1;
  for (int64_t ks = 1; ks <= kbt && ks <= 64; ++ks) {
    const int64_t kper = (kbt + ks - 1) / ks;
    const int64_t used = (kbt + kper - 1) / kper;      // non-empty ranges
    const int64_t waves = (tiles * used + sms - 1) / sms;
    const int64_t cost = waves * (kper + 2);
    if (best_cost < 0 || cost < best_cost) { best_cost = cost; best_ks = ks; }
  }
  q.ksplit = (int)best_ks;
  return wide ? launch_gemm_t<GM_REDUCE, 256, true, false>(q, l0, l1, r0, r1, num_sms, st)
              : launch_gemm_t<GM_REDUCE, 128, true, false>(q, l0, l1, r0, r1, num_sms, st);
}

}  // namespace hstu
