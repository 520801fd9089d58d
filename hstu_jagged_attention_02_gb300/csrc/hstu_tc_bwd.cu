// Tensor-core backward of HSTU jagged attention for sm_103a (BF16 inputs,
// d = 128).  Key-block stationary: each work item owns 128 key rows of one
// head and walks the 64-row query tiles the compound mask keeps.  A is
// recomputed, never stored (HSTU's memory design: sub-layer activations are
// not kept, ai6s.net survey section 2.1.3).
//
// Per query tile, with S^T, dA^T, dV, dK, dQ^T accumulated in TMEM (FP32):
//   S^T  = K Q^T                          (A = K, B = Q, both K-major)
//   dA^T = V dO^T                         (dO = dO_hi + dO_lo, two MMAs)
//   A    = mask ? SiLU(z) / N : 0,  z = alpha S + rab_pos[bp] + rab_time[bt]
//   dZ   = mask ? dA SiLU'(z) / N : 0,    SiLU'(z) = s (1 + z (1 - s))
//   dV  += A^T dO                         (A from TMEM as hi/lo pair)
//   dK  += dZ^T Q                         (dZ from TMEM as hi/lo pair)
//   dQ^T = K^T dZ^T                       (both MN-major in SMEM) -> FP32 red
//   d_rab[bucket] += dZ                   (shared-memory accumulators)
// Every derived operand (dO, A, dZ) enters the tensor core as a BF16 pair
// x = hi + lo; a single BF16 rounding of any of them costs ~1.5% of the
// output RMS on heavy-tailed batches.
//
// Roles (320 threads): warps 0-7 epilogue (TMEM lane quarter warp%4, column
// half warp/4), warp 8 TMA producer, warp 9 MMA issuer and TMEM owner.
#include "hstu_internal.h"
#include "tc_ptx.cuh"

namespace hstu {

namespace {

using namespace tc;

constexpr int D = 128;
constexpr int BQ = kTcBwdQTile;   // 64 query rows per tile
constexpr int BK = kTcTile;       // 128 key rows per item
constexpr int kEpiWarps = 8;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kThreads = 10 * 32;
constexpr int kQStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t DV_COL = 0, DK_COL = 128, S_COL = 256, DA_COL = 320, DQ_COL = 384;
constexpr float kLog2e = 1.4426950408889634f;

enum : int { BAR_KVFULL = 0, BAR_KVEMPTY, BAR_QFULL, BAR_QEMPTY = BAR_QFULL + kQStages,
             BAR_SFULL = BAR_QEMPTY + kQStages, BAR_PREADY, BAR_DQFULL, BAR_DQEMPTY, BAR_DKVFULL,
             BAR_DKVEMPTY, BAR_DRAIN, BAR_COUNT };

struct Lay {
  static constexpr int KBOX = BK * 128;            // 128 rows x 128 B = 16 KB
  static constexpr int QBOX = BQ * 128;            // 64 rows x 128 B = 8 KB
  static constexpr int K_OFF = 0;                  // K tile: 2 chunks of 16 KB
  static constexpr int V_OFF = K_OFF + 2 * KBOX;
  static constexpr int QS_OFF = V_OFF + 2 * KBOX;  // per stage: Q, dO_hi, dO_lo (2 chunks of 8 KB each)
  static constexpr int Q_BYTES = 2 * QBOX;
  static constexpr int QSTAGE = 3 * Q_BYTES;
  static constexpr int DZ_OFF = QS_OFF + kQStages * QSTAGE;  // dZ^T hi then lo: [128 key][64 query] bf16
  static constexpr int DZ_BYTES = BK * 128;
  static constexpr int TSQ_OFF = DZ_OFF + 2 * DZ_BYTES;      // int64 [kQStages][BQ]
  static constexpr int BAR_OFF = TSQ_OFF + kQStages * BQ * 8;
  static constexpr int MISC_OFF = BAR_OFF + BAR_COUNT * 8;
  static constexpr int TAB_OFF = MISC_OFF + 16;              // float [H][P+Tb] bias, then [H][P+Tb] d_rab
};

__device__ __forceinline__ float fast_sigmoid(float z) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-z * kLog2e));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return r;
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

struct Item {
  int b, h, k0;
  SeqInfo s;
};

__device__ __forceinline__ bool item_of(const AttnParams& p, int r, int nitems, Item& it) {
  const int G = gridDim.x;
  const int idx = r * G + ((r & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);  // snake order
  if (idx >= nitems) return false;
  const Block blk = p.blocks[idx / p.H];
  it.b = blk.b;
  it.h = idx % p.H;
  it.k0 = blk.blk * BK;
  it.s = seq_info(p.off, p.nt, p.nc, blk.b);
  return true;
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > 200000000ull) break;
  }
}

template <typename TO>
__global__ void __launch_bounds__(kThreads, 1)
hstu_bwd_tc_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmq,
                   const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const __grid_constant__ CUtensorMap tmdh, const __grid_constant__ CUtensorMap tmdl) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const uint32_t sK = base_u32 + Lay::K_OFF, sV = base_u32 + Lay::V_OFF;
  const uint32_t sQS = base_u32 + Lay::QS_OFF, sDZ = base_u32 + Lay::DZ_OFF;
  int64_t* tsq = reinterpret_cast<int64_t*>(base + Lay::TSQ_OFF);
  const uint32_t bar0 = base_u32 + Lay::BAR_OFF;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + Lay::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + Lay::MISC_OFF + 4);
  const int H = p.H, P = p.P, Tb = p.Tb, PT = p.P + p.Tb;
  float* tab = reinterpret_cast<float*>(base + Lay::TAB_OFF);
  float* drab = tab + H * PT;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool has_rp = p.rab_pos != nullptr, has_rt = p.rab_time != nullptr && p.ts != nullptr;
  const bool want_rp = has_rp && p.d_rab_pos, want_rt = has_rt && p.d_rab_time;

  if (threadIdx.x == 0) {
    mbar_init(bar(BAR_KVFULL), 1);
    mbar_init(bar(BAR_KVEMPTY), 1);
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(bar(BAR_QFULL + s), 1);
      mbar_init(bar(BAR_QEMPTY + s), 1);
    }
    mbar_init(bar(BAR_SFULL), 1);
    mbar_init(bar(BAR_PREADY), kEpiWarps);
    mbar_init(bar(BAR_DQFULL), 1);
    mbar_init(bar(BAR_DQEMPTY), kEpiWarps);
    mbar_init(bar(BAR_DKVFULL), 1);
    mbar_init(bar(BAR_DKVEMPTY), kEpiWarps);
    mbar_init(bar(BAR_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int x = threadIdx.x; x < H * PT; x += kThreads) {
    const int h = x / PT, e = x % PT;
    float v = 0.f;
    if (e < P) {
      if (has_rp) v = p.rab_pos[h * P + e];
    } else if (has_rt) {
      v = p.rab_time[h * Tb + (e - P)];
    }
    tab[x] = v;
    drab[x] = 0.f;
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmq);
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
    tma_prefetch_desc(&tmdh);
    tma_prefetch_desc(&tmdl);
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  Watchdog wd;
  wd.abort = abort_flag;
  wd.err = p.hdr_rw + WS_ERR;
  wd.err_info = p.hdr_rw + WS_ERR_INFO;
  wd.limit_ns = (p.flags & HSTU_FLAG_TEST_TIMEOUT) ? 1000000ull : 2000000000ull;
  const int nitems = p.hdr[WS_NBLK] * H;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    uint32_t item_it = 0, qt_it = 0, kv_armed = 0;
    uint32_t armed[kQStages] = {0, 0};
    bool ok = true;
    Item it;
    for (int r = 0; ok && item_of(p, r, nitems, it); ++r) {
      const int n = it.s.n;
      if (lane == 0) {
        ok = mbar_wait(bar(BAR_KVEMPTY), (item_it & 1) ^ 1, wd, 21);
        if (ok) {
          mbar_arrive_expect_tx(bar(BAR_KVFULL), 4 * Lay::KBOX);
          const int y = (int)(it.s.s0 + it.k0);
          for (int c = 0; c < 2; ++c) {
            tma_load_2d(sK + c * Lay::KBOX, &tmk, bar(BAR_KVFULL), it.h * D + c * 64, y);
            tma_load_2d(sV + c * Lay::KBOX, &tmv, bar(BAR_KVFULL), it.h * D + c * 64, y);
          }
          ++kv_armed;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      ++item_it;
      const int nqt = (n + BQ - 1) / BQ;
      for (int qt = bwd_q_begin(it.k0, it.s.c, BQ); ok && qt < nqt; ++qt) {
        const int q0 = qt * BQ;
        if (tile_class(q0, it.k0, BQ, BK, n, it.s.c, it.s.h_end) == 0) continue;
        const int stage = qt_it % kQStages;
        ok = mbar_wait(bar(BAR_QEMPTY + stage), ((qt_it / kQStages) & 1) ^ 1, wd, 22);
        if (!ok) break;
        for (int rr = lane; rr < BQ; rr += 32) {
          const int row = q0 + rr;
          tsq[stage * BQ + rr] = (p.ts && row < n) ? p.ts[it.s.s0 + row] : 0;
        }
        __syncwarp();
        if (lane == 0) {
          const uint32_t full = bar(BAR_QFULL + stage);
          mbar_arrive_expect_tx(full, Lay::QSTAGE);
          const uint32_t dst = sQS + stage * Lay::QSTAGE;
          const int y = (int)(it.s.s0 + q0);
          for (int c = 0; c < 2; ++c) {
            tma_load_2d(dst + c * Lay::QBOX, &tmq, full, it.h * D + c * 64, y);
            tma_load_2d(dst + Lay::Q_BYTES + c * Lay::QBOX, &tmdh, full, it.h * D + c * 64, y);
            tma_load_2d(dst + 2 * Lay::Q_BYTES + c * Lay::QBOX, &tmdl, full, it.h * D + c * 64, y);
          }
          armed[stage] += 1;
        }
        ++qt_it;
      }
    }
    if (lane == 0) {
      for (int s = 0; s < kQStages; ++s)
        if (armed[s]) drain_wait(bar(BAR_QFULL + s), (armed[s] - 1) & 1);
      if (kv_armed) drain_wait(bar(BAR_KVFULL), (kv_armed - 1) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(BK, BQ, false, false);    // M=128 keys, N=64 queries
      constexpr uint32_t IDESC_DVK = idesc_bf16(BK, D, false, true);    // A from TMEM, B MN-major
      constexpr uint32_t IDESC_DQ = idesc_bf16(D, BQ, true, true);      // A = K^T, B = dZ^T, MN-major
      uint32_t item_it = 0, qt_it = 0;
      bool ok = true;
      Item it;
      for (int r = 0; ok && item_of(p, r, nitems, it); ++r) {
        const int n = it.s.n;
        ok = mbar_wait(bar(BAR_KVFULL), item_it & 1, wd, 23) &&
             mbar_wait(bar(BAR_DKVEMPTY), (item_it & 1) ^ 1, wd, 24);
        if (!ok) break;
        fence_after_sync();
        bool first = true;
        const int nqt = (n + BQ - 1) / BQ;
        for (int qt = bwd_q_begin(it.k0, it.s.c, BQ); ok && qt < nqt; ++qt) {
          if (tile_class(qt * BQ, it.k0, BQ, BK, n, it.s.c, it.s.h_end) == 0) continue;
          const uint32_t stage = qt_it % kQStages;
          ok = mbar_wait(bar(BAR_QFULL + stage), (qt_it / kQStages) & 1, wd, 25);
          if (!ok) break;
          fence_after_sync();
          const uint32_t sQ = sQS + stage * Lay::QSTAGE;
          const uint32_t sDh = sQ + Lay::Q_BYTES, sDl = sQ + 2 * Lay::Q_BYTES;
          // S^T = K Q^T ; dA^T = V dO_hi^T + V dO_lo^T
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = (kk >> 2) * Lay::KBOX + (kk & 3) * 32;
            const uint32_t qb = (kk >> 2) * Lay::QBOX + (kk & 3) * 32;
            mma_ss(tmem + S_COL, sdesc_sw128(sK + ka, 16, 1024), sdesc_sw128(sQ + qb, 16, 1024), IDESC_S,
                   kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = (kk >> 2) * Lay::KBOX + (kk & 3) * 32;
            const uint32_t qb = (kk >> 2) * Lay::QBOX + (kk & 3) * 32;
            const uint64_t av = sdesc_sw128(sV + ka, 16, 1024);
            mma_ss(tmem + DA_COL, av, sdesc_sw128(sDh + qb, 16, 1024), IDESC_S, kk > 0 ? 1u : 0u);
            mma_ss(tmem + DA_COL, av, sdesc_sw128(sDl + qb, 16, 1024), IDESC_S, 1u);
          }
          mma_commit(bar(BAR_SFULL));
          ok = mbar_wait(bar(BAR_PREADY), qt_it & 1, wd, 26) &&
               mbar_wait(bar(BAR_DQEMPTY), (qt_it & 1) ^ 1, wd, 27);
          if (!ok) break;
          fence_after_sync();
          // dV += A^T dO ; dK += dZ^T Q   (K = 64 queries: 4 steps of 16)
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk) {
            const uint32_t a_hi = tmem + S_COL + 32u * (kk >> 1) + 8u * (kk & 1);
            const uint32_t z_hi = tmem + DA_COL + 32u * (kk >> 1) + 8u * (kk & 1);
            const uint64_t bdh = sdesc_sw128(sDh + kk * 2048, Lay::QBOX, 1024);
            const uint64_t bdl = sdesc_sw128(sDl + kk * 2048, Lay::QBOX, 1024);
            const uint64_t bq = sdesc_sw128(sQ + kk * 2048, Lay::QBOX, 1024);
            const uint32_t acc0 = (first && kk == 0) ? 0u : 1u;
            mma_ts(tmem + DV_COL, a_hi, bdh, IDESC_DVK, acc0);
            mma_ts(tmem + DV_COL, a_hi + 16, bdh, IDESC_DVK, 1u);
            mma_ts(tmem + DV_COL, a_hi, bdl, IDESC_DVK, 1u);
            mma_ts(tmem + DK_COL, z_hi, bq, IDESC_DVK, acc0);
            mma_ts(tmem + DK_COL, z_hi + 16, bq, IDESC_DVK, 1u);
          }
          // dQ^T = K^T dZ^T  (K = 128 keys: 8 steps of 16)
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ak = sdesc_sw128(sK + kk * 2048, Lay::KBOX, 1024);
            mma_ss(tmem + DQ_COL, ak, sdesc_sw128(sDZ + kk * 2048, Lay::DZ_BYTES, 1024), IDESC_DQ,
                   kk > 0 ? 1u : 0u);
            mma_ss(tmem + DQ_COL, ak, sdesc_sw128(sDZ + Lay::DZ_BYTES + kk * 2048, Lay::DZ_BYTES, 1024),
                   IDESC_DQ, 1u);
          }
          mma_commit(bar(BAR_DQFULL));
          mma_commit(bar(BAR_QEMPTY + stage));
          first = false;
          ++qt_it;
        }
        if (!ok) break;
        mma_commit(bar(BAR_DKVFULL));
        mma_commit(bar(BAR_KVEMPTY));
        ++item_it;
      }
      mma_commit(bar(BAR_DRAIN));
      drain_wait(bar(BAR_DRAIN), 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3, hh = warp >> 2;
    const int lrow = wq * 32 + lane;                  // TMEM lane: key row (S^T, dV, dK) or d (dQ^T)
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    const float alpha = p.alpha, inv_n = p.inv_n;
    uint32_t item_it = 0, qt_it = 0;
    bool ok = true;
    Item it;
    for (int r = 0; ok && item_of(p, r, nitems, it); ++r) {
      const int n = it.s.n, cx = it.s.c, h_end = it.s.h_end;
      const int j = it.k0 + lrow;
      const bool j_ok = j < n;
      const int pos_j = j < h_end ? j : h_end;
      const int64_t t_j = (p.ts && j_ok) ? p.ts[it.s.s0 + j] : 0;
      const float* tp = tab + it.h * PT;
      const float* tt = tp + P;
      float* drp = drab + it.h * PT;
      float* drt = drp + P;
      const int nqt = (n + BQ - 1) / BQ;
      for (int qt = bwd_q_begin(it.k0, cx, BQ); ok && qt < nqt; ++qt) {
        const int q0 = qt * BQ;
        const int cls = tile_class(q0, it.k0, BQ, BK, n, cx, h_end);
        if (cls == 0) continue;
        const uint32_t stage = qt_it % kQStages;
        ok = mbar_wait(bar(BAR_QFULL + stage), (qt_it / kQStages) & 1, wd, 28) &&
             mbar_wait(bar(BAR_SFULL), qt_it & 1, wd, 29);
        if (!ok) break;
        fence_after_sync();
        uint32_t sv[32], dav[32];
        tmem_ld32(lane_base + S_COL + hh * 32, sv);
        tmem_ld32(lane_base + DA_COL + hh * 32, dav);
        tmem_wait_ld();
        const int64_t* tq = tsq + stage * BQ + hh * 32;
        uint32_t ahi[16], alo[16], zhi[16], zlo[16];
        // d_rab partial sums: the clamped position bucket in a register, the
        // time bucket run-length along the row (timestamps are mostly sorted)
        float rp_far = 0.f, rt_run = 0.f;
        int rt_cur = -1;
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float av[2], zv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int i = q0 + hh * 32 + c + e;
            const int pi = i < h_end ? i : h_end;
            int dp = pi - pos_j;
            dp = dp < 0 ? -dp : dp;
            const int bp = dp < P - 1 ? dp : P - 1;
            const int64_t ti = tq[c + e];
            const uint64_t dt = ti >= t_j ? (uint64_t)(ti - t_j) : (uint64_t)(t_j - ti);
            int bt = 64 - __clzll((long long)dt);
            bt = bt < Tb - 1 ? bt : Tb - 1;
            const float z = fmaf(alpha, __uint_as_float(sv[c + e]), tp[bp] + tt[bt]);
            const float sg = fast_sigmoid(z);
            const bool valid = cls == 2 || (j_ok && i < n && allowed(i, j, cx, h_end));
            float a = 0.f, dz = 0.f;
            if (valid) {
              a = z * sg * inv_n;
              dz = __uint_as_float(dav[c + e]) * sg * fmaf(z, 1.f - sg, 1.f) * inv_n;
              if (want_rp) {
                if (bp == P - 1) rp_far += dz;
                else atomicAdd(drp + bp, dz);
              }
              if (want_rt) {
                if (bt == rt_cur) {
                  rt_run += dz;
                } else {
                  if (rt_cur >= 0) atomicAdd(drt + rt_cur, rt_run);
                  rt_cur = bt;
                  rt_run = dz;
                }
              }
            }
            av[e] = a;
            zv[e] = dz;
          }
          const uint32_t ah = pack_bf16(av[0], av[1]);
          const uint32_t zh = pack_bf16(zv[0], zv[1]);
          ahi[c >> 1] = ah;
          alo[c >> 1] = pack_bf16(av[0] - bf16_lo_f(ah), av[1] - bf16_hi_f(ah));
          zhi[c >> 1] = zh;
          zlo[c >> 1] = pack_bf16(zv[0] - bf16_lo_f(zh), zv[1] - bf16_hi_f(zh));
        }
        if (want_rt && rt_cur >= 0) atomicAdd(drt + rt_cur, rt_run);
        if (want_rp) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) rp_far += __shfl_xor_sync(0xffffffffu, rp_far, o);
          if (lane == 0 && rp_far != 0.f) atomicAdd(drp + (P - 1), rp_far);
        }
        // A and dZ back into TMEM: hi at [32 hh, 32 hh + 16), lo at [32 hh + 16, 32 hh + 32)
        tmem_st16(lane_base + S_COL + hh * 32, ahi);
        tmem_st16(lane_base + S_COL + hh * 32 + 16, alo);
        tmem_st16(lane_base + DA_COL + hh * 32, zhi);
        tmem_st16(lane_base + DA_COL + hh * 32 + 16, zlo);
        // dZ^T into SMEM (row = key, 64 queries = 128 B, 128-byte swizzle) for the dQ MMA
        {
          const uint32_t rowh = sDZ + (uint32_t)lrow * 128u, rowl = rowh + Lay::DZ_BYTES;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t chunk = (uint32_t)((hh * 4 + k) ^ (lrow & 7));
            st_shared_v4(rowh + chunk * 16, zhi[4 * k], zhi[4 * k + 1], zhi[4 * k + 2], zhi[4 * k + 3]);
            st_shared_v4(rowl + chunk * 16, zlo[4 * k], zlo[4 * k + 1], zlo[4 * k + 2], zlo[4 * k + 3]);
          }
        }
        fence_async_smem();
        tmem_wait_st();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_PREADY));
        // dQ^T drain: lane = d, columns = 32 queries of this half
        ok = mbar_wait(bar(BAR_DQFULL), qt_it & 1, wd, 30);
        if (!ok) break;
        fence_after_sync();
        uint32_t qv[32];
        tmem_ld32(lane_base + DQ_COL + hh * 32, qv);
        tmem_wait_ld();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_DQEMPTY));
        {
          const int ib = q0 + hh * 32;
          float* dst = p.dq_acc + ((size_t)(it.s.s0 + ib) * H + it.h) * D + lrow;
          const size_t ld = (size_t)H * D;
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (ib + c < n) atomicAdd(dst + c * ld, alpha * __uint_as_float(qv[c]));
        }
        ++qt_it;
      }
      if (!ok) break;
      // dV, dK out: lane = key row, columns half hh of d
      ok = mbar_wait(bar(BAR_DKVFULL), item_it & 1, wd, 31);
      if (!ok) break;
      fence_after_sync();
      const size_t g = ((size_t)(it.s.s0 + j) * H + it.h) * D + hh * 64;
      TO* dvp = static_cast<TO*>(p.dv) + g;
      TO* dkp = static_cast<TO*>(p.dk) + g;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const uint32_t col = (part == 0 ? DV_COL : DK_COL) + hh * 64;
        TO* dst = part == 0 ? dvp : dkp;
        const float scale = part == 0 ? 1.f : alpha;
#pragma unroll
        for (int c = 0; c < 64; c += 32) {
          uint32_t v[32];
          tmem_ld32(lane_base + col + c, v);
          tmem_wait_ld();
          if (j_ok) {
            if constexpr (sizeof(TO) == 4) {
              float4* o4 = reinterpret_cast<float4*>(dst + c);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                o4[e] = make_float4(scale * __uint_as_float(v[4 * e]), scale * __uint_as_float(v[4 * e + 1]),
                                    scale * __uint_as_float(v[4 * e + 2]), scale * __uint_as_float(v[4 * e + 3]));
            } else {
              uint4* o4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                o4[e] = make_uint4(
                    pack_bf16(scale * __uint_as_float(v[8 * e]), scale * __uint_as_float(v[8 * e + 1])),
                    pack_bf16(scale * __uint_as_float(v[8 * e + 2]), scale * __uint_as_float(v[8 * e + 3])),
                    pack_bf16(scale * __uint_as_float(v[8 * e + 4]), scale * __uint_as_float(v[8 * e + 5])),
                    pack_bf16(scale * __uint_as_float(v[8 * e + 6]), scale * __uint_as_float(v[8 * e + 7])));
            }
          }
        }
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_DKVEMPTY));
      ++item_it;
    }
  }

  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  // flush the per-CTA d_rab partial sums
  for (int x = threadIdx.x; x < H * PT; x += kThreads) {
    const float v = drab[x];
    if (v == 0.f) continue;
    const int h = x / PT, e = x % PT;
    if (e < P) {
      if (want_rp) atomicAdd(p.d_rab_pos + h * P + e, v);
    } else if (want_rt) {
      atomicAdd(p.d_rab_time + h * Tb + (e - P), v);
    }
  }
}

template <typename TO>
cudaError_t launch_t(const AttnParams& p, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mdh, mdl;
  const int64_t cols = (int64_t)p.H * D;
  const __nv_bfloat16* dh = static_cast<const __nv_bfloat16*>(p.dO);
  const __nv_bfloat16* dl = dh + (size_t)p.T * cols;
  if (!make_tmap_bf16(&mq, p.q, p.T, cols, BQ) || !make_tmap_bf16(&mk, p.k, p.T, cols, BK) ||
      !make_tmap_bf16(&mv, p.v, p.T, cols, BK) || !make_tmap_bf16(&mdh, dh, p.T, cols, BQ) ||
      !make_tmap_bf16(&mdl, dl, p.T, cols, BQ))
    return cudaErrorInvalidValue;
  const size_t smem = tc_bwd_smem_bytes(p.H, p.P, p.Tb);
  cudaError_t e = cudaFuncSetAttribute(hstu_bwd_tc_kernel<TO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t max_items = ((p.T + BK - 1) / BK + p.B) * (int64_t)p.H;
  const int grid = (int)(max_items < p.num_sms ? max_items : p.num_sms);
  hstu_bwd_tc_kernel<TO><<<grid, kThreads, smem, st>>>(p, mq, mk, mv, mdh, mdl);
  return cudaGetLastError();
}

}  // namespace

bool tc_bwd_supported(int dtype, int dqk, int dv) { return dtype == HSTU_BF16 && dqk == D && dv == D; }

size_t tc_bwd_smem_bytes(int H, int P, int Tb) {
  return Lay::TAB_OFF + 2 * sizeof(float) * (size_t)H * (P + Tb) + 1024;
}

cudaError_t launch_tc_bwd(const AttnParams& p, cudaStream_t st) {
  return p.out_dtype == HSTU_FP32 ? launch_t<float>(p, st) : launch_t<__nv_bfloat16>(p, st);
}

}  // namespace hstu
