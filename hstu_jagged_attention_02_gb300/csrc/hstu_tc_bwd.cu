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
//   dV  += A^T dO                         (A from its own TMEM buffer, hi/lo)
//   dK  += dZ^T Q                         (dZ^T staged in SMEM, hi/lo)
//   dQ^T = K^T dZ^T                       (both MN-major in SMEM) -> TMA reduce-add into FP32 dq
//   d_rab[bucket] += dZ                   (per-CTA partial sums, summed after)
// S^T and dA^T are released as soon as the epilogue has loaded them, so the
// next tile's S^T and dA^T are computed while this tile's A and dZ are; the
// dQ^T of a tile is drained in the middle of the next one.
// Every derived operand (dO, A, dZ) enters the tensor core as a BF16 pair
// x = hi + lo; a single BF16 rounding of any of them costs ~1.5% of the
// output RMS on heavy-tailed batches.
//
// Roles (576 threads): warps 0-15 epilogue (TMEM lane quarter warp%4, column
// quarter warp/4), warp 16 TMA producer, warp 17 MMA issuer and TMEM owner
// (the whole warp runs the issue loop, so its operands stay warp-uniform, and
// one elected lane issues each MMA and commit).
// The planner lists the key blocks longest-first and the producer takes its
// block index as its first work item and every later one from a global
// counter (greedy LPT), passing it to the other roles in a shared-memory slot
// with the item's key timestamps.
#include "hstu_internal.h"
#include "tc_ptx.cuh"

namespace hstu {

namespace {

using namespace tc;

constexpr int D = 128;
constexpr int BQ = kTcBwdQTile;   // 64 query rows per tile
constexpr int BK = kTcTile;       // 128 key rows per item
constexpr int kEpiWarps = 16;
constexpr int kProducerWarp = 16, kMmaWarp = 17;
constexpr int kThreads = 18 * 32;
constexpr int kQStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t DV_COL = 0, DK_COL = 128, S_COL = 256, DA_COL = 320, A_COL = 384, DQ_COL = 448;
constexpr float kLog2e = 1.4426950408889634f;

enum : int { BAR_KFULL = 0, BAR_KEMPTY, BAR_VFULL, BAR_VEMPTY, BAR_QFULL, BAR_QEMPTY = BAR_QFULL + kQStages,
             BAR_SFULL = BAR_QEMPTY + kQStages, BAR_SEMPTY, BAR_PREADY, BAR_DQFULL, BAR_DQEMPTY,
             BAR_DKVFULL, BAR_DKVEMPTY, BAR_DRAIN, BAR_COUNT };

// A work item as the producer hands it to the other roles.
struct __align__(16) ItemSlot {
  int64_t s0;     // first token of the sequence
  int64_t tbase;  // timestamp of that token (0 without timestamps)
  int valid;      // 0: no more work
  int h, k0, n, c, h_end;
  int wide;       // some key time of the item is 2^30 s or more from tbase
  int pad;
};

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
  static constexpr int TS64_OFF = DZ_OFF + 2 * DZ_BYTES;     // int64 [kQStages][BQ] absolute
  static constexpr int TS32_OFF = TS64_OFF + kQStages * BQ * 8;  // int32 [kQStages][BQ] relative
  static constexpr int CMM_OFF = TS32_OFF + kQStages * BQ * 4;   // int32 [kQStages][4 chunks][min, max] relative
  static constexpr int KTS_OFF = CMM_OFF + kQStages * 8 * 4;     // int64 [BK] key times of the item
  static constexpr int SLOT_OFF = KTS_OFF + BK * 8;              // ItemSlot
  static constexpr int BAR_OFF = SLOT_OFF + (int)sizeof(ItemSlot);
  static constexpr int MISC_OFF = BAR_OFF + BAR_COUNT * 8;
  // per epilogue warp: a 32-dim x 8-query FP32 block of dQ, the source of its
  // bulk reduce-add into dq
  static constexpr int DQS_OFF = (MISC_OFF + 16 + 127) / 128 * 128;
  static constexpr int DQS_WARP = 32 * 8 * 4;
  static constexpr int TAB_OFF = DQS_OFF + kEpiWarps * DQS_WARP;  // float [H][P+Tb] bias
};

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Fire-and-forget global float add when pred holds (no branch, no return value).
__device__ __forceinline__ void red_add(float* addr, float v, bool pred) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %2, 0;\n\t@p red.global.add.f32 [%0], %1;\n\t}" ::"l"(addr),
               "f"(v), "r"((int)pred)
               : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > 200000000ull) break;
  }
}

// Per-thread context of the epilogue: one key row j of the item.
struct KeyCtx {
  int j, h_end, pos_j;
  bool want_rp, want_rt;
  // the queries allowed to see this key under the compound mask: lo <= i <= hi
  int lo, hi;
  int32_t tj32;
  int64_t tj64;
  const float* tp;   // bias tables of the head, times -log2 e: position [0, P), time [P, P + Tb)
  float* drp;        // this CTA's d_rab partial sums of the head: position [0, P), time [P, P + Tb)
};

// d_rab partial sums one epilogue thread carries.  A thread owns one key row
// j and sees that row's query columns i in increasing order over the whole
// work item, so:
//  - the clamped position bucket (far from the diagonal) sums in rp_far;
//    the other position buckets go straight to the CTA's partial sums;
//  - the time bucket changes only where |t_i - t_j| crosses a power of two,
//    so a run sum (rt_cur, rt_run) rarely has to be flushed.
struct RabAcc {
  float rp_far, rt_run;
  int rt_cur;
};

// NC query columns ib.. of one key row: A and dZ as packed BF16 hi/lo pairs,
// plus the d_rab contributions; the mask is evaluated per element.  WIDE:
// 64-bit timestamp gaps.  (One code path for every tile class: the variants
// that skip the mask on full tiles cost more in instruction fetch than they
// save on heavy-tailed batches, where tile classes alternate.)
template <int NC, bool WIDE>
__device__ __forceinline__ void grad_cols(const AttnParams& p, const uint32_t (&sv)[NC], const uint32_t (&dav)[NC],
                                          uint32_t (&ahi)[NC / 2], uint32_t (&alo)[NC / 2], uint32_t (&zhi)[NC / 2],
                                          uint32_t (&zlo)[NC / 2], const KeyCtx& kc, int ib, const int32_t* ts32,
                                          const int64_t* ts64, RabAcc& acc) {
  int bps[NC], bts[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int i = ib + c;
    const int pi = i < kc.h_end ? i : kc.h_end;
    int dp = pi - kc.pos_j;
    dp = dp < 0 ? -dp : dp;
    const int bp = dp < p.P - 1 ? dp : p.P - 1;
    int bt;
    if (WIDE) {
      const int64_t ti = ts64[c];
      const uint64_t dt = ti >= kc.tj64 ? (uint64_t)(ti - kc.tj64) : (uint64_t)(kc.tj64 - ti);
      bt = 64 - __clzll((long long)dt);
    } else {
      int d = ts32[c] - kc.tj32;
      d = d < 0 ? -d : d;
      bt = 32 - __clz(d);
    }
    bt = bt < p.Tb - 1 ? bt : p.Tb - 1;
    bps[c] = bp;
    bts[c] = bt;
  }
  // Paired FP32 arithmetic (fma/mul/add on float2, one instruction for two
  // elements); each lane of a pair rounds exactly like the scalar operation,
  // and the products keep the scalar association.
  const float2 one2 = make_float2(1.f, 1.f);
#pragma unroll
  for (int c = 0; c < NC; c += 2) {
    const float2 b2 = __fadd2_rn(make_float2(kc.tp[bps[c]], kc.tp[bps[c + 1]]),
                                 make_float2(kc.tp[p.P + bts[c]], kc.tp[p.P + bts[c + 1]]));
    const float2 w2 = __ffma2_rn(p.kA2, make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), b2);
    const float2 d2 = __fadd2_rn(one2, make_float2(ex2_approx(w2.x), ex2_approx(w2.y)));
    const float2 sg2 = make_float2(rcp_approx(d2.x), rcp_approx(d2.y));
    const float2 z2 = make_float2(w2.x * p.kZ, w2.y * p.kZ);
    const float2 a2 = __fmul2_rn(make_float2(w2.x * p.kC, w2.y * p.kC), sg2);
    const float2 f2 = __ffma2_rn(z2, fsub2(one2, sg2), one2);  // 1 + z (1 - sg)
    const float2 h2 = __fmul2_rn(__fmul2_rn(make_float2(__uint_as_float(dav[c]), __uint_as_float(dav[c + 1])), sg2), f2);
    const float2 g2 = __fmul2_rn(h2, p.inv_n2);
    const float aa[2] = {a2.x, a2.y}, gg[2] = {g2.x, g2.y};
    float av[2], zv[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int i = ib + c + e;
      const bool valid = i >= kc.lo && i <= kc.hi;
      const float a = valid ? aa[e] : 0.f;
      const float dz = valid ? gg[e] : 0.f;
      av[e] = a;
      zv[e] = dz;
      if (kc.want_rp && valid) {
        if (bps[c + e] == p.P - 1) acc.rp_far += dz;
        else red_add(kc.drp + bps[c + e], dz, true);
      }
      if (kc.want_rt) {
        const bool flush = valid && bts[c + e] != acc.rt_cur;
        red_add(kc.drp + p.P + acc.rt_cur, acc.rt_run, flush && acc.rt_cur >= 0);
        acc.rt_run = flush ? dz : acc.rt_run + dz;
        acc.rt_cur = flush ? bts[c + e] : acc.rt_cur;
      }
    }
    const uint32_t ah = pack_bf16(av[0], av[1]);
    const uint32_t zh = pack_bf16(zv[0], zv[1]);
    ahi[c >> 1] = ah;
    zhi[c >> 1] = zh;
    const float2 al = bf16_residual2(make_float2(av[0], av[1]), ah);
    const float2 zl = bf16_residual2(make_float2(zv[0], zv[1]), zh);
    alo[c >> 1] = pack_bf16(al.x, al.y);
    zlo[c >> 1] = pack_bf16(zl.x, zl.y);
  }
}

// All 16 query columns of this thread's key row are allowed and see one
// bias value rb (scaled by -log2 e): the position bucket is saturated and the
// time bucket is the same for every column.  A and dZ as packed BF16 hi/lo
// pairs; returns the sum of the 16 dZ (their one d_rab bucket each).
// kC and inv_n are the score constants, or 0 for a key row past the
// sequence, which then yields exact zeros.
__device__ __forceinline__ float grad_fast16(const AttnParams& p, const uint32_t (&sv)[16], const uint32_t (&dav)[16],
                                             float rb, float kC, float inv_n, uint32_t (&ahi)[8], uint32_t (&alo)[8],
                                             uint32_t (&zhi)[8], uint32_t (&zlo)[8]) {
  const float2 b2 = make_float2(rb, rb), one2 = make_float2(1.f, 1.f), inv_n2 = make_float2(inv_n, inv_n);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < 16; c += 2) {
    const float2 w2 = __ffma2_rn(p.kA2, make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), b2);
    const float2 d2 = __fadd2_rn(one2, make_float2(ex2_approx(w2.x), ex2_approx(w2.y)));
    const float2 sg2 = make_float2(rcp_approx(d2.x), rcp_approx(d2.y));
    const float2 z2 = make_float2(w2.x * p.kZ, w2.y * p.kZ);
    const float2 a2 = __fmul2_rn(make_float2(w2.x * kC, w2.y * kC), sg2);
    const float2 f2 = __ffma2_rn(z2, fsub2(one2, sg2), one2);  // 1 + z (1 - sg)
    const float2 h2 = __fmul2_rn(__fmul2_rn(make_float2(__uint_as_float(dav[c]), __uint_as_float(dav[c + 1])), sg2), f2);
    const float2 g2 = __fmul2_rn(h2, inv_n2);
    acc = __fadd2_rn(acc, g2);
    const uint32_t ah = pack_bf16(a2.x, a2.y), zh = pack_bf16(g2.x, g2.y);
    ahi[c >> 1] = ah;
    zhi[c >> 1] = zh;
    const float2 al = bf16_residual2(a2, ah), zl = bf16_residual2(g2, zh);
    alo[c >> 1] = pack_bf16(al.x, al.y);
    zlo[c >> 1] = pack_bf16(zl.x, zl.y);
  }
  return acc.x + acc.y;
}

// All 16 query columns of this thread's key row are allowed and their
// position bucket is saturated (P - 1), but the time bucket may change along
// the columns: the bias is the far position term plus each column's time
// term.  A and dZ as packed BF16 hi/lo pairs; returns the sum of the 16 dZ
// (the far position bucket's share) and carries the time buckets' run sums
// in acc.  32-bit relative times only.
__device__ __forceinline__ float grad_time16(const AttnParams& p, const uint32_t (&sv)[16], const uint32_t (&dav)[16],
                                             float rbp, const float* tpt, const int32_t* ts32, int32_t tj32,
                                             float kC, float inv_n, bool want_rt, float* drt, RabAcc& acc,
                                             uint32_t (&ahi)[8], uint32_t (&alo)[8], uint32_t (&zhi)[8],
                                             uint32_t (&zlo)[8]) {
  const float2 one2 = make_float2(1.f, 1.f), inv_n2 = make_float2(inv_n, inv_n);
  float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < 16; c += 2) {
    int d0 = ts32[c] - tj32, d1 = ts32[c + 1] - tj32;
    d0 = d0 < 0 ? -d0 : d0;
    d1 = d1 < 0 ? -d1 : d1;
    int bt0 = 32 - __clz(d0), bt1 = 32 - __clz(d1);
    bt0 = bt0 < p.Tb - 1 ? bt0 : p.Tb - 1;
    bt1 = bt1 < p.Tb - 1 ? bt1 : p.Tb - 1;
    const float2 b2 = make_float2(rbp + tpt[bt0], rbp + tpt[bt1]);
    const float2 w2 = __ffma2_rn(p.kA2, make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), b2);
    const float2 d2 = __fadd2_rn(one2, make_float2(ex2_approx(w2.x), ex2_approx(w2.y)));
    const float2 sg2 = make_float2(rcp_approx(d2.x), rcp_approx(d2.y));
    const float2 z2 = make_float2(w2.x * p.kZ, w2.y * p.kZ);
    const float2 a2 = __fmul2_rn(make_float2(w2.x * kC, w2.y * kC), sg2);
    const float2 f2 = __ffma2_rn(z2, fsub2(one2, sg2), one2);  // 1 + z (1 - sg)
    const float2 h2 = __fmul2_rn(__fmul2_rn(make_float2(__uint_as_float(dav[c]), __uint_as_float(dav[c + 1])), sg2), f2);
    const float2 g2 = __fmul2_rn(h2, inv_n2);
    sum2 = __fadd2_rn(sum2, g2);
    if (want_rt) {
      const int bts[2] = {bt0, bt1};
      const float gs[2] = {g2.x, g2.y};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool flush = bts[e] != acc.rt_cur;
        red_add(drt + acc.rt_cur, acc.rt_run, flush && acc.rt_cur >= 0);
        acc.rt_run = flush ? gs[e] : acc.rt_run + gs[e];
        acc.rt_cur = bts[e];
      }
    }
    const uint32_t ah = pack_bf16(a2.x, a2.y), zh = pack_bf16(g2.x, g2.y);
    ahi[c >> 1] = ah;
    zhi[c >> 1] = zh;
    const float2 al = bf16_residual2(a2, ah), zl = bf16_residual2(g2, zh);
    alo[c >> 1] = pack_bf16(al.x, al.y);
    zlo[c >> 1] = pack_bf16(zl.x, zl.y);
  }
  return sum2.x + sum2.y;
}

// Warps are spread over the four SM sub-partitions, each with a quarter of the
// register file: with 18 warps two sub-partitions hold five,
// and 5 x 32 threads x 96 registers = 15360 <= 16384.
template <typename TO>
__global__ void __maxnreg__(96)
hstu_bwd_tc_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmq,
                   const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const __grid_constant__ CUtensorMap tmdh, const __grid_constant__ CUtensorMap tmdl,
                   const __grid_constant__ CUtensorMap tmdq) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const uint32_t sK = base_u32 + Lay::K_OFF, sV = base_u32 + Lay::V_OFF;
  const uint32_t sQS = base_u32 + Lay::QS_OFF, sDZ = base_u32 + Lay::DZ_OFF;
  int64_t* ts64_s = reinterpret_cast<int64_t*>(base + Lay::TS64_OFF);
  int32_t* ts32_s = reinterpret_cast<int32_t*>(base + Lay::TS32_OFF);
  int32_t* cmm_s = reinterpret_cast<int32_t*>(base + Lay::CMM_OFF);
  int64_t* kts_s = reinterpret_cast<int64_t*>(base + Lay::KTS_OFF);
  ItemSlot* slot = reinterpret_cast<ItemSlot*>(base + Lay::SLOT_OFF);
  const uint32_t bar0 = base_u32 + Lay::BAR_OFF;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + Lay::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + Lay::MISC_OFF + 4);
  int* stage_wide = reinterpret_cast<int*>(base + Lay::MISC_OFF + 8);  // [kQStages]: query times need 64 bits
  const int H = p.H, P = p.P, Tb = p.Tb, PT = p.P + p.Tb;
  float* tab = reinterpret_cast<float*>(base + Lay::TAB_OFF);
  float* drab = p.drab_partial + (size_t)blockIdx.x * H * PT;  // this CTA's partial sums

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool has_rp = p.rab_pos != nullptr, has_rt = p.rab_time != nullptr && p.ts != nullptr;
  const bool want_rp = has_rp && p.d_rab_pos, want_rt = has_rt && p.d_rab_time;

  if (threadIdx.x == 0) {
    mbar_init(bar(BAR_KFULL), 1);
    mbar_init(bar(BAR_KEMPTY), 1);
    mbar_init(bar(BAR_VFULL), 1);
    mbar_init(bar(BAR_VEMPTY), 1);
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(bar(BAR_QFULL + s), 1);
      mbar_init(bar(BAR_QEMPTY + s), 1);
    }
    mbar_init(bar(BAR_SFULL), 1);
    mbar_init(bar(BAR_SEMPTY), kEpiWarps);
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
    tab[x] = -kLog2e * v;
    if (want_rp || want_rt) drab[x] = 0.f;  // this CTA's partial sums start from zero
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
    uint32_t item_it = 0, qt_it = 0, k_phases = 0, v_phases = 0;
    bool k_copy = false;                  // the last KFULL phase carries a copy
    static_assert(kQStages == 2, "per-stage counters hold two stages");
    Count2 armed;
    bool ok = true;
    // The next work item is claimed only once the current one's loads are all
    // issued (claiming earlier pairs items up statically and loses the
    // longest-first balance); its planner record is one 48-byte load.  The
    // first item of CTA b is item b (no atomic on the way in); later claims
    // count on from the grid size.
    bool first_claim = true;
    while (ok) {
      int idx = (int)blockIdx.x;
      if (!first_claim) {
        if (lane == 0) idx = (int)gridDim.x + atomicAdd(p.hdr_rw + WS_NEXT, 1);
        idx = __shfl_sync(0xffffffffu, idx, 0);
      }
      first_claim = false;
      const bool valid = idx < nitems;
      PlanItem it{};
      if (valid) it = p.items[idx / H];
      const int h = idx % H, k0 = it.blk * BK, n = it.n;
      const int64_t tbase = it.tbase, s0 = it.s0;
      // key-row timestamps of the item: loads issued before waiting
      int64_t kv[BK / 32];
#pragma unroll
      for (int x = 0; x < BK / 32; ++x) {
        const int row = k0 + lane + 32 * x;
        kv[x] = (valid && p.ts && row < n) ? p.ts[s0 + row] : tbase;
      }
      // V first: its buffer is free once the previous item's last dA^T is
      // computed, a tile before K's (read by the last dQ^T)
      if (valid) {
        if (lane == 0) ok = mbar_wait(bar(BAR_VEMPTY), (v_phases & 1) ^ 1, wd, 33);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(BAR_VFULL), 2 * Lay::KBOX);
          const int y = (int)(s0 + k0);
          for (int c = 0; c < 2; ++c)
            tma_load_2d(sV + c * Lay::KBOX, &tmv, bar(BAR_VFULL), h * D + c * 64, y);
        }
        ++v_phases;
      }
      // K, the key timestamps and the slot, once the previous item's last
      // dQ^T is done: after the item's first query tile is on its way (so
      // that tile's copy overlaps the previous item's end), or now for an
      // item without tiles and for the final no-work slot
      bool k_done = false;
      auto stage_k = [&]() -> bool {
        if (lane == 0) ok = mbar_wait(bar(BAR_KEMPTY), (item_it & 1) ^ 1, wd, 34);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return false;
        // the K copy starts before the key timestamps are staged; the phase
        // completes with the copy and the arrive below
        if (lane == 0 && valid) {
          mbar_expect_tx(bar(BAR_KFULL), 2 * Lay::KBOX);
          const int y = (int)(s0 + k0);
          for (int c = 0; c < 2; ++c)
            tma_load_2d(sK + c * Lay::KBOX, &tmk, bar(BAR_KFULL), h * D + c * 64, y);
        }
        bool kw = false;
#pragma unroll
        for (int x = 0; x < BK / 32; ++x) kw |= ts_wide(kv[x] - tbase);
        const bool item_wide = __any_sync(0xffffffffu, kw);
#pragma unroll
        for (int x = 0; x < BK / 32; ++x) kts_s[lane + 32 * x] = kv[x];
        if (lane == 0) {
          slot->s0 = s0; slot->tbase = tbase; slot->valid = valid ? 1 : 0;
          slot->h = h; slot->k0 = k0; slot->n = n; slot->c = it.c; slot->h_end = it.h_end;
          slot->wide = item_wide ? 1 : 0;
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(BAR_KFULL));  // without a copy the slot says: no more work
          k_phases += 1;
          k_copy = valid;
        }
        k_done = true;
        return true;
      };
      if (!valid) {
        stage_k();
        break;
      }
      const int nqt = (n + BQ - 1) / BQ;
      for (int qt = bwd_q_begin(k0, it.c, BQ); ok && qt < nqt; ++qt) {
        const int q0 = qt * BQ;
        if (tile_class(q0, k0, BQ, BK, n, it.c, it.h_end) == 0) continue;
        const int stage = qt_it % kQStages;
        // query timestamps: loads issued before waiting for the stage, stored after
        int64_t tv[BQ / 32];
#pragma unroll
        for (int x = 0; x < BQ / 32; ++x) {
          const int row = q0 + lane + 32 * x;
          tv[x] = (p.ts && row < n) ? p.ts[s0 + row] : tbase;
        }
        ok = mbar_wait(bar(BAR_QEMPTY + stage), ((qt_it / kQStages) & 1) ^ 1, wd, 22);
        if (!ok) break;
        const uint32_t full = bar(BAR_QFULL + stage);
        if (lane == 0) {   // the copies start before the query timestamps arrive
          mbar_expect_tx(full, Lay::QSTAGE);
          const uint32_t dst = sQS + stage * Lay::QSTAGE;
          const int y = (int)(s0 + q0);
          for (int c = 0; c < 2; ++c) {
            tma_load_2d(dst + c * Lay::QBOX, &tmq, full, h * D + c * 64, y);
            tma_load_2d(dst + Lay::Q_BYTES + c * Lay::QBOX, &tmdh, full, h * D + c * 64, y);
            tma_load_2d(dst + 2 * Lay::Q_BYTES + c * Lay::QBOX, &tmdl, full, h * D + c * 64, y);
          }
          // (no L2 prefetch of later tiles: Q was read by the forward and dO
          // written just before, and prefetch requests only compete with the
          // copies: 202.7 -> 198.9 us without them)
        }
        bool qw = false;
#pragma unroll
        for (int x = 0; x < BQ / 32; ++x) {
          const int32_t r = (int32_t)(tv[x] - tbase);
          ts64_s[stage * BQ + lane + 32 * x] = tv[x];
          ts32_s[stage * BQ + lane + 32 * x] = r;
          qw |= ts_wide(tv[x] - tbase);
          // min and max relative time of each 16-query chunk (lanes 0-15
          // and 16-31 of this 32-query half), for the epilogue's test for a
          // time bucket that is the same across a chunk
          int mn = r, mx = r;
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) {
            mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          }
          if ((lane & 15) == 0) {
            cmm_s[stage * 8 + (2 * x + (lane >> 4)) * 2] = mn;
            cmm_s[stage * 8 + (2 * x + (lane >> 4)) * 2 + 1] = mx;
          }
        }
        qw = __any_sync(0xffffffffu, qw);
        if (lane == 0) stage_wide[stage] = qw ? 1 : 0;
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(full);
          armed.add(stage, 1);
        }
        ++qt_it;
        if (!k_done && !stage_k()) break;
      }
      if (ok && !k_done) ok = stage_k();   // an item without tiles (none is planned)
      ++item_it;
    }
    if (lane == 0) {
      for (int s = 0; s < kQStages; ++s)
        if (armed[s]) drain_wait(bar(BAR_QFULL + s), (armed[s] - 1) & 1);
      if (k_copy) drain_wait(bar(BAR_KFULL), (k_phases - 1) & 1);
      if (v_phases) drain_wait(bar(BAR_VFULL), (v_phases - 1) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    {   // the whole warp runs the issue loop (its values stay warp-uniform); one elected lane issues
      constexpr uint32_t IDESC_S = idesc_bf16(BK, BQ, false, false);    // M=128 keys, N=64 queries
      constexpr uint32_t IDESC_DVK = idesc_bf16(BK, D, false, true);    // A K-major, B MN-major
      constexpr uint32_t IDESC_DQ = idesc_bf16(D, BQ, true, true);      // A = K^T, B = dZ^T, MN-major
      uint32_t item_it = 0, qt_it = 0;
      bool ok = true;
      // Shared-memory descriptors, built once; every MMA below moves a start
      // address by a constant (one add on the low descriptor word).
      //  K-major operands (rows of 128 bytes): K, V, and per stage Q, dO_hi, dO_lo
      //  MN-major operands: K^T (dQ), dO_hi/lo (dV), Q (dK B), dZ^T (dQ B)
      const SDesc k_km = sdesc_w(sK, 16, 1024), v_km = sdesc_w(sV, 16, 1024);
      const SDesc q_km = sdesc_w(sQS, 16, 1024);
      const SDesc k_mn = sdesc_w(sK, Lay::KBOX, 1024);
      const SDesc q_mn = sdesc_w(sQS, Lay::QBOX, 1024);
      const SDesc zh_mn = sdesc_w(sDZ, Lay::DZ_BYTES, 1024), zl_mn = sdesc_w(sDZ + Lay::DZ_BYTES, Lay::DZ_BYTES, 1024);
      const SDesc zh_km = sdesc_w(sDZ, 16, 1024), zl_km = sdesc_w(sDZ + Lay::DZ_BYTES, 16, 1024);
      // dV += A^T dO (3 products: A_hi dO_hi, A_lo dO_hi, A_hi dO_lo) and
      // dK += dZ^T Q (2) of query tile g, which read the Q stage st; then
      // the stage is released, and dQ^T = K^T dZ^T (2) follows.  DQFULL
      // comes after all of them (A in TMEM and the dZ^T staging are free
      // again); on an item's last tile K/V is released after dQ^T.
      auto issue_grad = [&](uint32_t g, uint32_t st, bool first, bool last) -> bool {
        if (!mbar_wait(bar(BAR_PREADY), g & 1, wd, 26)) return false;
        if (first && !mbar_wait(bar(BAR_DKVEMPTY), (item_it & 1) ^ 1, wd, 24)) return false;
        fence_after_sync();
        const uint32_t so = st * Lay::QSTAGE;
        const SDesc q_s = q_mn + so, dh_s = q_mn + (so + Lay::Q_BYTES), dl_s = q_mn + (so + 2 * Lay::Q_BYTES);
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {   // K = 64 queries: 4 steps of 16
          const uint32_t a_hi = tmem + A_COL + 16u * kk;
          const uint32_t acc0 = (first && kk == 0) ? 0u : 1u;
          mma_ts_e(tmem + DV_COL, a_hi, dh_s + kk * 2048, IDESC_DVK, acc0);
          mma_ts_e(tmem + DV_COL, a_hi + 8, dh_s + kk * 2048, IDESC_DVK, 1u);
          mma_ts_e(tmem + DV_COL, a_hi, dl_s + kk * 2048, IDESC_DVK, 1u);
          mma_ss_e(tmem + DK_COL, zh_km + kk * 32, q_s + kk * 2048, IDESC_DVK, acc0);
          mma_ss_e(tmem + DK_COL, zl_km + kk * 32, q_s + kk * 2048, IDESC_DVK, 1u);
        }
        mma_commit_e(bar(BAR_QEMPTY + st));   // the Q / dO stage is read by no later MMA
        if (!mbar_wait(bar(BAR_DQEMPTY), (g & 1) ^ 1, wd, 27)) return false;
        fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {   // K = 128 keys: 8 steps of 16
          mma_ss_e(tmem + DQ_COL, k_mn + kk * 2048, zh_mn + kk * 2048, IDESC_DQ, kk > 0 ? 1u : 0u);
          mma_ss_e(tmem + DQ_COL, k_mn + kk * 2048, zl_mn + kk * 2048, IDESC_DQ, 1u);
        }
        if (last) mma_commit_e(bar(BAR_KEMPTY));   // K of this item is read by no later MMA
        mma_commit_e(bar(BAR_DQFULL));
        return true;
      };
      while (ok) {
        ok = mbar_wait(bar(BAR_KFULL), item_it & 1, wd, 23);
        if (!ok) break;
        fence_after_sync();
        const ItemSlot sl = *slot;
        if (!sl.valid) break;
        bool have_prev = false, first = true, v_ready = false;
        uint32_t prev = 0, prev_st = 0;
        const int nqt = (sl.n + BQ - 1) / BQ;
        const int qb0 = bwd_q_begin(sl.k0, sl.c, BQ);
        int q_last = nqt - 1;   // the item's last query tile the mask keeps (V is released after its dA^T)
        while (q_last >= qb0 && tile_class(q_last * BQ, sl.k0, BQ, BK, sl.n, sl.c, sl.h_end) == 0) --q_last;
        for (int qt = qb0; ok && qt < nqt; ++qt) {
          if (tile_class(qt * BQ, sl.k0, BQ, BK, sl.n, sl.c, sl.h_end) == 0) continue;
          const uint32_t stage = qt_it % kQStages;
          ok = mbar_wait(bar(BAR_QFULL + stage), (qt_it / kQStages) & 1, wd, 25) &&
               mbar_wait(bar(BAR_SEMPTY), (qt_it & 1) ^ 1, wd, 28);
          if (!ok) break;
          fence_after_sync();
          const uint32_t so = stage * Lay::QSTAGE;
          const SDesc q_s = q_km + so, dh_s = q_km + (so + Lay::Q_BYTES), dl_s = q_km + (so + 2 * Lay::Q_BYTES);
          // S^T = K Q^T ; dA^T = V dO_hi^T + V dO_lo^T
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = (kk >> 2) * Lay::KBOX + (kk & 3) * 32;
            const uint32_t qb = (kk >> 2) * Lay::QBOX + (kk & 3) * 32;
            mma_ss_e(tmem + S_COL, k_km + ka, q_s + qb, IDESC_S, kk > 0 ? 1u : 0u);
          }
          if (!v_ready) {
            ok = mbar_wait(bar(BAR_VFULL), item_it & 1, wd, 35);
            if (!ok) break;
            fence_after_sync();
            v_ready = true;
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = (kk >> 2) * Lay::KBOX + (kk & 3) * 32;
            const uint32_t qb = (kk >> 2) * Lay::QBOX + (kk & 3) * 32;
            mma_ss_e(tmem + DA_COL, v_km + ka, dh_s + qb, IDESC_S, kk > 0 ? 1u : 0u);
            mma_ss_e(tmem + DA_COL, v_km + ka, dl_s + qb, IDESC_S, 1u);
          }
          mma_commit_e(bar(BAR_SFULL));
          if (qt == q_last) mma_commit_e(bar(BAR_VEMPTY));   // V of this item is read by no later MMA
          if (have_prev) {
            ok = issue_grad(prev, prev_st, first, false);
            first = false;
          }
          have_prev = true;
          prev = qt_it;
          prev_st = stage;
          ++qt_it;
        }
        if (ok && have_prev) ok = issue_grad(prev, prev_st, first, true);
        if (!ok) break;
        if (!have_prev) {   // an item without tiles (none is planned): release its buffers as they are
          ok = mbar_wait(bar(BAR_VFULL), item_it & 1, wd, 35);
          if (!ok) break;
          mma_commit_e(bar(BAR_VEMPTY));
          mma_commit_e(bar(BAR_KEMPTY));
        }
        mma_commit_e(bar(BAR_DKVFULL));
        ++item_it;
      }
      mma_commit_e(bar(BAR_DRAIN));
      drain_wait(bar(BAR_DRAIN), 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3, hq = warp >> 2;
    const int lrow = wq * 32 + lane;                  // TMEM lane: key row (S^T, dV, dK) or d (dQ^T)
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    uint32_t item_it = 0, qt_it = 0;
    bool ok = true;
    KeyCtx kc;
    int n_seq = 0;  // tokens of the current item's sequence
    kc.want_rp = want_rp;
    kc.want_rt = want_rt;
    // the dQ^T of the previous query tile, drained in the middle of the next
    // dQ^T's columns are queries and its TMEM lanes dims: this warp holds dims
    // [32 wq, 32 wq + 32) of the 16 queries [qb0 + 16 hq, + 16).  They go
    // through the warp's staging block, 8 queries at a time, into one bulk
    // reduce-add each (tensor map [T][H][D] FP32).  Queries past the
    // sequence carry exact zeros (their dZ is masked), so the neighbouring
    // sequence's rows they land on are unchanged; rows past T are clipped.
    uint8_t* dqs = base + Lay::DQS_OFF + warp * Lay::DQS_WARP;
    const uint32_t dqs_u32 = base_u32 + Lay::DQS_OFF + warp * Lay::DQS_WARP;
    // The previous tile's gradient MMAs are complete once its dQ^T is: the A
    // buffer and the dZ^T staging are free again.
    auto wait_dq = [&](uint32_t g) -> bool {
      if (!mbar_wait(bar(BAR_DQFULL), g & 1, wd, 30)) return false;
      fence_after_sync();
      return true;
    };
    // dQ^T of tile g out of TMEM (its buffer released to the next dQ^T MMA)
    // and into dq; DQFULL of g has been seen
    auto drain_dq = [&](int qb0, int64_t s0, int hh) {
      uint32_t qv[16];
      tmem_ld16(lane_base + DQ_COL + hq * 16, qv);
      tmem_wait_ld();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_DQEMPTY));
      const float alpha = p.alpha;
      const int tok0 = (int)(s0 + qb0 + hq * 16);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (lane == 0) bulk_wait_read<0>();   // the block's previous reduce has read it
        __syncwarp();
        float* blk = reinterpret_cast<float*>(dqs) + lane;
#pragma unroll
        for (int c = 0; c < 8; ++c) blk[c * 32] = alpha * __uint_as_float(qv[8 * r + c]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (tok0 + 8 * r < p.T) tma_reduce_add_3d(&tmdq, dqs_u32, wq * 32, hh, tok0 + 8 * r);
          bulk_commit();
        }
      }
    };
    while (ok) {
      ok = mbar_wait(bar(BAR_KFULL), item_it & 1, wd, 32);
      if (!ok) break;
      // the slot stays until this item's last tile is handed over; keep what
      // the dV / dK write-out needs in registers
      const ItemSlot& sl = *slot;
      if (!sl.valid) break;
      const int64_t s0 = sl.s0;
      const int hh = sl.h, k0 = sl.k0;
      const bool item_wide = sl.wide != 0;
      n_seq = sl.n;
      const int cx = sl.c;
      kc.h_end = sl.h_end;
      kc.j = k0 + lrow;
      const bool j_ok = kc.j < n_seq;
      kc.pos_j = kc.j < kc.h_end ? kc.j : kc.h_end;
      // queries that see this key: a context key is seen by every row, a
      // history key by the rows at or after it, a candidate key by itself only
      kc.lo = !j_ok ? 1 : (kc.j >= kc.h_end ? kc.j : (kc.j < cx ? 0 : kc.j));
      kc.hi = !j_ok ? 0 : (kc.j >= kc.h_end ? kc.j : n_seq - 1);
      kc.tj64 = kts_s[lrow];
      kc.tj32 = (int32_t)(kc.tj64 - sl.tbase);
      kc.tp = tab + hh * PT;
      kc.drp = drab + hh * PT;
      RabAcc racc;
      racc.rp_far = racc.rt_run = 0.f;
      racc.rt_cur = -1;
      bool pend = false;    // a dQ^T of this item waits to be drained
      int pend_q0 = 0;
      const int nqt = (n_seq + BQ - 1) / BQ;
      for (int qt = bwd_q_begin(k0, cx, BQ); ok && qt < nqt; ++qt) {
        const int q0 = qt * BQ;
        const int cls = tile_class(q0, k0, BQ, BK, n_seq, cx, kc.h_end);
        if (cls == 0) continue;
        const uint32_t stage = qt_it % kQStages;
        ok = mbar_wait(bar(BAR_QFULL + stage), (qt_it / kQStages) & 1, wd, 28) &&
             mbar_wait(bar(BAR_SFULL), qt_it & 1, wd, 29);
        if (!ok) break;
        fence_after_sync();
        uint32_t svq[16], daq[16];
        tmem_ld16(lane_base + S_COL + hq * 16, svq);
        tmem_ld16(lane_base + DA_COL + hq * 16, daq);
        tmem_wait_ld();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_SEMPTY));   // S^T, dA^T may be overwritten now
        const int c0 = hq * 16;   // first query column of this thread within the tile
        const int ib = q0 + c0;
        const bool narrow = !item_wide && !stage_wide[stage];
        // Constant-bias test for this thread's 16 columns: all allowed, the
        // position bucket saturated for all (checked at both ends, positions
        // grow with the column), and the time bucket the same for all (the
        // chunk's times all on one side of t_j, and the bucket of the
        // nearest and of the farthest gap equal: buckets grow with the gap).
        bool fast = narrow && ib >= kc.lo && ib + 15 <= kc.hi;
        int btc = 0;
        if (fast && has_rp) {
          const int pa = ib < kc.h_end ? ib : kc.h_end;
          const int pb = ib + 15 < kc.h_end ? ib + 15 : kc.h_end;
          fast = pa - kc.pos_j >= P - 1 || kc.pos_j - pb >= P - 1;
        }
        // all allowed and the position bucket saturated: only the time bucket may vary
        const bool far_all = fast;
        if (fast && has_rt) {
          const int32_t cmin = cmm_s[stage * 8 + hq * 2], cmax = cmm_s[stage * 8 + hq * 2 + 1];
          int32_t dlo, dhi;
          if (kc.tj32 <= cmin) {
            dlo = cmin - kc.tj32;
            dhi = cmax - kc.tj32;
          } else if (kc.tj32 >= cmax) {
            dlo = kc.tj32 - cmax;
            dhi = kc.tj32 - cmin;
          } else {
            dlo = 0;
            dhi = 1;   // gaps of both signs: buckets differ
            fast = false;
          }
          const int blo = min(32 - __clz(dlo), Tb - 1), bhi = min(32 - __clz(dhi), Tb - 1);
          fast = fast && blo == bhi;
          btc = blo;
        }
        // a key row past the sequence takes the same path with zero
        // constants: its A and dZ (which the dQ products read) are exact zeros
        // (the warp takes the constant path when all its rows may, else the
        // far path with per-column time buckets when all its rows are far and
        // fully allowed, else the general path)
        const bool all_const = __all_sync(0xffffffffu, fast || !j_ok);
        if (all_const || (has_rt && narrow && __all_sync(0xffffffffu, far_all || !j_ok))) {
          uint32_t ahi[8], alo[8], zhi[8], zlo[8];
          float sum;
          if (all_const) {
            const float rb = kc.tp[P - 1] + kc.tp[P + btc];
            sum = grad_fast16(p, svq, daq, rb, j_ok ? p.kC : 0.f, j_ok ? p.inv_n : 0.f, ahi, alo, zhi, zlo);
            if (want_rt) {
              if (btc == racc.rt_cur) {
                racc.rt_run += sum;
              } else {
                red_add(kc.drp + P + racc.rt_cur, racc.rt_run, racc.rt_cur >= 0);
                racc.rt_cur = btc;
                racc.rt_run = sum;
              }
            }
          } else {
            sum = grad_time16(p, svq, daq, kc.tp[P - 1], kc.tp + P, ts32_s + stage * BQ + c0, kc.tj32,
                              j_ok ? p.kC : 0.f, j_ok ? p.inv_n : 0.f, want_rt, kc.drp + P, racc, ahi, alo, zhi, zlo);
          }
          if (want_rp) racc.rp_far += sum;
          if (pend) {
            ok = wait_dq(qt_it - 1);
            if (!ok) break;
          }
          tmem_st8(lane_base + A_COL + hq * 16, ahi);
          tmem_st8(lane_base + A_COL + hq * 16 + 8, alo);
          const uint32_t rowh = sDZ + (uint32_t)lrow * 128u, rowl = rowh + Lay::DZ_BYTES;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint32_t chunk = (uint32_t)((hq * 2 + half) ^ (lrow & 7));
            st_shared_v4(rowh + chunk * 16, zhi[4 * half], zhi[4 * half + 1], zhi[4 * half + 2], zhi[4 * half + 3]);
            st_shared_v4(rowl + chunk * 16, zlo[4 * half], zlo[4 * half + 1], zlo[4 * half + 2], zlo[4 * half + 3]);
          }
        } else {
          // computed and written out in two halves of 8 query columns
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int hc0 = c0 + half * 8;    // first query column of this half within the tile
            uint32_t sv[8], dav[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              sv[e] = svq[half * 8 + e];
              dav[e] = daq[half * 8 + e];
            }
            const int hib = q0 + hc0;
            const int32_t* t32 = ts32_s + stage * BQ + hc0;
            const int64_t* t64 = ts64_s + stage * BQ + hc0;
            uint32_t ahi[4], alo[4], zhi[4], zlo[4];
            if (narrow) grad_cols<8, false>(p, sv, dav, ahi, alo, zhi, zlo, kc, hib, t32, t64, racc);
            else grad_cols<8, true>(p, sv, dav, ahi, alo, zhi, zlo, kc, hib, t32, t64, racc);
            if (half == 0 && pend) {
              ok = wait_dq(qt_it - 1);
              if (!ok) break;
            }
            // A into its TMEM buffer.  Quarter hq owns columns [16 hq, 16 hq + 16):
            // hi pairs in the first 8, lo pairs in the last 8; this half's 8
            // queries are 4 packed columns of each.
            tmem_st4(lane_base + A_COL + hq * 16 + half * 4, ahi);
            tmem_st4(lane_base + A_COL + hq * 16 + 8 + half * 4, alo);
            // dZ^T into SMEM (row = key, 64 queries = 128 B, 128-byte swizzle) for the dK and dQ MMAs
            const uint32_t rowh = sDZ + (uint32_t)lrow * 128u, rowl = rowh + Lay::DZ_BYTES;
            const uint32_t chunk = (uint32_t)((hq * 2 + half) ^ (lrow & 7));
            st_shared_v4(rowh + chunk * 16, zhi[0], zhi[1], zhi[2], zhi[3]);
            st_shared_v4(rowl + chunk * 16, zlo[0], zlo[1], zlo[2], zlo[3]);
          }
        }
        if (!ok) break;
        fence_async_smem();
        tmem_wait_st();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_PREADY));
        // the previous tile's dQ^T goes out while this tile's gradient MMAs run
        if (pend) drain_dq(pend_q0, s0, hh);
        pend = true;
        pend_q0 = q0;
        ++qt_it;
      }
      if (!ok) break;
      if (pend) {
        ok = wait_dq(qt_it - 1);
        if (!ok) break;
        drain_dq(pend_q0, s0, hh);
      }
      // the item's remaining d_rab partial sums
      red_add(kc.drp + P + racc.rt_cur, racc.rt_run, want_rt && racc.rt_cur >= 0);
      if (want_rp) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) racc.rp_far += __shfl_xor_sync(0xffffffffu, racc.rp_far, o);
        red_add(kc.drp + (P - 1), racc.rp_far, lane == 0 && racc.rp_far != 0.f);
      }
      // dV, dK out: lane = key row, column quarter hq of d (32 columns each)
      ok = mbar_wait(bar(BAR_DKVFULL), item_it & 1, wd, 31);
      if (!ok) break;
      fence_after_sync();
      uint32_t vv[32], kv[32];
      tmem_ld32(lane_base + DV_COL + hq * 32, vv);
      tmem_ld32(lane_base + DK_COL + hq * 32, kv);
      tmem_wait_ld();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_DKVEMPTY));
      if (j_ok) {
        const size_t g = ((size_t)(s0 + kc.j) * H + hh) * D + hq * 32;
        TO* dvp = static_cast<TO*>(p.dv) + g;
        TO* dkp = static_cast<TO*>(p.dk) + g;
        const float alpha = p.alpha;
        if constexpr (sizeof(TO) == 4) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            reinterpret_cast<float4*>(dvp)[e] =
                make_float4(__uint_as_float(vv[4 * e]), __uint_as_float(vv[4 * e + 1]),
                            __uint_as_float(vv[4 * e + 2]), __uint_as_float(vv[4 * e + 3]));
            reinterpret_cast<float4*>(dkp)[e] =
                make_float4(alpha * __uint_as_float(kv[4 * e]), alpha * __uint_as_float(kv[4 * e + 1]),
                            alpha * __uint_as_float(kv[4 * e + 2]), alpha * __uint_as_float(kv[4 * e + 3]));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            reinterpret_cast<uint4*>(dvp)[e] =
                make_uint4(pack_bf16(__uint_as_float(vv[8 * e]), __uint_as_float(vv[8 * e + 1])),
                           pack_bf16(__uint_as_float(vv[8 * e + 2]), __uint_as_float(vv[8 * e + 3])),
                           pack_bf16(__uint_as_float(vv[8 * e + 4]), __uint_as_float(vv[8 * e + 5])),
                           pack_bf16(__uint_as_float(vv[8 * e + 6]), __uint_as_float(vv[8 * e + 7])));
            reinterpret_cast<uint4*>(dkp)[e] =
                make_uint4(pack_bf16(alpha * __uint_as_float(kv[8 * e]), alpha * __uint_as_float(kv[8 * e + 1])),
                           pack_bf16(alpha * __uint_as_float(kv[8 * e + 2]), alpha * __uint_as_float(kv[8 * e + 3])),
                           pack_bf16(alpha * __uint_as_float(kv[8 * e + 4]), alpha * __uint_as_float(kv[8 * e + 5])),
                           pack_bf16(alpha * __uint_as_float(kv[8 * e + 6]), alpha * __uint_as_float(kv[8 * e + 7])));
          }
        }
      }
      ++item_it;
    }
  }

  if (warp < kEpiWarps && lane == 0) bulk_wait_all();   // the dQ reduce-adds are complete
  __threadfence();   // this CTA's partial-sum reductions are performed before they are read back
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  // d_rab += this CTA's partial sums (the outputs were zeroed before the launch)
  if (want_rp || want_rt) {
    for (int x = threadIdx.x; x < H * PT; x += kThreads) {
      const float v = __ldcg(drab + x);
      const int h = x / PT, e = x % PT;
      if (e < P) red_add(p.d_rab_pos + h * P + e, v, want_rp && v != 0.f);
      else red_add(p.d_rab_time + h * Tb + (e - P), v, want_rt && v != 0.f);
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
  const void* fn = reinterpret_cast<const void*>(hstu_bwd_tc_kernel<TO>);
  cudaError_t e = cudaFuncSetAttribute(hstu_bwd_tc_kernel<TO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) {
    set_launch_detail(e, "hstu_bwd_tc_kernel (smem attribute)", fn, kThreads, smem);
    return e;
  }
  const int64_t max_items = ((p.T + BK - 1) / BK + p.B) * (int64_t)p.H;
  int grid = (int)(max_items < p.num_sms ? max_items : p.num_sms);
  if (grid > kDrabMaxCtas) grid = kDrabMaxCtas;  // one d_rab partial row per CTA
  // dq accumulator [T][H][D] FP32, 32-dim x 8-query reduce-add blocks
  CUtensorMap mdq;
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)p.H, (uint64_t)p.T};
    const uint64_t strides[2] = {(uint64_t)D * 4, (uint64_t)p.H * D * 4};
    const uint32_t box[3] = {32, 1, 8};
    if (!make_tmap_tile(&mdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.dq_acc, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  }
  hstu_bwd_tc_kernel<TO><<<grid, kThreads, smem, st>>>(p, mq, mk, mv, mdh, mdl, mdq);
  e = cudaGetLastError();
  if (e != cudaSuccess) set_launch_detail(e, "hstu_bwd_tc_kernel", fn, kThreads, smem);
  return e;
}

}  // namespace

bool tc_bwd_supported(int dtype, int dqk, int dv) { return dtype == HSTU_BF16 && dqk == D && dv == D; }

size_t tc_bwd_smem_bytes(int H, int P, int Tb) {
  return Lay::TAB_OFF + sizeof(float) * (size_t)H * (P + Tb) + 1024;
}

cudaError_t launch_tc_bwd(const AttnParams& p, cudaStream_t st) {
  return p.out_dtype == HSTU_FP32 ? launch_t<float>(p, st) : launch_t<__nv_bfloat16>(p, st);
}

}  // namespace hstu
