// Tensor-core forward of HSTU jagged attention for sm_103a (BF16 inputs,
// d in {64, 128}): tcgen05 MMA with FP32 accumulators in TMEM, operands
// staged by TMA, a fused score epilogue, persistent CTAs.
//
// Per work item (sequence b, head h, 128-row query block), for every key
// block the compound mask keeps:
//   S   = Q K^T                      tcgen05.mma, SMEM x SMEM -> TMEM (FP32)
//   P   = mask ? SiLU(alpha S + rab_pos[bp] + rab_time[bt]) / N : 0
//                                    epilogue warps, TMEM -> regs -> TMEM
//   O  += P V                        tcgen05.mma, TMEM x SMEM -> TMEM
// (HSTU spatial aggregation, ai6s.net survey section 2.1.2 eq. (2); tiling,
// Cube/Vector overlap and mask skipping follow the ideas of the Ascend HSTU
// fused operator on the wmrh.cn RecSDK page, re-planned for TMEM/TMA.)
//
// P is written back as two BF16 halves, P = P_hi + P_lo, and O accumulates
// P_hi V + P_lo V: one BF16 rounding of P alone costs ~1.5% of the output
// RMS on heavy-tailed batches, the pair keeps ~16 bits.
//
// Score arithmetic: with w = -log2(e) z, SiLU(z) / N = (w * c) / (1 + 2^w),
// c = -1 / (log2(e) N); the bias tables are stored pre-multiplied by
// -log2(e) so one FFMA gives w.
//
// Roles (640 threads): warps 0-15 epilogue (warp w reads TMEM lanes
// 32*(w%4).. and the 32-column quarter w/4 of each tile), warp 16 TMA
// producer of Q and K (plus the key timestamps), warp 17 S = Q K^T issuer
// and TMEM owner, warp 18 TMA producer of V, warp 19 O += P V issuer.  K
// and V have rings of their own: a K stage is free once its S = Q K^T is
// done, so the next tiles' K loads and S products never wait for the P V of
// the tile before, which is what a shared K/V stage made them do.
// TMEM columns: S/P buffers at 0 and 128, O buffers at 256 and 256 + d.
//
// Scheduling: the planner lists the query blocks longest-first; the producer
// of each CTA takes its block index as its first work item and every later
// one from a global counter (greedy LPT, dynamic), and passes it to the other roles through a shared-memory slot
// that travels with one of two Q buffers, so the next item's Q and first K/V
// are loading while the current item's last tiles are computed.
#include "hstu_internal.h"
#include "tc_ptx.cuh"

namespace hstu {

namespace {

using namespace tc;

constexpr int BM = kTcTile, BN = kTcTile;
constexpr int kEpiWarps = 16;
constexpr int kProducerWarp = 16, kMmaWarp = 17, kVProducerWarp = 18, kPvWarp = 19;
constexpr int kThreads = 20 * 32;
constexpr int kStages = 2;      // K ring and V ring, each
constexpr int kTsSlots = 4;     // key-timestamp slots, released by the epilogue
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSColStride = 128;  // S/P buffer sb starts at column sb * 128
constexpr float kLog2e = 1.4426950408889634f;

constexpr int kQBufs = 2;

enum : int { BAR_QFULL = 0, BAR_QEMPTY = BAR_QFULL + kQBufs, BAR_KFULL = BAR_QEMPTY + kQBufs,
             BAR_KEMPTY = BAR_KFULL + kStages, BAR_VFULL = BAR_KEMPTY + kStages, BAR_VEMPTY = BAR_VFULL + kStages,
             BAR_TSFULL = BAR_VEMPTY + kStages, BAR_TSEMPTY = BAR_TSFULL + kTsSlots,
             BAR_SFULL = BAR_TSEMPTY + kTsSlots, BAR_PREADY = BAR_SFULL + 2, BAR_OFULL = BAR_PREADY + 2,
             BAR_OEMPTY = BAR_OFULL + 2, BAR_SFREE = BAR_OEMPTY + 2, BAR_DRAIN = BAR_SFREE + 2, BAR_COUNT };

// A work item as the producer hands it to the other roles (one per Q buffer).
struct __align__(16) ItemSlot {
  int64_t s0;     // first token of the sequence
  int64_t tbase;  // timestamp of that token (0 without timestamps)
  int valid;      // 0: no more work
  int h, q0, n, c, h_end;
  int wide;       // some query time of the item is 2^30 s or more from tbase
  int L;          // delta forward: cached tokens of the sequence
  int64_t cs0;    // delta forward: first cached token of the sequence
  int64_t pad;
};

template <int D>
struct Layout {
  static constexpr int NCH = D / 64;            // 128-byte column chunks per row
  static constexpr int BOX = 128 * 128;         // one TMA box: 128 rows x 64 bf16 = 16 KB
  static constexpr int Q_BYTES = NCH * BOX;
  static constexpr int Q_OFF = 0;               // kQBufs Q buffers
  static constexpr int K_BYTES = NCH * BOX;     // one K or V stage
  static constexpr int K_OFF = Q_OFF + kQBufs * Q_BYTES;        // K ring
  static constexpr int V_OFF = K_OFF + kStages * K_BYTES;       // V ring
  static constexpr int TS64_OFF = V_OFF + kStages * K_BYTES;    // int64 [kTsSlots][BN] key times, absolute
  static constexpr int TS32_OFF = TS64_OFF + kTsSlots * BN * 8; // int32 [kTsSlots][BN] relative
  static constexpr int CMM_OFF = TS32_OFF + kTsSlots * BN * 4;  // int32 [kTsSlots][4 chunks][min, max] relative
  static constexpr int QTS_OFF = CMM_OFF + kTsSlots * 8 * 4;    // int64 [kQBufs][BM] query times
  static constexpr int SLOT_OFF = QTS_OFF + kQBufs * BM * 8;    // ItemSlot [kQBufs]
  static constexpr int BAR_OFF = SLOT_OFF + kQBufs * (int)sizeof(ItemSlot);
  static constexpr int MISC_OFF = BAR_OFF + BAR_COUNT * 8;      // tmem slot, abort flag, per-slot wide flags
  static constexpr int TAB_OFF = MISC_OFF + 32;                 // float [H][P + kTabTime]
  static constexpr uint32_t O_COL0 = 256, O_COL1 = 256 + D;
};

// Time-bias slots of a head's table after its P position entries, indexed by
// the count of leading zeros of the gap (bit length = width - clz), each
// holding bucket min(bit length, Tb - 1):
//   [0, 65)   64-bit gaps, clz in [0, 64]
//   [65, 98)  32-bit gaps, clz in [0, 32]
//   [98, 131) 32-bit gaps plus position bucket P - 1 (blocks far from the diagonal)
constexpr int kTabWide = 0, kTabNarrow = 65, kTabFar = 98, kTabTime = 131;

// waits for a phase, ignoring the abort flag (used to drain async copies)
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > 200000000ull) break;
  }
}

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

// Per-thread row context of the epilogue (one query row i of the item).
struct RowCtx {
  int i, h_end, pos_i;
  bool row_ok;
  // the row's allowed keys under the compound mask: j <= hi, and j == dg
  // (a candidate's own key); hi = -1, dg = -1 for rows past the sequence
  int hi, dg;
  int32_t ti32;      // timestamp relative to the sequence's first token
  int64_t ti64;      // absolute timestamp
  // bias tables of the head, pre-scaled by -log2(e): position [0, P), then the
  // kTabTime time slots
  const float* tp;
};

// Scores of 32 consecutive key columns jb.. of one row -> P_hi, P_lo packed
// pairs.  POS 1: every column is a history/context token at or before the
// row (position gap = pos_i - j >= 0); POS 2: besides, every gap of the
// warp's 32 x 32 block is at least P - 1 (one position bucket, folded into
// the far time table); POS 0: the general gap |pos_i - min(j, h_end)|.
// WIDE: 64-bit timestamp gaps.  PARTIAL: evaluate the mask per element.
// MODE (delta forward, candidate rows only): 1 = cached keys j < L (position
// gap L - j, rc.h_end = L), 2 = the candidates' own keys, where only the
// diagonal is allowed (gap 0).
template <int POS, bool WIDE, bool PARTIAL, int MODE = 0>
__device__ __forceinline__ void score32(const AttnParams& p, const uint32_t (&sv)[32], uint32_t (&hi)[16],
                                        uint32_t (&lo)[16], const RowCtx& rc, int jb, const int32_t* ts32,
                                        const int64_t* ts64) {
  // Paired FP32 arithmetic (fma/mul/add on float2, one instruction for two
  // elements); each lane of a pair rounds exactly like the scalar operation.
  const float2 kA2 = make_float2(p.kA, p.kA), kCi2 = make_float2(p.kCi, p.kCi);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float bias[16];
    int bps[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int cc = half * 16 + c;
      int bp = 0;
      if (MODE == 0 && POS == 2) {
        // no position term of its own
      } else if (MODE == 1) {
        int dp = rc.pos_i - (jb + cc);
        dp = dp < 0 ? 0 : dp;  // columns past the cache are masked below
        bp = dp < p.P - 1 ? dp : p.P - 1;
      } else if (MODE == 2) {
        bp = 0;
      } else if (POS == 1) {
        const int dp = rc.pos_i - (jb + cc);
        bp = dp < p.P - 1 ? dp : p.P - 1;
      } else {
        const int j = jb + cc;
        const int pj = j < rc.h_end ? j : rc.h_end;
        int dp = rc.pos_i - pj;
        dp = dp < 0 ? -dp : dp;
        bp = dp < p.P - 1 ? dp : p.P - 1;
      }
      int st;   // time slot: leading zeros of the gap, the tables map it to a bucket
      if (WIDE) {
        const int64_t tj = ts64[cc];
        const uint64_t dt = rc.ti64 >= tj ? (uint64_t)(rc.ti64 - tj) : (uint64_t)(tj - rc.ti64);
        st = kTabWide + __clzll((long long)dt);
      } else {
        int d = rc.ti32 - ts32[cc];
        d = d < 0 ? -d : d;
        st = (MODE == 0 && POS == 2 ? kTabFar : kTabNarrow) + __clz(d);
      }
      if (MODE == 0 && POS == 2) {
        bias[c] = rc.tp[p.P + st];
      } else {
        bps[c] = bp;
        bias[c] = rc.tp[p.P + st];
      }
    }
#pragma unroll
    for (int c = 0; c < 16; c += 2) {
      const int c0 = half * 16 + c;
      float2 b2 = make_float2(bias[c], bias[c + 1]);
      if (!(MODE == 0 && POS == 2)) b2 = __fadd2_rn(make_float2(rc.tp[bps[c]], rc.tp[bps[c + 1]]), b2);
      // SiLU(z)/N = w kC / (1 + 2^w), as w / (kCi + kCi 2^w)
      const float2 w2 = __ffma2_rn(kA2, make_float2(__uint_as_float(sv[c0]), __uint_as_float(sv[c0 + 1])), b2);
      const float2 den = __ffma2_rn(kCi2, make_float2(ex2_approx(w2.x), ex2_approx(w2.y)), kCi2);
      const float2 r2 = __fmul2_rn(w2, make_float2(rcp_approx(den.x), rcp_approx(den.y)));
      float a2[2] = {r2.x, r2.y};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int cc = c0 + e;
        float a = a2[e];
        if (MODE == 1) {
          a = (rc.row_ok && jb + cc < rc.h_end) ? a : 0.f;
        } else if (MODE == 2) {
          a = (rc.row_ok && jb + cc == rc.i) ? a : 0.f;
        } else if (PARTIAL) {
          const int j = jb + cc;
          const bool valid = j <= rc.hi || j == rc.dg;
          a = valid ? a : 0.f;
        }
        a2[e] = a;
      }
      const uint32_t h2 = pack_bf16(a2[0], a2[1]);
      hi[c0 >> 1] = h2;
      const float2 l2 = bf16_residual2(make_float2(a2[0], a2[1]), h2);
      lo[c0 >> 1] = pack_bf16(l2.x, l2.y);
    }
  }
}

// Scores of 32 key columns that are all allowed and share one bias value rb
// (scaled by -log2 e): position bucket saturated, one time bucket.  With so
// little else to do per score, the special-function unit (ex2 and rcp, two
// per score) would set the pace; so 7 of every 8 reciprocals are taken by
// Newton-Raphson on the FMA pipe instead (w is clamped at 64 there, where
// SiLU(z) / N has long been zero to within its rounding, so 1 + 2^w stays
// finite).  S is read and P written 16 columns at a time, which keeps few
// registers live: P_hi of columns [0, 16) goes to scol + [0, 8) and P_lo to
// scol + [16, 24), the columns of the second half's S, so that store waits
// until the second half is loaded.
__device__ __forceinline__ void score16_const(const AttnParams& p, const uint32_t (&sv)[16], uint32_t (&hi)[8],
                                              uint32_t (&lo)[8], float rb) {
  const float2 kA2 = make_float2(p.kA, p.kA), kC2 = make_float2(p.kC, p.kC), b2 = make_float2(rb, rb);
  const float2 one2 = make_float2(1.f, 1.f);
#pragma unroll
  for (int c = 0; c < 16; c += 2) {
    const float2 w2 = __ffma2_rn(kA2, make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), b2);
    float2 r2;
    if (c == 0) {
      const float2 den = __fadd2_rn(make_float2(ex2_approx(w2.x), ex2_approx(w2.y)), one2);
      r2 = __fmul2_rn(__fmul2_rn(w2, kC2), make_float2(rcp_approx(den.x), rcp_approx(den.y)));
    } else {
      const float2 den = __fadd2_rn(make_float2(ex2_approx(fminf(w2.x, 64.f)), ex2_approx(fminf(w2.y, 64.f))), one2);
      r2 = __fmul2_rn(__fmul2_rn(w2, kC2), rcp2_newton(den));
    }
    const uint32_t h2 = pack_bf16(r2.x, r2.y);
    hi[c >> 1] = h2;
    const float2 l2 = bf16_residual2(r2, h2);
    lo[c >> 1] = pack_bf16(l2.x, l2.y);
  }
}
__device__ __forceinline__ void score32_const(const AttnParams& p, uint32_t scol, float rb) {
  uint32_t sv[16], hi[8], lo0[8];
  tmem_ld16(scol, sv);
  tmem_wait_ld();
  score16_const(p, sv, hi, lo0, rb);
  tmem_st8(scol, hi);
  tmem_ld16(scol + 16, sv);
  tmem_wait_ld();
  tmem_st8(scol + 16, lo0);
  uint32_t lo[8];
  score16_const(p, sv, hi, lo, rb);
  tmem_st8(scol + 8, hi);
  tmem_st8(scol + 24, lo);
}

// Warps are spread over the four SM sub-partitions, each with a quarter of the
// register file: with 20 warps each sub-partition holds five,
// and 5 x 32 threads x 96 registers = 15360 <= 16384.
// DELTA: the delta forward (KV-cached candidates): work items are blocks of
// up to 128 candidates; their key tiles are every tile of the sequence's
// cached K/V (tmk2, tmv2, offsets p.off2, times p.ts2) and then one tile of
// the candidates' own K/V (tmk, tmv) for the diagonal.
template <int D, typename TO, bool DELTA>
__global__ void __maxnreg__(96)
hstu_fwd_tc_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmq,
                   const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const __grid_constant__ CUtensorMap tmk2, const __grid_constant__ CUtensorMap tmv2) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const uint32_t sQ0 = base_u32 + L::Q_OFF;
  const uint32_t sK0 = base_u32 + L::K_OFF, sV0 = base_u32 + L::V_OFF;
  int64_t* ts64_s = reinterpret_cast<int64_t*>(base + L::TS64_OFF);
  int32_t* ts32_s = reinterpret_cast<int32_t*>(base + L::TS32_OFF);
  int32_t* cmm_s = reinterpret_cast<int32_t*>(base + L::CMM_OFF);
  int64_t* qts_s = reinterpret_cast<int64_t*>(base + L::QTS_OFF);
  ItemSlot* slots = reinterpret_cast<ItemSlot*>(base + L::SLOT_OFF);
  const uint32_t bar0 = base_u32 + L::BAR_OFF;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L::MISC_OFF + 4);
  int* slot_wide = reinterpret_cast<int*>(base + L::MISC_OFF + 8);  // [kTsSlots]: key times need 64 bits
  float* tab = reinterpret_cast<float*>(base + L::TAB_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.H, P = p.P, Tb = p.Tb, PT = p.P + kTabTime;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQBufs; ++s) {
      mbar_init(bar(BAR_QFULL + s), 1);
      mbar_init(bar(BAR_QEMPTY + s), 2);   // the S issuer's last S and the P.V issuer's last P.V of the item
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(BAR_KFULL + s), 1);
      mbar_init(bar(BAR_KEMPTY + s), 1);
      mbar_init(bar(BAR_VFULL + s), 1);
      mbar_init(bar(BAR_VEMPTY + s), 1);
    }
    for (int s = 0; s < kTsSlots; ++s) {
      mbar_init(bar(BAR_TSFULL + s), 1);
      mbar_init(bar(BAR_TSEMPTY + s), kEpiWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(BAR_SFULL + s), 1);
      mbar_init(bar(BAR_PREADY + s), kEpiWarps);
      mbar_init(bar(BAR_OFULL + s), 1);
      mbar_init(bar(BAR_OEMPTY + s), kEpiWarps);
      mbar_init(bar(BAR_SFREE + s), 1);
    }
    mbar_init(bar(BAR_DRAIN), 2);   // both MMA issuers
    *abort_flag = 0;
    fence_mbar_init();
  }
  // bias tables of every head, times -log2(e): [h][0, P) position, then the
  // kTabTime time slots (wide, narrow, narrow plus position bucket P - 1)
  for (int x = threadIdx.x; x < H * PT; x += kThreads) {
    const int h = x / PT, e = x % PT;
    float v = 0.f;
    if (e < P) {
      if (p.rab_pos) v = p.rab_pos[h * P + e];
    } else {
      const int k = e - P;
      const int bits = k < kTabNarrow ? 64 - (k - kTabWide) : (k < kTabFar ? 32 - (k - kTabNarrow) : 32 - (k - kTabFar));
      if (p.rab_time && p.ts) v = p.rab_time[h * Tb + (bits < Tb - 1 ? bits : Tb - 1)];
      if (k >= kTabFar && p.rab_pos) v += p.rab_pos[h * P + P - 1];
    }
    tab[x] = -kLog2e * v;
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmq);
    tma_prefetch_desc(&tmk);
    if (DELTA) tma_prefetch_desc(&tmk2);
  }
  if (warp == kVProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmv);
    if (DELTA) tma_prefetch_desc(&tmv2);
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // the set-up above reads inputs only; the planner's work list and work
  // counter are read after it has completed (programmatic launch)
  pdl_wait();

  Watchdog wd;
  wd.abort = abort_flag;
  wd.err = p.hdr_rw + WS_ERR;
  wd.err_info = p.hdr_rw + WS_ERR_INFO;
  wd.limit_ns = (p.flags & HSTU_FLAG_TEST_TIMEOUT) ? 1000000ull : 2000000000ull;
  const int nitems = p.hdr[WS_NBLK] * H;

  if (warp == kProducerWarp) {
    // ------------------------------------------------- producer: Q, K, times
    uint32_t kv_it = 0, q_it = 0;
    static_assert(kStages == 2 && kQBufs == 2, "per-stage counters hold two stages");
    Count2 armed;       // K phases armed per stage
    Count2 q_phases;    // phases used per Q buffer (a copy or the final no-work arrive)
    Count2 q_copy;      // 1: the buffer's last phase carries a copy
    bool ok = true;
    // The next work item is claimed only once the current one's loads are all
    // issued (claiming earlier pairs items up statically and loses the
    // longest-first balance); its planner record is one 48-byte load.  The
    // first item of CTA b is item b (no atomic on the way in); later claims
    // count on from the grid size.
    bool first_claim = true;
    while (ok) {
      const int qb = (int)(q_it % kQBufs);
      int idx = (int)blockIdx.x;
      if (!first_claim) {
        if (lane == 0) idx = (int)gridDim.x + atomicAdd(p.hdr_rw + WS_NEXT, 1);
        idx = __shfl_sync(0xffffffffu, idx, 0);
      }
      first_claim = false;
      const bool valid = idx < nitems;
      PlanItem it{};
      if (valid) it = p.items[idx / H];
      const int h = idx % H, q0 = it.blk * BM, n = it.n, L = it.L;
      const int64_t tbase = it.tbase, s0 = it.s0, cs0 = it.cs0;
      // query-row timestamps: loads issued before waiting for the buffer
      int64_t qv[BM / 32];
#pragma unroll
      for (int x = 0; x < BM / 32; ++x) {
        const int row = q0 + lane + 32 * x;
        qv[x] = (valid && p.ts && row < n) ? p.ts[s0 + row] : tbase;
      }
      if (lane == 0) ok = mbar_wait(bar(BAR_QEMPTY + qb), ((q_it / kQBufs) & 1) ^ 1, wd, 1);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      // the Q copy starts before the timestamps arrive; the buffer's phase
      // completes with the copy and the arrive below, after they are staged
      if (lane == 0 && valid) {
        mbar_expect_tx(bar(BAR_QFULL + qb), L::Q_BYTES);
        for (int c = 0; c < L::NCH; ++c)
          tma_load_2d(sQ0 + qb * L::Q_BYTES + c * L::BOX, &tmq, bar(BAR_QFULL + qb), h * D + c * 64, (int)(s0 + q0));
      }
      bool qw = false;
#pragma unroll
      for (int x = 0; x < BM / 32; ++x) qw |= ts_wide(qv[x] - tbase);
      const bool item_wide = __any_sync(0xffffffffu, qw);
#pragma unroll
      for (int x = 0; x < BM / 32; ++x) qts_s[qb * BM + lane + 32 * x] = qv[x];
      if (lane == 0) {
        ItemSlot& sl = slots[qb];
        sl.s0 = s0; sl.tbase = tbase; sl.valid = valid ? 1 : 0;
        sl.h = h; sl.q0 = q0; sl.n = n; sl.c = it.c; sl.h_end = it.h_end; sl.wide = item_wide ? 1 : 0;
        sl.L = L; sl.cs0 = cs0;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(BAR_QFULL + qb));  // without a copy the slot says: no more work
        q_phases.add(qb, 1);
        q_copy.set(qb, valid ? 1u : 0u);
      }
      ++q_it;
      if (!valid) break;
      const int nkb = DELTA ? (L + BN - 1) / BN + 1 : fwd_kv_blocks(q0, n, it.c, BM, BN);
      // test only: the CTA that takes work item 0 withholds that item's first K load
      bool withhold_next = (p.flags & HSTU_FLAG_TEST_TIMEOUT) && idx == 0;
      for (int kb = 0; ok && kb < nkb; ++kb) {
        const bool self = DELTA && kb == nkb - 1;   // delta: the candidates' own keys
        const int k0 = self ? q0 : kb * BN;
        if (!DELTA && tile_class(q0, k0, BM, BN, n, it.c, it.h_end) == 0) continue;
        const int stage = kv_it % kStages, ts = kv_it % kTsSlots;
        // key timestamps: loads issued before waiting, stored after
        int64_t tv[BN / 32];
#pragma unroll
        for (int x = 0; x < BN / 32; ++x) {
          const int row = k0 + lane + 32 * x;
          if (DELTA && !self) tv[x] = (p.ts2 && row < L) ? p.ts2[cs0 + row] : tbase;
          else tv[x] = (p.ts && row < n) ? p.ts[s0 + row] : tbase;
        }
        ok = mbar_wait(bar(BAR_KEMPTY + stage), ((kv_it / kStages) & 1) ^ 1, wd, 2);
        if (!ok) break;
        const bool withhold = withhold_next;
        withhold_next = false;
        if (lane == 0 && !withhold) {   // withheld (test only): neither copy nor arrive
          const bool cached = DELTA && !self;
          mbar_arrive_expect_tx(bar(BAR_KFULL + stage), L::K_BYTES);
          const int y = (int)(cached ? cs0 + k0 : s0 + k0);
          for (int c = 0; c < L::NCH; ++c)
            tma_load_2d(sK0 + stage * L::K_BYTES + c * L::BOX, cached ? &tmk2 : &tmk, bar(BAR_KFULL + stage),
                        h * D + c * 64, y);
          armed.add(stage, 1);
          // delta forward: the cached K and V two tiles ahead into L2, so
          // their loads, issued once a stage frees up, do not wait on HBM
          // (the ordinary forward's K/V re-reads are L2 hits, and the
          // prefetch requests only compete with the copies: 70.3 -> 69.0 us
          // without them)
          if (DELTA && kb + 2 < nkb) {
            const bool self2 = DELTA && kb + 2 == nkb - 1, cached2 = DELTA && !self2;
            const int y2 = (int)(cached2 ? cs0 + (kb + 2) * BN : s0 + (self2 ? q0 : (kb + 2) * BN));
            for (int c = 0; c < L::NCH; ++c) {
              tma_prefetch_l2_2d(cached2 ? &tmk2 : &tmk, h * D + c * 64, y2);
              tma_prefetch_l2_2d(cached2 ? &tmv2 : &tmv, h * D + c * 64, y2);
            }
          }
        }
        ok = mbar_wait(bar(BAR_TSEMPTY + ts), ((kv_it / kTsSlots) & 1) ^ 1, wd, 11);
        if (!ok) break;
        bool kw = false;
#pragma unroll
        for (int x = 0; x < BN / 32; ++x) {
          const int32_t r = (int32_t)(tv[x] - tbase);
          ts64_s[ts * BN + lane + 32 * x] = tv[x];
          ts32_s[ts * BN + lane + 32 * x] = r;
          kw |= ts_wide(tv[x] - tbase);
          // min and max relative time of the 32-key chunk x, for the
          // epilogue's test for a time bucket that is the same across it
          int mn = r, mx = r;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          }
          if (lane == 0) {
            cmm_s[ts * 8 + 2 * x] = mn;
            cmm_s[ts * 8 + 2 * x + 1] = mx;
          }
        }
        kw = __any_sync(0xffffffffu, kw);
        if (lane == 0) slot_wide[ts] = kw ? 1 : 0;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_TSFULL + ts));
        ++kv_it;
      }
    }
    // make sure no copy is still landing in shared memory when the CTA ends
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s)
        if (armed[s]) drain_wait(bar(BAR_KFULL + s), (armed[s] - 1) & 1);
      // an earlier phase of a Q buffer completed before the buffer was reused
      for (int s = 0; s < kQBufs; ++s)
        if (q_copy[s]) drain_wait(bar(BAR_QFULL + s), (q_phases[s] - 1) & 1);
    }
  } else if (warp == kVProducerWarp) {
    // ------------------------------------------------------- producer: V
    // walks the items the Q/K producer publishes (each Q buffer's phase), so
    // it issues V loads as soon as a V stage is free, independently of K
    if (lane == 0) {
      uint32_t kv_it = 0, q_it = 0;
      Count2 armed;
      bool ok = true;
      while (ok) {
        const uint32_t qb = q_it % kQBufs;
        ok = mbar_wait(bar(BAR_QFULL + qb), (q_it / kQBufs) & 1, wd, 12);
        if (!ok) break;
        const ItemSlot sl = slots[qb];
        if (!sl.valid) break;
        const int nkb = DELTA ? (sl.L + BN - 1) / BN + 1 : fwd_kv_blocks(sl.q0, sl.n, sl.c, BM, BN);
        for (int kb = 0; ok && kb < nkb; ++kb) {
          const bool self = DELTA && kb == nkb - 1;
          const int k0 = self ? sl.q0 : kb * BN;
          if (!DELTA && tile_class(sl.q0, k0, BM, BN, sl.n, sl.c, sl.h_end) == 0) continue;
          const int stage = kv_it % kStages;
          ok = mbar_wait(bar(BAR_VEMPTY + stage), ((kv_it / kStages) & 1) ^ 1, wd, 13);
          if (!ok) break;
          const bool cached = DELTA && !self;
          mbar_arrive_expect_tx(bar(BAR_VFULL + stage), L::K_BYTES);
          const int y = (int)(cached ? sl.cs0 + k0 : sl.s0 + k0);
          for (int c = 0; c < L::NCH; ++c)
            tma_load_2d(sV0 + stage * L::K_BYTES + c * L::BOX, cached ? &tmv2 : &tmv, bar(BAR_VFULL + stage),
                        sl.h * D + c * 64, y);
          armed.add(stage, 1);
          ++kv_it;
        }
        ++q_it;
      }
      for (int s = 0; s < kStages; ++s)
        if (armed[s]) drain_wait(bar(BAR_VFULL + s), (armed[s] - 1) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------ MMA: S = Q K^T
    // Two warps issue the tensor-core work: this one S = Q K^T, warp kPvWarp
    // the P V products, each with its own barriers, so neither waits for the
    // other's issue.  S(t) goes into S/P buffer t % 2 once the P V of tile
    // t - 2 (the buffer's previous tile) is complete (SFREE); an item's Q
    // buffer is released by this warp's commit after its last S together
    // with the P V warp's arrival after its last P V.  This warp owns the
    // TMEM allocation.
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(BM, BN, false, false);
      const SDesc q_km = sdesc_w(sQ0, 16, 1024), k_km = sdesc_w(sK0, 16, 1024);
      uint32_t kv_it = 0, q_it = 0;
      bool ok = true;
      while (ok) {
        const uint32_t qb = q_it % kQBufs;
        ok = mbar_wait(bar(BAR_QFULL + qb), (q_it / kQBufs) & 1, wd, 3);
        if (!ok) break;
        fence_after_sync();
        const ItemSlot sl = slots[qb];
        if (!sl.valid) break;
        const SDesc q_s = q_km + qb * L::Q_BYTES;
        const int nkb = DELTA ? (sl.L + BN - 1) / BN + 1 : fwd_kv_blocks(sl.q0, sl.n, sl.c, BM, BN);
        for (int kb = 0; ok && kb < nkb; ++kb) {
          const int k0 = kb * BN;
          if (!DELTA && tile_class(sl.q0, k0, BM, BN, sl.n, sl.c, sl.h_end) == 0) continue;
          const uint32_t stage = kv_it % kStages, sb = kv_it & 1;
          ok = mbar_wait(bar(BAR_KFULL + stage), (kv_it / kStages) & 1, wd, 6) &&
               mbar_wait(bar(BAR_SFREE + sb), ((kv_it >> 1) & 1) ^ 1, wd, 15);
          if (!ok) break;
          fence_after_sync();
          const SDesc k_s = k_km + stage * L::K_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * L::BOX + (kk & 3) * 32;
            mma_ss_w(tmem + sb * kSColStride, q_s + off, k_s + off, IDESC_S, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(BAR_SFULL + sb));
          mma_commit(bar(BAR_KEMPTY + stage));   // K is read by no later MMA
          ++kv_it;
        }
        if (!ok) break;
        mma_commit(bar(BAR_QEMPTY + qb));   // Q is read by no later MMA
        ++q_it;
      }
      // every MMA issued by this thread is complete before TMEM is released
      mma_commit(bar(BAR_DRAIN));
      drain_wait(bar(BAR_DRAIN), 0);
    }
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------ MMA: O += P V
    if (lane == 0) {
      constexpr uint32_t IDESC_PV = idesc_bf16(BM, D, false, true);
      const SDesc v_mn = sdesc_w(sV0, L::BOX, 1024);
      uint32_t kv_it = 0, q_it = 0;
      bool ok = true;
      while (ok) {
        const uint32_t qb = q_it % kQBufs, ob = q_it & 1;
        ok = mbar_wait(bar(BAR_QFULL + qb), (q_it / kQBufs) & 1, wd, 16);
        if (!ok) break;
        fence_after_sync();
        const ItemSlot sl = slots[qb];
        if (!sl.valid) break;
        const uint32_t ocol = ob ? L::O_COL1 : L::O_COL0;
        // this item's P.V go into O buffer ob once the epilogue has written it out
        ok = mbar_wait(bar(BAR_OEMPTY + ob), ((q_it >> 1) & 1) ^ 1, wd, 4);
        if (!ok) break;
        fence_after_sync();
        bool first = true;
        const int nkb = DELTA ? (sl.L + BN - 1) / BN + 1 : fwd_kv_blocks(sl.q0, sl.n, sl.c, BM, BN);
        for (int kb = 0; ok && kb < nkb; ++kb) {
          const int k0 = kb * BN;
          if (!DELTA && tile_class(sl.q0, k0, BM, BN, sl.n, sl.c, sl.h_end) == 0) continue;
          // P of tile t: quarter k/2 of the S buffer, hi at [32 q, 32 q + 16), lo 16 columns later
          const uint32_t sb = kv_it & 1, stage = kv_it % kStages;
          ok = mbar_wait(bar(BAR_PREADY + sb), (kv_it >> 1) & 1, wd, 5) &&
               mbar_wait(bar(BAR_VFULL + stage), (kv_it / kStages) & 1, wd, 14);
          if (!ok) break;
          fence_after_sync();
          const SDesc v_s = v_mn + stage * L::K_BYTES;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint32_t a_hi = tmem + sb * kSColStride + 32u * (kk >> 1) + 8u * (kk & 1);
            mma_ts_w(tmem + ocol, a_hi, v_s + kk * 2048, IDESC_PV, (first && kk == 0) ? 0u : 1u);
            mma_ts_w(tmem + ocol, a_hi + 16, v_s + kk * 2048, IDESC_PV, 1u);
          }
          mma_commit(bar(BAR_VEMPTY + stage));
          mma_commit(bar(BAR_SFREE + sb));   // the S/P buffer may take the next S
          first = false;
          ++kv_it;
        }
        if (!ok) break;
        // the item's last P has been handed over: its slot is read by no one any more
        mbar_arrive(bar(BAR_QEMPTY + qb));
        mma_commit(bar(BAR_OFULL + ob));
        ++q_it;
      }
      mma_commit(bar(BAR_DRAIN));
      drain_wait(bar(BAR_DRAIN), 0);
    }
  } else if (warp < kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3, hq = warp >> 2;      // TMEM lane quarter, column quarter
    const int row = wq * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    uint32_t kv_it = 0, o_it = 0, q_it = 0;
    bool ok = true;
    RowCtx rc;
    // An item's O is written out after the next item's first P is handed
    // over (or when the work runs out), so the epilogue does not wait for the
    // item's last P.V: what the write-out needs is kept here.
    bool o_pend = false;
    uint32_t po_it = 0;
    int64_t po_row = 0;   // token of this thread's row, or -1
    int po_h = 0;
    auto write_o = [&]() -> bool {
      const uint32_t ob = po_it & 1;
      if (!mbar_wait(bar(BAR_OFULL + ob), (po_it >> 1) & 1, wd, 9)) return false;
      fence_after_sync();
      constexpr int QC = D / 4;  // columns per quarter
      const uint32_t ocol = lane_base + (ob ? L::O_COL1 : L::O_COL0) + hq * QC;
      uint32_t ov[32];
      if constexpr (QC == 32) {
        tmem_ld32(ocol, ov);
      } else {
        uint32_t o16[16];
        tmem_ld16(ocol, o16);
#pragma unroll
        for (int e = 0; e < 16; ++e) ov[e] = o16[e];
      }
      tmem_wait_ld();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_OEMPTY + ob));
      if (po_row >= 0) {
        TO* orow = static_cast<TO*>(p.o) + ((size_t)po_row * H + po_h) * D + hq * QC;
        if constexpr (sizeof(TO) == 4) {
          float4* dst = reinterpret_cast<float4*>(orow);
#pragma unroll
          for (int e = 0; e < QC / 4; ++e)
            dst[e] = make_float4(__uint_as_float(ov[4 * e]), __uint_as_float(ov[4 * e + 1]),
                                 __uint_as_float(ov[4 * e + 2]), __uint_as_float(ov[4 * e + 3]));
        } else {
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int e = 0; e < QC / 8; ++e)
            dst[e] = make_uint4(pack_bf16(__uint_as_float(ov[8 * e]), __uint_as_float(ov[8 * e + 1])),
                                pack_bf16(__uint_as_float(ov[8 * e + 2]), __uint_as_float(ov[8 * e + 3])),
                                pack_bf16(__uint_as_float(ov[8 * e + 4]), __uint_as_float(ov[8 * e + 5])),
                                pack_bf16(__uint_as_float(ov[8 * e + 6]), __uint_as_float(ov[8 * e + 7])));
        }
      }
      o_pend = false;
      return true;
    };
    while (ok) {
      const uint32_t qb = q_it % kQBufs;
      ok = mbar_wait(bar(BAR_QFULL + qb), (q_it / kQBufs) & 1, wd, 10);
      if (!ok) break;
      // the slot stays until this item's last P is handed over; keep what the
      // O write-out needs in registers
      const ItemSlot& sl = slots[qb];
      if (!sl.valid) break;
      const int64_t s0 = sl.s0;
      const int hh = sl.h, q0 = sl.q0;
      const bool item_wide = sl.wide != 0;
      const int n_seq = sl.n, cx = sl.c;
      rc.h_end = DELTA ? sl.L : sl.h_end;   // delta: the candidates' position is the cache length
      rc.i = q0 + row;
      rc.row_ok = rc.i < n_seq;
      rc.pos_i = DELTA ? rc.h_end : (rc.i < rc.h_end ? rc.i : rc.h_end);
      // allowed keys of this row: history/context rows see j <= i (context rows
      // the whole context), candidates see all of history/context and themselves
      rc.hi = !rc.row_ok ? -1 : (rc.i < rc.h_end ? (rc.i < cx ? cx - 1 : rc.i) : rc.h_end - 1);
      rc.dg = (rc.row_ok && rc.i >= rc.h_end) ? rc.i : -1;
      rc.ti64 = qts_s[qb * BM + row];
      rc.ti32 = (int32_t)(rc.ti64 - sl.tbase);
      rc.tp = tab + hh * PT;
      const int nkb = DELTA ? (rc.h_end + BN - 1) / BN + 1 : fwd_kv_blocks(q0, n_seq, cx, BM, BN);
      for (int kb = 0; ok && kb < nkb; ++kb) {
        const bool self = DELTA && kb == nkb - 1;
        const int k0 = self ? q0 : kb * BN;
        const int cls = DELTA ? 1 : tile_class(q0, k0, BM, BN, n_seq, cx, rc.h_end);
        if (cls == 0) continue;
        const uint32_t ts = kv_it % kTsSlots, sb = kv_it & 1;
        ok = mbar_wait(bar(BAR_TSFULL + ts), (kv_it / kTsSlots) & 1, wd, 7) &&
             mbar_wait(bar(BAR_SFULL + sb), (kv_it >> 1) & 1, wd, 8);
        if (!ok) break;
        fence_after_sync();
        const uint32_t scol = lane_base + sb * kSColStride + hq * 32;
        const int jb = k0 + hq * 32;
        const int32_t* t32 = ts32_s + ts * BN + hq * 32;
        const int64_t* t64 = ts64_s + ts * BN + hq * 32;
        uint32_t sv[32], hi[16], lo[16];
        bool stored = false;   // the constant-bias path loads S and stores P itself
        // Class of the warp's block (32 rows from r0, 32 keys from jb).  Rows
        // past the sequence only feed rows of O that are never written out,
        // so they do not limit it: the block is full when every key is a
        // history or context token that every row may see, i.e. all keys lie
        // at or before the first row, or all rows are candidates (which see
        // the whole history).  That holds on the ragged last block of a
        // sequence too, whose tiles are partial only by their missing rows.
        const int r0 = q0 + wq * 32, kend = jb + 31;
        const bool fast = kend < rc.h_end && (kend <= r0 || r0 >= rc.h_end);
        // the warp's rows start at position pos_lo (positions grow with the row)
        const int pos_lo = r0 < rc.h_end ? r0 : rc.h_end;
        const bool far = fast && pos_lo - kend >= p.P - 1;
        const bool narrow = !item_wide && !slot_wide[ts];
        if (DELTA) {
          tmem_ld32(scol, sv);
          tmem_wait_ld();
          if (self) {
            if (narrow) score32<0, false, false, 2>(p, sv, hi, lo, rc, jb, t32, t64);
            else score32<0, true, false, 2>(p, sv, hi, lo, rc, jb, t32, t64);
          } else {
            if (narrow) score32<0, false, false, 1>(p, sv, hi, lo, rc, jb, t32, t64);
            else score32<0, true, false, 1>(p, sv, hi, lo, rc, jb, t32, t64);
          }
        } else if (narrow) {
          // far blocks whose time bucket is also the same across the row's 32
          // keys (the keys' times all on one side of t_i, and the bucket of
          // the nearest and of the farthest gap equal): one bias per row
          bool cst = far;
          int slot = kTabFar;
          if (far && p.ts) {
            // gaps to the latest and the earliest key time of the chunk: of
            // one sign when t_i is not inside the chunk's time range, and then
            // the gaps of all its keys lie between them
            const int32_t d1 = rc.ti32 - cmm_s[ts * 8 + 2 * hq + 1], d2 = rc.ti32 - cmm_s[ts * 8 + 2 * hq];
            const int z1 = __clz(abs(d1)), z2 = __clz(abs(d2));
            cst = ((d1 ^ d2) >= 0 && min(32 - z1, Tb - 1) == min(32 - z2, Tb - 1)) || !rc.row_ok;
            slot = kTabFar + z1;   // a row past the sequence takes any bias
          }
          if (__all_sync(0xffffffffu, cst)) {
            score32_const(p, scol, rc.tp[P + slot]);
            stored = true;
          } else {
            tmem_ld32(scol, sv);
            tmem_wait_ld();
            if (far) score32<2, false, false>(p, sv, hi, lo, rc, jb, t32, t64);
            else if (fast) score32<1, false, false>(p, sv, hi, lo, rc, jb, t32, t64);
            else if (cls == 2) score32<0, false, false>(p, sv, hi, lo, rc, jb, t32, t64);
            else score32<0, false, true>(p, sv, hi, lo, rc, jb, t32, t64);
          }
        } else {
          tmem_ld32(scol, sv);
          tmem_wait_ld();
          if (cls == 2) score32<0, true, false>(p, sv, hi, lo, rc, jb, t32, t64);
          else score32<0, true, true>(p, sv, hi, lo, rc, jb, t32, t64);
        }
        // P_hi of this quarter at [32 hq, 32 hq + 16), P_lo at [32 hq + 16, 32 hq + 32)
        if (!stored) {
          tmem_st16(scol, hi);
          tmem_st16(scol + 16, lo);
        }
        tmem_wait_st();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(BAR_PREADY + sb));
          mbar_arrive(bar(BAR_TSEMPTY + ts));
        }
        ++kv_it;
        if (o_pend) {  // the previous item's O, now that this item's first P is out
          ok = write_o();
          if (!ok) break;
        }
      }
      if (!ok) break;
      if (o_pend) {  // an item without tiles (none is planned)
        ok = write_o();
        if (!ok) break;
      }
      o_pend = true;
      po_it = o_it;
      po_row = rc.row_ok ? s0 + rc.i : -1;
      po_h = hh;
      ++o_it;
      ++q_it;
    }
    if (ok && o_pend) ok = write_o();
  }

  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

}  // namespace

// 2-D BF16 tensor map over [rows, cols] (row-major), box 64 cols x box_rows
// rows, 128-byte swizzle, zero fill outside.
bool make_tmap_bf16(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of rank 2 or 3 for tile stores: dims innermost first, strides
// in bytes of dims 1..rank-1, the box, the swizzle; no L2 promotion.
bool make_tmap_tile(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* ptr, const uint64_t* dims,
                    const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rank < 2 || rank > 3) return false;
  cuuint64_t d[3], st[2];
  cuuint32_t b[3], e[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) { d[i] = dims[i]; b[i] = box[i]; }
  for (int i = 0; i < rank - 1; ++i) st[i] = strides[i];
  return fn(map, dt, rank, const_cast<void*>(ptr), d, st, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_fwd_supported(int dtype, int dqk, int dv) {
  return dtype == HSTU_BF16 && dqk == dv && (dqk == 64 || dqk == 128);
}

size_t tc_fwd_smem_bytes(int d, int H, int P, int Tb) {
  const size_t tab = sizeof(float) * (size_t)H * (P + kTabTime);
  return (d == 64 ? Layout<64>::TAB_OFF : Layout<128>::TAB_OFF) + tab + 1024;
}

template <int D, typename TO, bool DELTA>
static cudaError_t launch_fwd_t(const AttnParams& p, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mk2, mv2;
  const int64_t cols = (int64_t)p.H * D;
  if (!make_tmap_bf16(&mq, p.q, p.T, cols, BM) || !make_tmap_bf16(&mk, p.k, p.T, cols, BN) ||
      !make_tmap_bf16(&mv, p.v, p.T, cols, BN))
    return cudaErrorInvalidValue;
  if (DELTA && p.T2 > 0) {
    if (!make_tmap_bf16(&mk2, p.k2, p.T2, cols, BN) || !make_tmap_bf16(&mv2, p.v2, p.T2, cols, BN))
      return cudaErrorInvalidValue;
  } else {
    mk2 = mk;  // unused: no cached tiles
    mv2 = mv;
  }
  const size_t smem = tc_fwd_smem_bytes(D, p.H, p.P, p.Tb);
  const void* fn = reinterpret_cast<const void*>(hstu_fwd_tc_kernel<D, TO, DELTA>);
  cudaError_t e = cudaFuncSetAttribute(hstu_fwd_tc_kernel<D, TO, DELTA>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) {
    set_launch_detail(e, "hstu_fwd_tc_kernel (smem attribute)", fn, kThreads, smem);
    return e;
  }
  const int64_t max_items = ((p.T + BM - 1) / BM + p.B) * (int64_t)p.H;
  const int grid = (int)(max_items < p.num_sms ? max_items : p.num_sms);
  // launched programmatically after the planner: the set-up overlaps it
  e = launch_pdl(hstu_fwd_tc_kernel<D, TO, DELTA>, dim3(grid), dim3(kThreads), smem, st, p, mq, mk, mv, mk2, mv2);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) set_launch_detail(e, "hstu_fwd_tc_kernel", fn, kThreads, smem);
  return e;
}

template <bool DELTA>
static cudaError_t launch_any(const AttnParams& p, cudaStream_t st) {
  const bool f32 = p.out_dtype == HSTU_FP32;
  if (p.dqk == 128)
    return f32 ? launch_fwd_t<128, float, DELTA>(p, st) : launch_fwd_t<128, __nv_bfloat16, DELTA>(p, st);
  if (p.dqk == 64)
    return f32 ? launch_fwd_t<64, float, DELTA>(p, st) : launch_fwd_t<64, __nv_bfloat16, DELTA>(p, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_tc_fwd(const AttnParams& p, cudaStream_t st) { return launch_any<false>(p, st); }
cudaError_t launch_tc_fwd_delta(const AttnParams& p, cudaStream_t st) { return launch_any<true>(p, st); }

}  // namespace hstu
