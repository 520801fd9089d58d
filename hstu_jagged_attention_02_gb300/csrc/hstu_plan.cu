// Device tile planner.
//
// One CTA validates the jagged metadata, lists every query block (forward) or
// key block (backward) of every sequence, counts the tiles of each block that
// the compound mask does not skip, and orders the blocks longest-first
// (counting sort on the tile count), so a persistent grid that takes blocks in
// order gets an LPT-style balance.  This is the "greedy even core split" and
// "compound-mask skipping" of the Ascend HSTU fused operator (wmrh.cn RecSDK
// page, "HSTU acceleration operator" paragraph), done on the device so no
// host synchronisation is needed.  A forward that also plans the backward
// launches a second CTA, which plans the backward's tiling at the same time
// and records what it was made from, so the backward needs no planner launch.
#include "hstu_internal.h"

namespace hstu {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPlanWarps = kPlanThreads / 32;

// Exclusive prefix sum of v over the CTA (warp shuffles, two barriers); the
// CTA total goes to *total.  wsum holds kPlanWarps ints.
__device__ int cta_exclusive_scan(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    wsum[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  *total = wsum[kPlanWarps - 1];
  const int before = w > 0 ? wsum[w - 1] : 0;
  return before + x - v;
}

// Tiles of one block that lane gl of a group of G lanes counts (the group's
// sum is the block's cost).  Pass 2 (delta forward): a block of up to BM
// candidates sees every cached key tile of its sequence plus one tile of its
// own keys (the diagonal); cached_len is that sequence's cached-token count.
__device__ int block_cost_part(const SeqInfo& s, int blk, int pass, int BM, int BN, int cached_len, int gl, int G) {
  int cost = 0;
  if (pass == 2) {
    cost = gl == 0 ? (cached_len + BN - 1) / BN + 1 : 0;
  } else if (pass == 0) {
    const int q0 = blk * BM;
    const int nkb = fwd_kv_blocks(q0, s.n, s.c, BM, BN);
    for (int kb = gl; kb < nkb; kb += G) cost += tile_class(q0, kb * BN, BM, BN, s.n, s.c, s.h_end) != 0;
  } else {
    const int k0 = blk * BN;
    const int nqb = (s.n + BM - 1) / BM;
    for (int qb = bwd_q_begin(k0, s.c, BM) + gl; qb < nqb; qb += G)
      cost += tile_class(qb * BM, k0, BM, BN, s.n, s.c, s.h_end) != 0;
  }
  return cost;
}

// Dynamic shared memory: histogram, then (when they fit) the offsets, the
// block starts per sequence and the block records; otherwise the workspace
// scratch arrays stand in.  CTA 0 plans out[0]; with npass == 2, CTA 1 plans
// the backward's tiling into out[1] at the same time and keeps it for a later
// backward call (WS_PB_* words, the metadata it was made from).
__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(PlanParams p) {
  extern __shared__ __align__(16) uint8_t plan_smem[];
  __shared__ int sh_wsum[kPlanWarps];
  __shared__ int sh_bad, sh_bad_b;
  int* sh_hist = reinterpret_cast<int*>(plan_smem);
  uint8_t* cur = plan_smem + sizeof(int) * kCostBins;
  int64_t* off = const_cast<int64_t*>(p.off);
  if (p.stage_off) { off = reinterpret_cast<int64_t*>(cur); cur += sizeof(int64_t) * ((p.B + 2) & ~1); }
  int* start = nullptr;
  if (p.stage_off) { start = reinterpret_cast<int*>(cur); cur += sizeof(int) * ((p.B + 1 + 3) & ~3); }
  // the per-sequence counts and first timestamps, staged with the offsets
  const int32_t* nt = p.nt;
  const int32_t* nc = p.nc;
  int64_t* t0s = nullptr;
  if (p.stage_off) {
    t0s = reinterpret_cast<int64_t*>(cur); cur += sizeof(int64_t) * ((p.B + 1) & ~1);
    int32_t* nts = reinterpret_cast<int32_t*>(cur); cur += sizeof(int32_t) * ((p.B + 3) & ~3);
    int32_t* ncs = reinterpret_cast<int32_t*>(cur); cur += sizeof(int32_t) * ((p.B + 3) & ~3);
    for (int i = threadIdx.x; i < p.B; i += kPlanThreads) {
      nts[i] = p.nt ? p.nt[i] : 0;
      ncs[i] = p.nc ? p.nc[i] : 0;
    }
    nt = nts;
    nc = ncs;
  }
  const bool keep = blockIdx.x == 1;
  const PlanOut o = keep ? p.out[1] : p.out[0];
  if (!start) start = o.seq_start;
  Block* rec = p.stage_rec ? reinterpret_cast<Block*>(cur) : o.tmp;
  const int t = threadIdx.x;
  // the kernel that follows (launched programmatically) may start its own
  // set-up now; it waits for this grid before it reads the plan
  pdl_launch_dependents();

  if (t == 0) {
    if (!keep) {
      p.hdr[WS_ERR] = 0;
      p.hdr[WS_ERR_INFO] = 0;
      p.hdr[WS_NBLK] = 0;
      p.hdr[WS_NTILES] = 0;
      p.hdr[WS_FLAGS] = 0;
      p.hdr[WS_NEXT] = 0;
    }
    // a kept backward plan is void from here on: this launch either replaces
    // it (CTA 1) or plans another batch
    if (keep || p.npass == 1) p.hdr[WS_PB_VALID] = 0;
    sh_bad = 0;
    sh_bad_b = 0;
  }
  for (int i = t; i < kCostBins; i += kPlanThreads) sh_hist[i] = 0;
  if (p.stage_off)
    for (int i = t; i <= p.B; i += kPlanThreads) off[i] = p.off[i];
  __syncthreads();

  // 1. validation
  if (t == 0 && (off[0] != 0 || off[p.B] != p.T)) atomicExch(&sh_bad, 1);
  if (t == 0 && o.pass == 2 && (p.off2[0] != 0 || p.off2[p.B] != p.T2)) atomicExch(&sh_bad, 1);
  for (int b = t; b < p.B; b += kPlanThreads) {
    const int64_t n = off[b + 1] - off[b];
    const int64_t m = nt ? nt[b] : 0, c = nc ? nc[b] : 0;
    // pass 2: n candidates after L cached tokens, n + L <= N
    const int64_t L = o.pass == 2 ? p.off2[b + 1] - p.off2[b] : 0;
    if (n < 0 || L < 0 || n + L > p.max_n || m < 0 || c < 0 || m + c > n) {
      if (atomicExch(&sh_bad, 1) == 0) sh_bad_b = b;
    }
    if (keep) {
      p.sv_off[b] = off[b];
      p.sv_nt[b] = (int32_t)m;
      p.sv_nc[b] = (int32_t)c;
    }
  }
  if (keep && t == 0) p.sv_off[p.B] = off[p.B];
  __syncthreads();
  if (sh_bad) {
    if (t == 0 && !keep) {
      p.hdr[WS_ERR_INFO] = sh_bad_b;
      atomicCAS(p.hdr + WS_ERR, 0, HSTU_ERR_DEVICE_CHECK);
    }
    return;
  }
  // first timestamp of each sequence (the offsets are consistent now, so
  // every first token is in range): loads issued here, stored to shared
  // memory only before the scatter, so their latency overlaps steps 2-4
  int64_t my_t0 = 0;
  if (t0s && t < p.B && p.ts && off[t + 1] > off[t]) my_t0 = p.ts[off[t]];

  // 2. blocks per sequence -> exclusive prefix (start[b]), one chunk of
  // kPlanThreads sequences at a time
  const int BR = o.pass == 1 ? o.BN : o.BM;  // rows per block of this pass
  int carry = 0;
  for (int base = 0; base < p.B; base += kPlanThreads) {
    const int b = base + t;
    const int nb = b < p.B ? (int)((off[b + 1] - off[b] + BR - 1) / BR) : 0;
    int total;
    const int ex = cta_exclusive_scan(nb, sh_wsum, &total);
    if (b < p.B) start[b] = carry + ex;
    carry += total;
    __syncthreads();  // sh_wsum is reused by the next chunk
  }
  const int nblk = carry;
  if (t == 0) start[p.B] = nblk;
  if (nblk > p.cap_blocks) {  // cannot happen when off[B] == T; guard anyway
    if (t == 0) atomicCAS(p.hdr + WS_ERR, 0, HSTU_ERR_DEVICE_CHECK);
    return;
  }
  __syncthreads();

  // 3. cost of every block, histogram of costs.  While blocks are few, a
  // group of G lanes walks each block's tiles (a long sequence's blocks walk
  // up to N / 64 tiles); G = 1 once every thread has blocks of its own.
  {
    const int G = nblk <= kPlanThreads / 8 * 4 ? 8 : 1;
    const int gl = t % G;
    const unsigned gmask = G == 8 ? 0xffu << ((t & 31) & ~7) : 1u << (t & 31);
    for (int idx = t / G; idx < nblk; idx += kPlanThreads / G) {
      int lo = 0, hi = p.B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (start[mid] <= idx) lo = mid; else hi = mid - 1;
      }
      const int b = lo;  // the last sequence starting at or before idx (skips empty ones)
      SeqInfo s;
      s.s0 = off[b];
      s.n = (int)(off[b + 1] - s.s0);
      s.c = nc ? nc[b] : 0;
      s.h_end = s.n - (nt ? nt[b] : 0);
      const int blk = idx - start[b];
      const int cached_len = o.pass == 2 ? (int)(p.off2[b + 1] - p.off2[b]) : 0;
      int cost = block_cost_part(s, blk, o.pass, o.BM, o.BN, cached_len, gl, G);
      for (int x = 1; x < G; x <<= 1) cost += __shfl_xor_sync(gmask, cost, x);
      if (gl == 0) {
        Block r;
        r.b = b; r.blk = blk; r.cost = cost; r.pad = 0;
        rec[idx] = r;
        atomicAdd(&sh_hist[cost < kCostBins ? cost : kCostBins - 1], 1);
      }
    }
  }
  if (t0s) {
    if (t < p.B) t0s[t] = my_t0;
    for (int b = t + kPlanThreads; b < p.B; b += kPlanThreads)
      t0s[b] = (p.ts && off[b + 1] > off[b]) ? p.ts[off[b]] : 0;
  }
  __syncthreads();
  if (keep && t0s)
    for (int b = t; b < p.B; b += kPlanThreads) p.sv_t0[b] = t0s[b];
  if (keep && !t0s)
    for (int b = t; b < p.B; b += kPlanThreads) p.sv_t0[b] = (p.ts && off[b + 1] > off[b]) ? p.ts[off[b]] : 0;

  // 4. exclusive scan of the histogram in descending cost order: thread t
  // owns bins kCostBins-1-4t .. kCostBins-4-4t
  {
    constexpr int per = kCostBins / kPlanThreads;
    int local[per];
    int sum = 0;
#pragma unroll
    for (int r = 0; r < per; ++r) {
      local[r] = sh_hist[kCostBins - 1 - (t * per + r)];
      sum += local[r];
    }
    int total;
    const int ex = cta_exclusive_scan(sum, sh_wsum, &total);
    int run = ex;
#pragma unroll
    for (int r = 0; r < per; ++r) {
      sh_hist[kCostBins - 1 - (t * per + r)] = run;  // start of this bin
      run += local[r];
    }
  }
  __syncthreads();

  // 5. scatter into longest-first order, as block records and as full item
  // records (one load per item for the tensor-core kernels' producers)
  for (int idx = t; idx < nblk; idx += kPlanThreads) {
    const Block r = rec[idx];
    const int pos = atomicAdd(&sh_hist[r.cost < kCostBins ? r.cost : kCostBins - 1], 1);
    o.blocks[pos] = r;
    PlanItem it;
    it.b = r.b;
    it.blk = r.blk;
    it.s0 = off[r.b];
    it.n = (int)(off[r.b + 1] - it.s0);
    it.c = nc ? nc[r.b] : 0;
    it.h_end = it.n - (nt ? nt[r.b] : 0);
    it.tbase = t0s ? t0s[r.b] : ((p.ts && it.n > 0) ? p.ts[it.s0] : 0);
    it.cs0 = o.pass == 2 ? p.off2[r.b] : 0;
    it.L = o.pass == 2 ? (int)(p.off2[r.b + 1] - it.cs0) : 0;
    o.items[pos] = it;
  }
  if (t == 0) {
    if (!keep) {
      p.hdr[WS_NBLK] = nblk;
    } else {
      p.hdr[WS_PB_NBLK] = nblk;
      p.hdr[WS_PB_B] = p.B;
      p.hdr[WS_PB_T_LO] = (int)(uint32_t)p.T;
      p.hdr[WS_PB_T_HI] = (int)(p.T >> 32);
      p.hdr[WS_PB_TILE] = o.BM | (o.BN << 16);
      p.hdr[WS_PB_MAXN] = p.max_n;
      p.hdr[WS_PB_VALID] = kKeptPlanValid;
    }
  }
}

// Lists every non-skipped tile of every planned block, walking the blocks the
// same way the kernels do.  Record: b, q_block, k_block, class, query edge,
// key edge.
__global__ void debug_tiles_kernel(PlanParams p, int32_t* rec, int64_t cap) {
  const int nblk = p.hdr[WS_NBLK];
  const PlanOut& o = p.out[0];
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < nblk; idx += gridDim.x * blockDim.x) {
    const Block blk = o.blocks[idx];
    const SeqInfo s = seq_info(p.off, p.nt, p.nc, blk.b);
    if (o.pass == 0) {
      const int q0 = blk.blk * o.BM;
      const int nkb = fwd_kv_blocks(q0, s.n, s.c, o.BM, o.BN);
      for (int kb = 0; kb < nkb; ++kb) {
        const int cls = tile_class(q0, kb * o.BN, o.BM, o.BN, s.n, s.c, s.h_end);
        if (!cls) continue;
        const int slot = atomicAdd(p.hdr + WS_NTILES, 1);
        if (slot < cap) {
          int32_t* r = rec + (int64_t)slot * 6;
          r[0] = blk.b; r[1] = blk.blk; r[2] = kb; r[3] = cls; r[4] = o.BM; r[5] = o.BN;
        }
      }
    } else {
      const int k0 = blk.blk * o.BN;
      const int nqb = (s.n + o.BM - 1) / o.BM;
      for (int qb = bwd_q_begin(k0, s.c, o.BM); qb < nqb; ++qb) {
        const int cls = tile_class(qb * o.BM, k0, o.BM, o.BN, s.n, s.c, s.h_end);
        if (!cls) continue;
        const int slot = atomicAdd(p.hdr + WS_NTILES, 1);
        if (slot < cap) {
          int32_t* r = rec + (int64_t)slot * 6;
          r[0] = blk.b; r[1] = qb; r[2] = blk.blk; r[3] = cls; r[4] = o.BM; r[5] = o.BN;
        }
      }
    }
  }
}

}  // namespace

size_t plan_smem_bytes(const PlanParams& p) {
  size_t bytes = sizeof(int) * kCostBins;
  // every region a multiple of 16 bytes, so the 16-byte block records stay aligned
  if (p.stage_off)
    bytes += sizeof(int64_t) * ((p.B + 2) & ~1) + sizeof(int) * ((p.B + 1 + 3) & ~3) +
             sizeof(int64_t) * ((p.B + 1) & ~1) + 2 * sizeof(int32_t) * ((p.B + 3) & ~3);
  if (p.stage_rec) bytes += sizeof(Block) * (size_t)p.cap_blocks;
  return bytes;
}

cudaError_t launch_plan(const PlanParams& p_in, cudaStream_t stream) {
  PlanParams p = p_in;
  p.stage_off = p.B + 1 <= kPlanStageSeqs;
  p.stage_rec = p.cap_blocks <= kPlanStageBlocks;
  const size_t smem = plan_smem_bytes(p);
  cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  plan_kernel<<<p.npass == 2 ? 2 : 1, kPlanThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_debug_tiles(const PlanParams& p, int32_t* rec, int64_t cap, cudaStream_t stream) {
  debug_tiles_kernel<<<64, 256, 0, stream>>>(p, rec, cap);
  return cudaGetLastError();
}

}  // namespace hstu
