// Device tile planner.
//
// One CTA validates the jagged metadata, lists every query block (forward) or
// key block (backward) of every sequence, counts the tiles of each block that
// the compound mask does not skip, and orders the blocks longest-first
// (counting sort on the tile count), so a persistent grid that takes blocks in
// order gets an LPT-style balance.  This is the "greedy even core split" and
// "compound-mask skipping" of the Ascend HSTU fused operator (wmrh.cn RecSDK
// page, "HSTU acceleration operator" paragraph), done on the device so no
// host synchronisation is needed.
#include "hstu_internal.h"

namespace hstu {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kOffStage = 2048;  // sequence offsets staged in shared memory (B + 1 <= this)
constexpr int kUnroll = 8;       // tokens per thread in flight in the timestamp check

__device__ int block_scan_exclusive(int v, int* sh) {
  // inclusive scan of v over the CTA, returns the exclusive prefix; sh holds
  // kPlanThreads ints; the CTA total is left in sh[kPlanThreads - 1]
  const int t = threadIdx.x;
  sh[t] = v;
  __syncthreads();
  for (int off = 1; off < kPlanThreads; off <<= 1) {
    int x = t >= off ? sh[t - off] : 0;
    __syncthreads();
    sh[t] += x;
    __syncthreads();
  }
  return sh[t] - v;
}

__device__ int block_cost(const SeqInfo& s, int blk, int pass, int BM, int BN) {
  int cost = 0;
  if (pass == 0) {
    const int q0 = blk * BM;
    const int nkb = fwd_kv_blocks(q0, s.n, s.c, BM, BN);
    for (int kb = 0; kb < nkb; ++kb) cost += tile_class(q0, kb * BN, BM, BN, s.n, s.c, s.h_end) != 0;
  } else {
    const int k0 = blk * BN;
    const int nqb = (s.n + BM - 1) / BM;
    for (int qb = bwd_q_begin(k0, s.c, BM); qb < nqb; ++qb)
      cost += tile_class(qb * BM, k0, BM, BN, s.n, s.c, s.h_end) != 0;
  }
  return cost;
}

__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(PlanParams p) {
  __shared__ int sh_scan[kPlanThreads];
  __shared__ int sh_hist[kCostBins];
  __shared__ int sh_bad;
  __shared__ int64_t sh_off[kOffStage];
  const int t = threadIdx.x;
  if (t == 0) {
    p.hdr[WS_ERR] = 0;
    p.hdr[WS_ERR_INFO] = 0;
    p.hdr[WS_NBLK] = 0;
    p.hdr[WS_NTILES] = 0;
    p.hdr[WS_FLAGS] = 0;
    p.hdr[WS_NEXT] = 0;
    sh_bad = 0;
  }
  for (int i = t; i < kCostBins; i += kPlanThreads) sh_hist[i] = 0;
  __syncthreads();

  // 1. validation
  if (t == 0 && (p.off[0] != 0 || p.off[p.B] != p.T)) atomicExch(&sh_bad, 1);
  for (int b = t; b < p.B; b += kPlanThreads) {
    const int64_t n = p.off[b + 1] - p.off[b];
    const int64_t m = p.nt ? p.nt[b] : 0, c = p.nc ? p.nc[b] : 0;
    if (n < 0 || n > p.max_n || m < 0 || c < 0 || m + c > n) {
      if (atomicExch(&sh_bad, 1) == 0) p.hdr[WS_ERR_INFO] = b;
    }
  }
  __syncthreads();
  if (sh_bad) {
    if (t == 0) atomicCAS(p.hdr + WS_ERR, 0, HSTU_ERR_DEVICE_CHECK);
    return;
  }

  // 1b. can every timestamp be held relative to its sequence's first token in
  // 31 bits (so gaps fit in 32)?  Otherwise the kernels take their 64-bit path.
  // Token-parallel: each thread finds its tokens' sequences by binary search
  // over the offsets (staged in shared memory when they fit), kUnroll tokens
  // at a time so their loads overlap.
  if (p.ts) {
    const bool staged = p.B + 1 <= kOffStage;
    if (staged)
      for (int i = t; i <= p.B; i += kPlanThreads) sh_off[i] = p.off[i];
    __syncthreads();
    int wide = 0;
    for (int64_t base = t; base < p.T; base += (int64_t)kPlanThreads * kUnroll) {
      int64_t first[kUnroll], here[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t tok = base + (int64_t)u * kPlanThreads;
        first[u] = here[u] = 0;
        if (tok < p.T) {
          // the last b with off[b] <= tok (skips empty sequences)
          int lo = 0, hi = p.B - 1;
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            const int64_t o = staged ? sh_off[mid] : p.off[mid];
            if (o <= tok) lo = mid; else hi = mid - 1;
          }
          first[u] = p.ts[staged ? sh_off[lo] : p.off[lo]];
          here[u] = p.ts[tok];
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t d = here[u] - first[u];
        wide |= (d >= (int64_t)1 << 30 || d < -((int64_t)1 << 30));
      }
    }
    if (__syncthreads_or(wide) && t == 0) atomicOr(p.hdr + WS_FLAGS, WS_FLAG_WIDE_TS);
  }

  // 2. blocks per sequence -> exclusive prefix (seq_start[b]), chunked scan
  const int BR = p.pass == 0 ? p.BM : p.BN;  // rows per block of this pass
  int carry = 0;
  for (int base = 0; base < p.B; base += kPlanThreads) {
    const int b = base + t;
    int nb = 0;
    if (b < p.B) nb = (int)((p.off[b + 1] - p.off[b] + BR - 1) / BR);
    const int ex = block_scan_exclusive(nb, sh_scan);
    if (b < p.B) p.seq_start[b] = carry + ex;
    const int total = sh_scan[kPlanThreads - 1];
    __syncthreads();
    carry += total;
  }
  const int nblk = carry;
  if (t == 0) p.seq_start[p.B] = nblk;
  if (nblk > p.cap_blocks) {  // cannot happen when off[B] == T; guard anyway
    if (t == 0) atomicCAS(p.hdr + WS_ERR, 0, HSTU_ERR_DEVICE_CHECK);
    return;
  }
  __syncthreads();

  // 3. cost of every block, histogram of costs
  for (int idx = t; idx < nblk; idx += kPlanThreads) {
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.seq_start[mid] <= idx) lo = mid; else hi = mid - 1;
    }
    // skip empty sequences sharing the same start
    const int b = lo;
    const SeqInfo s = seq_info(p.off, p.nt, p.nc, b);
    const int blk = idx - p.seq_start[b];
    const int cost = block_cost(s, blk, p.pass, p.BM, p.BN);
    Block rec;
    rec.b = b; rec.blk = blk; rec.cost = cost; rec.pad = 0;
    p.tmp[idx] = rec;
    atomicAdd(&sh_hist[cost < kCostBins ? cost : kCostBins - 1], 1);
  }
  __syncthreads();

  // 4. exclusive scan of the histogram in descending cost order
  {
    constexpr int per = kCostBins / kPlanThreads;
    int local[per];
    int sum = 0;
    for (int r = 0; r < per; ++r) {
      local[r] = sh_hist[kCostBins - 1 - (t * per + r)];
      sum += local[r];
    }
    const int ex = block_scan_exclusive(sum, sh_scan);
    __syncthreads();
    int run = ex;
    for (int r = 0; r < per; ++r) {
      sh_hist[kCostBins - 1 - (t * per + r)] = run;  // start of this bin
      run += local[r];
    }
  }
  __syncthreads();

  // 5. scatter into longest-first order
  for (int idx = t; idx < nblk; idx += kPlanThreads) {
    const Block rec = p.tmp[idx];
    const int pos = atomicAdd(&sh_hist[rec.cost < kCostBins ? rec.cost : kCostBins - 1], 1);
    p.blocks[pos] = rec;
  }
  if (t == 0) p.hdr[WS_NBLK] = nblk;
}

// Lists every non-skipped tile of every planned block, walking the blocks the
// same way the kernels do.  Record: b, q_block, k_block, class, query edge,
// key edge.
__global__ void debug_tiles_kernel(PlanParams p, int32_t* rec, int64_t cap) {
  const int nblk = p.hdr[WS_NBLK];
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < nblk; idx += gridDim.x * blockDim.x) {
    const Block blk = p.blocks[idx];
    const SeqInfo s = seq_info(p.off, p.nt, p.nc, blk.b);
    if (p.pass == 0) {
      const int q0 = blk.blk * p.BM;
      const int nkb = fwd_kv_blocks(q0, s.n, s.c, p.BM, p.BN);
      for (int kb = 0; kb < nkb; ++kb) {
        const int cls = tile_class(q0, kb * p.BN, p.BM, p.BN, s.n, s.c, s.h_end);
        if (!cls) continue;
        const int slot = atomicAdd(p.hdr + WS_NTILES, 1);
        if (slot < cap) {
          int32_t* r = rec + (int64_t)slot * 6;
          r[0] = blk.b; r[1] = blk.blk; r[2] = kb; r[3] = cls; r[4] = p.BM; r[5] = p.BN;
        }
      }
    } else {
      const int k0 = blk.blk * p.BN;
      const int nqb = (s.n + p.BM - 1) / p.BM;
      for (int qb = bwd_q_begin(k0, s.c, p.BM); qb < nqb; ++qb) {
        const int cls = tile_class(qb * p.BM, k0, p.BM, p.BN, s.n, s.c, s.h_end);
        if (!cls) continue;
        const int slot = atomicAdd(p.hdr + WS_NTILES, 1);
        if (slot < cap) {
          int32_t* r = rec + (int64_t)slot * 6;
          r[0] = blk.b; r[1] = qb; r[2] = blk.blk; r[3] = cls; r[4] = p.BM; r[5] = p.BN;
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream) {
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_debug_tiles(const PlanParams& p, int32_t* rec, int64_t cap, cudaStream_t stream) {
  debug_tiles_kernel<<<64, 256, 0, stream>>>(p, rec, cap);
  return cudaGetLastError();
}

}  // namespace hstu
