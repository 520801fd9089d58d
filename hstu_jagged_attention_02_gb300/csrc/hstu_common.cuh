// Device-side pieces shared by every HSTU kernel: the compound mask, the
// position/time buckets, tile classification, the planner's block records and
// the workspace header.
//
// Mask and buckets follow the HSTU spatial-aggregation step (ai6s.net survey,
// section 2.1.2, eq. (2) and the ranking-task candidate rule) and the compound
// causal + context/target mask of the Ascend HSTU fused operator (wmrh.cn
// RecSDK page, "HSTU acceleration operator" paragraph).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "hstu_attn.h"  // include/ is on the include path

namespace hstu {

// ---------------------------------------------------------------- workspace
// int32 words at the start of every workspace
enum : int {
  WS_ERR = 0,       // first device error code (hstu_status_t), 0 = none
  WS_NBLK = 1,      // number of planner blocks of the current pass
  WS_ERR_INFO = 2,  // detail of the first error (sequence index or wait site)
  WS_NTILES = 3,    // debug-plan tile counter
  WS_FLAGS = 4,     // reserved (zero)
  WS_NEXT = 5,      // next work item of the tensor-core kernels (dynamic scheduling)
  WS_LAYER_ERR = 6, // layer input projection: first device error code (raised into WS_ERR later)
  WS_LAYER_INFO = 7,
  // the backward's tile plan kept by a forward called with HSTU_FLAG_PLAN_BWD
  // (second plan region of the workspace) and what it was made for
  WS_PB_VALID = 8,  // kKeptPlanValid while the kept plan is valid; every other planner launch clears it
  WS_PB_NBLK = 9,   // its block count
  WS_PB_B = 10,     // sequences
  WS_PB_T_LO = 11,  // tokens, low and high 32 bits
  WS_PB_T_HI = 12,
  WS_PB_TILE = 13,  // query-tile rows | key-tile rows << 16
  WS_PB_MAXN = 14,  // max_seq_len the metadata was validated against
};
// error detail (WS_ERR_INFO) of a backward whose kept plan does not match
constexpr int kPlanMismatchInfo = -1;
// Timestamps are staged relative to their sequence's first token; a tile
// whose relative times all lie within +-2^30 s computes its gaps in 32 bits,
// any other tile takes the 64-bit path.
constexpr int64_t kNarrowTsSpan = (int64_t)1 << 30;
__device__ __forceinline__ bool ts_wide(int64_t rel) { return rel >= kNarrowTsSpan || rel <= -kNarrowTsSpan; }
constexpr size_t kWsHeaderBytes = 256;
constexpr size_t kWsAlign = 256;
constexpr int kCostBins = 4096;  // planner histogram bins (cost = tiles per block)

// A planner block: one query block (forward) or one key block (backward) of
// one sequence; every head of it is a separate work item.
struct __align__(16) Block {
  int b;     // sequence
  int blk;   // block index within the sequence (rows blk*BM.. or cols blk*BN..)
  int cost;  // tiles that are not skipped
  int pad;
};

// The work-item record the planner writes for the tensor-core kernels, in
// longest-first order: everything a producer needs about an item in one
// 48-byte load (the sequence's first token and its timestamp, the counts,
// and for the delta forward the sequence's cached tokens).
struct __align__(16) PlanItem {
  int64_t s0;     // first token of the sequence (candidates' first token for the delta forward)
  int64_t tbase;  // timestamp of that token, 0 without timestamps
  int64_t cs0;    // delta forward: first cached token of the sequence
  int b, blk;     // sequence, block index within it
  int n, c, h_end;
  int L;          // delta forward: cached tokens of the sequence
};

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while its predecessor in the
// stream still runs; pdl_wait() blocks until the predecessor has completed
// and its memory is visible (it returns at once without such a predecessor).
// pdl_launch_dependents() lets the dependent start before this grid ends.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void set_error(int* hdr, int code, int info) {
  if (atomicCAS(hdr + WS_ERR, 0, code) == 0) hdr[WS_ERR_INFO] = info;
}

// -------------------------------------------------------------------- mask
// A sequence of n tokens: c context tokens, then history, then candidates
// from h_end = n - num_targets on.
__host__ __device__ __forceinline__ bool allowed(int i, int j, int c, int h_end) {
  return j >= h_end ? (i == j) : (j <= i || (i < c && j < c));
}

// Class of the BM x BN tile [q0, q0+BM) x [k0, k0+BN): 0 = no allowed
// in-sequence pair (skipped), 2 = every pair in the sequence and allowed,
// 1 = otherwise.  Exact interval reasoning on the mask above.
__host__ __device__ __forceinline__ int tile_class(int q0, int k0, int BM, int BN, int n, int c,
                                                   int h_end) {
  const int q1 = q0 + BM, k1 = k0 + BN;
  const int q1n = q1 < n ? q1 : n, k1n = k1 < n ? k1 : n;
  if (q0 >= q1n || k0 >= k1n) return 0;
  // full: all rows and columns inside, no candidate column, and every pair
  // causal or inside the context block
  if (q1 <= n && k1 <= h_end && (k1 - 1 <= q0 || k1 <= c)) return 2;
  // any allowed pair?
  const int kh = k1n < h_end ? k1n : h_end;          // history/context columns [k0, kh)
  const bool causal_any = k0 < kh && k0 <= q1n - 1;    // some j <= i with j < h_end
  const bool ctx_any = q0 < c && k0 < c;               // i < c and j < c
  int lo = q0 > k0 ? q0 : k0;
  lo = lo > h_end ? lo : h_end;
  int hi = q1n < k1n ? q1n : k1n;
  const bool diag_any = lo < hi;                       // candidate diagonal i == j >= h_end
  return (causal_any || ctx_any || diag_any) ? 1 : 0;
}

// Forward: the key blocks a query block may see are [0, fwd_kv_blocks).
__host__ __device__ __forceinline__ int fwd_kv_blocks(int q0, int n, int c, int BM, int BN) {
  int hi = q0 + BM < n ? q0 + BM : n;
  if (q0 < c && c > hi) hi = c;
  return (hi + BN - 1) / BN;
}

// Backward: the query blocks that may see key block k0 are
// [bwd_q_begin, ceil(n / BM)).
__host__ __device__ __forceinline__ int bwd_q_begin(int k0, int c, int BM) {
  return k0 < c ? 0 : k0 / BM;
}

// ----------------------------------------------------------------- buckets
__device__ __forceinline__ int pos_bucket(int i, int j, int h_end, int P) {
  int pi = i < h_end ? i : h_end;
  int pj = j < h_end ? j : h_end;
  int d = pi > pj ? pi - pj : pj - pi;
  return d < P - 1 ? d : P - 1;
}

// 0 for equal times, else floor(log2 |ti - tj|) + 1 (the bit length of the
// gap), clamped to Tb - 1.
__device__ __forceinline__ int time_bucket(int64_t ti, int64_t tj, int Tb) {
  uint64_t d = ti >= tj ? (uint64_t)ti - (uint64_t)tj : (uint64_t)tj - (uint64_t)ti;
  int bits = 64 - __clzll((long long)d);
  return bits < Tb - 1 ? bits : Tb - 1;
}

// ------------------------------------------------------------ element I/O
template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Per-sequence metadata of a block.
struct SeqInfo {
  int64_t s0;  // first token
  int n, c, h_end;
};

__device__ __forceinline__ SeqInfo seq_info(const int64_t* off, const int32_t* nt, const int32_t* nc,
                                            int b) {
  SeqInfo s;
  s.s0 = off[b];
  s.n = (int)(off[b + 1] - s.s0);
  s.c = nc ? nc[b] : 0;
  s.h_end = s.n - (nt ? nt[b] : 0);
  return s;
}

}  // namespace hstu
