// Internal launch interfaces between the C ABI (hstu_api.cu) and the kernels.
#pragma once

#include <cuda.h>

#include <utility>

#include "hstu_common.cuh"

namespace hstu {

// Where one pass of the planner writes its plan.
struct PlanOut {
  int pass;         // 0 forward (query blocks), 1 backward (key blocks), 2 delta forward (candidate blocks)
  int BM, BN;       // tile edges of the path that will run
  int* seq_start;   // [B+1] scratch
  Block* tmp;       // [cap_blocks] scratch
  Block* blocks;    // [cap_blocks] result, longest first
  PlanItem* items;  // [cap_blocks] the same blocks as full item records (tensor-core kernels)
};

struct PlanParams {
  const int64_t* off;
  const int32_t* nt;
  const int32_t* nc;
  const int64_t* ts;  // timestamps or NULL (span check only)
  int B;
  int64_t T;
  int max_n;
  const int64_t* off2;  // pass 2: cached-token offsets [B+1] (off: candidate offsets)
  int64_t T2;           // pass 2: cached tokens
  int* hdr;         // workspace header
  int cap_blocks;
  // 1: one CTA plans out[0].  2: a second CTA plans out[1] (the backward) at
  // the same time and keeps it for a later backward: the WS_PB_* header words
  // and the metadata below record what it was made from.
  int npass;
  PlanOut out[2];
  int64_t* sv_off;  // npass 2: [B+1] offsets
  int64_t* sv_t0;   // [B] timestamp of each sequence's first token (0 without timestamps or tokens)
  int32_t* sv_nt;   // [B] targets (0 when num_targets is NULL)
  int32_t* sv_nc;   // [B] contexts (0 when num_contexts is NULL)
  int stage_off;    // set by launch_plan: offsets and block starts staged in shared memory
  int stage_rec;    // set by launch_plan: block records staged in shared memory
};
// WS_PB_VALID while a kept backward plan is valid: a value that fresh or
// reused workspace memory is unlikely to hold by chance
constexpr int kKeptPlanValid = 0x4b505431;
// planner shared-memory staging limits (sequences, blocks)
constexpr int kPlanStageSeqs = 2048;
constexpr int kPlanStageBlocks = 8192;

// Everything a forward or backward attention kernel needs.
struct AttnParams {
  const int64_t* off;
  const int32_t* nt;
  const int32_t* nc;
  const int64_t* ts;     // NULL: no time bias
  const float* rab_pos;  // NULL: no position bias
  const float* rab_time; // NULL (or ts NULL): no time bias
  const void* q;
  const void* k;
  const void* v;
  void* o;               // forward output [T,H,dv]
  const void* dO;        // backward: gradient w.r.t. o [T,H,dv]
  void* dk;              // backward outputs [T,H,d]
  void* dv;
  float* dq_acc;         // backward: FP32 accumulator [T,H,dqk], zeroed before
  float* d_rab_pos;      // backward: [H,P] accumulated (zeroed before), or NULL
  float* d_rab_time;
  float* drab_partial;   // tensor-core backward: [kDrabMaxCtas][H][P+Tb] per-CTA partial sums
  const int* hdr;        // workspace header (block count)
  int* hdr_rw;           // same, writable (error word)
  const Block* blocks;
  const PlanItem* items;  // the planner's item records, same order as blocks
  // delta forward (KV-cached candidates): cached-token offsets [B+1], times
  // [T2] (or NULL) and K, V [T2, H, d]; q, k, v, o above are the candidates'
  const int64_t* off2;
  const int64_t* ts2;
  const void* k2;
  const void* v2;
  int64_t T2;
  int B, H, dqk, dv_dim;
  int dtype, out_dtype;  // hstu_dtype_t of the inputs / of the outputs
  int64_t T;
  float alpha, inv_n;
  // score constants of the tensor-core epilogues (w = -log2(e) z):
  // kA = -log2(e) alpha, kC = -1 / (log2(e) N), kZ = -1 / log2(e), kCi = 1 / kC
  float kA, kC, kZ, kCi;
  int P, Tb;
  uint32_t flags;
  int num_sms;
  // the same constants as lane pairs, for paired (f32x2) arithmetic
  float2 kA2, kC2, kZ2, kCi2, inv_n2;
};

struct NormParams {
  int dtype, out_dtype;  // u and dO have dtype; o, y, dy, du have out_dtype
  const void* o;
  const void* u;   // NULL: gate of one
  const void* dy;
  void* y;
  void* dO;        // backward: gradient w.r.t. o, FP32 [T, F] (split == 0) or the BF16 high part
  void* dO_lo;     // backward, split == 1: BF16 low part, dO ~= hi + lo
  int split;
  void* du;
  float* mean;
  float* rstd;
  // backward only, or NULL: FP32 buffers the kernel zeroes on the way (the
  // tensor-core backward's dq accumulator [T, zero_F], and the two d_rab tables)
  float* zero_rows;
  int zero_F;
  float* zero_a;
  int zero_a_n;
  float* zero_b;
  int zero_b_n;
  // fused dropout on y (forward) / dy (backward): keep iff the element's
  // Philox4x64-10 word >= drop_thr, kept values times drop_scale
  int drop;
  uint32_t drop_thr;
  float drop_scale;
  uint64_t drop_seed, drop_offset;
  int64_t T;
  int F;           // H * d_v
  int norm;
  float eps;
  // backward with a kept plan (HSTU_FLAG_REUSE_PLAN): one warp checks that
  // the plan in the workspace was made for this call's descriptor and
  // metadata, then arms it for the attention backward (block count, work
  // counter), or records HSTU_ERR_DEVICE_CHECK and leaves it no work
  int* pc_hdr;     // workspace header, or NULL (no check)
  const int64_t* pc_off;
  const int32_t* pc_nt;
  const int32_t* pc_nc;
  const int64_t* pc_ts;
  const int64_t* pc_sv_off;
  const int64_t* pc_sv_t0;
  const int32_t* pc_sv_nt;
  const int32_t* pc_sv_nc;
  int pc_B;
  int pc_tile;     // query-tile rows | key-tile rows << 16 of the backward this call runs
  int pc_max_n;
};

// Diagnostics behind HSTU_ERR_CUDA (read with hstu_last_error_detail):
// the failing call, or the kernel launch with its resource attributes.
void set_error_detail(cudaError_t e, const char* where);
void set_launch_detail(cudaError_t e, const char* kernel, const void* func, int threads, size_t smem);
void set_detail_message(const char* msg);
// adds n kernels of a composite call (the layer) to hstu_last_launch_count
void note_launches(int32_t n);

// Launches kernel<<<grid, block, smem, st>>>(args...) with programmatic
// stream serialization: it may start while the previous kernel in the stream
// runs, and must call pdl_wait() before it reads that kernel's outputs or
// writes what that kernel reads.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream);
cudaError_t launch_debug_tiles(const PlanParams& p, int32_t* rec, int64_t cap, cudaStream_t stream);

// CUDA-core path (FP32 and BF16), 32 x 32 tiles
constexpr int kSimtTile = 32;
cudaError_t launch_simt_fwd(const AttnParams& p, int max_items, cudaStream_t stream);
cudaError_t launch_simt_bwd(const AttnParams& p, int max_items, cudaStream_t stream);

// norm + gate, forward and backward; dq FP32 -> dtype
cudaError_t launch_norm_gate_fwd(const NormParams& p, cudaStream_t stream);
cudaError_t launch_norm_gate_bwd(const NormParams& p, cudaStream_t stream);
cudaError_t launch_convert_f32(const float* src, void* dst, int64_t count, int dtype, cudaStream_t stream);

// Tensor-core path (BF16): forward d in {64, 128} on 128 x 128 tiles;
// backward d = 128 on 64 (query) x 128 (key) tiles
constexpr int kTcTile = 128;
constexpr int kTcBwdQTile = 64;
constexpr int kDrabMaxCtas = 256;  // tensor-core backward grid cap (one d_rab partial row each)
bool make_tmap_bf16(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int box_rows);
bool make_tmap_tile(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* ptr, const uint64_t* dims,
                    const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle sw);
size_t tc_bwd_smem_bytes(int H, int P, int Tb);
bool tc_fwd_supported(int dtype, int dqk, int dv);
size_t tc_fwd_smem_bytes(int d, int H, int P, int Tb);
constexpr size_t kMaxSmemPerCta = 227 * 1024;
bool tc_bwd_supported(int dtype, int dqk, int dv);
cudaError_t launch_tc_fwd(const AttnParams& p, cudaStream_t stream);
// delta forward: candidate blocks against cached K/V (p.off2, p.ts2, p.k2, p.v2, p.T2)
cudaError_t launch_tc_fwd_delta(const AttnParams& p, cudaStream_t stream);
cudaError_t launch_tc_bwd(const AttnParams& p, cudaStream_t stream);

// Tensor-core GEMMs of the layer with fused epilogues (BF16 operands, FP32
// accumulation).  C [M, N] = sum over passes of A_p B_p, A [M, K], B [K, N];
// A is read K-major (a row-major [M, K] array) or MN-major (a row-major
// [K, M] array, i.e. the transpose of a stored matrix), B MN-major (row-major
// [K, N]) or K-major (row-major [N, K]).  M % 128 == 0 unless the output rows
// are clipped (row-major outputs), N % 128 == 0; K needs no alignment (the
// last 64-block is zero-filled).
struct GemmParams {
  int64_t M;
  int N;
  int64_t K;
  int D;
  int npass;            // passes over K into one accumulator: the two halves of a BF16 operand pair
  int pair_b;           // 0: pass p reads A_p (and B_0); 1: pass p reads B_p (and A_0)
  int ksplit;           // K cut into ksplit ranges of whole 64-blocks, one work item each (reduce epilogue)
  int test_timeout;     // test only: CTA 0 never loads its first stage; waits give up after ~1 ms
  int* err;             // first error code (HSTU_ERR_TIMEOUT) and its wait site
  int* err_info;
  const int* carry_err; // error words of an earlier GEMM, raised into err at launch (or NULL)
  float* z1;            // f1: [M, 4D] FP32
  float* u;             // f1: [M, D] FP32
  __nv_bfloat16* vqk;   // f1: [3][M][D] BF16 (V, Q, K)
  const __nv_bfloat16* x; // f2: [M, N] BF16 residual
  const float* res;     // FP32 residual [M, N] (dX = dOut + dZ1 W1^T)
  float* out;           // [M, N] FP32 output (stored, residual-added or reduce-added)
};
bool gemm_tc_supported(int D);
// f1: z1 = X W1; u = SiLU(z1[:, :D]); V | Q | K = BF16(SiLU(z1[:, D:]))
cudaError_t launch_gemm_f1(const GemmParams& p, const void* x, const void* w1, int num_sms, cudaStream_t st);
// f2: out = X + y_hi W2 + y_lo W2
cudaError_t launch_gemm_f2(const GemmParams& p, const void* y_hi, const void* y_lo, const void* w2, int num_sms,
                           cudaStream_t st);
// out = A W^T with A [M, K] row-major and W [N, K] row-major (dy = dOut W2^T);
// with res: out = res + sum_p A_p W^T (dX = dOut + dZ1_hi W1^T + dZ1_lo W1^T)
cudaError_t launch_gemm_nt(const GemmParams& p, const void* a0, const void* a1, const void* w, int num_sms,
                           cudaStream_t st);
// out += sum_p L_p^T R_p over K = rows of L and R (L [K, M], R [K, N] row-major),
// split over K: the weight gradients dW2 = y^T dOut and dW1 = X^T dZ1.  out
// must hold its initial value (zero) before the launch.
cudaError_t launch_gemm_tn_reduce(const GemmParams& p, const void* l0, const void* l1, const void* r0,
                                  const void* r1, int num_sms, cudaStream_t st);

}  // namespace hstu
