/*
 * hstu_attn.h -- C ABI of the GB300 (sm_103a) HSTU jagged attention library
 * (libhstu_attn.so).
 *
 * The operation (HSTU "Spatial Aggregation" and "Pointwise Transformation",
 * ai6s.net generative-recommendation survey, section 2.1.2, equations (2)
 * and (3); the equations are images on the page, the prose describes a
 * softmax-free "pointwise aggregated attention" with a position/time bias and
 * a U gate):
 *
 *   for each sequence b and head h, tokens i, j of the sequence:
 *     z_ij = alpha * <q_i, k_j> + rab_pos[h][bp(i,j)] + rab_time[h][bt(i,j)]
 *     o_i  = sum over allowed j of SiLU(z_ij) / N * v_j        (no softmax)
 *   y_t = Norm(concat_h o_t) * u_t
 *
 * Jagged layout (KeyedJaggedTensor convention, same survey, section 3.1.2):
 * tokens of all sequences are packed back to back, row-major, no padding;
 * seq_offsets[b] is the first token of sequence b, seq_offsets[B] == T.
 *   q, k     [T, H, d_qk]     v, o  [T, H, d_v]     u, y, dy, du  [T, H*d_v]
 * Every row is dense and contiguous; every tensor pointer must be 16-byte
 * aligned.  q, k, v, u have the element type `dtype`; o, y, dy and the
 * gradients have `out_dtype` (BF16 inputs with FP32 outputs keep the final
 * rounding out of the result; BF16 outputs halve the output traffic).
 *
 * Mask (the ranking task's candidates, section 2.1.2, and the compound
 * causal + context/target mask of the Ascend HSTU fused operator, wmrh.cn
 * RecSDK page, "HSTU acceleration operator" paragraph).  A sequence of n
 * tokens has c = num_contexts[b] context tokens in front and
 * m = num_targets[b] candidates at the end; h_end = n - m:
 *   j >= h_end : allowed iff i == j
 *   j <  h_end : allowed iff j <= i  or  (i < c and j < c)
 * Buckets: pos(i) = min(i, h_end);  bp = min(|pos(i) - pos(j)|, P - 1);
 *          bt = 0 if t_i == t_j else min(Tb - 1, floor(log2|t_i - t_j|) + 1).
 * Norm:    LAYERNORM normalises each token's H*d_v features (population
 *          variance, eps = ln_eps, no affine); NONE leaves them as they are.
 *
 * Conventions
 *  - Every pointer is a device pointer except the host_* outputs of
 *    hstu_attn_debug_plan and hstu_get_device_error.  The caller owns every
 *    buffer, including the workspace; the library never allocates device
 *    memory and keeps no state between calls.  The one exception is
 *    hstu_attn_fwd_noalloc: it uses a fixed buffer built into the library
 *    in place of a workspace, shared by all its calls on a device (its own
 *    comment gives the size limit and the race between overlapping calls).
 *    What one call leaves in a workspace for a later one is the caller's
 *    to keep: the backward's plan kept with HSTU_FLAG_PLAN_BWD.
 *  - Calls are stream-ordered and return without synchronising, except
 *    hstu_attn_debug_plan and hstu_get_device_error, which synchronise the
 *    given stream.  Concurrent calls must use distinct workspaces.
 *  - Host-side checks return an error code before anything is launched.
 *    Problems seen on the device (inconsistent offsets or counts, a pipeline
 *    wait that ran out) are recorded in the workspace and read back with
 *    hstu_get_device_error; outputs are undefined then.  The library never
 *    traps or aborts.
 */
#ifndef HSTU_ATTN_H_
#define HSTU_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HSTU_ATTN_ABI_VERSION 2

typedef struct CUstream_st* hstu_stream_t; /* same type as cudaStream_t; NULL = legacy default stream */

typedef enum {
  HSTU_OK = 0,
  HSTU_ERR_INVALID_ARG = 1,   /* a NULL required pointer, bad size or misalignment */
  HSTU_ERR_UNSUPPORTED = 2,   /* a valid request this build does not implement */
  HSTU_ERR_WORKSPACE = 3,     /* workspace NULL, misaligned or too small */
  HSTU_ERR_CUDA = 4,          /* a CUDA runtime call failed */
  HSTU_ERR_TIMEOUT = 5,       /* device: a pipeline wait ran out of its limit */
  HSTU_ERR_DEVICE_CHECK = 6   /* device: offsets/counts inconsistent with the descriptor */
} hstu_status_t;

typedef enum { HSTU_BF16 = 0, HSTU_FP32 = 1 } hstu_dtype_t;
typedef enum { HSTU_NORM_NONE = 0, HSTU_NORM_LAYERNORM = 1 } hstu_norm_t;

/* Flags */
#define HSTU_FLAG_FORCE_SIMT (1u << 0)   /* use the CUDA-core kernels even where the tensor-core path applies;
                                            BF16 work the tensor-core kernels do not take (the backward
                                            needs d = 128, the forward d = 64 or 128) runs only with this
                                            flag, else the call returns HSTU_ERR_UNSUPPORTED */
#define HSTU_FLAG_TEST_TIMEOUT (1u << 1) /* test only: the tensor-core forward withholds one load (the
                                            first K/V tile of work item 0) and its waits give up after about
                                            a millisecond, so the timeout path runs without a hang; the
                                            result is HSTU_ERR_TIMEOUT.  In hstu_layer_fwd it applies to the
                                            tensor-core input projection instead (its CTA 0 skips its first
                                            load), and hstu_layer_bwd rejects it */
#define HSTU_FLAG_U_FP32 (1u << 2)       /* u is FP32 whatever dtype is (requires out_dtype FP32).  The
                                            gate multiplies y element by element, so a BF16 rounding of u
                                            is never averaged out; q, k, v stay in dtype */
#define HSTU_FLAG_PLAN_BWD (1u << 3)     /* hstu_attn_fwd only: its planner launch also plans the
                                            backward's tiling (a second CTA of the same launch) and keeps
                                            it in the workspace, which must then have the backward's size */
#define HSTU_FLAG_REUSE_PLAN (1u << 4)   /* hstu_attn_bwd only: launch no planner and use the plan kept by
                                            the last hstu_attn_fwd with HSTU_FLAG_PLAN_BWD on this
                                            workspace.  The backward checks on the device that the plan was
                                            made for the same B, total_tokens, max_seq_len and path, from
                                            the same seq_offsets, num_targets, num_contexts and first
                                            timestamp of every sequence; otherwise it computes nothing and
                                            records HSTU_ERR_DEVICE_CHECK.  A kept plan serves any number of
                                            backward calls until another planner launch on the workspace
                                            (any forward, a backward without this flag, a debug plan)
                                            voids it.  Rejected by the layer, delta and no-alloc calls */

typedef struct {
  uint32_t struct_size;     /* sizeof(hstu_attn_desc) */
  int32_t dtype;            /* hstu_dtype_t of the inputs q, k, v, u */
  int32_t out_dtype;        /* hstu_dtype_t of o, y, dy, dq, dk, dv, du; FP32 when dtype is FP32 */
  int32_t B;                /* number of sequences, >= 0 */
  int32_t H;                /* heads, >= 1 */
  int32_t d_qk, d_v;        /* head dims; this build: d_qk == d_v in {32, 64, 128} */
  int64_t total_tokens;     /* T == seq_offsets[B] */
  int32_t max_seq_len;      /* N of the 1/N scale; every sequence must have n <= N */
  float alpha;              /* scale of <q, k> */
  int32_t num_pos_buckets;  /* P >= 1 (128 in the reference workloads) */
  int32_t num_time_buckets; /* Tb >= 1 (64) */
  int32_t norm;             /* hstu_norm_t */
  float ln_eps;             /* LayerNorm epsilon (1e-5) */
  uint32_t flags;           /* HSTU_FLAG_* */
  float dropout_p;          /* fused dropout on y, 0 <= p < 1 (0: none); see below */
  uint32_t reserved;        /* must be 0 */
} hstu_attn_desc;

/* Fused dropout (ai6s.net survey, section 2.1.3, "memory optimisation":
 * dropout fused with its neighbouring operators).  With dropout_p = p > 0
 * the forward's y becomes dropout(Norm(o) * u) and the backward takes dy as
 * the gradient of that dropped-out y.  The keep decision of element (t, f)
 * of the [T, F] output (F = H * d_v) comes from the counter-based generator
 * Philox4x64-10 (Salmon, Moraes, Dror, Shaw, SC 2011):
 *
 *   e = t F + f;  r = Philox4x64-10(counter (e >> 3, dropout_offset, 0, 0),
 *                                   key (dropout_seed, 0))
 *   w = 32-bit word (e & 7) of r[0..3] (low half of each 64-bit word first)
 *   keep iff w >= floor(p 2^32); kept elements are multiplied by 1 / (1 - p)
 *
 * so the backward regenerates the forward's mask from the same seed and
 * offset (a caller advances the offset, or changes the seed, per step).  The
 * mask does not depend on the batch's split into sequences. */

typedef struct {
  const int64_t* seq_offsets;  /* [B+1], non-decreasing, seq_offsets[0] == 0 */
  const int32_t* num_targets;  /* [B] candidates at the end of each sequence, or NULL (none) */
  const int32_t* num_contexts; /* [B] context tokens at the front, or NULL (none) */
  const int64_t* timestamps;   /* [T] integer seconds, or NULL (no time bias) */
  const float* rab_pos;        /* [H, P] position-bucket bias, or NULL */
  const float* rab_time;       /* [H, Tb] time-bucket bias, or NULL; ignored without timestamps */
  const void* q;               /* [T, H, d_qk] */
  const void* k;               /* [T, H, d_qk] */
  const void* v;               /* [T, H, d_v] */
  const void* u;               /* [T, H*d_v] gate, or NULL (gate of one); FP32 with HSTU_FLAG_U_FP32 */
  void* o;                     /* out [T, H, d_v]: A.V, kept for the backward */
  void* y;                     /* out [T, H*d_v]: Norm(o) * u, or NULL (not produced) */
  float* ln_mean;              /* out [T] or NULL: per-token mean of o (LAYERNORM) */
  float* ln_rstd;              /* out [T] or NULL: per-token 1/sqrt(var + eps) (LAYERNORM) */
  uint64_t dropout_seed;       /* fused dropout (desc->dropout_p > 0): generator key */
  uint64_t dropout_offset;     /* and counter word 1 */
} hstu_attn_fwd_args;

typedef struct {
  /* the forward's inputs, unchanged */
  const int64_t* seq_offsets;
  const int32_t* num_targets;
  const int32_t* num_contexts;
  const int64_t* timestamps;
  const float* rab_pos;
  const float* rab_time;
  const void* q;
  const void* k;
  const void* v;
  const void* u;
  const void* o;               /* the forward's o */
  const void* dy;              /* [T, H*d_v] gradient of the loss w.r.t. y */
  /* outputs, overwritten (not accumulated) */
  void* dq;                    /* [T, H, d_qk] */
  void* dk;                    /* [T, H, d_qk] */
  void* dv;                    /* [T, H, d_v] */
  void* du;                    /* [T, H*d_v]; required iff u != NULL */
  float* d_rab_pos;            /* [H, P] or NULL (not wanted) */
  float* d_rab_time;           /* [H, Tb] or NULL */
  uint64_t dropout_seed;       /* the forward's dropout seed and offset */
  uint64_t dropout_offset;
} hstu_attn_bwd_args;

/* Workspace bytes the forward and the backward need for this descriptor
 * (a bound valid for any seq_offsets consistent with it).  The workspace must
 * be 256-byte aligned.  Either output pointer may be NULL. */
hstu_status_t hstu_attn_workspace_size(const hstu_attn_desc* desc, size_t* fwd_bytes, size_t* bwd_bytes);

/* Forward: o = A.V and, if y != NULL, y = Norm(o) * u (eqs. (2), (3)).
 * One planner launch, the attention kernel and (with y or the statistics) the
 * norm-gate kernel.  With HSTU_FLAG_PLAN_BWD the planner also plans the
 * backward, so a training step (forward, then the backward with
 * HSTU_FLAG_REUSE_PLAN on the same workspace) launches one planner. */
hstu_status_t hstu_attn_fwd(const hstu_attn_desc* desc, const hstu_attn_fwd_args* args,
                            void* workspace, size_t workspace_bytes, hstu_stream_t stream);

/* Backward: dq, dk, dv, du, d_rab_pos, d_rab_time from dy; A is recomputed
 * tile by tile, never stored (HSTU's memory design, section 2.1.3 "memory
 * optimisation": sub-layer activations are not kept). */
hstu_status_t hstu_attn_bwd(const hstu_attn_desc* desc, const hstu_attn_bwd_args* args,
                            void* workspace, size_t workspace_bytes, hstu_stream_t stream);

/* The tile plan of one pass, as the kernels walk it (compound-mask tile
 * skipping, wmrh.cn RecSDK page, "HSTU acceleration operator" paragraph).
 * pass 0 = forward (query-block work items), 1 = backward (key-block items).
 * Writes up to host_capacity records of 6 int32 (b, q_block, k_block, class,
 * q_rows, k_rows) to host_tiles for every tile that is not skipped; class 1 =
 * partial, 2 = full; q_rows x k_rows = the tile shape of the path this
 * descriptor selects (tensor-core or CUDA-core).  *n_tiles receives the total
 * count.  The workspace must hold the forward workspace plus
 * 24 * host_capacity bytes (rounded up to 256).  Synchronises the stream. */
hstu_status_t hstu_attn_debug_plan(const hstu_attn_desc* desc, const int64_t* seq_offsets,
                                   const int32_t* num_targets, const int32_t* num_contexts, int32_t pass,
                                   void* workspace, size_t workspace_bytes, int32_t* host_tiles,
                                   int64_t host_capacity, int64_t* n_tiles, hstu_stream_t stream);

/* Forward without a caller workspace, for callers that are not allowed to
 * allocate device memory (a framework that owns all device memory through its
 * own pool, a latency-bound server that cannot afford an allocation, an
 * integration with no allocator at hand).  The pages describe no counterpart;
 * this is a library convenience.
 *
 * Same operation, arguments and outputs as hstu_attn_fwd; the caller still
 * passes every input and output buffer.  The scratch comes from a 1 MiB
 * buffer built into the library (every GPU that loads the library holds it
 * until the process exits).  The plan of T tokens in B sequences needs
 * 256 + 4 (B + 1) + 80 (ceil(T / 32) + B) bytes (each part rounded up to
 * 256), roughly 2.5 T + 84 B + 1 KiB, which must fit in 1 MiB: e.g. 250,000
 * tokens in 4,000 sequences.  Larger problems return HSTU_ERR_WORKSPACE
 * (hstu_last_error_detail says how much was needed) without launching.
 *
 * Each call looks up the buffer's device address (cudaGetSymbolAddress) with
 * the current device, which must be the stream's device (else
 * HSTU_ERR_INVALID_ARG).  The address is not cached, so a device reset
 * between calls does not leave a stale pointer behind.  The first call on a
 * device may load the library's device code, so make that first call before
 * any stream capture.  Every call shares the one buffer: calls that may
 * overlap on the GPU (other streams, other host threads) race and must be
 * serialised by the caller.  The buffer keeps the last call's contents; the
 * planner rewrites everything it reads on every call.
 *
 * host_device_error: NULL, or a host int32 that receives the call's device
 * error code (as hstu_get_device_error reports it); non-NULL makes the call
 * synchronise the stream. */
hstu_status_t hstu_attn_fwd_noalloc(const hstu_attn_desc* desc, const hstu_attn_fwd_args* args,
                                    hstu_stream_t stream, int32_t* host_device_error);

/* ------------------------------------------------------------------------
 * The full HSTU layer around the attention (ai6s.net survey, section 2.1.2,
 * equations (1)-(3), with the residual connection between layers; section
 * 2.1.3: two linear layers per block).  With D = H * d_v (= H * d_qk):
 *
 *   Z1 = X W1                                   [T, 4D]  (FP32 accumulation)
 *   U | V | Q | K = SiLU(Z1), column blocks of width D in that order
 *   o, y = attention(Q, K, V, U) as in hstu_attn_fwd (y = Norm(o) * U)
 *   out  = X + y W2                             [T, D]
 *
 * Precision: X, W1, W2 BF16; V, Q, K = SiLU(Z1) are rounded to BF16 (the
 * attention's MMA operands) while the gate U stays FP32 (it scales y element
 * by element, where a rounding is never averaged out).  The computed GEMM
 * operands y (y W2, y^T dout) and dZ1 (X^T dZ1, dZ1 W1^T) enter as BF16
 * pairs hi + lo (about 16 bits, two accumulating GEMMs each); dout is
 * rounded to BF16 for dout W2^T and y^T dout.  Every accumulation, o, y,
 * out, dx and all gradients are FP32.  The descriptor is the
 * attention's and must have dtype BF16, out_dtype FP32, d_qk == d_v.
 *
 * When D is a multiple of 128 the forward's two projections are this
 * library's tensor-core GEMMs: Z1 = X W1 with the SiLU split in its epilogue
 * (z1, U, V, Q, K written once), and out = X + y_hi W2 + y_lo W2 with the
 * residual in its epilogue.  Otherwise, and for the backward's GEMMs, they
 * are plain cuBLAS GEMMs (BF16 x BF16 -> FP32) around this library's
 * element-wise kernels.  cuBLAS's scratch comes from the caller's
 * workspace, but the first call on each (host thread, device) that uses
 * cuBLAS creates a cuBLAS handle, which allocates cuBLAS's own small state:
 * make that first call outside any stream capture.
 * ------------------------------------------------------------------------ */
typedef struct {
  const int64_t* seq_offsets;  /* as hstu_attn_fwd_args */
  const int32_t* num_targets;
  const int32_t* num_contexts;
  const int64_t* timestamps;
  const float* rab_pos;
  const float* rab_time;
  const void* x;               /* [T, D] BF16 layer input */
  const void* w1;              /* [D, 4D] BF16, row-major (x W1) */
  const void* w2;              /* [D, D] BF16, row-major (y W2) */
  float* out;                  /* out [T, D] FP32: x + y W2 */
  float* z1;                   /* out [T, 4D] FP32: x W1, kept for the backward */
  float* u;                    /* out [T, D] FP32: the gate U */
  void* vqk;                   /* out [3, T, D] BF16: V, Q, K, each [T, H, d] */
  void* o;                     /* out [T, D] FP32: A.V, kept for the backward */
  void* y;                     /* out [T, D] FP32: Norm(o) * U (dropped out when desc->dropout_p > 0) */
  uint64_t dropout_seed;       /* fused dropout on y, as hstu_attn_fwd_args */
  uint64_t dropout_offset;
} hstu_layer_fwd_args;

typedef struct {
  const int64_t* seq_offsets;  /* the forward's inputs, unchanged */
  const int32_t* num_targets;
  const int32_t* num_contexts;
  const int64_t* timestamps;
  const float* rab_pos;
  const float* rab_time;
  const void* x;
  const void* w1;
  const void* w2;
  const float* z1;             /* the forward's z1, u, vqk, o, y */
  const float* u;
  const void* vqk;
  const void* o;
  const void* y;
  const float* dout;           /* [T, D] FP32 gradient of the loss w.r.t. out */
  float* dx;                   /* out [T, D]: dout + dZ1 W1^T */
  float* dw1;                  /* out [D, 4D]: X^T dZ1 */
  float* dw2;                  /* out [D, D]: y^T dout */
  float* d_rab_pos;            /* out [H, P] or NULL */
  float* d_rab_time;           /* out [H, Tb] or NULL */
  uint64_t dropout_seed;       /* the forward's dropout seed and offset */
  uint64_t dropout_offset;
} hstu_layer_bwd_args;

/* Workspace bytes of hstu_layer_fwd / hstu_layer_bwd (256-byte aligned
 * workspace; either output may be NULL).  HSTU_ERR_UNSUPPORTED unless dtype
 * is BF16, out_dtype FP32 and D a multiple of 8. */
hstu_status_t hstu_layer_workspace_size(const hstu_attn_desc* desc, size_t* fwd_bytes, size_t* bwd_bytes);

/* Layer forward (above).  All pointers device, 16-byte aligned; outputs are
 * overwritten.  Device-side problems (the attention's, or a tensor-core
 * projection's wait that ran out: HSTU_ERR_TIMEOUT) land in the error word
 * at the start of the workspace (hstu_get_device_error). */
hstu_status_t hstu_layer_fwd(const hstu_attn_desc* desc, const hstu_layer_fwd_args* args,
                             void* workspace, size_t workspace_bytes, hstu_stream_t stream);

/* Layer backward: dx, dw1, dw2 and the bias-table gradients, recomputing the
 * attention tile by tile from the saved u, vqk and o.  All pointers device,
 * 16-byte aligned; outputs are overwritten.  With D % 128 == 0 the four
 * GEMMs run on the library's tensor-core kernels: dw1 and dw2 are then sums
 * over ranges of tokens added in no fixed order (FP32 rounding may differ
 * from call to call); otherwise on cuBLAS.  A tensor-core GEMM's wait that
 * runs out is reported as HSTU_ERR_TIMEOUT in the workspace's error word. */
hstu_status_t hstu_layer_bwd(const hstu_attn_desc* desc, const hstu_layer_bwd_args* args,
                             void* workspace, size_t workspace_bytes, hstu_stream_t stream);

/* ------------------------------------------------------------------------
 * Delta forward: KV-cached, candidate-only inference (P2 "HSTU acceleration
 * operator" paragraph: variable-length sequences with a KV cache; P1 section
 * 2.1.2: the ranking task scores all candidates of a request in one pass).
 *
 * Sequence b has L_b cached tokens (its context and history, already
 * processed: their K and V are kept) and m_b new candidates.  The call
 * computes, for the candidates only, exactly the candidate rows of
 * hstu_attn_fwd on the whole sequence (n = L_b + m_b, num_targets = m_b):
 * candidate r attends every cached token j < L_b (position bucket
 * min(L_b - j, P - 1)) and itself (position bucket 0), never another
 * candidate; o and y as in hstu_attn_fwd.  num_contexts play no part (a
 * candidate sees all cached tokens either way).
 *
 * The descriptor is hstu_attn_fwd's with total_tokens = T_cand (candidates
 * in the batch); max_seq_len = N must bound every L_b + m_b.  Workspace: the
 * forward size from hstu_attn_workspace_size.  Tensor-core path only: BF16,
 * d_qk = d_v in {64, 128}, T_cand >= 128 and T_cache == 0 or >= 128, and no
 * dropout (inference), else HSTU_ERR_UNSUPPORTED.  Offsets inconsistent with the counts are reported
 * through the workspace error word (HSTU_ERR_DEVICE_CHECK).
 * ------------------------------------------------------------------------ */
typedef struct {
  const int64_t* cand_offsets;      /* [B+1] candidates of each sequence, packed; [B] == T_cand */
  const int64_t* cache_offsets;     /* [B+1] cached tokens of each sequence, packed; [B] == cache_tokens */
  int64_t cache_tokens;             /* T_cache */
  const int64_t* cand_timestamps;   /* [T_cand] or NULL (no time bias) */
  const int64_t* cache_timestamps;  /* [T_cache]; NULL iff cand_timestamps is NULL (when T_cache > 0) */
  const float* rab_pos;             /* [H, P] or NULL */
  const float* rab_time;            /* [H, Tb] or NULL */
  const void* q;                    /* [T_cand, H, d] candidates */
  const void* k;                    /* [T_cand, H, d] candidates' own keys */
  const void* v;                    /* [T_cand, H, d] */
  const void* u;                    /* [T_cand, H*d] gate or NULL */
  const void* k_cache;              /* [T_cache, H, d] */
  const void* v_cache;              /* [T_cache, H, d] */
  void* o;                          /* out [T_cand, H, d] */
  void* y;                          /* out [T_cand, H*d] or NULL */
  float* ln_mean;                   /* out [T_cand] or NULL */
  float* ln_rstd;                   /* out [T_cand] or NULL */
} hstu_attn_delta_args;

hstu_status_t hstu_attn_fwd_delta(const hstu_attn_desc* desc, const hstu_attn_delta_args* args,
                                  void* workspace, size_t workspace_bytes, hstu_stream_t stream);

/* Reads the device error word of the last call that used this workspace
 * (HSTU_OK when none).  Synchronises the stream. */
hstu_status_t hstu_get_device_error(const void* workspace, hstu_stream_t stream, int32_t* code);

/* Static string for a status code. */
const char* hstu_status_string(hstu_status_t status);

/* After HSTU_ERR_CUDA: the failing CUDA call of the last call on this thread,
 * by name, or the kernel launch with its resource attributes (registers,
 * threads per block, shared memory).  Empty when the last call did not fail
 * in CUDA.  The string belongs to the library and lives until the next call
 * on this thread. */
const char* hstu_last_error_detail(void);

/* Number of this library's kernels that the last successful hstu_attn_fwd,
 * hstu_attn_bwd, hstu_attn_fwd_delta, hstu_layer_fwd or hstu_layer_bwd call
 * on this thread launched (for launch accounting; cuBLAS's kernels inside
 * the layer calls are not counted). */
int32_t hstu_last_launch_count(void);

/* Measurement hook.  start_event and stop_event are cudaEvent_t handles (or
 * both NULL to clear).  The next hstu_attn_fwd or hstu_attn_bwd call on this
 * thread records start_event on its stream right before launching its
 * attention kernel and stop_event right after, then forgets them.  Under
 * stream capture they are recorded as external event nodes, so each replay
 * of the graph timestamps them. */
hstu_status_t hstu_time_next_attention_kernel(void* start_event, void* stop_event);

#ifdef __cplusplus
}
#endif

#endif /* HSTU_ATTN_H_ */
