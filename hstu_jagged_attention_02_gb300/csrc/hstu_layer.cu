// The full HSTU layer around the jagged attention (ai6s.net survey, section
// 2.1.2: pointwise projection eq. (1), spatial aggregation eq. (2), pointwise
// transformation eq. (3), residual connections between layers; section 2.1.3:
// two linear layers, no stored sub-layer activations beyond what the
// backward needs):
//
//   Z1 = X W1; U | V | Q | K = SiLU(Z1)   one tensor-core GEMM (hstu_gemm_tc.cu)
//                                         whose epilogue writes z1 [T, 4D] FP32,
//                                         U FP32 [T, D] and V, Q, K BF16 3 x [T, D]
//   o, y = attention(Q, K, V, U)          hstu_attn_fwd (norm and gate per desc)
//   out = X + y W2                        one tensor-core GEMM, residual in its epilogue
//
// and its backward: dW2 = y^T dOut and dW1 = X^T dZ1 (split-K, reduce-added),
// dy = dOut W2^T and dX = dOut + dZ1 W1^T, on the same tensor-core GEMM
// kernel, around this file's element-wise kernels (SiLU', BF16 pairs).
// Where D is not a multiple of 128 both passes take the library route:
// cuBLAS GEMMs (their workspace taken from the caller's workspace), then the
// SiLU split and the residual as separate kernels.
//
// Precision: V, Q, K are BF16 (the attention's MMA operands); the gate U and
// every accumulation stay FP32.  The computed GEMM operands y and dZ1 enter
// their GEMMs as BF16 pairs (hi + lo, about 16 bits) so that no single BF16
// rounding of a computed value reaches an output; dout, an input, is rounded
// to BF16 once.
#include <cublas_v2.h>

#include <mutex>

#include "hstu_internal.h"

using namespace hstu;

namespace hstu {
namespace {

size_t align_up(size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }

constexpr size_t kCublasWsBytes = size_t(32) << 20;

// -------------------------------------------------------------- kernels

__device__ __forceinline__ float sigmoid_acc(float z) { return 1.0f / (1.0f + expf(-z)); }

// [U | V | Q | K] = SiLU(Z1): z1 [T, 4D] FP32 -> u [T][D] FP32 (the gate keeps
// FP32) and vqk [3][T][D] BF16 (the attention's MMA operands)
__global__ void silu_split_kernel(const float* __restrict__ z1, float* __restrict__ u,
                                  __nv_bfloat16* __restrict__ vqk, int64_t T, int D) {
  const int64_t n4 = T * (int64_t)D;  // elements per part
  const int64_t total = 4 * n4 / 4;   // float4 groups over [T, 4D]
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = g * 4;               // first element, row-major in [T, 4D]
    const int64_t t = e / (4 * D);
    const int col = (int)(e % (4 * D));
    const int part = col / D, f = col % D;  // D % 4 == 0: a group never straddles parts
    const float4 z = *reinterpret_cast<const float4*>(z1 + e);
    const float4 a4 = make_float4(z.x * sigmoid_acc(z.x), z.y * sigmoid_acc(z.y), z.z * sigmoid_acc(z.z),
                                  z.w * sigmoid_acc(z.w));
    if (part == 0) {
      *reinterpret_cast<float4*>(u + t * D + f) = a4;
      continue;
    }
    const __nv_bfloat162 a = __floats2bfloat162_rn(a4.x, a4.y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(a4.z, a4.w);
    __nv_bfloat16* dst = vqk + (part - 1) * n4 + t * D + f;
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&a);
    w.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(dst) = w;
  }
}

// BF16 pair of an FP32 value: hi = bf16(x), lo = bf16(x - hi) (about 16 bits)
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __low2float(h), x1 - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// dZ1 = [du | dv | dq | dk] * SiLU'(Z1), SiLU'(z) = s (1 + z (1 - s)):
// grads [4][T][D] FP32, z1 [T, 4D] FP32 -> dz1 [T, 4D] as a BF16 pair
__global__ void silu_grad_kernel(const float* __restrict__ grads, const float* __restrict__ z1,
                                 __nv_bfloat16* __restrict__ dz1_hi, __nv_bfloat16* __restrict__ dz1_lo,
                                 int64_t T, int D) {
  const int64_t n4 = T * (int64_t)D;
  const int64_t total = n4;  // float4 groups over [T, 4D]
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = g * 4;
    const int64_t t = e / (4 * D);
    const int col = (int)(e % (4 * D));
    const int part = col / D, f = col % D;
    const float4 z = *reinterpret_cast<const float4*>(z1 + e);
    const float4 d = *reinterpret_cast<const float4*>(grads + part * n4 + t * D + f);
    float s;
    float r[4];
    s = sigmoid_acc(z.x); r[0] = d.x * s * (1.f + z.x * (1.f - s));
    s = sigmoid_acc(z.y); r[1] = d.y * s * (1.f + z.y * (1.f - s));
    s = sigmoid_acc(z.z); r[2] = d.z * s * (1.f + z.z * (1.f - s));
    s = sigmoid_acc(z.w); r[3] = d.w * s * (1.f + z.w * (1.f - s));
    uint2 h, l;
    split2(r[0], r[1], h.x, l.x);
    split2(r[2], r[3], h.y, l.y);
    *reinterpret_cast<uint2*>(dz1_hi + e) = h;
    *reinterpret_cast<uint2*>(dz1_lo + e) = l;
  }
}

// dst FP32 = src BF16 (the residual term before out += y W2)
__global__ void bf16_to_f32_kernel(const __nv_bfloat16* __restrict__ src, float* __restrict__ dst, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = __bfloat162float(src[i]);
}

__global__ void f32_to_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = __float2bfloat16_rn(src[i]);
}

// FP32 [n] -> BF16 pair (hi, lo); n a multiple of 4, 16-byte aligned
__global__ void f32_to_bf16_pair_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ hi,
                                        __nv_bfloat16* __restrict__ lo, int64_t n4) {
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < n4; g += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = reinterpret_cast<const float4*>(src)[g];
    uint2 h, l;
    split2(v.x, v.y, h.x, l.x);
    split2(v.z, v.w, h.y, l.y);
    reinterpret_cast<uint2*>(hi)[g] = h;
    reinterpret_cast<uint2*>(lo)[g] = l;
  }
}

unsigned grid_for(int64_t work) {
  int64_t g = (work + 255) / 256;
  if (g > 152 * 32) g = 152 * 32;
  return (unsigned)(g < 1 ? 1 : g);
}

// ------------------------------------------------------------- cuBLAS

// One handle per (thread, device), created on first use.
cublasHandle_t handle_for_device(int dev) {
  static thread_local cublasHandle_t handles[64] = {};
  if (dev < 0 || dev >= 64) return nullptr;
  if (!handles[dev]) {
    cublasHandle_t h = nullptr;
    if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS) return nullptr;
    handles[dev] = h;
  }
  return handles[dev];
}

// Row-major C[M, N] = op(A)[M, K] op(B)[K, N] (+ beta C), BF16 operands, FP32
// accumulation and FP32 C.  lda/ldb/ldc are the row-major leading dimensions.
bool gemm_rm(cublasHandle_t h, bool ta, bool tb, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
             const void* B, int64_t ldb, float beta, float* C, int64_t ldc) {
  const float alpha = 1.f;
  // column-major view: C^T[N, M] = op(B)^T op(A)^T
  return cublasGemmEx_64(h, tb ? CUBLAS_OP_T : CUBLAS_OP_N, ta ? CUBLAS_OP_T : CUBLAS_OP_N, N, M, K, &alpha, B,
                         CUDA_R_16BF, ldb, A, CUDA_R_16BF, lda, &beta, C, CUDA_R_32F, ldc, CUBLAS_COMPUTE_32F,
                         CUBLAS_GEMM_DEFAULT) == CUBLAS_STATUS_SUCCESS;
}

struct LayerWs {
  size_t cublas, attn, y_hi, y_lo, dout_bf, dy, grads, dz1_hi, dz1_lo, total;
  size_t attn_bytes;
};

LayerWs layer_ws(const hstu_attn_desc* d, bool bwd) {
  LayerWs L{};
  size_t fwd_attn = 0, bwd_attn = 0;
  hstu_attn_workspace_size(d, &fwd_attn, &bwd_attn);
  const size_t TD = (size_t)d->total_tokens * (size_t)(d->H * d->d_v);
  size_t off = 0;
  L.attn = off;   L.attn_bytes = bwd ? bwd_attn : fwd_attn;  off = align_up(off + L.attn_bytes);
  L.cublas = off; off = align_up(off + kCublasWsBytes);
  L.y_hi = off;   off = align_up(off + 2 * TD);
  L.y_lo = off;   off = align_up(off + 2 * TD);
  if (bwd) {
    L.dout_bf = off; off = align_up(off + 2 * TD);
    L.dy = off;      off = align_up(off + 4 * TD);
    L.grads = off;   off = align_up(off + 4 * 4 * TD);
    L.dz1_hi = off;  off = align_up(off + 2 * 4 * TD);
    L.dz1_lo = off;  off = align_up(off + 2 * 4 * TD);
  }
  L.total = off;
  return L;
}

hstu_status_t check_layer_desc(const hstu_attn_desc* d) {
  size_t f = 0, b = 0;
  const hstu_status_t s = hstu_attn_workspace_size(d, &f, &b);
  if (s != HSTU_OK) return s;
  if (d->dtype != HSTU_BF16 || d->out_dtype != HSTU_FP32) return HSTU_ERR_UNSUPPORTED;
  // HSTU_FLAG_TEST_TIMEOUT reaches only the forward's tensor-core input projection
  if ((d->H * d->d_v) % 8 != 0) return HSTU_ERR_UNSUPPORTED;
  return HSTU_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// the attention's descriptor inside the layer: the gate U is FP32
hstu_attn_desc attn_desc(const hstu_attn_desc* d) {
  hstu_attn_desc a = *d;
  a.flags |= HSTU_FLAG_U_FP32;
  a.flags &= ~HSTU_FLAG_TEST_TIMEOUT;
  return a;
}

#define LAYER_CUDA(expr)                                                         \
  do {                                                                           \
    cudaError_t e_ = (expr);                                                     \
    if (e_ != cudaSuccess) { (void)cudaGetLastError(); set_error_detail(e_, #expr); return HSTU_ERR_CUDA; } \
  } while (0)

#define LAYER_CUBLAS(ok)                                                          \
  do {                                                                            \
    if (!(ok)) { set_detail_message("cuBLAS GEMM failed: " #ok); return HSTU_ERR_CUDA; } \
  } while (0)

cublasHandle_t prepare_cublas(cudaStream_t st, void* ws) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  cublasHandle_t h = handle_for_device(dev);
  if (!h) return nullptr;
  if (cublasSetStream(h, st) != CUBLAS_STATUS_SUCCESS) return nullptr;
  if (cublasSetWorkspace(h, ws, kCublasWsBytes) != CUBLAS_STATUS_SUCCESS) return nullptr;
  return h;
}

}  // namespace
}  // namespace hstu

extern "C" {

hstu_status_t hstu_layer_workspace_size(const hstu_attn_desc* desc, size_t* fwd_bytes, size_t* bwd_bytes) {
  const hstu_status_t s = check_layer_desc(desc);
  if (s != HSTU_OK) return s;
  if (fwd_bytes) *fwd_bytes = layer_ws(desc, false).total;
  if (bwd_bytes) *bwd_bytes = layer_ws(desc, true).total;
  return HSTU_OK;
}

hstu_status_t hstu_layer_fwd(const hstu_attn_desc* d, const hstu_layer_fwd_args* a, void* workspace,
                             size_t workspace_bytes, hstu_stream_t stream) {
  hstu_status_t s = check_layer_desc(d);
  if (s != HSTU_OK) return s;
  // the layer plans its attention itself: the plan-keeping flags are not for it
  if (d->flags & (HSTU_FLAG_PLAN_BWD | HSTU_FLAG_REUSE_PLAN)) return HSTU_ERR_INVALID_ARG;
  if (!a || !a->seq_offsets ||
      (d->total_tokens > 0 &&
       (!a->x || !a->w1 || !a->w2 || !a->out || !a->z1 || !a->u || !a->vqk || !a->o || !a->y)))
    return HSTU_ERR_INVALID_ARG;
  for (const void* p : {a->x, a->w1, a->w2, (const void*)a->out, (const void*)a->z1, (const void*)a->u,
                        (const void*)a->vqk, (const void*)a->o, (const void*)a->y})
    if (p && !aligned16(p)) return HSTU_ERR_INVALID_ARG;
  const LayerWs L = layer_ws(d, false);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kWsAlign - 1)) || workspace_bytes < L.total)
    return HSTU_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const int64_t T = d->total_tokens;
  const int D = d->H * d->d_v;
  const size_t TD = (size_t)T * D;
  if (T == 0) return HSTU_OK;
  const bool fused = gemm_tc_supported(D);
  if ((d->flags & HSTU_FLAG_TEST_TIMEOUT) && !fused) return HSTU_ERR_UNSUPPORTED;
  cublasHandle_t h = nullptr;
  if (!fused) {
    h = prepare_cublas(st, ws + L.cublas);
    if (!h) { set_detail_message("cuBLAS handle set-up failed"); return HSTU_ERR_CUDA; }
  }

  // Z1 = X W1 ; U | V | Q | K = SiLU(Z1): one tensor-core GEMM whose epilogue
  // writes z1, U and V, Q, K (D % 128 == 0), else cuBLAS + the split kernel
  __nv_bfloat16* vqk = static_cast<__nv_bfloat16*>(a->vqk);
  int32_t* hdr = reinterpret_cast<int32_t*>(ws + L.attn);
  GemmParams gp{};
  gp.M = T; gp.D = D; gp.K = D;
  int sms = 0;
  if (fused) {
    int dev = 0;
    LAYER_CUDA(cudaGetDevice(&dev));
    LAYER_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    LAYER_CUDA(cudaMemsetAsync(hdr + WS_LAYER_ERR, 0, 2 * sizeof(int32_t), st));
    gp.N = 4 * D; gp.npass = 1;
    gp.test_timeout = (d->flags & HSTU_FLAG_TEST_TIMEOUT) ? 1 : 0;
    gp.err = hdr + WS_LAYER_ERR; gp.err_info = hdr + WS_LAYER_INFO;
    gp.z1 = a->z1; gp.u = a->u; gp.vqk = vqk;
    LAYER_CUDA(launch_gemm_f1(gp, a->x, a->w1, sms, st));
  } else {
    LAYER_CUBLAS(gemm_rm(h, false, false, T, 4 * D, D, a->x, D, a->w1, 4 * D, 0.f, a->z1, 4 * D));
    silu_split_kernel<<<grid_for(TD), 256, 0, st>>>(a->z1, a->u, vqk, T, D);
    LAYER_CUDA(cudaGetLastError());
  }

  // attention: o, y
  hstu_attn_fwd_args fa{};
  fa.seq_offsets = a->seq_offsets; fa.num_targets = a->num_targets; fa.num_contexts = a->num_contexts;
  fa.timestamps = a->timestamps; fa.rab_pos = a->rab_pos; fa.rab_time = a->rab_time;
  fa.u = a->u; fa.v = vqk; fa.q = vqk + TD; fa.k = vqk + 2 * TD;
  fa.o = a->o; fa.y = a->y;
  fa.dropout_seed = a->dropout_seed; fa.dropout_offset = a->dropout_offset;
  const hstu_attn_desc ad = attn_desc(d);
  s = hstu_attn_fwd(&ad, &fa, ws + L.attn, L.attn_bytes, stream);
  if (s != HSTU_OK) return s;

  // out = X + y W2, y entering the GEMM as a BF16 pair: out = X + y_hi W2 + y_lo W2
  __nv_bfloat16* y_hi = reinterpret_cast<__nv_bfloat16*>(ws + L.y_hi);
  __nv_bfloat16* y_lo = reinterpret_cast<__nv_bfloat16*>(ws + L.y_lo);
  f32_to_bf16_pair_kernel<<<grid_for(TD / 4), 256, 0, st>>>(static_cast<const float*>(a->y), y_hi, y_lo,
                                                           (int64_t)(TD / 4));
  LAYER_CUDA(cudaGetLastError());
  if (fused) {
    // one tensor-core GEMM over both halves of the pair, the residual added in its epilogue;
    // an error of the first GEMM is raised into the workspace's error word here
    gp.N = D; gp.npass = 2; gp.test_timeout = 0;
    gp.err = hdr + WS_ERR; gp.err_info = hdr + WS_ERR_INFO; gp.carry_err = hdr + WS_LAYER_ERR;
    gp.z1 = nullptr; gp.u = nullptr; gp.vqk = nullptr;
    gp.x = static_cast<const __nv_bfloat16*>(a->x); gp.out = static_cast<float*>(a->out);
    LAYER_CUDA(launch_gemm_f2(gp, y_hi, y_lo, a->w2, sms, st));
    note_launches(3);  // f1, the y pair, f2
    return HSTU_OK;
  }
  bf16_to_f32_kernel<<<grid_for(TD), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(a->x),
                                                    static_cast<float*>(a->out), (int64_t)TD);
  LAYER_CUDA(cudaGetLastError());
  LAYER_CUBLAS(gemm_rm(h, false, false, T, D, D, y_hi, D, a->w2, D, 1.f, static_cast<float*>(a->out), D));
  LAYER_CUBLAS(gemm_rm(h, false, false, T, D, D, y_lo, D, a->w2, D, 1.f, static_cast<float*>(a->out), D));
  note_launches(3);  // SiLU split, the y pair, the residual copy (cuBLAS's own kernels not counted)
  return HSTU_OK;
}

hstu_status_t hstu_layer_bwd(const hstu_attn_desc* d, const hstu_layer_bwd_args* a, void* workspace,
                             size_t workspace_bytes, hstu_stream_t stream) {
  hstu_status_t s = check_layer_desc(d);
  if (s != HSTU_OK) return s;
  if (d->flags & HSTU_FLAG_TEST_TIMEOUT) return HSTU_ERR_UNSUPPORTED;   // a forward-only test mode
  if (d->flags & (HSTU_FLAG_PLAN_BWD | HSTU_FLAG_REUSE_PLAN)) return HSTU_ERR_INVALID_ARG;
  if (!a || !a->seq_offsets ||
      (d->total_tokens > 0 && (!a->x || !a->w1 || !a->w2 || !a->z1 || !a->u || !a->vqk || !a->o || !a->y || !a->dout ||
                               !a->dx || !a->dw1 || !a->dw2)))
    return HSTU_ERR_INVALID_ARG;
  for (const void* p : {a->x, a->w1, a->w2, (const void*)a->z1, (const void*)a->u, a->vqk, a->o, a->y, (const void*)a->dout,
                        (const void*)a->dx, (const void*)a->dw1, (const void*)a->dw2})
    if (p && !aligned16(p)) return HSTU_ERR_INVALID_ARG;
  const LayerWs L = layer_ws(d, true);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kWsAlign - 1)) || workspace_bytes < L.total)
    return HSTU_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const int64_t T = d->total_tokens;
  const int D = d->H * d->d_v;
  const size_t TD = (size_t)T * D;
  if (T == 0) {
    if (a->dw1) LAYER_CUDA(cudaMemsetAsync(a->dw1, 0, sizeof(float) * (size_t)D * 4 * D, st));
    if (a->dw2) LAYER_CUDA(cudaMemsetAsync(a->dw2, 0, sizeof(float) * (size_t)D * D, st));
    if (a->d_rab_pos) LAYER_CUDA(cudaMemsetAsync(a->d_rab_pos, 0, sizeof(float) * d->H * d->num_pos_buckets, st));
    if (a->d_rab_time) LAYER_CUDA(cudaMemsetAsync(a->d_rab_time, 0, sizeof(float) * d->H * d->num_time_buckets, st));
    return HSTU_OK;
  }
  // the four GEMMs run on the tensor-core kernel when D % 128 == 0, else on cuBLAS
  const bool fused = gemm_tc_supported(D);
  cublasHandle_t h = nullptr;
  int32_t* hdr = reinterpret_cast<int32_t*>(ws + L.attn);
  int sms = 0;
  if (fused) {
    int dev = 0;
    LAYER_CUDA(cudaGetDevice(&dev));
    LAYER_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    LAYER_CUDA(cudaMemsetAsync(hdr + WS_LAYER_ERR, 0, 2 * sizeof(int32_t), st));
    // the weight gradients are reduce-added over ranges of tokens: start from zero
    LAYER_CUDA(cudaMemsetAsync(a->dw1, 0, sizeof(float) * (size_t)D * 4 * D, st));
    LAYER_CUDA(cudaMemsetAsync(a->dw2, 0, sizeof(float) * (size_t)D * D, st));
  } else {
    h = prepare_cublas(st, ws + L.cublas);
    if (!h) { set_detail_message("cuBLAS handle set-up failed"); return HSTU_ERR_CUDA; }
  }
  const __nv_bfloat16* vqk = static_cast<const __nv_bfloat16*>(a->vqk);
  __nv_bfloat16* y_hi = reinterpret_cast<__nv_bfloat16*>(ws + L.y_hi);
  __nv_bfloat16* y_lo = reinterpret_cast<__nv_bfloat16*>(ws + L.y_lo);
  __nv_bfloat16* doutbf = reinterpret_cast<__nv_bfloat16*>(ws + L.dout_bf);
  float* dy = reinterpret_cast<float*>(ws + L.dy);
  float* grads = reinterpret_cast<float*>(ws + L.grads);  // du | dv | dq | dk
  __nv_bfloat16* dz1_hi = reinterpret_cast<__nv_bfloat16*>(ws + L.dz1_hi);
  __nv_bfloat16* dz1_lo = reinterpret_cast<__nv_bfloat16*>(ws + L.dz1_lo);

  // dW2 = y^T dOut (y as a BF16 pair) ; dy = dOut W2^T
  f32_to_bf16_pair_kernel<<<grid_for(TD / 4), 256, 0, st>>>(static_cast<const float*>(a->y), y_hi, y_lo,
                                                           (int64_t)(TD / 4));
  LAYER_CUDA(cudaGetLastError());
  f32_to_bf16_kernel<<<grid_for(TD), 256, 0, st>>>(static_cast<const float*>(a->dout), doutbf, (int64_t)TD);
  LAYER_CUDA(cudaGetLastError());
  GemmParams gp{};
  gp.D = D;
  gp.err = hdr + WS_LAYER_ERR; gp.err_info = hdr + WS_LAYER_INFO;
  if (fused) {
    gp.M = D; gp.N = D; gp.K = T; gp.out = a->dw2;
    LAYER_CUDA(launch_gemm_tn_reduce(gp, y_hi, y_lo, doutbf, nullptr, sms, st));
    gp.M = T; gp.N = D; gp.K = D; gp.out = dy;
    LAYER_CUDA(launch_gemm_nt(gp, doutbf, nullptr, a->w2, sms, st));
  } else {
    LAYER_CUBLAS(gemm_rm(h, true, false, D, D, T, y_hi, D, doutbf, D, 0.f, a->dw2, D));
    LAYER_CUBLAS(gemm_rm(h, true, false, D, D, T, y_lo, D, doutbf, D, 1.f, a->dw2, D));
    LAYER_CUBLAS(gemm_rm(h, false, true, T, D, D, doutbf, D, a->w2, D, 0.f, dy, D));
  }

  // attention backward: du, dv, dq, dk (FP32), d_rab
  hstu_attn_bwd_args ba{};
  ba.seq_offsets = a->seq_offsets; ba.num_targets = a->num_targets; ba.num_contexts = a->num_contexts;
  ba.timestamps = a->timestamps; ba.rab_pos = a->rab_pos; ba.rab_time = a->rab_time;
  ba.u = a->u; ba.v = vqk; ba.q = vqk + TD; ba.k = vqk + 2 * TD;
  ba.o = a->o; ba.dy = dy;
  ba.du = grads; ba.dv = grads + TD; ba.dq = grads + 2 * TD; ba.dk = grads + 3 * TD;
  ba.d_rab_pos = a->d_rab_pos; ba.d_rab_time = a->d_rab_time;
  ba.dropout_seed = a->dropout_seed; ba.dropout_offset = a->dropout_offset;
  const hstu_attn_desc ad = attn_desc(d);
  s = hstu_attn_bwd(&ad, &ba, ws + L.attn, L.attn_bytes, stream);
  if (s != HSTU_OK) return s;

  // dZ1 = [du|dv|dq|dk] * SiLU'(Z1) ; dW1 = X^T dZ1 ; dX = dOut + dZ1 W1^T
  silu_grad_kernel<<<grid_for(TD), 256, 0, st>>>(grads, a->z1, dz1_hi, dz1_lo, T, D);
  LAYER_CUDA(cudaGetLastError());
  float* dx = static_cast<float*>(a->dx);
  if (fused) {
    // an error of the two GEMMs before the attention is raised into the
    // workspace's error word here (the attention's plan cleared it)
    gp.err = hdr + WS_ERR; gp.err_info = hdr + WS_ERR_INFO; gp.carry_err = hdr + WS_LAYER_ERR;
    gp.M = D; gp.N = 4 * D; gp.K = T; gp.out = a->dw1;
    LAYER_CUDA(launch_gemm_tn_reduce(gp, a->x, nullptr, dz1_hi, dz1_lo, sms, st));
    gp.M = T; gp.N = D; gp.K = 4 * D; gp.out = dx; gp.res = static_cast<const float*>(a->dout);
    LAYER_CUDA(launch_gemm_nt(gp, dz1_hi, dz1_lo, a->w1, sms, st));
    note_launches(7);  // the y pair, dout to BF16, dW2, dy, SiLU', dW1, dX
    return HSTU_OK;
  }
  LAYER_CUBLAS(gemm_rm(h, true, false, D, 4 * D, T, a->x, D, dz1_hi, 4 * D, 0.f, a->dw1, 4 * D));
  LAYER_CUBLAS(gemm_rm(h, true, false, D, 4 * D, T, a->x, D, dz1_lo, 4 * D, 1.f, a->dw1, 4 * D));
  LAYER_CUDA(cudaMemcpyAsync(a->dx, a->dout, sizeof(float) * TD, cudaMemcpyDeviceToDevice, st));
  LAYER_CUBLAS(gemm_rm(h, false, true, T, D, 4 * D, dz1_hi, 4 * D, a->w1, 4 * D, 1.f, dx, D));
  LAYER_CUBLAS(gemm_rm(h, false, true, T, D, 4 * D, dz1_lo, 4 * D, a->w1, 4 * D, 1.f, dx, D));
  note_launches(3);  // the y pair, dout to BF16, SiLU' (cuBLAS's own kernels not counted)
  return HSTU_OK;
}

}  // extern "C"
