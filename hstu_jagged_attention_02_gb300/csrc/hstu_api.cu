// C ABI entry points of libhstu_attn.so (declared in include/hstu_attn.h):
// argument checks, workspace layout, path selection and the stream-ordered
// launch sequence of each pass.  No device memory is allocated here.
#include <cmath>
#include <cstdio>
#include <cstring>

#include "hstu_internal.h"

using namespace hstu;

namespace {

thread_local int32_t g_launches = 0;
thread_local cudaEvent_t g_ev_start = nullptr, g_ev_stop = nullptr;
thread_local char g_detail[320] = {0};

bool detail_is_set() { return g_detail[0] != 0; }
void clear_detail() { g_detail[0] = 0; }

// Records the measurement-hook events around one launch, then clears them.
// Records the hook's events around one launch.  Under stream capture they
// become external event-record nodes, so each replay of the graph
// timestamps them; outside capture they are plain records.
void record_hook_event(cudaEvent_t e, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
  else
    cudaEventRecord(e, st);
}

struct KernelTimer {
  cudaStream_t st;
  cudaEvent_t a, b;
  explicit KernelTimer(cudaStream_t s) : st(s), a(g_ev_start), b(g_ev_stop) {
    g_ev_start = g_ev_stop = nullptr;
    if (a) record_hook_event(a, st);
  }
  ~KernelTimer() { if (b) record_hook_event(b, st); }
};

constexpr uint32_t kKnownFlags = HSTU_FLAG_FORCE_SIMT | HSTU_FLAG_TEST_TIMEOUT | HSTU_FLAG_U_FP32 |
                                  HSTU_FLAG_PLAN_BWD | HSTU_FLAG_REUSE_PLAN;

size_t align_up(size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }
size_t esize(int dtype) { return dtype == HSTU_BF16 ? 2 : 4; }

struct WsLayout {
  size_t seq_start, tmp, blocks, items, plan_end, dO, dq_acc, drab_part, drab_part_bytes, total;
  // backward layout only: the second plan region, where a forward called with
  // HSTU_FLAG_PLAN_BWD keeps the backward's plan, and the metadata it was made from
  size_t pb_seq_start, pb_tmp, pb_blocks, pb_items, sv_off, sv_t0, sv_nt, sv_nc;
  int cap_blocks;
};

WsLayout ws_layout(const hstu_attn_desc* d, bool bwd) {
  WsLayout L{};
  const int64_t cap = (d->total_tokens + kSimtTile - 1) / kSimtTile + d->B;  // blocks at the smallest edge
  L.cap_blocks = (int)cap;
  size_t off = kWsHeaderBytes;
  L.seq_start = off; off = align_up(off + sizeof(int) * (size_t)(d->B + 1));
  L.tmp = off;       off = align_up(off + sizeof(Block) * (size_t)cap);
  L.blocks = off;    off = align_up(off + sizeof(Block) * (size_t)cap);
  L.items = off;     off = align_up(off + sizeof(PlanItem) * (size_t)cap);
  L.plan_end = off;
  if (bwd) {
    const size_t rows = (size_t)d->total_tokens * (size_t)d->H;
    L.dO = off;     off = align_up(off + sizeof(float) * rows * (size_t)d->d_v);  // FP32 or a BF16 pair
    L.dq_acc = off; off = align_up(off + sizeof(float) * rows * (size_t)d->d_qk);
    L.drab_part_bytes = sizeof(float) * kDrabMaxCtas * (size_t)d->H * (d->num_pos_buckets + d->num_time_buckets);
    L.drab_part = off; off = align_up(off + L.drab_part_bytes);
    L.pb_seq_start = off; off = align_up(off + sizeof(int) * (size_t)(d->B + 1));
    L.pb_tmp = off;       off = align_up(off + sizeof(Block) * (size_t)cap);
    L.pb_blocks = off;    off = align_up(off + sizeof(Block) * (size_t)cap);
    L.pb_items = off;     off = align_up(off + sizeof(PlanItem) * (size_t)cap);
    L.sv_off = off;       off = align_up(off + sizeof(int64_t) * (size_t)(d->B + 1));
    L.sv_t0 = off;        off = align_up(off + sizeof(int64_t) * (size_t)d->B);
    L.sv_nt = off;        off = align_up(off + sizeof(int32_t) * (size_t)d->B);
    L.sv_nc = off;        off = align_up(off + sizeof(int32_t) * (size_t)d->B);
  }
  L.total = off;
  return L;
}

hstu_status_t check_desc(const hstu_attn_desc* d) {
  if (!d || d->struct_size != sizeof(hstu_attn_desc)) return HSTU_ERR_INVALID_ARG;
  if (d->dtype != HSTU_BF16 && d->dtype != HSTU_FP32) return HSTU_ERR_INVALID_ARG;
  if (d->out_dtype != HSTU_BF16 && d->out_dtype != HSTU_FP32) return HSTU_ERR_INVALID_ARG;
  if (d->dtype == HSTU_FP32 && d->out_dtype != HSTU_FP32) return HSTU_ERR_UNSUPPORTED;
  if (d->B < 0 || d->H < 1 || d->total_tokens < 0 || d->d_qk < 1 || d->d_v < 1) return HSTU_ERR_INVALID_ARG;
  if (d->max_seq_len < 1 || d->num_pos_buckets < 1 || d->num_time_buckets < 1) return HSTU_ERR_INVALID_ARG;
  if (d->norm != HSTU_NORM_NONE && d->norm != HSTU_NORM_LAYERNORM) return HSTU_ERR_INVALID_ARG;
  if (d->norm == HSTU_NORM_LAYERNORM && !(d->ln_eps > 0.f && std::isfinite(d->ln_eps))) return HSTU_ERR_INVALID_ARG;
  if (!std::isfinite(d->alpha)) return HSTU_ERR_INVALID_ARG;
  if (!(d->dropout_p >= 0.f && d->dropout_p < 1.f) || d->reserved != 0) return HSTU_ERR_INVALID_ARG;
  if (d->flags & ~kKnownFlags) return HSTU_ERR_INVALID_ARG;
  if ((d->flags & HSTU_FLAG_U_FP32) && d->out_dtype != HSTU_FP32) return HSTU_ERR_UNSUPPORTED;
  if (d->d_qk != d->d_v || (d->d_qk != 32 && d->d_qk != 64 && d->d_qk != 128)) return HSTU_ERR_UNSUPPORTED;
  if (d->H * d->d_v > 2048) return HSTU_ERR_UNSUPPORTED;
  if (d->max_seq_len > kCostBins * kSimtTile) return HSTU_ERR_UNSUPPORTED;
  if (d->num_pos_buckets > 4096 || d->num_time_buckets > 4096) return HSTU_ERR_UNSUPPORTED;
  if ((d->total_tokens + kSimtTile - 1) / kSimtTile + d->B > (int64_t)0x3fffffff / d->H) return HSTU_ERR_UNSUPPORTED;
  return HSTU_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Fused dropout constants of the norm-gate kernels: keep iff the element's
// 32-bit generator word >= floor(p 2^32); kept values times 1 / (1 - p).
void set_dropout(NormParams& np, const hstu_attn_desc* d, uint64_t seed, uint64_t offset) {
  if (!(d->dropout_p > 0.f)) return;
  const double p = (double)d->dropout_p;
  np.drop = 1;
  np.drop_thr = (uint32_t)std::floor(p * 4294967296.0);
  np.drop_scale = (float)(1.0 / (1.0 - p));
  np.drop_seed = seed;
  np.drop_offset = offset;
}

// Score constants of the tensor-core epilogues (w = -log2(e) z form).
void set_score_constants(AttnParams& p) {
  const float log2e = 1.4426950408889634f;
  p.kA = -log2e * p.alpha;
  p.kC = -p.inv_n / log2e;
  p.kZ = -1.0f / log2e;
  p.kCi = 1.0f / p.kC;
  p.kA2 = make_float2(p.kA, p.kA);
  p.kC2 = make_float2(p.kC, p.kC);
  p.kZ2 = make_float2(p.kZ, p.kZ);
  p.kCi2 = make_float2(p.kCi, p.kCi);
  p.inv_n2 = make_float2(p.inv_n, p.inv_n);
}

hstu_status_t check_ws(void* ws, size_t bytes, size_t need) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kWsAlign - 1)) != 0) return HSTU_ERR_WORKSPACE;
  if (bytes < need) return HSTU_ERR_WORKSPACE;
  return HSTU_OK;
}

// Device properties, cached per device.
struct DevInfo { int cc = -1; int sms = 0; };
DevInfo dev_info() {
  static DevInfo cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DevInfo{};
  if (cache[dev].cc < 0) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cache[dev].sms = sms;
    cache[dev].cc = major * 10 + minor;
  }
  return cache[dev];
}

bool use_tc(const hstu_attn_desc* d, bool bwd) {
  if (d->flags & HSTU_FLAG_FORCE_SIMT) return false;
  if (d->total_tokens < kTcTile) return false;  // TMA boxes of 128 rows
  if (dev_info().cc != 103) return false;
  if (bwd)
    return tc_bwd_supported(d->dtype, d->d_qk, d->d_v) &&
           tc_bwd_smem_bytes(d->H, d->num_pos_buckets, d->num_time_buckets) <= kMaxSmemPerCta;
  return tc_fwd_supported(d->dtype, d->d_qk, d->d_v) &&
         tc_fwd_smem_bytes(d->d_qk, d->H, d->num_pos_buckets, d->num_time_buckets) <= kMaxSmemPerCta;
}

// BF16 work the tensor-core kernels do not take (head sizes other than 128,
// or 64 in the forward; bias tables too large for shared memory) would run
// on the CUDA-core kernels, some thirty times slower.  That happens only when
// the caller asks for it with HSTU_FLAG_FORCE_SIMT; otherwise the call is
// refused.  Problems under 128 tokens take the CUDA-core kernels either way
// (they last microseconds).
hstu_status_t check_tc_shape(const hstu_attn_desc* d, bool bwd) {
  if (d->dtype != HSTU_BF16 || (d->flags & HSTU_FLAG_FORCE_SIMT)) return HSTU_OK;
  const bool ok = bwd ? tc_bwd_supported(d->dtype, d->d_qk, d->d_v) &&
                            tc_bwd_smem_bytes(d->H, d->num_pos_buckets, d->num_time_buckets) <= kMaxSmemPerCta
                      : tc_fwd_supported(d->dtype, d->d_qk, d->d_v) &&
                            tc_fwd_smem_bytes(d->d_qk, d->H, d->num_pos_buckets, d->num_time_buckets) <= kMaxSmemPerCta;
  if (ok) return HSTU_OK;
  set_detail_message(bwd ? "BF16 backward without a tensor-core kernel for this shape (d = 128 only); "
                           "HSTU_FLAG_FORCE_SIMT runs it on the CUDA-core kernels"
                         : "BF16 forward without a tensor-core kernel for this shape (d = 64 or 128); "
                           "HSTU_FLAG_FORCE_SIMT runs it on the CUDA-core kernels");
  return HSTU_ERR_UNSUPPORTED;
}

// One pass's tiling (the path's tile edges) and the plan region it is written to.
PlanOut plan_out(int pass, bool tc, char* ws, size_t seq_start, size_t tmp, size_t blocks, size_t items) {
  PlanOut o{};
  if (!tc) {
    o.BM = o.BN = kSimtTile;
  } else if (pass == 0 || pass == 2) {
    o.BM = o.BN = kTcTile;
  } else {
    o.BM = kTcBwdQTile;  // the tensor-core backward walks 64-row query tiles per 128-row key block
    o.BN = kTcTile;
  }
  o.pass = pass;
  o.seq_start = reinterpret_cast<int*>(ws + seq_start);
  o.tmp = reinterpret_cast<Block*>(ws + tmp);
  o.blocks = reinterpret_cast<Block*>(ws + blocks);
  o.items = reinterpret_cast<PlanItem*>(ws + items);
  return o;
}

PlanParams plan_params(const hstu_attn_desc* d, const int64_t* off, const int32_t* nt, const int32_t* nc,
                       const int64_t* ts, int pass, bool tc, char* ws, const WsLayout& L) {
  PlanParams p{};
  p.off = off; p.nt = nt; p.nc = nc; p.ts = ts;
  p.B = d->B; p.T = d->total_tokens; p.max_n = d->max_seq_len;
  p.hdr = reinterpret_cast<int*>(ws);
  p.cap_blocks = L.cap_blocks;
  p.npass = 1;
  p.out[0] = plan_out(pass, tc, ws, L.seq_start, L.tmp, L.blocks, L.items);
  return p;
}

// The kept backward plan (second plan region of a backward-sized workspace).
PlanOut kept_plan_out(const hstu_attn_desc* d, char* ws, const WsLayout& L) {
  return plan_out(1, use_tc(d, true), ws, L.pb_seq_start, L.pb_tmp, L.pb_blocks, L.pb_items);
}

#define HSTU_CUDA_TRY(expr)                                    \
  do {                                                         \
    cudaError_t e_ = (expr);                                   \
    if (e_ != cudaSuccess) {                                   \
      (void)cudaGetLastError();                                \
      if (!detail_is_set()) set_error_detail(e_, #expr);       \
      return HSTU_ERR_CUDA;                                    \
    }                                                          \
  } while (0)

}  // namespace

namespace hstu {

void set_error_detail(cudaError_t e, const char* where) {
  snprintf(g_detail, sizeof(g_detail), "%s in %s", cudaGetErrorName(e), where);
}

void set_detail_message(const char* msg) { snprintf(g_detail, sizeof(g_detail), "%s", msg); }

void set_launch_detail(cudaError_t e, const char* kernel, const void* func, int threads, size_t smem) {
  cudaFuncAttributes fa{};
  const cudaError_t ea = cudaFuncGetAttributes(&fa, func);
  (void)cudaGetLastError();
  if (ea == cudaSuccess)
    snprintf(g_detail, sizeof(g_detail),
             "%s launching %s: %d threads, %zu B dynamic smem; kernel uses %d registers, "
             "allows %d threads per block, %zu B static smem",
             cudaGetErrorName(e), kernel, threads, smem, fa.numRegs, fa.maxThreadsPerBlock, fa.sharedSizeBytes);
  else
    snprintf(g_detail, sizeof(g_detail), "%s launching %s (%d threads, %zu B smem)", cudaGetErrorName(e), kernel,
             threads, smem);
}

}  // namespace hstu

namespace hstu {
void note_launches(int32_t n) { g_launches += n; }
}  // namespace hstu

extern "C" {

const char* hstu_last_error_detail(void) { return g_detail; }

const char* hstu_status_string(hstu_status_t s) {
  switch (s) {
    case HSTU_OK: return "ok";
    case HSTU_ERR_INVALID_ARG: return "invalid argument";
    case HSTU_ERR_UNSUPPORTED: return "unsupported configuration";
    case HSTU_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case HSTU_ERR_CUDA: return "CUDA runtime error";
    case HSTU_ERR_TIMEOUT: return "device pipeline wait timed out";
    case HSTU_ERR_DEVICE_CHECK: return "device check failed: offsets or counts inconsistent";
  }
  return "unknown status";
}

int32_t hstu_last_launch_count(void) { return g_launches; }

hstu_status_t hstu_time_next_attention_kernel(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr)) return HSTU_ERR_INVALID_ARG;
  g_ev_start = static_cast<cudaEvent_t>(start_event);
  g_ev_stop = static_cast<cudaEvent_t>(stop_event);
  return HSTU_OK;
}

hstu_status_t hstu_attn_workspace_size(const hstu_attn_desc* desc, size_t* fwd_bytes, size_t* bwd_bytes) {
  const hstu_status_t s = check_desc(desc);
  if (s != HSTU_OK) return s;
  if (fwd_bytes) *fwd_bytes = ws_layout(desc, false).total;
  if (bwd_bytes) *bwd_bytes = ws_layout(desc, true).total;
  return HSTU_OK;
}

hstu_status_t hstu_attn_fwd(const hstu_attn_desc* d, const hstu_attn_fwd_args* a, void* workspace,
                            size_t workspace_bytes, hstu_stream_t stream) {
  hstu_status_t s = check_desc(d);
  if (s != HSTU_OK) return s;
  // token tensors may be NULL only when there are no tokens
  if (!a || !a->seq_offsets || (d->total_tokens > 0 && (!a->q || !a->k || !a->v || !a->o)))
    return HSTU_ERR_INVALID_ARG;
  if (d->flags & HSTU_FLAG_REUSE_PLAN) return HSTU_ERR_INVALID_ARG;  // a backward-only flag
  for (const void* ptr : {a->q, a->k, a->v, (const void*)a->o, a->u, (const void*)a->y})
    if (ptr && !aligned16(ptr)) return HSTU_ERR_INVALID_ARG;
  clear_detail();
  if ((s = check_tc_shape(d, false)) != HSTU_OK) return s;
  // keeping the backward's plan takes the backward's workspace
  const bool keep_bwd = (d->flags & HSTU_FLAG_PLAN_BWD) != 0;
  const WsLayout L = ws_layout(d, keep_bwd);
  if ((s = check_ws(workspace, workspace_bytes, L.total)) != HSTU_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  g_launches = 0;

  const bool tc = use_tc(d, false);
  PlanParams pp = plan_params(d, a->seq_offsets, a->num_targets, a->num_contexts, a->timestamps, 0, tc, ws, L);
  if (keep_bwd) {  // a second CTA of the same launch plans the backward
    pp.npass = 2;
    pp.out[1] = kept_plan_out(d, ws, L);
    pp.sv_off = reinterpret_cast<int64_t*>(ws + L.sv_off);
    pp.sv_t0 = reinterpret_cast<int64_t*>(ws + L.sv_t0);
    pp.sv_nt = reinterpret_cast<int32_t*>(ws + L.sv_nt);
    pp.sv_nc = reinterpret_cast<int32_t*>(ws + L.sv_nc);
  }
  HSTU_CUDA_TRY(launch_plan(pp, st));
  ++g_launches;

  AttnParams p{};
  p.off = a->seq_offsets; p.nt = a->num_targets; p.nc = a->num_contexts;
  p.ts = a->timestamps; p.rab_pos = a->rab_pos; p.rab_time = a->timestamps ? a->rab_time : nullptr;
  p.q = a->q; p.k = a->k; p.v = a->v; p.o = a->o;
  p.hdr = pp.hdr; p.hdr_rw = pp.hdr; p.blocks = pp.out[0].blocks; p.items = pp.out[0].items;
  p.B = d->B; p.H = d->H; p.dqk = d->d_qk; p.dv_dim = d->d_v; p.T = d->total_tokens;
  p.dtype = d->dtype; p.out_dtype = d->out_dtype;
  p.alpha = d->alpha; p.inv_n = 1.0f / (float)d->max_seq_len;
  set_score_constants(p);
  p.P = d->num_pos_buckets; p.Tb = d->num_time_buckets; p.flags = d->flags;
  p.num_sms = dev_info().sms;
  if (d->total_tokens > 0) {
    {
      KernelTimer timer(st);
      if (tc) {
        HSTU_CUDA_TRY(launch_tc_fwd(p, st));
      } else {
        const int max_items = ((int)((d->total_tokens + kSimtTile - 1) / kSimtTile) + d->B) * d->H;
        HSTU_CUDA_TRY(launch_simt_fwd(p, max_items, st));
      }
    }
    ++g_launches;
    if (a->y || a->ln_mean || a->ln_rstd) {
      NormParams np{};
      np.dtype = (d->flags & HSTU_FLAG_U_FP32) ? HSTU_FP32 : d->dtype; np.out_dtype = d->out_dtype;
      np.o = a->o; np.u = a->u; np.y = a->y; np.mean = a->ln_mean; np.rstd = a->ln_rstd;
      np.T = d->total_tokens; np.F = d->H * d->d_v; np.norm = d->norm; np.eps = d->ln_eps;
      set_dropout(np, d, a->dropout_seed, a->dropout_offset);
      HSTU_CUDA_TRY(launch_norm_gate_fwd(np, st));
      ++g_launches;
    }
  }
  return HSTU_OK;
}

hstu_status_t hstu_attn_bwd(const hstu_attn_desc* d, const hstu_attn_bwd_args* a, void* workspace,
                            size_t workspace_bytes, hstu_stream_t stream) {
  hstu_status_t s = check_desc(d);
  if (s != HSTU_OK) return s;
  if (!a || !a->seq_offsets ||
      (d->total_tokens > 0 && (!a->q || !a->k || !a->v || !a->o || !a->dy || !a->dq || !a->dk || !a->dv)))
    return HSTU_ERR_INVALID_ARG;
  if (d->total_tokens > 0 && (a->u == nullptr) != (a->du == nullptr)) return HSTU_ERR_INVALID_ARG;
  if (d->flags & HSTU_FLAG_PLAN_BWD) return HSTU_ERR_INVALID_ARG;  // a forward-only flag
  for (const void* ptr : {a->q, a->k, a->v, a->o, a->u, a->dy, (const void*)a->dq, (const void*)a->dk,
                          (const void*)a->dv, (const void*)a->du})
    if (ptr && !aligned16(ptr)) return HSTU_ERR_INVALID_ARG;
  clear_detail();
  if ((s = check_tc_shape(d, true)) != HSTU_OK) return s;
  const WsLayout L = ws_layout(d, true);
  if ((s = check_ws(workspace, workspace_bytes, L.total)) != HSTU_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  g_launches = 0;

  const bool tc = use_tc(d, true);
  // with HSTU_FLAG_REUSE_PLAN no planner runs: the norm-gate backward checks
  // the plan a forward kept in the second plan region and arms it
  const bool reuse = (d->flags & HSTU_FLAG_REUSE_PLAN) != 0;
  const PlanParams pp =
      plan_params(d, a->seq_offsets, a->num_targets, a->num_contexts, a->timestamps, 1, tc, ws, L);
  const PlanOut plan = reuse ? kept_plan_out(d, ws, L) : pp.out[0];
  if (!reuse) {
    HSTU_CUDA_TRY(launch_plan(pp, st));
    ++g_launches;
  }

  const size_t rows = (size_t)d->total_tokens * (size_t)d->H;
  // dq is reduced in FP32: straight into the output when it is FP32, else in
  // the workspace and converted at the end
  const bool dq_direct = d->out_dtype == HSTU_FP32;
  float* dq_acc = dq_direct ? static_cast<float*>(a->dq) : reinterpret_cast<float*>(ws + L.dq_acc);
  const bool has_rp = a->rab_pos != nullptr;
  const bool has_rt = a->rab_time != nullptr && a->timestamps != nullptr;
  // d_rab outputs and the dq accumulator start from zero: on the tensor-core
  // path the norm-gate backward kernel zeroes them on its way (the attention
  // kernel then adds each CTA's d_rab partial sums), otherwise memsets do
  const bool fused_zero = tc && d->total_tokens > 0;
  if (!fused_zero) {
    if (a->d_rab_pos)
      HSTU_CUDA_TRY(cudaMemsetAsync(a->d_rab_pos, 0, sizeof(float) * d->H * d->num_pos_buckets, st));
    if (a->d_rab_time)
      HSTU_CUDA_TRY(cudaMemsetAsync(a->d_rab_time, 0, sizeof(float) * d->H * d->num_time_buckets, st));
  }
  if (d->total_tokens == 0) return HSTU_OK;
  if (!fused_zero) HSTU_CUDA_TRY(cudaMemsetAsync(dq_acc, 0, sizeof(float) * rows * d->d_qk, st));
  // per-CTA d_rab partial sums: each tensor-core CTA zeroes its own row first
  float* drab_partial = reinterpret_cast<float*>(ws + L.drab_part);

  // gradient w.r.t. o, in the input type (an MMA operand of the attention backward)
  {
    NormParams np{};
    np.dtype = (d->flags & HSTU_FLAG_U_FP32) ? HSTU_FP32 : d->dtype; np.out_dtype = d->out_dtype;
    np.o = a->o; np.u = a->u; np.dy = a->dy; np.dO = ws + L.dO; np.du = a->du;
    np.split = tc ? 1 : 0;
    np.dO_lo = ws + L.dO + sizeof(__nv_bfloat16) * rows * (size_t)d->d_v;
    np.T = d->total_tokens; np.F = d->H * d->d_v; np.norm = d->norm; np.eps = d->ln_eps;
    set_dropout(np, d, a->dropout_seed, a->dropout_offset);
    if (fused_zero) {  // d_qk == d_v and H * d_qk % 4 == 0 on this path
      np.zero_rows = dq_acc; np.zero_F = d->H * d->d_qk;
      np.zero_a = a->d_rab_pos; np.zero_a_n = a->d_rab_pos ? d->H * d->num_pos_buckets : 0;
      np.zero_b = a->d_rab_time; np.zero_b_n = a->d_rab_time ? d->H * d->num_time_buckets : 0;
    }
    if (reuse) {
      np.pc_hdr = pp.hdr;
      np.pc_off = a->seq_offsets; np.pc_nt = a->num_targets; np.pc_nc = a->num_contexts;
      np.pc_ts = a->timestamps;
      np.pc_sv_off = reinterpret_cast<const int64_t*>(ws + L.sv_off);
      np.pc_sv_t0 = reinterpret_cast<const int64_t*>(ws + L.sv_t0);
      np.pc_sv_nt = reinterpret_cast<const int32_t*>(ws + L.sv_nt);
      np.pc_sv_nc = reinterpret_cast<const int32_t*>(ws + L.sv_nc);
      np.pc_B = d->B;
      np.pc_tile = plan.BM | (plan.BN << 16);
      np.pc_max_n = d->max_seq_len;
    }
    HSTU_CUDA_TRY(launch_norm_gate_bwd(np, st));
    ++g_launches;
  }
  const void* dO = ws + L.dO;  // FP32, or the hi part followed by the lo part

  AttnParams p{};
  p.off = a->seq_offsets; p.nt = a->num_targets; p.nc = a->num_contexts;
  p.ts = a->timestamps; p.rab_pos = a->rab_pos; p.rab_time = has_rt ? a->rab_time : nullptr;
  p.q = a->q; p.k = a->k; p.v = a->v; p.dO = dO; p.dk = a->dk; p.dv = a->dv; p.dq_acc = dq_acc;
  p.d_rab_pos = has_rp ? a->d_rab_pos : nullptr;
  p.d_rab_time = has_rt ? a->d_rab_time : nullptr;
  p.drab_partial = drab_partial;
  p.hdr = pp.hdr; p.hdr_rw = pp.hdr; p.blocks = plan.blocks; p.items = plan.items;
  p.B = d->B; p.H = d->H; p.dqk = d->d_qk; p.dv_dim = d->d_v; p.T = d->total_tokens;
  p.dtype = d->dtype; p.out_dtype = d->out_dtype;
  p.alpha = d->alpha; p.inv_n = 1.0f / (float)d->max_seq_len;
  set_score_constants(p);
  p.P = d->num_pos_buckets; p.Tb = d->num_time_buckets; p.flags = d->flags;
  p.num_sms = dev_info().sms;
  {
    KernelTimer timer(st);
    if (tc) {
      HSTU_CUDA_TRY(launch_tc_bwd(p, st));  // its CTAs add their d_rab partial sums at exit
    } else {
      const int max_items = ((int)((d->total_tokens + kSimtTile - 1) / kSimtTile) + d->B) * d->H;
      HSTU_CUDA_TRY(launch_simt_bwd(p, max_items, st));
    }
  }
  ++g_launches;
  if (!dq_direct) {
    HSTU_CUDA_TRY(launch_convert_f32(dq_acc, a->dq, (int64_t)(rows * d->d_qk), d->out_dtype, st));
    ++g_launches;
  }
  return HSTU_OK;
}

hstu_status_t hstu_attn_fwd_delta(const hstu_attn_desc* d, const hstu_attn_delta_args* a, void* workspace,
                                  size_t workspace_bytes, hstu_stream_t stream) {
  hstu_status_t s = check_desc(d);
  if (s != HSTU_OK) return s;
  if (!a || !a->cand_offsets || !a->cache_offsets || a->cache_tokens < 0) return HSTU_ERR_INVALID_ARG;
  if (d->dropout_p > 0.f) return HSTU_ERR_UNSUPPORTED;  // inference: no dropout
  if (d->flags & (HSTU_FLAG_PLAN_BWD | HSTU_FLAG_REUSE_PLAN)) return HSTU_ERR_INVALID_ARG;
  if (d->total_tokens > 0 && (!a->q || !a->k || !a->v || !a->o)) return HSTU_ERR_INVALID_ARG;
  if (d->total_tokens > 0 && a->cache_tokens > 0 && (!a->k_cache || !a->v_cache)) return HSTU_ERR_INVALID_ARG;
  if (a->cache_tokens > 0 && (a->cand_timestamps == nullptr) != (a->cache_timestamps == nullptr))
    return HSTU_ERR_INVALID_ARG;
  for (const void* ptr : {a->q, a->k, a->v, a->u, a->k_cache, a->v_cache, (const void*)a->o, (const void*)a->y})
    if (ptr && !aligned16(ptr)) return HSTU_ERR_INVALID_ARG;
  // tensor-core path only: 128-row TMA boxes over both token tensors
  if ((d->flags & HSTU_FLAG_FORCE_SIMT) || dev_info().cc != 103 || !tc_fwd_supported(d->dtype, d->d_qk, d->d_v) ||
      tc_fwd_smem_bytes(d->d_qk, d->H, d->num_pos_buckets, d->num_time_buckets) > kMaxSmemPerCta ||
      (d->total_tokens > 0 && d->total_tokens < kTcTile) || (a->cache_tokens > 0 && a->cache_tokens < kTcTile) ||
      a->cache_tokens > (int64_t)0x7fffffff)
    return HSTU_ERR_UNSUPPORTED;
  const WsLayout L = ws_layout(d, false);
  if ((s = check_ws(workspace, workspace_bytes, L.total)) != HSTU_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  g_launches = 0;
  clear_detail();

  PlanParams pp = plan_params(d, a->cand_offsets, nullptr, nullptr, a->cand_timestamps, 2, true, ws, L);
  pp.off2 = a->cache_offsets;
  pp.T2 = a->cache_tokens;
  HSTU_CUDA_TRY(launch_plan(pp, st));
  ++g_launches;
  if (d->total_tokens == 0) return HSTU_OK;

  AttnParams p{};
  p.off = a->cand_offsets; p.nt = nullptr; p.nc = nullptr;
  p.ts = a->cand_timestamps; p.rab_pos = a->rab_pos;
  p.rab_time = a->cand_timestamps ? a->rab_time : nullptr;
  p.q = a->q; p.k = a->k; p.v = a->v; p.o = a->o;
  p.off2 = a->cache_offsets; p.ts2 = a->cache_timestamps; p.k2 = a->k_cache; p.v2 = a->v_cache;
  p.T2 = a->cache_tokens;
  p.hdr = pp.hdr; p.hdr_rw = pp.hdr; p.blocks = pp.out[0].blocks; p.items = pp.out[0].items;
  p.B = d->B; p.H = d->H; p.dqk = d->d_qk; p.dv_dim = d->d_v; p.T = d->total_tokens;
  p.dtype = d->dtype; p.out_dtype = d->out_dtype;
  p.alpha = d->alpha; p.inv_n = 1.0f / (float)d->max_seq_len;
  set_score_constants(p);
  p.P = d->num_pos_buckets; p.Tb = d->num_time_buckets; p.flags = d->flags;
  p.num_sms = dev_info().sms;
  {
    KernelTimer timer(st);
    HSTU_CUDA_TRY(launch_tc_fwd_delta(p, st));
  }
  ++g_launches;
  if (a->y || a->ln_mean || a->ln_rstd) {
    NormParams np{};
    np.dtype = (d->flags & HSTU_FLAG_U_FP32) ? HSTU_FP32 : d->dtype; np.out_dtype = d->out_dtype;
    np.o = a->o; np.u = a->u; np.y = a->y; np.mean = a->ln_mean; np.rstd = a->ln_rstd;
    np.T = d->total_tokens; np.F = d->H * d->d_v; np.norm = d->norm; np.eps = d->ln_eps;
    HSTU_CUDA_TRY(launch_norm_gate_fwd(np, st));
    ++g_launches;
  }
  return HSTU_OK;
}

hstu_status_t hstu_attn_debug_plan(const hstu_attn_desc* d, const int64_t* seq_offsets,
                                   const int32_t* num_targets, const int32_t* num_contexts, int32_t pass,
                                   void* workspace, size_t workspace_bytes, int32_t* host_tiles,
                                   int64_t host_capacity, int64_t* n_tiles, hstu_stream_t stream) {
  hstu_status_t s = check_desc(d);
  if (s != HSTU_OK) return s;
  if (!seq_offsets || !n_tiles || (pass != 0 && pass != 1) || host_capacity < 0 ||
      (host_capacity > 0 && !host_tiles))
    return HSTU_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(d, false);
  const size_t need = L.plan_end + align_up(sizeof(int32_t) * 6 * (size_t)host_capacity);
  if ((s = check_ws(workspace, workspace_bytes, need)) != HSTU_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const bool tc = use_tc(d, pass == 1);
  const PlanParams pp = plan_params(d, seq_offsets, num_targets, num_contexts, nullptr, pass, tc, ws, L);
  int32_t* rec = reinterpret_cast<int32_t*>(ws + L.plan_end);
  HSTU_CUDA_TRY(launch_plan(pp, st));
  HSTU_CUDA_TRY(launch_debug_tiles(pp, rec, host_capacity, st));
  int32_t hdr[4] = {0, 0, 0, 0};
  HSTU_CUDA_TRY(cudaMemcpyAsync(hdr, ws, sizeof(hdr), cudaMemcpyDeviceToHost, st));
  HSTU_CUDA_TRY(cudaStreamSynchronize(st));
  if (hdr[WS_ERR] != 0) return (hstu_status_t)hdr[WS_ERR];
  *n_tiles = hdr[WS_NTILES];
  const int64_t copy = hdr[WS_NTILES] < host_capacity ? hdr[WS_NTILES] : host_capacity;
  if (copy > 0) {
    HSTU_CUDA_TRY(cudaMemcpyAsync(host_tiles, rec, sizeof(int32_t) * 6 * (size_t)copy,
                                  cudaMemcpyDeviceToHost, st));
    HSTU_CUDA_TRY(cudaStreamSynchronize(st));
  }
  return HSTU_OK;
}

hstu_status_t hstu_get_device_error(const void* workspace, hstu_stream_t stream, int32_t* code) {
  if (!workspace || !code) return HSTU_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  HSTU_CUDA_TRY(cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st));
  HSTU_CUDA_TRY(cudaStreamSynchronize(st));
  *code = v;
  return HSTU_OK;
}

}  // extern "C"
