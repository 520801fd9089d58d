// Forward entry point for callers that cannot allocate device memory.
//
// Some callers of this library are not allowed to call cudaMalloc: a host
// framework that owns every byte of device memory through its own pool, a
// serving process whose latency budget cannot absorb an allocation (which can
// synchronise the device), or an integration that simply has no allocator to
// hand.  hstu_attn_fwd_noalloc takes the forward pass's scratch (the tile
// plan: workspace header, per-sequence block starts, block lists) from a
// fixed buffer compiled into the library instead of a caller workspace.
//
// The buffer is a file-scope __device__ array of kScratchBytes; every GPU that
// loads the library holds it until the process exits.  Host code cannot hand
// the array's name to a kernel (on the host it is only a stand-in, not a
// device address), so every call looks its device address up with
// cudaGetSymbolAddress while the stream's device is current.  The lookup is a
// host call and is not cached: a cached address would outlive a device reset
// (cudaDeviceReset) or a new context and then point at freed memory.
#include <cstdio>

#include "hstu_internal.h"

static constexpr size_t kScratchBytes = size_t(1) << 20;  // 1 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

extern "C" hstu_status_t hstu_attn_fwd_noalloc(const hstu_attn_desc* desc, const hstu_attn_fwd_args* args,
                                               hstu_stream_t stream, int32_t* host_device_error) {
  size_t need = 0;
  hstu_status_t s = hstu_attn_workspace_size(desc, &need, nullptr);
  if (s != HSTU_OK) return s;
  // the built-in scratch holds a forward plan only
  if (desc->flags & (HSTU_FLAG_PLAN_BWD | HSTU_FLAG_REUSE_PLAN)) return HSTU_ERR_INVALID_ARG;
  if (need > kScratchBytes) {
    char msg[160];
    snprintf(msg, sizeof(msg), "this problem needs %zu bytes of forward scratch; the built-in buffer holds %zu",
             need, kScratchBytes);
    hstu::set_detail_message(msg);
    return HSTU_ERR_WORKSPACE;
  }
  // the scratch belongs to the current device: a stream of another device
  // would run the kernels against memory of the wrong GPU
  int dev = -1, stream_dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaStreamGetDevice(reinterpret_cast<cudaStream_t>(stream), &stream_dev);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    hstu::set_error_detail(e, "cudaGetDevice / cudaStreamGetDevice before the built-in forward scratch");
    return HSTU_ERR_CUDA;
  }
  if (stream_dev != dev) {
    hstu::set_detail_message("the stream belongs to another device than the current one");
    return HSTU_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  e = cudaGetSymbolAddress(&scratch, g_noalloc_scratch);
  if (e != cudaSuccess || scratch == nullptr) {
    (void)cudaGetLastError();
    hstu::set_error_detail(e, "cudaGetSymbolAddress of the built-in forward scratch");
    return HSTU_ERR_CUDA;
  }
  // The planner rewrites the whole plan region, header first, on every call,
  // so nothing left by an earlier call is read.
  s = hstu_attn_fwd(desc, args, scratch, kScratchBytes, stream);
  if (s != HSTU_OK || host_device_error == nullptr) return s;
  return hstu_get_device_error(scratch, stream, host_device_error);
}
