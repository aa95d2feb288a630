// attn_fwd_noalloc: the attention forward for callers that cannot hand the
// library a workspace.
//
// attn_fwd needs 256 bytes of device scratch (the persistent scheduler's
// work counter and the device error record), which the caller normally
// allocates once and passes in. Some callers have no way to do that: code
// embedded in a host framework that owns every device allocation through its
// own pool and exposes only tensors and a stream, or serving loops that are
// not allowed to allocate after start-up. For them this entry point keeps the
// scratch in a fixed array inside the library instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds its own copy until the process exits. Host code cannot use
// the array's name as a device address; its device address is looked up with
// cudaGetSymbolAddress (with the device current). The first call on a device
// does that set-up; make it before any stream capture begins. Later calls
// look the address up again whenever their stream is not capturing (the
// lookup allocates nothing), so a context that was torn down and recreated
// (cudaDeviceReset) never receives a stale address; while a capture is
// running they reuse the address found before it.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = ATTN_FWD_STATIC_WORKSPACE_BYTES;
static_assert(kStaticWorkspaceBytes >= af::kWsWords * sizeof(uint32_t), "static workspace too small");

static __device__ __align__(256) uint32_t g_static_workspace[kStaticWorkspaceBytes / sizeof(uint32_t)];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_workspace_ptr[kMaxDevices] = {};

// Device address of the current device's copy of the array: looked up again
// on every call made outside a stream capture, reused from the last lookup
// inside one.
attn_status static_workspace(cudaStream_t stream, void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return af::report_error(ATTN_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return af::report_error(ATTN_ERR_UNSUPPORTED, "device index %d beyond the %d devices supported", dev, kMaxDevices);
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &capture);
  if (e != cudaSuccess)
    return af::report_error(ATTN_ERR_CUDA, "cudaStreamIsCapturing failed: %s", cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (capture != cudaStreamCaptureStatusNone && g_workspace_ptr[dev] == nullptr)
    return af::report_error(ATTN_ERR_INVALID_ARG, "the first attn_fwd_noalloc call on a device must come before "
                            "any stream capture (it looks up the static workspace's address)");
  if (capture == cudaStreamCaptureStatusNone) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_workspace);
    if (e != cudaSuccess || ptr == nullptr)
      return af::report_error(ATTN_ERR_CUDA, "cudaGetSymbolAddress of the static workspace failed: %s",
                              cudaGetErrorString(e));
    g_workspace_ptr[dev] = ptr;
  }
  *out = g_workspace_ptr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_fwd_noalloc(const attn_fwd_params* p, attn_stream_t stream) {
  if (p == nullptr) return af::report_error(ATTN_ERR_INVALID_ARG, "params is NULL");
  attn_fwd_params q = *p;
  // Split-KV partial results do not fit the fixed array: the automatic
  // choice becomes "no split" here, and an explicit split count is refused
  // below as needing more scratch.
  if (q.num_splits == 0) q.num_splits = 1;
  const size_t need = attn_fwd_workspace_bytes(&q);
  if (need > kStaticWorkspaceBytes)
    return af::report_error(ATTN_ERR_UNSUPPORTED,
                            "this call needs %zu bytes of scratch, more than the %zu-byte static workspace", need,
                            kStaticWorkspaceBytes);
  void* ws = nullptr;
  attn_status st = static_workspace(reinterpret_cast<cudaStream_t>(stream), &ws);
  if (st != ATTN_OK) return st;
  q.workspace = ws;
  q.workspace_bytes = kStaticWorkspaceBytes;
  attn_fwd_plan_info info;
  st = attn_fwd_plan(&q, &info);   // validate before anything is enqueued
  if (st != ATTN_OK) return st;
  // The array keeps whatever the previous call left; the scheduler counters
  // and the error record must start at zero.
  cudaError_t e = cudaMemsetAsync(ws, 0, af::kWsWords * sizeof(uint32_t), reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return af::report_error(ATTN_ERR_CUDA, "clearing the static workspace failed: %s", cudaGetErrorString(e));
  return attn_fwd(&q, stream);
}
