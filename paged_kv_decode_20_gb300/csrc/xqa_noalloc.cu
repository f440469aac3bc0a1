// xqa_decode_noalloc: the grouped-query decode call with its scratch memory
// (split-KV partials and reduction tickets) taken from a fixed array that is
// part of this library, so the caller passes only inputs and outputs.
//
// Who needs it: callers that cannot hand the library a workspace because they
// may not allocate device memory at the point of the call -- for example a
// serving runtime that reserves nearly all device memory for its KV-cache pool
// up front and forbids further allocations, or a host application whose device
// allocator is owned by someone else and is not reachable from this call site.
//
// The scratch is a file-scope __device__ array of fixed size.  Every GPU that
// loads this library keeps it for the life of the process (64 MiB + 64 KiB),
// whether or not this entry point is ever called.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "xqa.h"
#include "xqa_internal.h"

namespace {

constexpr size_t kScratchWorkspaceBytes = size_t(64) << 20;  // split partials
constexpr size_t kScratchSemaphores = size_t(16) << 10;      // reduction tickets

static __device__ __align__(256) unsigned char g_scratch_workspace[kScratchWorkspaceBytes];
static __device__ __align__(256) uint32_t g_scratch_semaphores[kScratchSemaphores];

constexpr int kMaxDevices = 64;

struct DeviceScratch {
  void* workspace = nullptr;
  uint32_t* semaphores = nullptr;
};

// Device addresses of the two arrays on device `dev` (the current device),
// looked up on the first call that succeeds and kept from then on; a failed
// lookup (for example one attempted during a stream capture) is not kept, so
// a later call tries again.  The host-side symbols are stand-ins and must
// never be passed to a kernel.
cudaError_t scratch_for(int dev, DeviceScratch* out) {
  static DeviceScratch table[kMaxDevices];
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  DeviceScratch& d = table[dev];
  if (!d.workspace || !d.semaphores) {
    DeviceScratch fresh;
    cudaError_t e = cudaGetSymbolAddress(&fresh.workspace, g_scratch_workspace);
    if (e == cudaSuccess)
      e = cudaGetSymbolAddress(reinterpret_cast<void**>(&fresh.semaphores), g_scratch_semaphores);
    if (e != cudaSuccess) return e;
    d = fresh;
  }
  *out = d;
  return cudaSuccess;
}

xqa_status fail(xqa_status st, const char* msg) {
  xqa::set_last_error(msg);
  return st;
}

}  // namespace

extern "C" xqa_status xqa_decode_noalloc(const xqa_params* params, xqa_stream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(XQA_ERR_CUDA, "xqa_decode_noalloc: no current device");
  if (dev < 0 || dev >= kMaxDevices) return fail(XQA_ERR_UNSUPPORTED, "xqa_decode_noalloc: device index too large");
  const size_t need_ws = xqa_workspace_size(params, 0);
  if (need_ws == size_t(-1)) return xqa_decode(params, nullptr, 0, nullptr, stream);  // reports why
  const size_t need_sems = xqa_semaphore_count(params);
  if (need_ws > kScratchWorkspaceBytes || need_sems > kScratchSemaphores) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "xqa_decode_noalloc: problem needs %zu workspace bytes and %zu semaphores; the built-in "
             "scratch holds %zu bytes and %zu semaphores (use xqa_decode with your own buffers)",
             need_ws, need_sems, kScratchWorkspaceBytes, kScratchSemaphores);
    return fail(XQA_ERR_WORKSPACE_TOO_SMALL, msg);
  }
  DeviceScratch s;
  e = scratch_for(dev, &s);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof msg, "xqa_decode_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
    return fail(XQA_ERR_CUDA, msg);
  }
  // Tickets must start at zero; a call that was cut short could have left some set.
  e = cudaMemsetAsync(s.semaphores, 0, need_sems * sizeof(uint32_t), reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(XQA_ERR_CUDA, "xqa_decode_noalloc: clearing the tickets failed");
  return xqa_decode(params, s.workspace, kScratchWorkspaceBytes, s.semaphores, stream);
}
