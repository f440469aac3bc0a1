// A read-only streaming kernel: the HBM read rate that the decode kernels,
// which read the cache and write little, are measured beside.  Not part of
// the decode path.
#include <cuda_runtime.h>
#include <stdint.h>

#include "xqa.h"
#include "xqa_internal.h"

namespace {

constexpr int kThreads = 512;
constexpr int kUnroll = 4;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Every thread folds kUnroll 16-byte loads per step of a grid-stride loop
// into one word; the word is stored only if it equals `never`, which keeps
// the loads without writing.
__global__ void __launch_bounds__(kThreads) read_stream_kernel(const uint4* __restrict__ p, size_t n16,
                                                               uint32_t* sink, uint32_t never) {
  uint32_t acc = 0;
  const size_t stride = size_t(gridDim.x) * kThreads;
  size_t i = size_t(blockIdx.x) * kThreads + threadIdx.x;
  for (; i + (kUnroll - 1) * stride < n16; i += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream(p + i + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = ld_stream(p + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == never) sink[blockIdx.x] = acc;
}

}  // namespace

extern "C" xqa_status xqa_read_bandwidth_probe(const void* buf, size_t bytes, uint32_t* sink, int sink_words,
                                               xqa_stream_t stream) {
  if (!buf || !sink || bytes == 0 || (bytes & 15) || (reinterpret_cast<uintptr_t>(buf) & 15) || sink_words <= 0) {
    xqa::set_last_error("read probe: buf and sink non-null, bytes a non-zero multiple of 16, buf 16-byte aligned");
    return XQA_ERR_INVALID_ARG;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess) {
    xqa::set_last_error("read probe: cannot query the device");
    return XQA_ERR_CUDA;
  }
  const int grid = sms * 4 < sink_words ? sms * 4 : sink_words;
  read_stream_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(buf), bytes / 16, sink, 0x9e3779b9u);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    xqa::set_last_error(cudaGetErrorString(e));
    return XQA_ERR_CUDA;
  }
  return XQA_OK;
}
