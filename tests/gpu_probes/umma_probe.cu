// Single-CTA checks of the tcgen05 building blocks in csrc/umma.cuh: shared
// memory descriptors (K-major and MN-major, 128-byte swizzle), the kind::f16
// instruction descriptor, A from tensor memory, commit and 32x32b loads.
// Every operand buffer is sized so that any reading of the descriptor stays
// inside this kernel's shared memory.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "umma.cuh"

using namespace xqa;

namespace {

constexpr int kA = 0;            // A: 128 rows x 64 elements, 16 KB
constexpr int kB = 16384;        // B: up to 48 KB
constexpr int kBar = 16384 + 49152;
constexpr int kSmem = kBar + 64 + 1024;

__device__ void fill_rows(uint8_t* dst, const __nv_bfloat16* src, int rows, int row_elems_src,
                          int col0) {
  // row r of the tile = src[r * row_elems_src + col0 .. +64], swizzled 128B
  for (int idx = threadIdx.x; idx < rows * 8; idx += blockDim.x) {
    const int r = idx >> 3, u = idx & 7;
    const uint4 v = *reinterpret_cast<const uint4*>(src + size_t(r) * row_elems_src + col0 + 8 * u);
    *reinterpret_cast<uint4*>(dst + umma::sw128(r, u)) = v;
  }
}

// rows of 64 bytes with the 64-byte swizzle (row r of the tile = src row r)
__device__ void fill_rows64(uint8_t* dst, const uint8_t* src, int rows) {
  for (int idx = threadIdx.x; idx < rows * 4; idx += blockDim.x) {
    const int r = idx >> 2, u = idx & 3;
    const uint4 v = *reinterpret_cast<const uint4*>(src + size_t(r) * 64 + 16 * u);
    *reinterpret_cast<uint4*>(dst + umma::sw64(r, u)) = v;
  }
}

// mode 0: D[128x64] = A . B^T, A and B K-major in shared memory
// mode 1: D[128x256] = A . V, V [64 x 256] MN-major (4 chunks of 64 columns)
// mode 2: D[128x64] = A . B^T with A in tensor memory
// mode 3: as mode 0 with E4M3 A [128 x 128] and B [64 x 128] (kind::f8f6f4,
//         K = 32 per instruction, 128-byte swizzle)
// mode 4: as mode 3 with A in tensor memory (four codes per column)
// mode 5: E4M3 A [128 x 64] and B [64 x 64], rows of 64 bytes with the 64-byte swizzle
// mode 6: as mode 1 with f16 A and V
__global__ void probe_kernel(int mode, const __nv_bfloat16* A, const __nv_bfloat16* B, float* D,
                             int lbo, int sbo, int* status) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + kBar + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    umma::tmem_alloc(tslot, 512);
    umma::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (mode == 5) {
    fill_rows64(sm + kA, reinterpret_cast<const uint8_t*>(A), 128);
    fill_rows64(sm + kB, reinterpret_cast<const uint8_t*>(B), 64);
  } else {
    // (an E4M3 row of 128 codes is 128 bytes, filled like 64 16-bit elements)
    fill_rows(sm + kA, A, 128, 64, 0);
    if (mode == 1 || mode == 6) {
      for (int c = 0; c < 4; ++c) fill_rows(sm + kB + c * 8192, B, 64, 256, 64 * c);
    } else {
      fill_rows(sm + kB, B, 64, 64, 0);
    }
  }
  umma::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tslot;
  const int N = (mode == 1 || mode == 6) ? 256 : 64;
  if (mode == 2 || mode == 4) {
    // row t of A into lane t, columns 256.. (two bf16 per 32-bit column)
    uint32_t w[32];
    const uint32_t* src = reinterpret_cast<const uint32_t*>(A + size_t(threadIdx.x) * 64);
    for (int i = 0; i < 32; ++i) w[i] = src[i];
    umma::tmem_st32(tmem + (uint32_t(32 * warp) << 16) + 256, w);
    umma::tmem_st_wait();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
  }
  if (threadIdx.x == 0) {
    const uint32_t a0 = smem_u32(sm + kA), b0 = smem_u32(sm + kB);
    for (int k = 0; k < 4; ++k) {
      if (mode == 0) {
        umma::mma_ss(tmem, umma::smem_desc(a0 + 32 * k, 16, 1024, umma::kSw128),
                     umma::smem_desc(b0 + 32 * k, 16, 1024, umma::kSw128),
                     umma::idesc_f16(128, 64, true, false, false), k > 0);
      } else if (mode == 1) {
        umma::mma_ss(tmem, umma::smem_desc(a0 + 32 * k, 16, 1024, umma::kSw128),
                     umma::smem_desc(b0 + 2048 * k, lbo, sbo, umma::kSw128),
                     umma::idesc_f16(128, 256, true, false, true), k > 0);
      } else if (mode == 2) {
        umma::mma_ts(tmem, tmem + 256 + 8 * k, umma::smem_desc(b0 + 32 * k, 16, 1024, umma::kSw128),
                     umma::idesc_f16(128, 64, true, false, false), k > 0);
      } else if (mode == 3) {
        umma::mma_ss_f8(tmem, umma::smem_desc(a0 + 32 * k, 16, 1024, umma::kSw128),
                        umma::smem_desc(b0 + 32 * k, 16, 1024, umma::kSw128),
                        umma::idesc_e4m3(128, 64, false, false), k > 0);
      } else if (mode == 4) {
        umma::mma_ts_f8(tmem, tmem + 256 + 8 * k, umma::smem_desc(b0 + 32 * k, 16, 1024, umma::kSw128),
                        umma::idesc_e4m3(128, 64, false, false), k > 0);
      } else if (mode == 5) {
        if (k < 2)
          umma::mma_ss_f8(tmem, umma::smem_desc(a0 + 32 * k, 16, 512, umma::kSw64),
                          umma::smem_desc(b0 + 32 * k, 16, 512, umma::kSw64),
                          umma::idesc_e4m3(128, 64, false, false), k > 0);
      } else {
        umma::mma_ss(tmem, umma::smem_desc(a0 + 32 * k, 16, 1024, umma::kSw128),
                     umma::smem_desc(b0 + 2048 * k, lbo, sbo, umma::kSw128),
                     umma::idesc_f16(128, 256, false, false, true), k > 0);
      }
    }
    umma::commit(bar);
  }
  const bool ok = mbar_wait(bar, 0);
  if (!ok && lane == 0) atomicOr(status, 1);
  umma::fence_after_sync();
  if (ok) {
    for (int c = 0; c < N; c += 32) {
      float v[32];
      umma::tmem_ld32(tmem + (uint32_t(32 * warp) << 16) + c, v);
      umma::tmem_ld_wait();
      for (int i = 0; i < 32; ++i) D[size_t(threadIdx.x) * N + c + i] = v[i];
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 0) umma::tmem_dealloc(tmem, 512);
}

}  // namespace

extern "C" int umma_probe(int mode, const void* A, const void* B, void* D, int lbo, int sbo,
                          int* status) {
  cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  probe_kernel<<<1, 128, kSmem>>>(mode, static_cast<const __nv_bfloat16*>(A),
                                  static_cast<const __nv_bfloat16*>(B), static_cast<float*>(D), lbo,
                                  sbo, status);
  cudaError_t e = cudaDeviceSynchronize();
  return int(e);
}
