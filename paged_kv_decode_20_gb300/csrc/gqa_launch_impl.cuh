// Shared body of the per-dtype launch functions.
#pragma once
#include "gqa_kernel.cuh"
#include "gqa_launch.h"

namespace xqa {

template <int KV, int D, int RB, int WR>
cudaError_t gqa_launch_one(bool launch, dim3 grid, const CUtensorMap* tk, const CUtensorMap* tv,
                           const DecodeArgs* args, cudaStream_t stream, int* ctas_per_sm) {
  const bool pdl = args && args->pdl;
  using C = GqaCfg<KV, D, RB, WR>;
  auto kern = gqa_decode_kernel<KV, D, RB, WR>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  if (ctas_per_sm) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, kern, C::kThreads, C::kSmem);
    if (e != cudaSuccess) return e;
  }
  if (!launch) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, *tk, *tv, *args);
}

}  // namespace xqa
