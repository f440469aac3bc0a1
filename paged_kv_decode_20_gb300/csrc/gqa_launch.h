// Host-side entry points of the grouped-query decode kernels (one translation
// unit per KV element type, so they compile in parallel).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "kernel_args.h"

namespace xqa {

// kv: 0 f16, 1 bf16, 2 e4m3.  row_blocks: 16-row MMA blocks per consumer
// warp; warp_rows: warp row groups splitting a CTA's rows (1, 2 or 4; built
// for e4m3 K/V only, since larger 16-bit tiles take the tensor-core kernel).
// Returns cudaErrorInvalidValue when no kernel is built for (kv, head_dim,
// row_blocks, warp_rows).  With launch == false only the occupancy (CTAs per
// SM) is reported.
cudaError_t gqa_launch_f16(int head_dim, int row_blocks, int warp_rows, bool launch, dim3 grid,
                           const CUtensorMap* tk, const CUtensorMap* tv, const DecodeArgs* args,
                           cudaStream_t stream, int* ctas_per_sm);
cudaError_t gqa_launch_bf16(int head_dim, int row_blocks, int warp_rows, bool launch, dim3 grid,
                            const CUtensorMap* tk, const CUtensorMap* tv, const DecodeArgs* args,
                            cudaStream_t stream, int* ctas_per_sm);
cudaError_t gqa_launch_e4m3(int head_dim, int row_blocks, int warp_rows, bool launch, dim3 grid,
                            const CUtensorMap* tk, const CUtensorMap* tv, const DecodeArgs* args,
                            cudaStream_t stream, int* ctas_per_sm);

// The tensor-core grouped-query kernel (16-bit K/V, head_dim 64 or 128) for
// more than 16 (head_dim 128) or 32 (head_dim 64) query rows per kv head: 128
// rows per CTA, one CTA per SM.
cudaError_t gqa_tc_launch(bool bf16, int head_dim, bool launch, dim3 grid, const CUtensorMap* tk,
                          const CUtensorMap* tv, const DecodeArgs* args, cudaStream_t stream, int* ctas_per_sm);

}  // namespace xqa
