// Grouped-query decode kernels with f16 K/V (and f16 q / output).
#include "gqa_launch_impl.cuh"

namespace xqa {

cudaError_t gqa_launch_f16(int head_dim, int row_blocks, int warp_rows, bool launch, dim3 grid,
                            const CUtensorMap* tk, const CUtensorMap* tv, const DecodeArgs* args,
                            cudaStream_t stream, int* ctas_per_sm) {
  if (head_dim == 64 && row_blocks == 1 && warp_rows == 1)
    return gqa_launch_one<kKvF16, 64, 1, 1>(launch, grid, tk, tv, args, stream, ctas_per_sm);
  if (head_dim == 64 && row_blocks == 2 && warp_rows == 1)
    return gqa_launch_one<kKvF16, 64, 2, 1>(launch, grid, tk, tv, args, stream, ctas_per_sm);
  if (head_dim == 128 && row_blocks == 1 && warp_rows == 1)
    return gqa_launch_one<kKvF16, 128, 1, 1>(launch, grid, tk, tv, args, stream, ctas_per_sm);
  return cudaErrorInvalidValue;
}

}  // namespace xqa
