// Grouped-query decode kernels with float8 e4m3 K/V ("fp8 compute": K/V are
// widened to f16 in registers; a bf16 query is rescaled into f16 exactly).
#include "gqa_launch_impl.cuh"

namespace xqa {

cudaError_t gqa_launch_e4m3(int head_dim, int row_blocks, int warp_rows, bool launch, dim3 grid,
                            const CUtensorMap* tk, const CUtensorMap* tv, const DecodeArgs* args,
                            cudaStream_t stream, int* ctas_per_sm) {
  if (head_dim == 128 && row_blocks == 1 && warp_rows == 1)
    return gqa_launch_one<kKvE4m3, 128, 1, 1>(launch, grid, tk, tv, args, stream, ctas_per_sm);
  if (head_dim == 128 && row_blocks == 1 && warp_rows == 2)
    return gqa_launch_one<kKvE4m3, 128, 1, 2>(launch, grid, tk, tv, args, stream, ctas_per_sm);
  if (head_dim == 128 && row_blocks == 1 && warp_rows == 4)
    return gqa_launch_one<kKvE4m3, 128, 1, 4>(launch, grid, tk, tv, args, stream, ctas_per_sm);
  return cudaErrorInvalidValue;
}

}  // namespace xqa
