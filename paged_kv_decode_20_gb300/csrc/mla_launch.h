// Host-side entry of the MLA latent decode kernel (one 576-wide latent kv
// head, V = its first 512 elements).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

#include "xqa.h"

namespace xqa {

size_t mla_workspace_size(const xqa_params* p, int v_head_dim, int sm_count);
size_t mla_semaphore_count(const xqa_params* p, int v_head_dim);
xqa_status mla_decode(const xqa_params* p, int v_head_dim, void* ws, size_t ws_bytes,
                      uint32_t* sems, cudaStream_t stream, char* err, size_t err_len);

}  // namespace xqa
