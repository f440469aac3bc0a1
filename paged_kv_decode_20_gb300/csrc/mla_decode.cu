// MLA latent decode (vLLM Kimi-K3 MultiHeadLatentAttention page: forward_mqa
// on the absorbed query; head_size = kv_lora_rank + qk_rope_head_dim).
#include <stdio.h>

#include "mla_launch.h"

namespace xqa {

size_t mla_workspace_size(const xqa_params*, int, int) { return size_t(-1); }
size_t mla_semaphore_count(const xqa_params*, int) { return size_t(-1); }

xqa_status mla_decode(const xqa_params*, int, void*, size_t, uint32_t*, cudaStream_t, char* err,
                      size_t err_len) {
  snprintf(err, err_len, "the MLA latent kernel is not built yet");
  return XQA_ERR_UNSUPPORTED;
}

}  // namespace xqa
