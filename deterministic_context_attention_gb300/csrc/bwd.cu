// bwd.cu -- deterministic backward (placeholder until the kernels land).
#include <cuda_runtime.h>

#include "../../include/rlk_attn.h"
#include "rlk_internal.h"

namespace rlk {

size_t backward_workspace_bytes(const rlk_attn_params* prm, const int32_t* cu) {
  const size_t rows = static_cast<size_t>(cu[prm->num_seqs]);
  return (rows * prm->num_q_heads * sizeof(float) + 255) / 256 * 256;
}

rlk_status run_backward(const rlk_attn_params*, const void*, const void*, const void*, const float*, const void*,
                        const float*, const int32_t*, int32_t, float*, float*, float*, void*, size_t, cudaStream_t) {
  return RLK_ERR_UNSUPPORTED;
}

}  // namespace rlk
