// attn_bwd.cu -- fused main + KL backward (placeholder until the kernels land).
#include "common.cuh"
#include "kernels.h"

namespace msa {

size_t bwd_ws_bytes(const Shape& s) { return plan_bytes(s); }

cudaError_t run_bwd(const Shape&, const void*, const void*, const void*, const void*,
                    const float*, const void*, const void*, const void*, const int32_t*,
                    const float*, float, void*, void*, void*, void*, void*, float*, void*,
                    const Ctx&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace msa
