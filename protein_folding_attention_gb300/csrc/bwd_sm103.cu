// EvoAttention backward on sm_103a (placeholder until the kernels land).
#include "sm103.h"

namespace evo {

size_t bf16_bwd_workspace_bytes(const Problem& P, unsigned) {
  return (size_t)P.rows() * 4 + 256;
}

cudaError_t bf16_bwd(const Problem&, const Bf16Ptrs&, unsigned, void*, unsigned int*,
                     cudaStream_t, bool*) {
  return cudaErrorNotSupported;
}

}  // namespace evo
