// attn_bwd.cu — backward pass (placeholder until the kernels land).
#include "kernels.h"

namespace sdpa {

size_t bwd_smem_bytes(int) { return 0; }

cudaError_t launch_bwd(int, bool, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                       const CUtensorMap&, const CUtensorMap&, const BwdParams&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace sdpa
