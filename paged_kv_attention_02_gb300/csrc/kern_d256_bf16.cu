// Kernel instantiations for head_dim 256, bf16 KV pools.
#include "launch.cuh"

namespace rad {
cudaError_t launch_d256_bf16(int family, const CUtensorMap& tk, const CUtensorMap& tv,
                           const AttnParams& p, int grid, cudaStream_t st) {
    return launch_family<256, false>(family, tk, tv, p, grid, st);
}
}  // namespace rad
