// Kernel instantiations for head_dim 256, fp8 KV pools.
#include "launch.cuh"

namespace rad {
cudaError_t launch_d256_fp8(int family, const CUtensorMap& tk, const CUtensorMap& tv,
                           const AttnParams& p, int grid, cudaStream_t st) {
    return launch_family<256, true>(family, tk, tv, p, grid, st);
}
}  // namespace rad
