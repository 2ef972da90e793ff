// Kernel instantiations for head_dim 128, fp8 KV pools.
#include "launch.cuh"

namespace rad {
cudaError_t launch_d128_fp8(int family, const CUtensorMap& tk, const CUtensorMap& tv,
                           const AttnParams& p, int grid, cudaStream_t st) {
    return launch_family<128, true>(family, tk, tv, p, grid, st);
}
}  // namespace rad
