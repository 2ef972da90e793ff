// Kernel instantiations for head_dim 128, bf16 KV pools.
#include "launch.cuh"

namespace rad {
cudaError_t launch_d128_bf16(int family, const CUtensorMap& tk, const CUtensorMap& tv,
                           const AttnParams& p, int grid, cudaStream_t st) {
    return launch_family<128, false>(family, tk, tv, p, grid, st);
}
}  // namespace rad
