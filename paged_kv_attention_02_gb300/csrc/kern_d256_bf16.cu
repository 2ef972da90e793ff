// Kernel instantiations for head_dim 256, bf16 KV pools.
#include "launch.cuh"

namespace rad {
cudaError_t launch_d256_bf16(int family, const AttnParams& p, int sms, cudaStream_t st) {
    return launch_family<256, false>(family, p, sms, st);
}
}  // namespace rad
