// Kernel instantiations for head_dim 256, fp8 KV pools.
#include "launch.cuh"

namespace rad {
cudaError_t launch_d256_fp8(int family, const AttnParams& p, int sms, cudaStream_t st) {
    return launch_family<256, true>(family, p, sms, st);
}
}  // namespace rad
