// Kernel instantiations for head_dim 128, fp8 KV pools.
#include "launch.cuh"

namespace rad {
cudaError_t launch_d128_fp8(int family, const AttnParams& p, int sms, cudaStream_t st) {
    return launch_family<128, true>(family, p, sms, st);
}
}  // namespace rad
