// Launcher of the tcgen05 prefill kernel for fp8-e4m3 pools (head_dim 256).
#include <cuda_runtime.h>

#include "prefill_fp8.cuh"
#include "tile_configs.cuh"

namespace rad {

cudaError_t launch_prefill_fp8_d256(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int sms,
                                    cudaStream_t st) {
    return launch_prefill_fp8_dim<256>(tk, tv, p, sms, st);
}

}  // namespace rad
