// Launcher of the tcgen05 prefill kernel (head_dim 256, bf16 KV pools).
#include <cuda_runtime.h>

#include "prefill_tc05.cuh"
#include "tile_configs.cuh"

namespace rad {

cudaError_t launch_prefill_tc05_d256(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                     const AttnParams& p, int sms, cudaStream_t st) {
    return launch_prefill_tc05_dim<256>(tq, tk, tv, p, sms, st);
}

}  // namespace rad
