// Launcher of the tcgen05 prefill kernel for fp8-e4m3 pools (head_dim 128).
#include <cuda_runtime.h>

#include "prefill_fp8.cuh"
#include "tile_configs.cuh"

namespace rad {

cudaError_t launch_prefill_fp8(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int sms,
                               cudaStream_t st) {
    return launch_prefill_fp8_dim<128>(tk, tv, p, sms, st);
}

// Keys per tile of the fp8 prefill kernel's build for this head_dim.
int prefill_fp8_tile_keys(int head_dim) {
    return head_dim == 256 ? PrefillFp8CfgD<256>::BN : PrefillFp8CfgD<128>::BN;
}

}  // namespace rad
