// Launcher of the tcgen05 prefill kernel (head_dim 128, bf16 KV pools).
#include <cuda_runtime.h>

#include "prefill_tc05.cuh"
#include "tile_configs.cuh"

namespace rad {

static_assert(PrefillTileKeys == PrefillCfg::BN, "host and kernel agree on the key tile");

cudaError_t launch_prefill_tc05(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const AttnParams& p, int sms, cudaStream_t st) {
    return launch_prefill_tc05_dim<128>(tq, tk, tv, p, sms, st);
}

// Keys per tile of the bf16 prefill kernel's build for this head_dim.
int prefill_tc05_tile_keys(int head_dim) {
    return head_dim == 256 ? PrefillCfgD<256>::BN : PrefillCfgD<128>::BN;
}

}  // namespace rad
