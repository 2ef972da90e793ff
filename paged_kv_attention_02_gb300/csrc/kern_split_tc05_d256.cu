// Launcher of the tcgen05 split kernel for fp8 KV pools with head_dim 256
// (decode and verify calls) and of the split combine after it.
#include <cuda_runtime.h>

#include "launch.cuh"
#include "split_tc05.cuh"
#include "tile_configs.cuh"

namespace rad {

// Decode and verify calls share one form: at head_dim 256 both take three K
// and two V stages.
cudaError_t launch_split_tc05_d256(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int sms,
                                   cudaStream_t st) {
    const cudaError_t e = launch_split_tc05_form<false, 256>(tk, tv, p, sms, st);
    if (e != cudaSuccess || p.max_splits <= 1) return e;
    return launch_combine<256>(p, st);
}

}  // namespace rad
