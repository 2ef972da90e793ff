// Launcher of the tcgen05 split kernel for fp8 KV pools with head_dim 128
// (decode and verify calls) and of the split combine after it.
#include <cuda_runtime.h>

#include "launch.cuh"
#include "split_tc05.cuh"
#include "tile_configs.cuh"

namespace rad {

TileInfo split_tc05_info(bool few, int head_dim) {
    if (head_dim == 256) {
        using C = SplitTcCfg<false, 256>;   // one form: both take the same stages
        return TileInfo{256, 1, 4, 0, 0, C::BK, C::NSK, C::QT, C::NTHREADS, C::SMEM_BYTES, 1};
    }
    if (few) {
        using C = SplitTcCfg<true, 128>;
        return TileInfo{128, 1, 4, 0, 0, C::BK, C::NSK, C::QT, C::NTHREADS, C::SMEM_BYTES, 1};
    }
    using C = SplitTcCfg<false, 128>;
    return TileInfo{128, 1, 4, 0, 0, C::BK, C::NSK, C::QT, C::NTHREADS, C::SMEM_BYTES, 1};
}

// Calls with at most 8 query rows per KV head take the decode form's stages.
cudaError_t launch_split_tc05(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int sms,
                              cudaStream_t st, bool few) {
    const cudaError_t e = few ? launch_split_tc05_form<true, 128>(tk, tv, p, sms, st)
                              : launch_split_tc05_form<false, 128>(tk, tv, p, sms, st);
    if (e != cudaSuccess || p.max_splits <= 1) return e;
    return launch_combine<128>(p, st);
}

}  // namespace rad
