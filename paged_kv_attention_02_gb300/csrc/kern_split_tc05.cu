// Launcher of the tcgen05 split kernel (head_dim 128, fp8 KV pools) and of
// the split combine after it.
#include <cuda_runtime.h>

#include "launch.cuh"
#include "split_tc05.cuh"
#include "tile_configs.cuh"

namespace rad {

namespace {

template <bool FEW>
cudaError_t launch_form(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int sms, cudaStream_t st) {
    using C = SplitTcCfg<FEW>;
    auto kern = p.window > 0  ? attn_split_tc05_kernel<kModeWindow, FEW>
                : p.tree_mask ? attn_split_tc05_kernel<kModeTree, FEW>
                              : attn_split_tc05_kernel<kModeCausal, FEW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    long long grid = sms;   // one CTA per SM (shared memory, all of TMEM), persistent over the items
    if (grid > p.n_items) grid = p.n_items;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(C::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

}  // namespace

TileInfo split_tc05_info(bool few) {
    if (few) {
        using C = SplitTcCfg<true>;
        return TileInfo{128, 1, 4, 0, 0, C::BK, C::NSK, C::QT, C::NTHREADS, C::SMEM_BYTES, 1};
    }
    using C = SplitTcCfg<false>;
    return TileInfo{128, 1, 4, 0, 0, C::BK, C::NSK, C::QT, C::NTHREADS, C::SMEM_BYTES, 1};
}

// Calls with at most 8 query rows per KV head take the decode form's stages.
cudaError_t launch_split_tc05(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int sms,
                              cudaStream_t st, bool few) {
    const cudaError_t e = few ? launch_form<true>(tk, tv, p, sms, st) : launch_form<false>(tk, tv, p, sms, st);
    if (e != cudaSuccess || p.max_splits <= 1) return e;
    return launch_combine<128>(p, st);
}

}  // namespace rad
