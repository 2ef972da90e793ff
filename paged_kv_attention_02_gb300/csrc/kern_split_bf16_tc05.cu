// Launcher of the tcgen05 split kernel for bf16 KV pools (head_dim 128,
// verify-shaped calls) and of the split combine after it.
#include <cuda_runtime.h>

#include "launch.cuh"
#include "split_bf16_tc05.cuh"
#include "tile_configs.cuh"

namespace rad {

TileInfo split_bf16_tc05_info() {
    using C = SplitBf16Cfg;
    return TileInfo{128, 1, 4, 0, 0, C::BK, C::NSK, C::QT, C::NTHREADS, C::SMEM_BYTES, 1};
}

cudaError_t launch_split_bf16_tc05(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int sms,
                                   cudaStream_t st) {
    using C = SplitBf16Cfg;
    auto kern = p.window > 0  ? attn_split_bf16_tc05_kernel<kModeWindow>
                : p.tree_mask ? attn_split_bf16_tc05_kernel<kModeTree>
                              : attn_split_bf16_tc05_kernel<kModeCausal>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    long long grid = sms;   // one CTA per SM (shared memory, TMEM), persistent over the items
    if (grid > p.n_items) grid = p.n_items;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(C::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = st;
    e = cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
    if (e != cudaSuccess || p.max_splits <= 1) return e;
    return launch_combine<128>(p, st);
}

}  // namespace rad
