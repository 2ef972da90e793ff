// Launcher of the tcgen05 prefill kernel for fp8-e4m3 pools (head_dim 128).
#include <cuda_runtime.h>

#include "prefill_fp8.cuh"
#include "tile_configs.cuh"

namespace rad {

cudaError_t launch_prefill_fp8(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int sms,
                               cudaStream_t st) {
    // the window build for a sliding window, else the lean one (a scale <= 0
    // needs nothing special here: logits are scaled before their max)
    auto kern = p.window > 0 ? attn_prefill_fp8_kernel<true> : attn_prefill_fp8_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PrefillFp8Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    long long grid = sms;   // one CTA per SM, persistent over the items
    if (grid > p.n_items) grid = p.n_items;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(PrefillFp8Cfg::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = PrefillFp8Cfg::SMEM_BYTES;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

}  // namespace rad
