// Launcher of the tcgen05 prefill kernel (head_dim 128, bf16 KV pools).
#include <cuda_runtime.h>

#include "prefill_tc05.cuh"
#include "tile_configs.cuh"

namespace rad {

static_assert(PrefillTileKeys == PrefillCfg::BN, "host and kernel agree on the key tile");

cudaError_t launch_prefill_tc05(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const AttnParams& p, int sms, cudaStream_t st) {
    // the general kernel for a sliding window or a scale <= 0, else the lean one
    auto kern = (p.window > 0 || p.scale_log2 <= 0.f) ? attn_prefill_tc05_kernel<true>
                                                      : attn_prefill_tc05_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PrefillCfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    long long grid = (long long)sms * PrefillCfg::CTAS;
    if (grid > p.n_items) grid = p.n_items;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(PrefillCfg::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = PrefillCfg::SMEM_BYTES;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p);
}

}  // namespace rad
