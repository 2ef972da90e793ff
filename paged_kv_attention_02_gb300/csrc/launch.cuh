// Launch helper shared by the kernel translation units.
#pragma once
#include <cuda_runtime.h>

#include "tile_configs.cuh"

namespace rad {

template <class C>
cudaError_t launch_cfg(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int grid,
                       cudaStream_t st) {
    auto kern = attn_tile_kernel<C>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(C::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

template <int D, bool FP8>
cudaError_t launch_family(int family, const CUtensorMap& tk, const CUtensorMap& tv,
                          const AttnParams& p, int grid, cudaStream_t st) {
    switch (family) {
        case kFamDecode: return launch_cfg<typename Pick<D, FP8, kFamDecode>::T>(tk, tv, p, grid, st);
        case kFamVerify: return launch_cfg<typename Pick<D, FP8, kFamVerify>::T>(tk, tv, p, grid, st);
        default: return launch_cfg<typename Pick<D, FP8, kFamWide>::T>(tk, tv, p, grid, st);
    }
}

}  // namespace rad
