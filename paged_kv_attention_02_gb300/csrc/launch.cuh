// Launch helper shared by the kernel translation units.
#pragma once
#include <cuda_runtime.h>

#include "combine.cuh"
#include "tile_configs.cuh"

namespace rad {

// Persistent launch: as many CTAs as fit on the device at once (never more
// than there are work items).  Calls with a sliding window run the kernel
// built with the window terms, calls with tree masks the one with the mask
// test, others the plain causal one.
template <class C>
cudaError_t launch_cfg(const AttnParams& p, int sms, cudaStream_t st) {
    auto kern = p.window > 0  ? attn_tile_kernel<C, kModeWindow>
                : p.tree_mask ? attn_tile_kernel<C, kModeTree>
                              : attn_tile_kernel<C, kModeCausal>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::NTHREADS, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    long long grid = (long long)sms * per_sm;
    if (grid > p.n_items) grid = p.n_items;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(C::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

// The split combine: one CTA per (sequence, KV head, query tile, group of
// kCombineCols rows); CTAs of sequences with a single split exit at once.
template <int D>
cudaError_t launch_combine(const AttnParams& p, cudaStream_t st) {
    const long long n_cg = (p.qt_rows + kCombineCols - 1) / kCombineCols;
    const long long n_gq = (long long)(p.tile_map ? 1 : p.groups) * p.n_head_kv * p.n_qtiles;
    const long long grid = n_gq * n_cg;
    if (grid > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kCombineThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, attn_combine_kernel<D>, p);
}

template <int D, bool FP8>
cudaError_t launch_family(int family, const AttnParams& p, int sms, cudaStream_t st) {
    cudaError_t e;
    switch (family) {
        case kFamDecode: e = launch_cfg<typename Pick<D, FP8, kFamDecode>::T>(p, sms, st); break;
        case kFamVerify: e = launch_cfg<typename Pick<D, FP8, kFamVerify>::T>(p, sms, st); break;
        default: e = launch_cfg<typename Pick<D, FP8, kFamWide>::T>(p, sms, st); break;
    }
    if (e != cudaSuccess || p.split_len == 0 || p.max_splits <= 1) return e;
    return launch_combine<D>(p, st);
}

}  // namespace rad
