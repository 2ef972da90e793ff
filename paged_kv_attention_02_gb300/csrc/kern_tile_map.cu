// The tile map of a ragged call (calls with cu_seqlens): which sequence and
// query tile each tile of the call's work list is.
#include <cuda_runtime.h>

#include "attn_tile.cuh"
#include "tile_configs.cuh"

namespace rad {

// The tile map of a ragged call: one CTA writes (sequence, query tile) for
// each query tile of the call, sequences in order, and (-1, 0) for the rest of
// the n_qtiles bound.  Sequences with malformed offsets get no tiles and raise
// RAD_ERRW_CUSEQ here, as does a call whose tiles overrun the bound (the
// caller's row total was short): tiles past it are not run.
__global__ void __launch_bounds__(kTileMapThreads) ragged_tile_map_kernel(const __grid_constant__ AttnParams p,
                                                                          int2* map, int qt_rows) {
    __shared__ int part[kTileMapThreads];
    const int tid = threadIdx.x;
    const int per = (p.groups + kTileMapThreads - 1) / kTileMapThreads;
    const int g0 = min(p.groups, tid * per), g1 = min(p.groups, g0 + per);
    uint32_t err = 0;
    int sum = 0;
    for (int g = g0; g < g1; ++g) {
        GroupRows gr;
        if (group_rows(p, g, gr))
            sum += (gr.n * p.ratio + qt_rows - 1) / qt_rows;
        else
            err |= kErrCuSeq;
    }
    part[tid] = sum;
    __syncthreads();
    for (int off = 1; off < kTileMapThreads; off <<= 1) {   // inclusive scan
        const int v = tid >= off ? part[tid - off] : 0;
        __syncthreads();
        part[tid] += v;
        __syncthreads();
    }
    const int total = part[kTileMapThreads - 1];
    int t = part[tid] - sum;
    for (int g = g0; g < g1; ++g) {
        GroupRows gr;
        if (!group_rows(p, g, gr)) continue;
        const int n = (gr.n * p.ratio + qt_rows - 1) / qt_rows;
        for (int i = 0; i < n; ++i, ++t)
            if (t < p.n_qtiles) map[t] = make_int2(g, i);
    }
    for (int i = total + tid; i < p.n_qtiles; i += kTileMapThreads) map[i] = make_int2(-1, 0);
    if (total > p.n_qtiles) err |= kErrCuSeq;
    if (err && p.err_word) atomicOr(p.err_word, err);
}

cudaError_t launch_ragged_tile_map(const AttnParams& p, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(kTileMapThreads, 1, 1);
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, ragged_tile_map_kernel, p, const_cast<int2*>(p.tile_map), p.qt_rows);
}

}  // namespace rad
