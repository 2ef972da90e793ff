// The tile map of a ragged call (calls with cu_seqlens): which sequence and
// query tile each tile of the call's work lists is.
#include <cuda_runtime.h>

#include "attn_tile.cuh"
#include "tile_configs.cuh"

namespace rad {

// One CTA writes, for each class of sequences, (sequence, query tile) of each
// of the class's query tiles in sequence order and (-1, 0) for the rest of
// the class's bound.  With two maps, sequences of at most `split_m` query rows
// per KV head (decode-shaped) form class 0 and the rest class 1; with one, all
// are class 0.  Sequences with malformed offsets get no tiles and raise
// RAD_ERRW_CUSEQ here, as does a class whose tiles overrun its bound (the
// caller's row total was short): tiles past it are not run.
__global__ void __launch_bounds__(kTileMapThreads) ragged_tile_map_kernel(const __grid_constant__ AttnParams p,
                                                                          const RaggedMaps m) {
    __shared__ int part[2][kTileMapThreads];
    const int tid = threadIdx.x;
    const int per = (p.groups + kTileMapThreads - 1) / kTileMapThreads;
    const int g0 = min(p.groups, tid * per), g1 = min(p.groups, g0 + per);
    const bool two = m.map[1] != nullptr;
    uint32_t err = 0;
    int sum[2] = {0, 0};
    for (int g = g0; g < g1; ++g) {
        GroupRows gr;
        if (!group_rows(p, g, gr)) {
            err |= kErrCuSeq;
            continue;
        }
        const int rows_kv = gr.n * p.ratio;
        const int c = (two && rows_kv > m.split_m) ? 1 : 0;
        sum[c] += (rows_kv + m.qt[c] - 1) / m.qt[c];
    }
    part[0][tid] = sum[0];
    part[1][tid] = sum[1];
    __syncthreads();
    for (int off = 1; off < kTileMapThreads; off <<= 1) {   // inclusive scans
        const int v0 = tid >= off ? part[0][tid - off] : 0;
        const int v1 = tid >= off ? part[1][tid - off] : 0;
        __syncthreads();
        part[0][tid] += v0;
        part[1][tid] += v1;
        __syncthreads();
    }
    int t[2] = {part[0][tid] - sum[0], part[1][tid] - sum[1]};
    for (int g = g0; g < g1; ++g) {
        GroupRows gr;
        if (!group_rows(p, g, gr)) continue;
        const int rows_kv = gr.n * p.ratio;
        const int c = (two && rows_kv > m.split_m) ? 1 : 0;
        const int n = (rows_kv + m.qt[c] - 1) / m.qt[c];
        for (int i = 0; i < n; ++i, ++t[c])
            if (t[c] < m.bound[c]) m.map[c][t[c]] = make_int2(g, i);
    }
    for (int c = 0; c < (two ? 2 : 1); ++c) {
        const int total = part[c][kTileMapThreads - 1];
        for (int i = total + tid; i < m.bound[c]; i += kTileMapThreads) m.map[c][i] = make_int2(-1, 0);
        if (total > m.bound[c]) err |= kErrCuSeq;
    }
    if (err && p.err_word) atomicOr(p.err_word, err);
}

cudaError_t launch_ragged_tile_map(const AttnParams& p, const RaggedMaps& m, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(kTileMapThreads, 1, 1);
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, ragged_tile_map_kernel, p, m);
}

}  // namespace rad
