// Launcher of the paired-query-tile tcgen05 prefill kernel (head_dim 128, bf16
// KV pools).
#include <cuda_runtime.h>

#include "prefill_pair.cuh"
#include "tile_configs.cuh"

namespace rad {

// `p` as planned for the one-tile kernel (n_items = groups x n_head_kv x
// query tiles); the pair kernel runs over pairs of query tiles.
cudaError_t launch_prefill_tc05_pair(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                     const AttnParams& p, int sms, cudaStream_t st) {
    AttnParams pp = p;
    const long long n_pairs = (p.n_qtiles + 1) / 2;
    pp.n_items = (int)((long long)p.groups * p.n_head_kv * n_pairs);
    return launch_prefill_pair(tq, tk, tv, pp, sms, st);
}

}  // namespace rad
