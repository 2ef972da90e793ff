// Tile shapes per (head_dim, KV dtype, call family).  The family is chosen
// from call scalars only (rows * n_head/n_head_kv), so a row's arithmetic never
// depends on the other sequences in the call.
#pragma once
#include "attn_tile.cuh"

namespace rad {

enum Family : int { kFamDecode = 0, kFamVerify = 1, kFamWide = 2, kFamPrefillTC = 3, kFamSplitTC = 4, kFamSplitBf = 5 };

// Split calls (decode and verify shapes) with head_dim 128 and fp8 pools run
// on the tcgen05 split kernel (split_tc05.cuh); 0 keeps them on the mma.sync
// tile kernel.
#ifndef RAD_SPLIT_TC05
#define RAD_SPLIT_TC05 1
#endif
// Split calls (decode and verify shapes) with head_dim 128 and bf16 pools run
// on the bf16 tcgen05 split kernel (split_bf16_tc05.cuh); 0 keeps them on the
// mma.sync tile kernel.
#ifndef RAD_SPLIT_BF16_TC05
#define RAD_SPLIT_BF16_TC05 1
#endif
// The same for head_dim 256 with bf16 pools, and with fp8 pools.
#ifndef RAD_SPLIT_BF16_TC05_D256
#define RAD_SPLIT_BF16_TC05_D256 1
#endif
#ifndef RAD_SPLIT_TC05_D256
#define RAD_SPLIT_TC05_D256 1
#endif
// Prefill chunks with head_dim 256 over bf16 (fp8) pools run on the tcgen05
// prefill kernels' head_dim-256 builds; 0 keeps them on the mma.sync wide tile.
#ifndef RAD_PREFILL_TC05_D256
#define RAD_PREFILL_TC05_D256 1
#endif
#ifndef RAD_PREFILL_FP8_D256
#define RAD_PREFILL_FP8_D256 1
#endif
// Prefill chunks with head_dim 128 over bf16 pools run two query tiles per
// work item (prefill_pair.cuh); 0 keeps one tile per item (prefill_tc05.cuh).
#ifndef RAD_PREFILL_PAIR
#define RAD_PREFILL_PAIR 1
#endif

// Keys per split for calls of up to kSplitMaxRows rows; longer calls (prefill
// chunks) run one range per query tile.  A multiple of every tile's KS.
#ifndef RAD_SPLIT_LEN
#define RAD_SPLIT_LEN 1024
#endif
constexpr int kSplitLen = RAD_SPLIT_LEN;
// Keys per split of the tcgen05 split kernels: each work item pays a fixed cost
// (query rows, the merge of its four quarters, the wait for its last PV) that
// longer splits spread over more key tiles, and fewer, longer items spread
// less evenly over the SMs.  One length per kernel family and head_dim: a row's
// bits depend on it, so decode and verify calls of one family share it.
#ifndef RAD_SPLITTC_LEN
#define RAD_SPLITTC_LEN 4096   // e4m3 pools, head_dim 128
#endif
constexpr int kSplitLenTC = RAD_SPLITTC_LEN;
#ifndef RAD_SPLITTC_LEN_E4M3_D256
#define RAD_SPLITTC_LEN_E4M3_D256 2048   // e4m3 pools, head_dim 256
#endif
constexpr int kSplitLenTC_E4M3_256 = RAD_SPLITTC_LEN_E4M3_D256;
#ifndef RAD_SPLITBF_LEN
#define RAD_SPLITBF_LEN 2048   // bf16 pools, head_dim 128
#endif
constexpr int kSplitLenBf = RAD_SPLITBF_LEN;
#ifndef RAD_SPLITTC_LEN_D256
#define RAD_SPLITTC_LEN_D256 2048   // bf16 pools, head_dim 256
#endif
constexpr int kSplitLenTC256 = RAD_SPLITTC_LEN_D256;
constexpr int kSplitMaxRows = 256;
// The tcgen05 split kernels take their items from a counter shared by all
// CTAs (sched.cuh); 0 gives every CTA a fixed stride of items instead.
#ifndef RAD_SPLIT_DYNAMIC
#define RAD_SPLIT_DYNAMIC 1
#endif
// ... heaviest first (an order kernel sorts the items by key tiles before
// the split kernel runs); 0 hands them out in split order.
#ifndef RAD_ITEM_ORDER
#define RAD_ITEM_ORDER 1
#endif

// Tile shapes: WQ, NQW, WK, KS, NS, CTAs per SM (see TileCfg).  Each can be
// overridden at compile time (-DRAD_TILE_...="...") for tuning sweeps.
#ifndef RAD_TILE_D128_BF16_DEC
#define RAD_TILE_D128_BF16_DEC 1, 1, 2, 32, 3, 3
#endif
#ifndef RAD_TILE_D128_BF16_VER
#define RAD_TILE_D128_BF16_VER 4, 1, 2, 64, 2, 2
#endif
#ifndef RAD_TILE_D128_BF16_WIDE
#define RAD_TILE_D128_BF16_WIDE 4, 2, 1, 64, 4, 1
#endif
#ifndef RAD_TILE_D128_FP8_DEC
#define RAD_TILE_D128_FP8_DEC 1, 1, 2, 64, 6, 2
#endif
#ifndef RAD_TILE_D128_FP8_VER
#define RAD_TILE_D128_FP8_VER 2, 2, 2, 64, 3, 2
#endif
#ifndef RAD_TILE_D128_FP8_WIDE
#define RAD_TILE_D128_FP8_WIDE 4, 2, 1, 64, 8, 1
#endif
#ifndef RAD_TILE_D256_BF16_DEC
#define RAD_TILE_D256_BF16_DEC 1, 1, 2, 32, 3, 2
#endif
#ifndef RAD_TILE_D256_BF16_VER
#define RAD_TILE_D256_BF16_VER 4, 1, 2, 32, 3, 1
#endif
#ifndef RAD_TILE_D256_BF16_WIDE
#define RAD_TILE_D256_BF16_WIDE 4, 1, 1, 32, 4, 1
#endif
#ifndef RAD_TILE_D256_FP8_DEC
#define RAD_TILE_D256_FP8_DEC 1, 1, 2, 32, 4, 2
#endif
#ifndef RAD_TILE_D256_FP8_VER
#define RAD_TILE_D256_FP8_VER 4, 1, 2, 32, 7, 1
#endif
#ifndef RAD_TILE_D256_FP8_WIDE
#define RAD_TILE_D256_FP8_WIDE 4, 1, 1, 32, 8, 1
#endif

template <int D, bool FP8, int F> struct Pick;
template <> struct Pick<128, false, kFamDecode> { using T = TileCfg<128, false, RAD_TILE_D128_BF16_DEC>; };
template <> struct Pick<128, false, kFamVerify> { using T = TileCfg<128, false, RAD_TILE_D128_BF16_VER>; };
template <> struct Pick<128, false, kFamWide>   { using T = TileCfg<128, false, RAD_TILE_D128_BF16_WIDE>; };
template <> struct Pick<128, true,  kFamDecode> { using T = TileCfg<128, true,  RAD_TILE_D128_FP8_DEC>; };
template <> struct Pick<128, true,  kFamVerify> { using T = TileCfg<128, true,  RAD_TILE_D128_FP8_VER>; };
template <> struct Pick<128, true,  kFamWide>   { using T = TileCfg<128, true,  RAD_TILE_D128_FP8_WIDE>; };
template <> struct Pick<256, false, kFamDecode> { using T = TileCfg<256, false, RAD_TILE_D256_BF16_DEC>; };
template <> struct Pick<256, false, kFamVerify> { using T = TileCfg<256, false, RAD_TILE_D256_BF16_VER>; };
template <> struct Pick<256, false, kFamWide>   { using T = TileCfg<256, false, RAD_TILE_D256_BF16_WIDE>; };
template <> struct Pick<256, true,  kFamDecode> { using T = TileCfg<256, true,  RAD_TILE_D256_FP8_DEC>; };
template <> struct Pick<256, true,  kFamVerify> { using T = TileCfg<256, true,  RAD_TILE_D256_FP8_VER>; };
template <> struct Pick<256, true,  kFamWide>   { using T = TileCfg<256, true,  RAD_TILE_D256_FP8_WIDE>; };

// tcgen05 prefill kernel: keys per tile (64 or 128), K/V stages, CTAs per SM.
#ifndef RAD_PREFILL_BN
#define RAD_PREFILL_BN 128
#endif
#ifndef RAD_PREFILL_NSK
#define RAD_PREFILL_NSK 2   // K stages of the bf16 tcgen05 prefill kernel
#endif
#ifndef RAD_PREFILL_NSV
#define RAD_PREFILL_NSV 2   // V stages
#endif
#ifndef RAD_PREFILL_FP8_NSK
#define RAD_PREFILL_FP8_NSK 4   // K stages of the fp8 tcgen05 prefill kernel
#endif
#ifndef RAD_PREFILL_FP8_NSV
#define RAD_PREFILL_FP8_NSV 3   // V stages
#endif
#ifndef RAD_PREFILL_CTAS
#define RAD_PREFILL_CTAS 1
#endif
constexpr int PrefillTileKeys = RAD_PREFILL_BN;
// The prefill kernels' K producer hands out the CTA's next item this many key
// tiles before it issues the current item's last one.
#ifndef RAD_PREFILL_PUBLISH_LEAD
#define RAD_PREFILL_PUBLISH_LEAD 0
#endif

// Split calls (decode and verify shapes) share one key schedule: two key
// warps take alternate 16-key sub-tiles in key order, so a query row's
// arithmetic is the same in every split tile -- a verified row equals the
// decode step's row at its position bit for bit ("Adding a model", step 4).
template <int D, bool FP8>
constexpr bool same_key_schedule() {
    using Dec = typename Pick<D, FP8, kFamDecode>::T;
    using Ver = typename Pick<D, FP8, kFamVerify>::T;
    return Dec::WK == 2 && Ver::WK == 2;
}
static_assert(same_key_schedule<128, false>() && same_key_schedule<128, true>() &&
                  same_key_schedule<256, false>() && same_key_schedule<256, true>(),
              "decode and verify tiles must share the key schedule");

struct TileInfo {
    int D, fp8, WQ, NQW, WK, KS, NS, QT, threads, smem, minb;
};

template <class C>
constexpr TileInfo info_of() {
    return TileInfo{C::D, C::FP8 ? 1 : 0, C::WQ, C::NQW, C::WK, C::KS, C::NS, C::QT, C::NTHREADS,
                    C::SMEM_BYTES, C::MINB};
}

template <int D, bool FP8>
inline TileInfo tile_info(int family) {
    switch (family) {
        case kFamDecode: return info_of<typename Pick<D, FP8, kFamDecode>::T>();
        case kFamVerify: return info_of<typename Pick<D, FP8, kFamVerify>::T>();
        default: return info_of<typename Pick<D, FP8, kFamWide>::T>();
    }
}

// One launcher per (head_dim, dtype) translation unit.
cudaError_t launch_d128_bf16(int family, const AttnParams& p, int sms, cudaStream_t st);
cudaError_t launch_d128_fp8(int family, const AttnParams& p, int sms, cudaStream_t st);
cudaError_t launch_d256_bf16(int family, const AttnParams& p, int sms, cudaStream_t st);
cudaError_t launch_d256_fp8(int family, const AttnParams& p, int sms, cudaStream_t st);
cudaError_t launch_prefill_tc05(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const AttnParams& p, int sms, cudaStream_t st);
cudaError_t launch_prefill_tc05_d256(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                     const AttnParams& p, int sms, cudaStream_t st);
cudaError_t launch_prefill_tc05_pair(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                     const AttnParams& p, int sms, cudaStream_t st);
int prefill_tc05_tile_keys(int head_dim);
cudaError_t launch_prefill_fp8(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int sms,
                               cudaStream_t st);
cudaError_t launch_prefill_fp8_d256(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int sms,
                                    cudaStream_t st);
int prefill_fp8_tile_keys(int head_dim);
cudaError_t launch_split_tc05(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int sms,
                              cudaStream_t st, bool few);
cudaError_t launch_split_tc05_d256(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int sms,
                                   cudaStream_t st);
TileInfo split_tc05_info(bool few, int head_dim);
cudaError_t launch_split_bf16_tc05(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int sms,
                                   cudaStream_t st, bool few);
cudaError_t launch_split_bf16_tc05_d256(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int sms,
                                        cudaStream_t st, bool few);
TileInfo split_bf16_tc05_info(bool few, int head_dim);
// Ragged calls: the tile maps (one CTA), before the tile kernels.  map[1]
// null: one class; else sequences with at most split_m query rows per KV head
// go to map[0] (tiles of qt[0] rows), the rest to map[1].
constexpr int kTileMapThreads = 1024;
struct RaggedMaps {
    int2* map[2];
    int qt[2];
    int bound[2];
    int split_m;
};
cudaError_t launch_ragged_tile_map(const AttnParams& p, const RaggedMaps& m, cudaStream_t st);

}  // namespace rad
