// Tile shapes per (head_dim, KV dtype, call family).  The family is chosen
// from call scalars only (rows * n_head/n_head_kv), so a row's arithmetic never
// depends on the other sequences in the call.
#pragma once
#include "attn_tile.cuh"

namespace rad {

enum Family : int { kFamDecode = 0, kFamVerify = 1, kFamWide = 2 };

// Keys per split for calls of up to kSplitMaxRows rows; longer calls (prefill
// chunks) run one range per query tile.  A multiple of every tile's KS.
constexpr int kSplitLen = 512;
constexpr int kSplitMaxRows = 256;

template <int D, bool FP8, int F> struct Pick;
//                                         D    FP8   WQ NQW WK  KS  NS  CTAs/SM
template <> struct Pick<128, false, kFamDecode> { using T = TileCfg<128, false, 1, 1, 2, 32, 6, 2>; };
template <> struct Pick<128, false, kFamVerify> { using T = TileCfg<128, false, 2, 2, 2, 64, 5>; };
template <> struct Pick<128, false, kFamWide>   { using T = TileCfg<128, false, 4, 2, 1, 64, 4>; };
template <> struct Pick<128, true,  kFamDecode> { using T = TileCfg<128, true,  1, 1, 4, 64, 8>; };
template <> struct Pick<128, true,  kFamVerify> { using T = TileCfg<128, true,  2, 2, 2, 64, 8>; };
template <> struct Pick<128, true,  kFamWide>   { using T = TileCfg<128, true,  4, 2, 1, 64, 8>; };
template <> struct Pick<256, false, kFamDecode> { using T = TileCfg<256, false, 1, 1, 2, 32, 6>; };
template <> struct Pick<256, false, kFamVerify> { using T = TileCfg<256, false, 4, 1, 2, 32, 3>; };
template <> struct Pick<256, false, kFamWide>   { using T = TileCfg<256, false, 4, 1, 1, 32, 4>; };
template <> struct Pick<256, true,  kFamDecode> { using T = TileCfg<256, true,  1, 1, 4, 64, 5>; };
template <> struct Pick<256, true,  kFamVerify> { using T = TileCfg<256, true,  4, 1, 2, 32, 7>; };
template <> struct Pick<256, true,  kFamWide>   { using T = TileCfg<256, true,  4, 1, 1, 32, 8>; };

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

}  // namespace rad
