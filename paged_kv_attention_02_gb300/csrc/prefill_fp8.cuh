// Prefill-chunk attention over fp8-e4m3 KV pools on the 5th-generation tensor
// cores (tcgen05, TMEM): the e4m3 tensor-core prefill the pages name
// (`attn_prefill_fp8`, "Radiance architecture plugins", section "Declare: the
// metadata"), with every product exact.
//
// Work items, masks and the item order are those of the bf16 tcgen05 prefill
// kernel (prefill_tc05.cuh): (sequence g, KV head kvh, 128 query rows), keys
// 0 .. kmax-1, causal per row, an optional sliding window.  The CTAs take the
// items, heavier query tiles first, from a counter shared by all CTAs
// (sched.cuh), the K producer handing each CTA's items to its other warps.
//
//   S_j  = Q K_j^T     kind::f8f6f4, M 128 query rows, N 128 keys, K = head_dim:
//                      K straight from the TMA-staged e4m3 rows; each query row
//                      q split as q * 2^k = hi + lo, both e4m3 (hi: 4
//                      significant bits, lo: the remainder of a bf16 value,
//                      which then fits e4m3 exactly outside its subnormal
//                      range); logits scaled back by 2^-k and by the page's K
//                      scale of their key
//   O   += P_j V_j     kind::f16, A = P in f16 from TMEM (p times the page's V
//                      scale), B = V converted e4m3 -> f16 (exact) into a
//                      128-byte-swizzled MN-major tile
//
// Warp roles (one CTA per SM, persistent, heavier query tiles first):
//   warp 6      K producer: page ids and per-page K/V scales (the scales of a
//               tile's pages into the K stage's meta block), TMA loads of every
//               page's e4m3 K rows (one 3-D box per page: P rows x 128 bytes)
//               into a ring of K stages, each free once its QK is done and the
//               softmax has read its scales; pages outside the tile's range
//               load from an out-of-range coordinate (zero fill).
//   warp 7      V producer: the same for V rows into a ring of V stages, each
//               free once converted.
//   warp 4      QK: lane 0 issues QK per tile (2 terms x 4 K-steps) into TMEM
//               buffer j & 1 once K_j landed and PV_{j-2} is done; then the
//               warp turns key rows 0-63 of the staged e4m3 V_j into f16
//               buffer j & 1 (zeros for keys outside the sequence or below the
//               tile's window) while the softmax works on S_j.
//   warp 5      V: converts key rows 64-127 the same way, then, once P_j is
//               written and the QK warp's rows are converted, lane 0 issues
//               PV.  (One warp converting all 128 rows measured 8% slower: it
//               then noticed P_j late.)
//   warps 0-3   softmax: thread t owns query row t; per item it splits its row
//               of Q into the two e4m3 terms; per tile it reads S_j, scales
//               and masks the logits, keeps the running max (lazy rescale of O
//               past 2^8, warp-wide), writes P over S_j and finally O / l.
// PV of tile t completes a phase of pv_done[t & 1]; every wait on it is at most
// one phase ahead (see prefill_tc05.cuh).  The QK warp's conversion of tile t
// completes a phase of v16_full[t & 1]; it starts only after PV(t-2), which
// waited for tile t-2's phase, so the V warp's wait on it is never two phases
// behind either.  Every wait is bounded.
#pragma once
#include <cuda.h>

#include "prefill_tc05.cuh"
#include "sched.cuh"
#include "tc05.cuh"

namespace rad {

// D: head_dim 128 or 256.  At 256 a key tile holds 64 keys (16 KB of e4m3 K or
// V rows, as a 128-key tile at 128) in two 128-byte column blocks, the query
// terms take 64 KB, and each converting warp turns 32 rows of a tile into f16.
template <int D_>
struct PrefillFp8CfgD {
    static constexpr int D = D_;
    static constexpr int BM = 128;                  // query rows per item
    static constexpr int BN = D == 128 ? 128 : 64;  // keys per tile
    static constexpr int NKB = D / 128;             // 128-byte column blocks of an e4m3 row
    static constexpr int NSK = D == 128 ? RAD_PREFILL_FP8_NSK : 3;   // K stages (with the tile's page scales)
    static constexpr int NSV = D == 128 ? RAD_PREFILL_FP8_NSV : 3;   // V stages
    static constexpr int QK_VROWS = BN / 2;         // V rows the QK warp converts per tile (the V warp: the rest)
    static constexpr int Q8_BLK = BM * 128;         // one 128-byte column block of a query term: [row][128 B]
    static constexpr int Q8_TERM = NKB * Q8_BLK;    // one e4m3 term of the query tile
    static constexpr int KBLK = BN * 128;           // one 128-byte column block of a K or V tile
    static constexpr int KV_TILE = NKB * KBLK;      // e4m3 K or V rows of one tile
    static constexpr int ATOM = BN * 128;           // one 64-column block of the f16 V tile
    static constexpr int V16_BYTES = (D / 64) * ATOM;
    static constexpr int META_STRIDE = 64;          // ks[8], vs[8] of a tile's pages
    static constexpr int OFF_Q8 = 0;
    static constexpr int OFF_K = OFF_Q8 + 2 * Q8_TERM;
    static constexpr int OFF_V = OFF_K + NSK * KV_TILE;
    static constexpr int OFF_V16 = OFF_V + NSV * KV_TILE;
    static constexpr int OFF_META = OFF_V16 + 2 * V16_BYTES;
    static constexpr int OFF_BARS = OFF_META + NSK * META_STRIDE;
    // q8_full, q8_empty, k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV], s_full[2], p_full[2],
    // pv_done[2], v16_full[2], o_free, final[2]
    static constexpr int NBARS = 2 + 2 * NSK + 2 * NSV + 2 + 2 + 2 + 2 + 1 + 2;
    static constexpr int OFF_RING = OFF_BARS + NBARS * 8;     // the item ring (sched.cuh)
    static constexpr int OFF_MISC = OFF_RING + kRingBytesNoTaken;
    static constexpr int RING_CONSUMERS = 7;                 // every warp but the K producer, which fills it
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;   // 1 KB alignment of the swizzled tiles
    static constexpr int NTHREADS = 8 * 32;   // 8 warps: the softmax threads keep 255 registers
    static constexpr int W_QK = 4, W_V = 5, W_PROD_K = 6, W_PROD_V = 7;
    // a K stage is free once QK read its K (a commit) and the softmax warps read its scales
    static constexpr int K_EMPTY_ARRIVALS = 1 + 4;
    static constexpr uint32_t TMEM_COLS = 512;      // O in [0, D), S buffer b in [D + BN b, ...)
    static constexpr float RESCALE_LOG2 = 8.f;
    static_assert(D == 128 || D == 256, "head_dim 128 or 256");
    static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && OFF_V16 % 1024 == 0 && KV_TILE % 1024 == 0, "1 KB tiles");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(QK_VROWS % 32 == 0 && QK_VROWS > 0 && QK_VROWS < BN, "both warps convert whole 32-row groups");
    static_assert(D + 2 * BN <= (int)TMEM_COLS, "tensor memory budget");
};
using PrefillFp8Cfg = PrefillFp8CfgD<128>;

// Key rows row0 + lane + 32 i (i < n) of a staged e4m3 V tile -> the f16
// MN-major tile PV reads (128-byte swizzle, 64-column blocks); keys outside
// [zlo, L) become zeros.  Each 128-code column block of a row goes to its
// pair of f16 blocks.
template <class C>
__device__ __forceinline__ void convert_v_rows(const uint8_t* stage, uint8_t* v16, int row0, int n, int key0, int zlo,
                                               int L, int lane) {
    const uint32_t sw = (uint32_t)(lane & 7);   // (row0 + lane + 32 i) & 7: row0 is a multiple of 32
#pragma unroll 1
    for (int i = 0; i < n; ++i) {
        const int row = row0 + lane + 32 * i;
        const int key = key0 + row;
        const bool zero = key < zlo || key >= L;
#pragma unroll
        for (int kb = 0; kb < C::NKB; ++kb) {
            const uint8_t* src = stage + kb * C::KBLK + row * 128;
            uint8_t* dst = v16 + 2 * kb * C::ATOM + row * 128;
            uint4 in[8];   // the row's loads first: stores below may alias them as far as the compiler knows
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
                in[ch] = zero ? make_uint4(0u, 0u, 0u, 0u)
                              : *reinterpret_cast<const uint4*>(src + (((uint32_t)ch ^ sw) << 4));
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                // codes 16ch .. 16ch+15 -> f16 chunks 2ch, 2ch+1 of the row, column block ch / 4
                const uint4 v = in[ch];
                const uint32_t h0 = e4m3x2_to_f16x2((uint16_t)(v.x & 0xFFFFu));
                const uint32_t h1 = e4m3x2_to_f16x2((uint16_t)(v.x >> 16));
                const uint32_t h2 = e4m3x2_to_f16x2((uint16_t)(v.y & 0xFFFFu));
                const uint32_t h3 = e4m3x2_to_f16x2((uint16_t)(v.y >> 16));
                const uint32_t h4 = e4m3x2_to_f16x2((uint16_t)(v.z & 0xFFFFu));
                const uint32_t h5 = e4m3x2_to_f16x2((uint16_t)(v.z >> 16));
                const uint32_t h6 = e4m3x2_to_f16x2((uint16_t)(v.w & 0xFFFFu));
                const uint32_t h7 = e4m3x2_to_f16x2((uint16_t)(v.w >> 16));
                uint8_t* blk = dst + (ch >> 2) * C::ATOM;
                const uint32_t c2 = (uint32_t)((ch & 3) * 2);
                *reinterpret_cast<uint4*>(blk + ((c2 ^ sw) << 4)) = make_uint4(h0, h1, h2, h3);
                *reinterpret_cast<uint4*>(blk + (((c2 + 1) ^ sw) << 4)) = make_uint4(h4, h5, h6, h7);
            }
        }
    }
}

template <bool GEN, int D = 128>
__global__ void __launch_bounds__(PrefillFp8CfgD<D>::NTHREADS, 1)
    attn_prefill_fp8_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ AttnParams p) {
    using C = PrefillFp8CfgD<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_addr);

    const uint32_t bar_q8_full = base + C::OFF_BARS;
    const uint32_t bar_q8_empty = bar_q8_full + 8;
    const uint32_t bar_k_full = bar_q8_empty + 8;
    const uint32_t bar_k_empty = bar_k_full + 8 * C::NSK;
    const uint32_t bar_v_full = bar_k_empty + 8 * C::NSK;
    const uint32_t bar_v_empty = bar_v_full + 8 * C::NSV;
    const uint32_t bar_s_full = bar_v_empty + 8 * C::NSV;   // [2]
    const uint32_t bar_p_full = bar_s_full + 16;            // [2]
    const uint32_t bar_pv_done = bar_p_full + 16;           // [2], by tile parity
    const uint32_t bar_v16_full = bar_pv_done + 16;         // [2], by tile parity: the QK warp's V rows converted
    const uint32_t bar_o_free = bar_v16_full + 16;
    const uint32_t bar_final = bar_o_free + 8;
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);  // [0] tmem, [1] abort
    const ItemRing iring(smem + C::OFF_RING, base + C::OFF_RING);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar_q8_full, 4);
        mbar_init(bar_q8_empty, 1);
        for (int i = 0; i < C::NSK; ++i) {
            mbar_init(bar_k_full + 8 * i, 1);
            mbar_init(bar_k_empty + 8 * i, C::K_EMPTY_ARRIVALS);
        }
        for (int i = 0; i < C::NSV; ++i) {
            mbar_init(bar_v_full + 8 * i, 1);
            mbar_init(bar_v_empty + 8 * i, 2);   // both converting warps
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_s_full + 8 * i, 1);
            mbar_init(bar_p_full + 8 * i, 4);
            mbar_init(bar_pv_done + 8 * i, 1);
            mbar_init(bar_v16_full + 8 * i, 1);
        }
        mbar_init(bar_o_free, 4);
        mbar_init(bar_final, 1);
        mbar_init(bar_final + 8, 1);
        iring.init(C::RING_CONSUMERS, false);
        misc[1] = 0;
        fence_mbarrier_init();
    }
    if (warp == C::W_QK) {
        tmem_alloc(base + C::OFF_MISC, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const uint32_t t_o = tmem;
    const uint32_t t_s = tmem + C::D;   // S buffer b at t_s + BN*b

    const int P = p.page_size;
    const int ppt = C::BN / P;       // pages per key tile (8 or 4)
    bool abort = false;

    if (warp == C::W_PROD_K || warp == C::W_PROD_V) {
        // ===================================================== producers: K (+ the tile's scales), V
        const bool is_k = warp == C::W_PROD_K;
        const int NSX = is_k ? C::NSK : C::NSV;
        const uint32_t bar_full = is_k ? bar_k_full : bar_v_full;
        const uint32_t bar_empty = is_k ? bar_k_empty : bar_v_empty;
        const uint32_t ring = base + (is_k ? C::OFF_K : C::OFF_V);
        const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
        const uint64_t pol = policy_evict_last();   // K/V tiles are re-read by every query tile
        const int oob_tok = p.num_pages * P;
        uint32_t sc = 0;
        if (lane == 0) prefetch_tmap(tm);
        // The K producer fills the item ring (sched.cuh): entry n + 1 right after
        // it issued entry n's last tile (at once for an invalid sequence).
        ItemRing::Cursor cur;
        int next = -1;
        const auto publish_next = [&](uint32_t m) {
            bool ok = true;
            if (lane == 0) {
                next = iring.fetch_if(p, cur, misc + 1, [](int) { return true; });
                ok = iring.publish(m, next, p.wait_ns);
            }
            next = __shfl_sync(0xffffffffu, next, 0);
            return __shfl_sync(0xffffffffu, ok, 0);
        };
        if (is_k && !publish_next(0)) abort = true;
        for (uint32_t n = 0; !abort; ++n) {
            int item = -1;
            if (is_k) {
                item = next;
            } else if (!iring.take(n, item, p.wait_ns, false)) {
                abort = true;
                break;
            }
            if (item < 0) break;
            const PrefItem it = plan_prefill<GEN, C::BM, C::BN>(item, p);
            if (!it.seq_ok) {
                if (is_k && !publish_next(n + 1)) abort = true;
                continue;
            }
            const int page_hi = (it.kmax + P - 1) / P;
            const int page_lo = GEN ? it.klo / P : 0;   // pages below hold no visible key: never read
            const int32_t* trow = p.page_table + (long long)it.g * p.pages_per_seq;
            int batch0 = -1 << 30, my_pg = 0;
            float my_ks = 1.f, my_vs = 1.f;
            for (int j = 0; j < it.T; ++j) {
                const uint32_t st = sc % (uint32_t)NSX, use = sc / (uint32_t)NSX;
                if (use >= 1 && !mbar_wait_bounded(bar_empty + 8 * st, (use - 1) & 1u, p.wait_ns)) {
                    abort = true;
                    break;
                }
                const int pstart = (it.kt0 + j) * ppt;
                if (pstart + ppt > batch0 + 32) {
                    batch0 = pstart;
                    const int pi = batch0 + lane;
                    my_pg = 0;
                    my_ks = my_vs = 1.f;
                    if ((!GEN || pi >= page_lo) && pi < page_hi) {
                        const int pg = __ldg(trow + pi);
                        my_pg = (pg < 0 || pg >= p.num_pages) ? 0 : pg;
                        if (is_k) {
                            my_ks = __ldg(p.k_scales + my_pg);
                            my_vs = __ldg(p.v_scales + my_pg);
                        }
                    }
                }
                float kss[8], vss[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int src = (pstart - batch0 + (i < ppt ? i : 0)) & 31;
                    kss[i] = __shfl_sync(0xffffffffu, my_ks, src);
                    vss[i] = __shfl_sync(0xffffffffu, my_vs, src);
                }
                const uint32_t dst = ring + st * C::KV_TILE;
                if (lane == 0) {
                    if (is_k) {
                        // the tile's page scales, released with the K-full arrive below
                        float* meta = reinterpret_cast<float*>(smem + C::OFF_META + st * C::META_STRIDE);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            meta[i] = kss[i];
                            meta[8 + i] = vss[i];
                        }
                    }
                    mbar_arrive_expect_tx(bar_full + 8 * st, C::KV_TILE);
                }
                for (int i = 0; i < ppt; ++i) {
                    const int pi = pstart + i;
                    const int pg = __shfl_sync(0xffffffffu, my_pg, (pi - batch0) & 31);
                    const int tok = ((!GEN || pi >= page_lo) && pi < page_hi) ? pg * P : oob_tok;
                    if (lane == 0) {
#pragma unroll
                        for (int kb = 0; kb < C::NKB; ++kb)
                            tma_load_3d(dst + (uint32_t)(kb * C::KBLK + i * P * 128), tm, bar_full + 8 * st, kb * 128,
                                        it.kvh, tok, pol);
                    }
                }
                ++sc;
                // the next item, RAD_PREFILL_PUBLISH_LEAD tiles before this one's last
                if (is_k && j == it.T - 1 - RAD_PREFILL_PUBLISH_LEAD && !publish_next(n + 1)) {
                    abort = true;
                    break;
                }
            }
            // the next item, if this one had too few tiles to hand it out earlier
            if (is_k && !abort && it.T <= RAD_PREFILL_PUBLISH_LEAD && !publish_next(n + 1)) abort = true;
            if (misc[1]) abort = true;
        }
        // drain: nothing may still be landing in shared memory at exit
        if (lane == 0) {
            const uint32_t first = sc > (uint32_t)NSX ? sc - NSX : 0u;
            for (uint32_t c = first; c < sc; ++c)
                mbar_wait_bounded(bar_full + 8 * (c % NSX), (c / NSX) & 1u, p.wait_ns);
        }
    } else if (warp == C::W_QK) {
        // ===================================================== QK issue
        constexpr uint32_t idesc_qk = umma_idesc_e4m3(C::BM, C::BN);
        uint32_t sc = 0, tc = 0, ic = 0;
        bool issued = false;
        for (uint32_t n = 0; !abort; ++n) {
            int item;
            if (!iring.take(n, item, p.wait_ns, false)) {
                abort = true;
                break;
            }
            if (item < 0) break;
            const PrefItem it = plan_prefill<GEN, C::BM, C::BN>(item, p);
            if (!it.seq_ok) continue;
            if (!mbar_wait_bounded(bar_q8_full, ic & 1u, p.wait_ns)) {
                abort = true;
                break;
            }
            tc_fence_after();
            for (int j = 0; j < it.T; ++j) {
                const uint32_t s_ = sc + j, st = s_ % C::NSK, tcj = tc + j, b = tcj & 1u;
                // K landed, and S buffer b is free: PV(tcj - 2) read the P it held
                bool ok = mbar_wait_bounded(bar_k_full + 8 * st, (s_ / C::NSK) & 1u, p.wait_ns);
                if (ok && tcj >= 2) ok = mbar_wait_bounded(bar_pv_done + 8 * b, ((tcj - 2) >> 1) & 1u, p.wait_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    abort = true;
                    break;
                }
                tc_fence_after();
                const uint32_t kb = base + C::OFF_K + st * C::KV_TILE;
                if (lane == 0) {
#pragma unroll
                    for (int term = 0; term < 2; ++term)
#pragma unroll
                        for (int kk = 0; kk < C::D / 32; ++kk)
                            tc_mma_ss_f8(t_s + C::BN * b,
                                         umma_desc_sw128(base + C::OFF_Q8 + term * C::Q8_TERM + (kk >> 2) * C::Q8_BLK +
                                                             (kk & 3) * 32,
                                                         16, 1024),
                                         umma_desc_sw128(kb + (kk >> 2) * C::KBLK + (kk & 3) * 32, 16, 1024), idesc_qk,
                                         (term > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(bar_s_full + 8 * b);
                    tc_commit(bar_k_empty + 8 * st);
                    if (j == it.T - 1) tc_commit(bar_q8_empty);   // the item's query terms are read
                    issued = true;
                }
                __syncwarp();
                // key rows 0 .. QK_VROWS-1 of V_j -> f16 buffer b (free: PV(tcj - 2) is done)
                // while the softmax works on S_j
                const uint32_t sv = s_ % C::NSV;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar_v_full + 8 * sv, (s_ / C::NSV) & 1u, p.wait_ns))) {
                    abort = true;
                    break;
                }
                convert_v_rows<C>(smem + C::OFF_V + sv * C::KV_TILE, smem + C::OFF_V16 + b * C::V16_BYTES, 0,
                               C::QK_VROWS / 32, (it.kt0 + j) * C::BN, GEN ? it.klo : 0, it.L, lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar_v16_full + 8 * b);
                    mbar_arrive(bar_v_empty + 8 * sv);
                }
            }
            sc += it.T;
            tc += it.T;
            ++ic;
            if (misc[1]) abort = true;
        }
        // every MMA this thread issued is complete before TMEM is released
        if (lane == 0 && issued) {
            tc_commit(bar_final);
            mbar_wait_bounded(bar_final, 0, p.wait_ns);
        }
        __syncwarp();
    } else if (warp == C::W_V) {
        // ===================================================== V: conversion and PV issue
        constexpr uint32_t idesc_pv = umma_idesc_f16(C::BM, C::D, 0, 1);
        uint32_t sc = 0, tc = 0, ic = 0;
        bool issued = false;
        for (uint32_t n = 0; !abort; ++n) {
            int item;
            if (!iring.take(n, item, p.wait_ns, false)) {
                abort = true;
                break;
            }
            if (item < 0) break;
            const PrefItem it = plan_prefill<GEN, C::BM, C::BN>(item, p);
            if (!it.seq_ok) continue;
            const int zlo = GEN ? it.klo : 0;   // keys below the tile's window may hold anything
            for (int j = 0; j < it.T; ++j) {
                const uint32_t s_ = sc + j, st = s_ % C::NSV, tcj = tc + j, b = tcj & 1u;
                bool ok = mbar_wait_bounded(bar_v_full + 8 * st, (s_ / C::NSV) & 1u, p.wait_ns);
                // f16 buffer b was last read by PV(tcj - 2)
                if (ok && tcj >= 2)
                    ok = mbar_wait_bounded(bar_pv_done + 8 * b, ((tcj - 2) >> 1) & 1u, p.wait_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    abort = true;
                    break;
                }
                // key rows QK_VROWS .. 127 of the staged tile -> f16 (the QK warp converts the rows below)
                convert_v_rows<C>(smem + C::OFF_V + st * C::KV_TILE, smem + C::OFF_V16 + b * C::V16_BYTES, C::QK_VROWS,
                               (C::BN - C::QK_VROWS) / 32,
                               (it.kt0 + j) * C::BN, zlo, it.L, lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_v_empty + 8 * st);   // the staged V tile is read
                // PV once P is written (and, at an item's first tile, O was read out)
                ok = mbar_wait_bounded(bar_p_full + 8 * b, (tcj >> 1) & 1u, p.wait_ns);
                if (ok) ok = mbar_wait_bounded(bar_v16_full + 8 * b, (tcj >> 1) & 1u, p.wait_ns);
                if (ok && j == 0 && ic >= 1) ok = mbar_wait_bounded(bar_o_free, (ic - 1) & 1u, p.wait_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    abort = true;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sp = t_s + C::BN * b;
                    const uint32_t vb = base + C::OFF_V16 + b * C::V16_BYTES;
#pragma unroll
                    for (int kk = 0; kk < C::BN / 16; ++kk)
                        tc_mma_ts(t_o, sp + kk * 8, umma_desc_sw128(vb + kk * 16 * 128, C::ATOM, 1024), idesc_pv,
                                  (j > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(bar_pv_done + 8 * b);
                    issued = true;
                }
                __syncwarp();
            }
            sc += it.T;
            tc += it.T;
            ++ic;
            if (__any_sync(0xffffffffu, misc[1] != 0)) abort = true;
        }
        if (lane == 0 && issued) {
            tc_commit(bar_final + 8);
            mbar_wait_bounded(bar_final + 8, 0, p.wait_ns);
        }
        __syncwarp();
    } else {
        // ===================================================== softmax (warps 0-3)
        const int t = threadIdx.x;                                  // query row of the tile
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;      // this warp's TMEM lanes
        const int lp = (P == 16) ? 4 : 5;
        uint32_t sc = 0, tc = 0, ic = 0;
        for (uint32_t n = 0; !abort; ++n) {
            int item;
            if (!iring.take(n, item, p.wait_ns, false)) {
                abort = true;
                break;
            }
            if (item < 0) break;
            const PrefItem it = plan_prefill<GEN, C::BM, C::BN>(item, p);
            const int m = it.m0 + t;
            const bool valid = m < it.m_end;
            const int r = m / p.ratio, hl = m - r * p.ratio;
            __nv_bfloat16* orow = p.out + (((long long)it.g * p.rows + r) * p.n_head + it.kvh * p.ratio + hl) * C::D;
            if (!it.seq_ok) {
                if (valid)
                    for (int i = 0; i < C::D / 8; ++i) reinterpret_cast<uint4*>(orow)[i] = make_uint4(0, 0, 0, 0);
                if (t == 0 && p.err_word) atomicOr(p.err_word, kErrSeqLen);
                continue;
            }
            // ---- the row's query as two e4m3 terms, written once the previous item's
            // QKs are done (the row is loaded and its scale found before that wait)
            float isq = 1.f;   // 2^-k: the row's logits scale back
            {
                const uint4* qrow = reinterpret_cast<const uint4*>(
                    p.q + (((long long)it.g * p.rows + r) * p.n_head + it.kvh * p.ratio + hl) * C::D);
                // the row's largest magnitude, 128 elements at a time (head_dim 256: the
                // second pass reads the row again, from L1)
                uint4 qv[16];
                float amax = 0.f;
#pragma unroll
                for (int h = 0; h < C::D / 128; ++h) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) qv[i] = valid ? __ldg(qrow + 16 * h + i) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint32_t x[4] = {qv[i].x, qv[i].y, qv[i].z, qv[i].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(x[e])), fabsf(bf16_hi(x[e]))));
                    }
                }
                // 2^k with amax * 2^k in [128, 256): k = 7 - floor(log2 amax), kept a normal float
                const int ex = amax > 0.f ? (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127 : 7;
                const int kx = max(-126, min(127, 7 - ex));
                const float sq = __uint_as_float((uint32_t)(kx + 127) << 23);
                isq = __uint_as_float((uint32_t)(127 - kx) << 23);
                if (ic >= 1 &&
                    !__all_sync(0xffffffffu, mbar_wait_bounded(bar_q8_empty, (ic - 1) & 1u, p.wait_ns))) {
                    abort = true;
                    break;
                }
#pragma unroll
                for (int h = 0; h < C::D / 128; ++h) {
                    if (C::D > 128) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) qv[i] = valid ? __ldg(qrow + 16 * h + i) : make_uint4(0u, 0u, 0u, 0u);
                    }
                    // column block h of each term: [row][128 B]
                    uint8_t* q8 = smem + C::OFF_Q8 + h * C::Q8_BLK + t * 128;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        // elements 128h + 16i .. 128h + 16i+15: chunk i of the block's row
                        uint32_t w[2][4];
                        const uint32_t words[8] = {qv[2 * i].x,     qv[2 * i].y,     qv[2 * i].z,     qv[2 * i].w,
                                                   qv[2 * i + 1].x, qv[2 * i + 1].y, qv[2 * i + 1].z, qv[2 * i + 1].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const uint32_t x0 = words[2 * e], x1 = words[2 * e + 1];
                            const float v0 = bf16_lo(x0) * sq, v1 = bf16_hi(x0) * sq;
                            const float v2 = bf16_lo(x1) * sq, v3 = bf16_hi(x1) * sq;
                            const uint32_t h01 = f32x2_to_e4m3x2(v0, v1), h23 = f32x2_to_e4m3x2(v2, v3);
                            const float2 a01 = e4m3x2_to_f32x2(h01), a23 = e4m3x2_to_f32x2(h23);
                            const uint32_t l01 = f32x2_to_e4m3x2(v0 - a01.x, v1 - a01.y);
                            const uint32_t l23 = f32x2_to_e4m3x2(v2 - a23.x, v3 - a23.y);
                            w[0][e] = h01 | (h23 << 16);
                            w[1][e] = l01 | (l23 << 16);
                        }
                        const uint32_t off = (((uint32_t)i ^ (uint32_t)(t & 7)) << 4);
#pragma unroll
                        for (int term = 0; term < 2; ++term)
                            *reinterpret_cast<uint4*>(q8 + term * C::Q8_TERM + off) =
                                make_uint4(w[term][0], w[term][1], w[term][2], w[term][3]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_q8_full);
                ++ic;
            }
            // every page id the sequence's rows need must be valid, or all its rows are zero
            bool bad = false;
            const int npg = (it.L + P - 1) / P;
            const int pg0 = GEN ? first_visible_key(it.L, p.rows, 0, p.window) / P : 0;
            const int32_t* trow = p.page_table + (long long)it.g * p.pages_per_seq;
            for (int i = pg0 + t; i < npg; i += 128) {
                const int pg = __ldg(trow + i);
                bad |= (pg < 0 || pg >= p.num_pages);
            }
            bad = named_barrier_or(1, 128, bad);
            const int nk = valid ? it.L - p.rows + r + 1 : it.L;
            const int nlo = (GEN && valid) ? first_visible_key(it.L, p.rows, r, p.window) : 0;   // row sees nlo .. nk-1
            const float crow = p.scale_log2 * isq;
            float m_run = -CUDART_INF_F, l_run = 0.f;
            for (int j = 0; j < it.T; ++j) {
                const uint32_t tcj = tc + j, b = tcj & 1u;
                const uint32_t s_ = sc + j, st = s_ % C::NSK;
                // S_j landed, and the K stage's scales are visible (its K-full phase is
                // complete: QK waited for it); the stage is released after the reads
                bool ok = mbar_wait_bounded(bar_s_full + 8 * b, (tcj >> 1) & 1u, p.wait_ns);
                if (ok) ok = mbar_wait_bounded(bar_k_full + 8 * st, (s_ / C::NSK) & 1u, p.wait_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    abort = true;
                    break;
                }
                const float* meta = reinterpret_cast<const float*>(smem + C::OFF_META + st * C::META_STRIDE);
                float kf[C::BN / 16], vf[C::BN / 16];   // per 16-key block of the tile
#pragma unroll
                for (int q16 = 0; q16 < C::BN / 16; ++q16) {
                    kf[q16] = crow * meta[(q16 * 16) >> lp];
                    vf[q16] = meta[8 + ((q16 * 16) >> lp)];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_k_empty + 8 * st);
                tc_fence_after();
                const uint32_t sc_addr = t_s + C::BN * b + lane_off;
                uint32_t sv[C::BN];
                if constexpr (C::BN == 128) {
                    tmem_ld128(sc_addr, *reinterpret_cast<uint32_t(*)[128]>(sv));
                } else {
                    tmem_ld64(sc_addr, *reinterpret_cast<uint32_t(*)[64]>(sv));
                }
                // the logits in log2 units, in place
#pragma unroll
                for (int e = 0; e < C::BN; ++e) sv[e] = __float_as_uint(__uint_as_float(sv[e]) * kf[e >> 4]);
#define X(e) __uint_as_float(sv[e])
                const int key0 = (it.kt0 + j) * C::BN;
                const int lim = nk - key0, lim_lo = nlo - key0;   // columns outside [lim_lo, lim) are masked
                if (lim < C::BN || (GEN && lim_lo > 0)) {
#pragma unroll
                    for (int e = 0; e < C::BN; ++e)
                        if (e >= lim || (GEN && e < lim_lo)) sv[e] = __float_as_uint(-CUDART_INF_F);
                }
                float mx8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = X(i);
#pragma unroll
                for (int e = 8; e < C::BN; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], X(e));
                const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
                // lazy rescale past 2^8, warp-wide (tcgen05.ld/st are warp-collective)
                bool need = false;
                float alpha = 1.f, m_new = m_run;
                if (mx != -CUDART_INF_F) {
                    if (m_run == -CUDART_INF_F) {
                        m_run = mx;
                    } else if (mx > m_run + C::RESCALE_LOG2) {
                        need = true;
                        alpha = exp2f(m_run - mx);
                        m_new = mx;
                    }
                }
                if (__any_sync(0xffffffffu, need)) {
                    const uint32_t tp = tcj - 1;   // the previous tile's PV
                    const bool okw = mbar_wait_bounded(bar_pv_done + 8 * (tp & 1u), (tp >> 1) & 1u, p.wait_ns);
                    if (!__all_sync(0xffffffffu, okw)) {
                        abort = true;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int q = 0; q < C::D / 32; ++q) {
                        uint32_t ov[32];
                        tmem_ld32(t_o + lane_off + 32 * q, ov);
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                        tmem_st32(t_o + lane_off + 32 * q, ov);
                    }
                    tmem_wait_st();
                    if (need) {
                        l_run *= alpha;
                        m_run = m_new;
                    }
                }
                const float m_use = (m_run == -CUDART_INF_F) ? 0.f : m_run;
                float ps8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int q = 0; q < C::BN / 64; ++q) {
                    uint32_t pk[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int k0 = 64 * q + 2 * e;
                        const float p0 = exp2f(X(k0) - m_use), p1 = exp2f(X(k0 + 1) - m_use);
                        ps8[e & 7] += p0 + p1;
                        pk[e] = pack_f16x2(p0 * vf[k0 >> 4], p1 * vf[k0 >> 4]);
                    }
                    tmem_st32(sc_addr + 32 * q, pk);
                }
#undef X
                l_run += ((ps8[0] + ps8[1]) + (ps8[2] + ps8[3])) + ((ps8[4] + ps8[5]) + (ps8[6] + ps8[7]));
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_p_full + 8 * b);
                if (__any_sync(0xffffffffu, misc[1] != 0)) {
                    abort = true;
                    break;
                }
            }
            if (named_barrier_or(1, 128, abort)) {
                abort = true;
                break;
            }
            // ---- epilogue: O / l -> bf16
            const uint32_t tcl = tc + it.T - 1;
            if (!mbar_wait_bounded(bar_pv_done + 8 * (tcl & 1u), (tcl >> 1) & 1u, p.wait_ns)) abort = true;
            tc_fence_after();
            const float inv = (bad || l_run == 0.f) ? 0.f : 1.f / l_run;
#pragma unroll
            for (int q = 0; q < C::D / 32; ++q) {
                uint32_t ov[32];
                tmem_ld32(t_o + lane_off + 32 * q, ov);
                if (valid) {
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        w[e] = bad ? 0u
                                   : pack_bf16x2(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
                    uint4* dst = reinterpret_cast<uint4*>(orow + 32 * q);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) dst[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
                }
            }
            if (bad && t == 0 && p.err_word) atomicOr(p.err_word, kErrPage);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_o_free);
            tc += it.T;
            sc += it.T;
            if (named_barrier_or(1, 128, abort)) {
                abort = true;
                break;
            }
        }
    }
    if (abort) {
        misc[1] = 1;
        if (lane == 0 && p.err_word) atomicOr(p.err_word, kErrTimeout);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::W_QK) tmem_dealloc(tmem, C::TMEM_COLS);
}

// The launch: one CTA per SM, persistent over the items; the window build for
// a sliding window, else the lean one (a scale <= 0 needs nothing special
// here: logits are scaled before their max).
template <int D>
cudaError_t launch_prefill_fp8_dim(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int sms,
                                   cudaStream_t st) {
    using C = PrefillFp8CfgD<D>;
    auto kern = p.window > 0 ? attn_prefill_fp8_kernel<true, D> : attn_prefill_fp8_kernel<false, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    long long grid = sms;
    if (grid > p.n_items) grid = p.n_items;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(C::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

}  // namespace rad
