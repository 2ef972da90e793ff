// Split-call attention on the 5th-generation tensor cores (tcgen05, TMEM) for
// bf16 KV pools with head_dim 128 or 256, the query rows on the MMA's M: the
// decode and verify call shapes ("kern manifest v7", $defs.Batch) of the
// `attn_paged` op.
//
// The same item plan, partials and combine as attn_tile.cuh, and the same
// structure as the e4m3 split kernel (split_tc05.cuh): the item's up to 32
// query rows are copied into the four 32-lane quarters of M = 128, and softmax
// warp w owns keys KW*w .. KW*w+KW-1 of every BK-key tile (BK = 128, KW = 32
// with head_dim 128; BK = 64, KW = 16 with head_dim 256, so a K or V tile is
// 32 KB either way), with its own running max and sum; the four partials of a
// row are merged once per item, in warp order.  With bf16 pools nothing is
// converted:
//   S  = Q K^T   kind::f16, bf16 A (Q, exact) and B (the staged K rows,
//                K-major, head_dim/64 64-column blocks), M 128, N BK,
//                K = head_dim
//   O += P V     kind::f16, A = P from TMEM as bf16 hi + lo (two MMAs, the
//                pair carries p to ~16 bits), B = the staged V rows as the
//                MN-major operand, N = head_dim
// P is written over S in TMEM (S buffer b's BK columns hold P_hi in the first
// BK/2 and P_lo in the last BK/2; in lane 32w + r only warp w's keys are
// non-zero), so TMEM holds two O buffers (by item parity) with head_dim 128, one
// with head_dim 256 (256 columns), and two S/P buffers (by tile parity).
//
// Warp roles (one CTA per SM, persistent):
//   warps 0-3   softmax (quarter w, thread = query row r); at an item's end
//               they hand its (max, sum) per quarter and its error bits to the
//               epilogue warps and go on with the next item.
//   warp 4      QK: once K_j landed and PV_{j-2} is done (S/P buffer j & 1
//               free), lane 0 issues QK_j.
//   warp 5      PV: once P_j is written and V_j landed, lane 0 issues PV_j into
//               the item's O buffer (at an item's first tile, once the epilogue
//               has read that buffer out); its commit also frees the V stage.
//               On a tile that straddles the item's key range it first zeroes
//               the V rows outside it.
//   warps 6, 7  K and V producers: page ids, one TMA box per page and 64-column
//               block (page_size rows x 128 bytes of the KV head), issued by
//               lanes 0 .. (head_dim/64) * pages - 1; pages outside the item's
//               range load zeros.
//   warp 8      query rows: the item's rows, four copies, in the 128-byte
//               swizzled K-major layout, once the previous item's QKs are done.
//   warps 9-12  epilogue: warp 9 + i reads TMEM lane quarter (9 + i) & 3 of
//               the item's O buffer, and the four merge the quarters of each row
//               in warp order (a 16 KB scratch), then store the row or the
//               split's partial; an item's merge overlaps the next item's tiles.
//   warp 13     scheduler: takes the CTA's items from the counter shared by all
//               CTAs and hands them to the other warps (sched.cuh).
// PV of tile t completes a phase of pv_done[t & 1]; a thread that has seen
// S(t) knows PV(t-2) is done (QK(t) waited for it), so no wait on pv_done is
// two phases ahead of its barrier.  The O buffers' barriers (o_full, ml_full,
// o_free) complete once per item of that buffer, and each role waits on them
// in order: the PV warp and the softmax hand-off wait for the read-out of the
// item NOB back (NOB = the O buffers), so no waiter falls two phases behind.
// Every wait is bounded; a time-out sets RAD_ERRW_TIMEOUT and the roles
// unwind.
#pragma once
#include <cuda.h>

#include "attn_tile.cuh"
#include "sched.cuh"
#include "tc05.cuh"

#ifndef RAD_SPLITBF_NSK
#define RAD_SPLITBF_NSK 3
#endif
#ifndef RAD_SPLITBF_NSV
#define RAD_SPLITBF_NSV 2
#endif
// Stages of the form for calls with at most 8 query rows per KV head, whose
// query rows take 2 KB instead of 32 KB.
#ifndef RAD_SPLITBF_FEW_NSK
#define RAD_SPLITBF_FEW_NSK 3
#endif
#ifndef RAD_SPLITBF_FEW_NSV
#define RAD_SPLITBF_FEW_NSV 3
#endif
// head_dim 256: the four query copies take 64 KB (the FEW form's 8 rows 4 KB).
#ifndef RAD_SPLITBF256_NSK
#define RAD_SPLITBF256_NSK 2
#endif
#ifndef RAD_SPLITBF256_NSV
#define RAD_SPLITBF256_NSV 2
#endif
#ifndef RAD_SPLITBF256_FEW_NSK
#define RAD_SPLITBF256_FEW_NSK 3
#endif
#ifndef RAD_SPLITBF256_FEW_NSV
#define RAD_SPLITBF256_FEW_NSV 3
#endif

namespace rad {

// FEW: every item has at most 8 query rows (calls with at most 8 query rows
// per KV head).  The query operand then holds those 8 rows once, and its
// descriptor's 8-row group stride is 0, so all 16 groups of M = 128 read them:
// lane 32w + r holds row r % 8, the item's row r for r < 8, and the rows
// beyond are masked as before.  Nothing else changes, so a row's bits are
// those of the other form.
template <bool FEW, int D_ = 128>
struct SplitBf16Cfg {
    static constexpr int D = D_;                    // head dim: 128 or 256
    static constexpr int BK = D == 128 ? 128 : 64;  // keys per tile (a K or V tile is 32 KB)
    static constexpr int NBLK = D / 64;             // 64-column blocks of a row
    static constexpr int KW = BK / 4;               // keys of a tile per softmax warp
    static constexpr int NOB = D == 128 ? 2 : 1;    // O buffers in TMEM
    static constexpr int QT = 32;                   // (item planner) query rows per item
    static constexpr int KS = BK;                   // (item planner) keys per stage
    static constexpr int NSK = D == 128 ? (FEW ? RAD_SPLITBF_FEW_NSK : RAD_SPLITBF_NSK)
                                        : (FEW ? RAD_SPLITBF256_FEW_NSK : RAD_SPLITBF256_NSK);   // K stages
    static constexpr int NSV = D == 128 ? (FEW ? RAD_SPLITBF_FEW_NSV : RAD_SPLITBF_NSV)
                                        : (FEW ? RAD_SPLITBF256_FEW_NSV : RAD_SPLITBF256_NSV);   // V stages
    static constexpr int BLK = BK * 128;            // one 64-column block of a K or V tile: [key][128 B]
    static constexpr int KV_TILE = NBLK * BLK;
    static constexpr int Q_ROWS = FEW ? 8 : 128;    // query operand rows held: 8, or four copies of 32
    static constexpr int Q_BLK = Q_ROWS * 128;      // one 64-column block of them
    static constexpr uint32_t Q_SBO = FEW ? 0u : 1024u;   // the A descriptor's 8-row group stride
    static constexpr int MAXPG = BK / 16;           // pages per tile
    static constexpr int META_STRIDE = 128;         // [16]: the tile's page-id flag
    static constexpr int SCR_BYTES = 4 * 32 * 128;  // the merge: [warp][row][32 floats], chunks swizzled
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + NBLK * Q_BLK;    // 1 KB-aligned
    static constexpr int OFF_V = OFF_K + NSK * KV_TILE;
    static constexpr int OFF_SCR = OFF_V + NSV * KV_TILE;
    static constexpr int OFF_ML = OFF_SCR + SCR_BYTES;      // [hand-off slot][max, sum][quarter][32 rows]
    static constexpr int OFF_FLAGS = OFF_ML + 2 * 2 * 4 * 32 * 4;   // [hand-off slot]: the item's error bits
    static constexpr int OFF_META = OFF_FLAGS + 16;
    static constexpr int OFF_BARS = OFF_META + NSK * META_STRIDE;
    // q_full, q_empty, k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV], s_full[2], p_full[2],
    // pv_done[2], o_full[2], ml_full[2], o_free[2], final[2]
    static constexpr int NBARS = 2 + 2 * NSK + 2 * NSV + 2 + 2 + 2 + 2 + 2 + 2 + 2;
    static constexpr int OFF_RING = OFF_BARS + NBARS * 8;     // the item ring (sched.cuh)
    static constexpr int OFF_MISC = OFF_RING + kRingBytes;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;   // 1 KB alignment of the swizzled tiles
    static constexpr int NTHREADS = 14 * 32;
    static constexpr int W_QK = 4, W_PV = 5, W_PROD_K = 6, W_PROD_V = 7, W_Q = 8, W_EPI = 9, W_SCHED = 13;
    static constexpr int RING_CONSUMERS = 13;                 // every warp but the scheduler
    static constexpr int K_EMPTY_ARRIVALS = 1 + 4;            // the QK commit + the softmax warps' flag reads
    static constexpr uint32_t TMEM_COLS = 512;   // O_b [D b, ...), S/P_b [NOB D + BK b, ...)
    static_assert(D == 128 || D == 256, "head_dim 128 or 256");
    static_assert(NOB * D + 2 * BK <= (int)TMEM_COLS, "tensor memory budget");
    static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && KV_TILE % 1024 == 0, "1 KB tiles");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// MODE: kModeCausal, kModeWindow or kModeTree (draft-tree rows, uniform row
// counts: bit i of a row's mask word lets it see the call's key i).
template <int MODE, bool FEW, int D = 128>
__global__ void __launch_bounds__(SplitBf16Cfg<FEW, D>::NTHREADS, 1)
    attn_split_bf16_tc05_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                                const __grid_constant__ AttnParams p) {
    using C = SplitBf16Cfg<FEW, D>;
    constexpr bool WIN = MODE == kModeWindow;
    constexpr bool TREE = MODE == kModeTree;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_addr);

    const uint32_t bar_q_full = base + C::OFF_BARS;
    const uint32_t bar_q_empty = bar_q_full + 8;
    const uint32_t bar_k_full = bar_q_empty + 8;
    const uint32_t bar_k_empty = bar_k_full + 8 * C::NSK;
    const uint32_t bar_v_full = bar_k_empty + 8 * C::NSK;
    const uint32_t bar_v_empty = bar_v_full + 8 * C::NSV;
    const uint32_t bar_s_full = bar_v_empty + 8 * C::NSV;   // [2]
    const uint32_t bar_p_full = bar_s_full + 16;            // [2]
    const uint32_t bar_pv_done = bar_p_full + 16;           // [2], by tile parity
    const uint32_t bar_o_full = bar_pv_done + 16;           // [NOB], by O buffer: the item's last PV done
    const uint32_t bar_ml_full = bar_o_full + 16;           // [NOB], by O buffer: the softmax's hand-off
    const uint32_t bar_o_free = bar_ml_full + 16;           // [NOB], by O buffer: read out by the epilogue
    const uint32_t bar_final = bar_o_free + 16;             // [2]: QK warp, PV warp
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);  // [0] tmem, [1] abort
    const ItemRing iring(smem + C::OFF_RING, base + C::OFF_RING);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar_q_full, 1);
        mbar_init(bar_q_empty, 1);   // the item's last QK commit
        for (int i = 0; i < C::NSK; ++i) {
            mbar_init(bar_k_full + 8 * i, 1);
            mbar_init(bar_k_empty + 8 * i, C::K_EMPTY_ARRIVALS);
        }
        for (int i = 0; i < C::NSV; ++i) {
            mbar_init(bar_v_full + 8 * i, 1);
            mbar_init(bar_v_empty + 8 * i, 1);   // the PV commit
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_s_full + 8 * i, 1);
            mbar_init(bar_p_full + 8 * i, 4);
            mbar_init(bar_pv_done + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_o_full + 8 * i, 1);
            mbar_init(bar_ml_full + 8 * i, 4);
            mbar_init(bar_o_free + 8 * i, 4);
        }
        reinterpret_cast<uint32_t*>(smem + C::OFF_FLAGS)[0] = 0u;
        reinterpret_cast<uint32_t*>(smem + C::OFF_FLAGS)[1] = 0u;
        mbar_init(bar_final, 1);
        mbar_init(bar_final + 8, 1);
        iring.init(C::RING_CONSUMERS, true);
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
    const uint32_t t_o = tmem;                   // O buffer b (item ic: b = ic % NOB) at t_o + D b
    const uint32_t t_s = tmem + C::NOB * C::D;   // S/P buffer b (by tile parity) at t_s + BK b
    bool abort = false;

    // items that run the pipeline: active, a valid sequence length, keys to see
    const auto real = [&](const ItemPlan& it) { return it.active && it.seq_ok && it.n_stages > 0; };

    if (warp == C::W_SCHED) {
        // ===================================================== scheduler (lane 0)
        if (lane == 0 && !iring.run<C, WIN>(p, misc + 1)) abort = true;
        __syncwarp();
    } else if (warp == C::W_PROD_K || warp == C::W_PROD_V) {
        // ===================================================== producers
        const bool is_k = warp == C::W_PROD_K;
        const int NSX = is_k ? C::NSK : C::NSV;
        const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
        const uint32_t bar_full = is_k ? bar_k_full : bar_v_full;
        const uint32_t bar_empty = is_k ? bar_k_empty : bar_v_empty;
        const uint32_t ring = base + (is_k ? C::OFF_K : C::OFF_V);
        const uint64_t pol_kv = policy_evict_first();
        const int P = p.page_size;
        const int ppt = C::BK / P;
        const int oob_tok = p.num_pages * P;   // a row past the pool: TMA fills the box with zeros
        uint32_t sc = 0;
        if (lane == 0) prefetch_tmap(tm);
        for (uint32_t n = 0; !abort; ++n) {
            int item;
            if (!iring.take(n, item, p.wait_ns, is_k)) {
                abort = true;
                break;
            }
            if (item < 0) break;
            const ItemPlan it = plan_item<C, WIN>(item, p);
            if (!real(it)) continue;
            const int page_hi = (it.k1 + P - 1) / P;
            const int page_lo = WIN ? it.klo / P : 0;
            const int32_t* trow = p.page_table + (long long)it.g * p.pages_per_seq;
            int batch0 = -1 << 30, my_pg = 0;
            bool my_bad = false;
            for (int j = 0; j < it.n_stages; ++j) {
                const int pstart = (it.k0 + j * C::BK) / P;
                if (pstart + ppt > batch0 + 32) {
                    batch0 = pstart;
                    const int pi = batch0 + lane;
                    my_bad = false;
                    my_pg = 0;
                    if ((!WIN || pi >= page_lo) && pi < page_hi) {
                        const int pg = __ldg(trow + pi);
                        my_bad = (pg < 0 || pg >= p.num_pages);
                        my_pg = my_bad ? 0 : pg;
                    }
                }
                const uint32_t st = sc % (uint32_t)NSX, use = sc / (uint32_t)NSX;
                if (use >= 1 && !mbar_wait_bounded(bar_empty + 8 * st, (use - 1) & 1u, p.wait_ns)) {
                    abort = true;
                    break;
                }
                // lane i < NBLK * ppt: page i % ppt of the tile, 64-column block i / ppt
                const int pl = lane % ppt, blk = lane / ppt;
                const int pi = pstart + pl;
                const int srcl = (pstart - batch0 + pl) & 31;
                const int pg = __shfl_sync(0xffffffffu, my_pg, srcl);
                const bool mine = lane < C::NBLK * ppt;
                const bool live = mine && (!WIN || pi >= page_lo) && pi < page_hi;
                if (is_k) {
                    // the tile's page-id flag, released by the arrive below
                    const bool badl = __shfl_sync(0xffffffffu, (uint32_t)my_bad, srcl) != 0u;
                    const bool bad_any = __any_sync(0xffffffffu, lane < ppt && pi < page_hi && badl);
                    if (lane == 0)
                        reinterpret_cast<uint32_t*>(smem + C::OFF_META + st * C::META_STRIDE)[16] =
                            bad_any ? kErrPage : 0u;
                }
                // (a test's injected fault: CTA 0 leaves its first K tile unissued)
                const bool skip = is_k && p.fault == kFaultSkipFirstKTile && blockIdx.x == 0 && sc == 0;
                if (lane == 0 && !skip) mbar_arrive_expect_tx(bar_full + 8 * st, (uint32_t)C::KV_TILE);
                __syncwarp();
                if (mine && !skip)
                    tma_load_3d(ring + st * C::KV_TILE + (uint32_t)(blk * C::BLK + pl * P * 128), tm,
                                bar_full + 8 * st, blk * 64, it.kvh, live ? pg * P : oob_tok, pol_kv);
                __syncwarp();
                ++sc;
            }
            if (misc[1]) abort = true;
        }
        // drain: nothing may still be landing in shared memory at exit
        if (lane == 0) {
            const uint32_t first = sc > (uint32_t)NSX ? sc - NSX : 0u;
            for (uint32_t c = first; c < sc; ++c)
                mbar_wait_bounded(bar_full + 8 * (c % NSX), (c / NSX) & 1u, p.wait_ns);
        }
        __syncwarp();
    } else if (warp == C::W_Q) {
        // ===================================================== query rows
        uint32_t ic = 0;
        for (uint32_t n = 0; !abort; ++n) {
            int item;
            if (!iring.take(n, item, p.wait_ns, false)) {
                abort = true;
                break;
            }
            if (item < 0) break;
            const ItemPlan it = plan_item<C, WIN>(item, p);
            if (!real(it)) continue;
            // lane r: query row r of the item (zeros past its rows), loaded before the
            // previous item's QKs are done, stored after
            const int m = it.m0 + lane;
            const bool valid = lane < it.m_end - it.m0;
            const int tok = m / p.ratio, hl = m - tok * p.ratio;
            const __nv_bfloat16* qrow = p.q + ((it.qrow0 + tok) * p.n_head + it.kvh * p.ratio + hl) * C::D;
            // the row in pieces of 16 x 16 bytes (128 columns); the first is loaded
            // before the wait
            bool wait_ok = true;
#pragma unroll 1
            for (int h = 0; h < C::D / 128; ++h) {
                uint4 qv[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    qv[i] = valid ? __ldg(reinterpret_cast<const uint4*>(qrow) + 16 * h + i) : make_uint4(0u, 0u, 0u, 0u);
                if (h == 0 && ic >= 1 &&
                    !__all_sync(0xffffffffu, mbar_wait_bounded(bar_q_empty, (ic - 1) & 1u, p.wait_ns))) {
                    wait_ok = false;
                    break;
                }
                // copy c at rows 32c + r of the M = 128 operand (FEW: rows 0-7 once);
                // elements 8i .. 8i+7 in block i / 8, 16-byte chunk i % 8 (swizzled by
                // the row)
#pragma unroll
                for (int c = 0; c < (FEW ? 1 : 4); ++c) {
                    const int qr = 32 * c + lane;
                    if (FEW && lane >= 8) break;
                    uint8_t* dst = smem + C::OFF_Q + qr * 128;
#pragma unroll
                    for (int i0 = 0; i0 < 16; ++i0) {
                        const int i = 16 * h + i0;
                        *reinterpret_cast<uint4*>(dst + (i >> 3) * C::Q_BLK +
                                                  ((((uint32_t)i & 7u) ^ (uint32_t)(qr & 7)) << 4)) = qv[i0];
                    }
                }
            }
            if (!wait_ok) {
                abort = true;
                break;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_q_full);
            ++ic;
            if (__any_sync(0xffffffffu, misc[1] != 0)) abort = true;
        }
    } else if (warp == C::W_QK) {
        // ===================================================== QK issue
        constexpr uint32_t idesc_qk = umma_idesc_bf16(128, C::BK, 0, 0);
        uint32_t tc = 0, ic = 0;
        bool issued = false;
        for (uint32_t n = 0; !abort; ++n) {
            int item;
            if (!iring.take(n, item, p.wait_ns, false)) {
                abort = true;
                break;
            }
            if (item < 0) break;
            const ItemPlan it = plan_item<C, WIN>(item, p);
            if (!real(it)) continue;
            const int T = it.n_stages;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar_q_full, ic & 1u, p.wait_ns))) {
                abort = true;
                break;
            }
            tc_fence_after();
            for (int j = 0; j < T; ++j) {
                const uint32_t tcj = tc + j, b = tcj & 1u, sk = tcj % C::NSK;
                // K landed, and S/P buffer b is free: PV(tcj - 2) is done
                bool ok = mbar_wait_bounded(bar_k_full + 8 * sk, (tcj / C::NSK) & 1u, p.wait_ns);
                if (ok && tcj >= 2) ok = mbar_wait_bounded(bar_pv_done + 8 * b, ((tcj - 2) >> 1) & 1u, p.wait_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    abort = true;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t kb = base + C::OFF_K + sk * C::KV_TILE;
#pragma unroll
                    for (int kk = 0; kk < C::D / 16; ++kk) {
                        const uint32_t off = (uint32_t)((kk >> 2) * C::BLK + (kk & 3) * 32);
                        tc_mma_ss(t_s + C::BK * b,
                                  umma_desc_sw128(base + C::OFF_Q + (uint32_t)((kk >> 2) * C::Q_BLK + (kk & 3) * 32), 16,
                                                  C::Q_SBO),
                                  umma_desc_sw128(kb + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(bar_s_full + 8 * b);
                    tc_commit(bar_k_empty + 8 * sk);
                    if (j == T - 1) tc_commit(bar_q_empty);   // the item's query rows are read
                    issued = true;
                }
                __syncwarp();
            }
            tc += T;
            ++ic;
            if (misc[1]) abort = true;
        }
        // every MMA this thread issued is complete before TMEM is released
        if (lane == 0 && issued) {
            tc_commit(bar_final);
            mbar_wait_bounded(bar_final, 0, p.wait_ns);
        }
        __syncwarp();
    } else if (warp == C::W_PV) {
        // ===================================================== PV issue
        constexpr uint32_t idesc_pv = umma_idesc_bf16(128, C::D, 0, 1);
        uint32_t tc = 0, ic = 0;
        bool issued = false;
        for (uint32_t n = 0; !abort; ++n) {
            int item;
            if (!iring.take(n, item, p.wait_ns, false)) {
                abort = true;
                break;
            }
            if (item < 0) break;
            const ItemPlan it = plan_item<C, WIN>(item, p);
            if (!real(it)) continue;
            const int T = it.n_stages;
            for (int j = 0; j < T; ++j) {
                const uint32_t tcj = tc + j, b = tcj & 1u, sv = tcj % C::NSV;
                // P_j written, V_j landed, and at an item's first tile its O buffer read out
                // (the item NOB before)
                const uint32_t ob = ic % C::NOB;
                const uint32_t t_ob = t_o + C::D * ob;
                bool ok = mbar_wait_bounded(bar_p_full + 8 * b, (tcj >> 1) & 1u, p.wait_ns);
                if (ok) ok = mbar_wait_bounded(bar_v_full + 8 * sv, (tcj / C::NSV) & 1u, p.wait_ns);
                if (ok && j == 0 && ic >= (uint32_t)C::NOB)
                    ok = mbar_wait_bounded(bar_o_free + 8 * ob, ((ic - C::NOB) / C::NOB) & 1u, p.wait_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    abort = true;
                    break;
                }
                // V rows outside the item's keys [klo, k1) may hold anything (slots past
                // the sequence); P is 0 there, so they are zeroed: 0 x NaN is not 0
                const int key0 = it.k0 + j * C::BK;
                const int zlo = it.klo - key0, zhi = it.k1 - key0;
                if (zlo > 0 || zhi < C::BK) {
                    uint8_t* vt = smem + C::OFF_V + sv * C::KV_TILE;
                    constexpr int CPR = C::NBLK * 8;   // 16-byte chunks per row
                    for (int idx = lane; idx < C::BK * CPR; idx += 32) {
                        const int row = idx / CPR, ch = idx % CPR;
                        if (row < zlo || row >= zhi)
                            *reinterpret_cast<uint4*>(vt + (ch >> 3) * C::BLK + row * 128 + ((ch & 7) << 4)) =
                                make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t vb = base + C::OFF_V + sv * C::KV_TILE;
                    const uint32_t tp = t_s + C::BK * b;
#pragma unroll
                    for (int kk = 0; kk < C::BK / 16; ++kk) {
                        const uint64_t bd = umma_desc_sw128(vb + kk * 16 * 128, C::BLK, 1024);
                        tc_mma_ts(t_ob, tp + kk * 8, bd, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);   // P_hi
                        tc_mma_ts(t_ob, tp + C::BK / 2 + kk * 8, bd, idesc_pv, 1u);               // P_lo
                    }
                    tc_commit(bar_pv_done + 8 * b);
                    tc_commit(bar_v_empty + 8 * sv);
                    if (j == T - 1) tc_commit(bar_o_full + 8 * ob);
                    issued = true;
                }
                __syncwarp();
            }
            tc += T;
            ++ic;
            if (__any_sync(0xffffffffu, misc[1] != 0)) abort = true;
        }
        if (lane == 0 && issued) {
            tc_commit(bar_final + 8);
            mbar_wait_bounded(bar_final + 8, 0, p.wait_ns);
        }
        __syncwarp();
    } else if (warp >= C::W_EPI) {
        // ===================================================== epilogue (warps 9-12)
        // Warp 9 + i reads TMEM lane quarter w = (9 + i) & 3: the O of softmax warp w.
        const int w = warp & 3;
        const int r = lane;                                     // query row r of the item
        const uint32_t lane_off = (uint32_t)(w * 32) << 16;
        const int t = threadIdx.x - C::W_EPI * 32;              // 0 .. 127
        float* const ml = reinterpret_cast<float*>(smem + C::OFF_ML);
        uint32_t* const flags = reinterpret_cast<uint32_t*>(smem + C::OFF_FLAGS);
        uint8_t* const scr = smem + C::OFF_SCR;
        uint32_t ic = 0;
        for (uint32_t n = 0; !abort; ++n) {
            int item;
            if (!iring.take(n, item, p.wait_ns, false)) {
                abort = true;
                break;
            }
            if (item < 0) break;
            const ItemPlan it = plan_item<C, WIN>(item, p);
            if (!real(it)) continue;
            // the item's last PV done and the softmax warps' hand-off
            const uint32_t ob = ic % C::NOB, hs = ic & 1u;   // O buffer, hand-off slot
            bool ok = mbar_wait_bounded(bar_o_full + 8 * ob, (ic / C::NOB) & 1u, p.wait_ns);
            if (ok) ok = mbar_wait_bounded(bar_ml_full + 8 * ob, (ic / C::NOB) & 1u, p.wait_ns);
            if (named_barrier_or(2, 128, !__all_sync(0xffffffffu, ok) || misc[1] != 0)) {   // all leave together
                abort = true;
                break;
            }
            tc_fence_after();
            const float* const mlb = ml + hs * 256;
            const int nrows = it.m_end - it.m0;
            const int m = it.m0 + r;
            const bool valid = r < nrows;
            const int tok = m / p.ratio, hl = m - tok * p.ratio;
            const long long orow = (it.qrow0 + tok) * p.n_head + it.kvh * p.ratio + hl;   // q/out row
            const long long slot_idx = it.gq * p.max_splits + it.s;
            // ---- the four quarters' (max, sum, O) of row r, merged in warp order
            const uint32_t item_bits = flags[hs];
            const bool page_bad = (item_bits & kErrPage) != 0;
            const bool mask_bad = TREE && (item_bits & kErrMask) != 0;
            const bool item_bad = page_bad || mask_bad;
            const uint32_t bad_bits = (page_bad ? kErrPage : 0u) | (mask_bad ? kErrMask : 0u);
            float mq[4], M = -CUDART_INF_F;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                mq[q] = mlb[q * 32 + r];
                M = fmaxf(M, mq[q]);
            }
            const float mu = (M == -CUDART_INF_F) ? 0.f : M;
            float L = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) L += exp2f(mq[q] - mu) * mlb[128 + q * 32 + r];
            const float f_me = exp2f(mq[w] - mu);
            const bool final_write = it.n_splits - it.s_first == 1;
            const float inv = L == 0.f ? 0.f : 1.f / L;
            float* pacc = p.part_acc + slot_idx * p.qtv * C::D;
            for (int c = 0; c < C::D / 32; ++c) {
                // quarter w's scaled O of row r, columns 32c .. 32c+31, 16-byte chunks
                // swizzled by the row
                uint32_t ov[32];
                tmem_ld32(t_o + C::D * ob + lane_off + 32 * c, ov);
                float4* mine = reinterpret_cast<float4*>(scr + (w * 32 + r) * 128);
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4)
                    mine[e4 ^ (r & 7)] = make_float4(__uint_as_float(ov[4 * e4]) * f_me, __uint_as_float(ov[4 * e4 + 1]) * f_me,
                                                     __uint_as_float(ov[4 * e4 + 2]) * f_me,
                                                     __uint_as_float(ov[4 * e4 + 3]) * f_me);
                if (c == C::D / 32 - 1) {
                    // O is read out: the next item's first PV may overwrite it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_o_free + 8 * ob);
                }
                named_barrier_sync(2, 128);
                if (c == 0 && t == 0) flags[hs] = 0u;   // read by all: reset for the item two on
                // row r, columns 32c + 8w .. 32c + 8w + 7: the four quarters summed in order
                float a[8];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float4 s4 = reinterpret_cast<const float4*>(scr + r * 128)[(2 * w + h) ^ (r & 7)];
#pragma unroll
                    for (int q = 1; q < 4; ++q) {
                        const float4 v4 = reinterpret_cast<const float4*>(scr + (q * 32 + r) * 128)[(2 * w + h) ^ (r & 7)];
                        s4.x += v4.x;
                        s4.y += v4.y;
                        s4.z += v4.z;
                        s4.w += v4.w;
                    }
                    a[4 * h] = s4.x;
                    a[4 * h + 1] = s4.y;
                    a[4 * h + 2] = s4.z;
                    a[4 * h + 3] = s4.w;
                }
                const int d0 = 32 * c + 8 * w;
                if (valid) {
                    if (final_write) {
                        // acc * (1/l), the combine kernel's form; a bad item's rows are zeros
                        uint4 o = make_uint4(0u, 0u, 0u, 0u);
                        if (!item_bad) {
                            o.x = pack_bf16x2(a[0] * inv, a[1] * inv);
                            o.y = pack_bf16x2(a[2] * inv, a[3] * inv);
                            o.z = pack_bf16x2(a[4] * inv, a[5] * inv);
                            o.w = pack_bf16x2(a[6] * inv, a[7] * inv);
                        }
                        *reinterpret_cast<uint4*>(p.out + orow * C::D + d0) = o;
                    } else {
                        __stcg(reinterpret_cast<float4*>(pacc + r * C::D + d0), make_float4(a[0], a[1], a[2], a[3]));
                        __stcg(reinterpret_cast<float4*>(pacc + r * C::D + d0) + 1, make_float4(a[4], a[5], a[6], a[7]));
                    }
                }
                named_barrier_sync(2, 128);   // the scratch is free for the next chunk
            }
            if (final_write) {
                if (item_bad && t == 0 && p.err_word) atomicOr(p.err_word, bad_bits);
            } else {
                float* pml = p.part_ml + slot_idx * p.qtv * 2;
                if (w == 0 && valid) __stcg(reinterpret_cast<float2*>(pml) + r, make_float2(L == 0.f ? -CUDART_INF_F : M, L));
                if (t == 0) __stcg(p.part_flag + slot_idx, bad_bits);
            }
            ++ic;
        }
    } else {
        // ===================================================== softmax (warps 0-3)
        const int w = warp;                                     // quarter: keys KW w .. KW w + KW-1 of a tile
        const int r = lane;                                     // query row r of the item
        const uint32_t lane_off = (uint32_t)(w * 32) << 16;     // this warp's TMEM lanes
        const int t = threadIdx.x;                              // 0 .. 127
        float* const ml = reinterpret_cast<float*>(smem + C::OFF_ML);
        uint32_t* const flags = reinterpret_cast<uint32_t*>(smem + C::OFF_FLAGS);
        uint32_t tc = 0, ic = 0;
        for (uint32_t n = 0; !abort; ++n) {
            int item;
            if (!iring.take(n, item, p.wait_ns, false)) {
                abort = true;
                break;
            }
            if (item < 0) break;
            const ItemPlan it = plan_item<C, WIN>(item, p);
            if (!it.active) continue;
            const int nrows = it.m_end - it.m0;
            const int m = it.m0 + r;
            const bool valid = r < nrows;
            const int tok = m / p.ratio, hl = m - tok * p.ratio;
            const long long orow = (it.qrow0 + tok) * p.n_head + it.kvh * p.ratio + hl;   // q/out row
            const long long slot_idx = it.gq * p.max_splits + it.s;
            if (!it.seq_ok) {
                // an invalid sequence length: the group's rows are zeros (malformed
                // offsets name no rows: only the error bit)
                if (w == 0 && valid)
                    for (int i = 0; i < C::D / 8; ++i)
                        reinterpret_cast<uint4*>(p.out + orow * C::D)[i] = make_uint4(0u, 0u, 0u, 0u);
                if (t == 0 && p.err_word) atomicOr(p.err_word, it.cu_ok ? kErrSeqLen : kErrCuSeq);
                continue;
            }
            if (it.n_stages == 0) {
                // a later split none of whose keys the tile's rows see: an empty partial
                float* pacc = p.part_acc + slot_idx * p.qtv * C::D;
                float* pml = p.part_ml + slot_idx * p.qtv * 2;
                if (valid) {
                    for (int i = w; i < C::D / 4; i += 4)
                        __stcg(reinterpret_cast<float4*>(pacc + r * C::D) + i, make_float4(0.f, 0.f, 0.f, 0.f));
                    if (w == 0) __stcg(reinterpret_cast<float2*>(pml) + r, make_float2(-CUDART_INF_F, 0.f));
                }
                if (t == 0) __stcg(p.part_flag + slot_idx, 0u);
                continue;
            }
            const int T = it.n_stages;
            uint32_t bad = 0;
            // pages the group needs that no item of this query tile loads
            if (it.s == it.s_first) {
                const int P_ = p.page_size;
                const int glo = WIN ? first_visible_key(it.L, it.qlen, 0, p.window) / P_ : 0;
                const int tlo = it.klo / P_, thi = (it.kmax + P_ - 1) / P_, ghi = (it.L + P_ - 1) / P_;
                const int32_t* trow = p.page_table + (long long)it.g * p.pages_per_seq;
                const int n_below = tlo - glo;
                for (int i = t; i < n_below + (ghi - thi); i += 128) {
                    const int pi = i < n_below ? glo + i : thi + (i - n_below);
                    const int pg = __ldg(trow + pi);
                    bad |= (pg < 0 || pg >= p.num_pages) ? kErrPage : 0u;
                }
            }
            // every item checks all mask words of its group, so a malformed word
            // zeroes every row of the group: a word holds its own row's bit and
            // no later row's
            uint32_t tmw = 0;
            if (TREE) {
                if (t < it.qlen) {
                    const uint32_t wd = __ldg(p.tree_mask + it.qrow0 + t);
                    if ((wd >> t) != 1u) bad |= kErrMask;
                }
                tmw = valid ? __ldg(p.tree_mask + it.qrow0 + tok) : 0u;
            }
            // keys row r sees: [nlo, nk) (tree rows: every cached key, of the call's
            // keys only their paths), within the item's [klo, k1)
            const int nk = valid ? min(it.L - it.qlen + tok + 1, it.k1) : 0;
            const int nlo = max(it.klo, (WIN && valid) ? first_visible_key(it.L, it.qlen, tok, p.window) : 0);
            const int n_full = TREE ? it.L - it.qlen : nk;   // keys below: no tree bit to test
            const float crow = p.scale_log2;
            float m_run = -CUDART_INF_F, l_run = 0.f;
            for (int j = 0; j < T; ++j) {
                const uint32_t tcj = tc + j, b = tcj & 1u, sk = tcj % C::NSK;
                // S_j landed, and the K stage's scales are visible (QK waited for its K-full
                // phase); the stage is released after the reads
                bool ok = mbar_wait_bounded(bar_s_full + 8 * b, (tcj >> 1) & 1u, p.wait_ns);
                if (ok) ok = mbar_wait_bounded(bar_k_full + 8 * sk, (tcj / C::NSK) & 1u, p.wait_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    abort = true;
                    break;
                }
                bad |= reinterpret_cast<const uint32_t*>(smem + C::OFF_META + sk * C::META_STRIDE)[16];
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_k_empty + 8 * sk);
                tc_fence_after();
                constexpr int KW = C::KW;
                uint32_t sv[KW];
                tmem_ld_cols<KW>(t_s + C::BK * b + KW * w + lane_off, sv);
#pragma unroll
                for (int e = 0; e < KW; ++e) sv[e] = __float_as_uint(__uint_as_float(sv[e]) * crow);
#define X(e) __uint_as_float(sv[e])
                const int key0 = it.k0 + j * C::BK + KW * w;
                const int lim = nk - key0, lim_lo = nlo - key0;   // columns outside [lim_lo, lim) are masked
                if (TREE && key0 + KW > n_full) {
                    // key0 + e < n_full: a cached key; else the call's key i = key0 + e - n_full
                    // (a tile of cached keys only takes the plain test below: i < 0 there)
                    const int ib = key0 - n_full;
#pragma unroll
                    for (int e = 0; e < KW; ++e) {
                        const int i = ib + e;
                        const bool vis = e < lim && e >= lim_lo && (i < 0 || ((tmw >> (i & 31)) & 1u));
                        if (!vis) sv[e] = __float_as_uint(-CUDART_INF_F);
                    }
                } else if (lim < KW || lim_lo > 0) {
#pragma unroll
                    for (int e = 0; e < KW; ++e)
                        if (e >= lim || e < lim_lo) sv[e] = __float_as_uint(-CUDART_INF_F);
                }
                float mx8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = X(i);
#pragma unroll
                for (int e = 8; e < KW; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], X(e));
                const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
                // lazy rescale of this quarter's O past 2^8, warp-wide (tcgen05.ld/st are
                // warp-collective)
                bool need = false;
                float alpha = 1.f, m_new = m_run;
                if (mx != -CUDART_INF_F) {
                    if (m_run == -CUDART_INF_F) {
                        m_run = mx;
                    } else if (mx > m_run + kLazyRescaleLog2) {
                        need = true;
                        alpha = exp2f(m_run - mx);
                        m_new = mx;
                    }
                }
                if (__any_sync(0xffffffffu, need)) {
                    const uint32_t tp = tcj - 1;   // the previous tile's PV
                    const bool okw = j == 0 || mbar_wait_bounded(bar_pv_done + 8 * (tp & 1u), (tp >> 1) & 1u, p.wait_ns);
                    if (!__all_sync(0xffffffffu, okw)) {
                        abort = true;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int q = 0; q < C::D / 32; ++q) {
                        uint32_t ov[32];
                        tmem_ld32(t_o + C::D * (ic % C::NOB) + lane_off + 32 * q, ov);
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                        tmem_st32(t_o + C::D * (ic % C::NOB) + lane_off + 32 * q, ov);
                    }
                    tmem_wait_st();
                    if (need) {
                        l_run *= alpha;
                        m_run = m_new;
                    }
                }
                const float m_use = (m_run == -CUDART_INF_F) ? 0.f : m_run;
                float ps8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                uint32_t ph[KW / 2], plo[KW / 2];   // p as bf16 hi + lo
#pragma unroll
                for (int e = 0; e < KW / 2; ++e) {
                    const float p0 = exp2f(X(2 * e) - m_use), p1 = exp2f(X(2 * e + 1) - m_use);
                    ps8[e & 7] += p0 + p1;
                    const uint32_t hv = pack_bf16x2(p0, p1);
                    ph[e] = hv;
                    plo[e] = pack_bf16x2(p0 - bf16_lo(hv), p1 - bf16_hi(hv));
                }
#undef X
                {
                    // P over S in this warp's lanes: P_hi in columns [0, BK/2), P_lo in
                    // [BK/2, BK); this quarter's keys at columns KW/2 w .. KW/2 w + KW/2-1
                    // of each, zeros elsewhere (its S reads are complete)
                    uint32_t z[KW / 2];
#pragma unroll
                    for (int e = 0; e < KW / 2; ++e) z[e] = 0u;
                    const uint32_t tp = t_s + C::BK * b + lane_off;
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        if (h == w) {
                            tmem_st_cols<KW / 2>(tp + (KW / 2) * h, ph);
                            tmem_st_cols<KW / 2>(tp + C::BK / 2 + (KW / 2) * h, plo);
                        } else {
                            tmem_st_cols<KW / 2>(tp + (KW / 2) * h, z);
                            tmem_st_cols<KW / 2>(tp + C::BK / 2 + (KW / 2) * h, z);
                        }
                    }
                }
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
            if (abort) break;
            // ---- hand-off: this quarter's (max, sum) of row r and the item's error bits
            // go to the epilogue warps, once they have read out the item NOB before (its
            // O buffer is this item's; its hand-off slot was read before that)
            const uint32_t ob = ic % C::NOB, hs = ic & 1u;
            if (ic >= (uint32_t)C::NOB &&
                !__all_sync(0xffffffffu,
                            mbar_wait_bounded(bar_o_free + 8 * ob, ((ic - C::NOB) / C::NOB) & 1u, p.wait_ns))) {
                abort = true;
                break;
            }
            ml[hs * 256 + w * 32 + r] = m_run;
            ml[hs * 256 + 128 + w * 32 + r] = l_run;
            const uint32_t bad_w = __reduce_or_sync(0xffffffffu, bad);
            if (lane == 0 && bad_w) atomicOr(flags + hs, bad_w);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_ml_full + 8 * ob);
            tc += T;
            ++ic;
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

// Launch of one form: one CTA per SM (shared memory, TMEM), persistent over
// the items; calls with a sliding window run the window build, calls with
// tree masks the tree build, others the causal one.
template <bool FEW, int D>
cudaError_t launch_split_bf16_form(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int sms,
                                   cudaStream_t st) {
    using C = SplitBf16Cfg<FEW, D>;
    auto kern = p.window > 0  ? attn_split_bf16_tc05_kernel<kModeWindow, FEW, D>
                : p.tree_mask ? attn_split_bf16_tc05_kernel<kModeTree, FEW, D>
                              : attn_split_bf16_tc05_kernel<kModeCausal, FEW, D>;
    cudaError_t e = launch_item_order<C>(p, st);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
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
