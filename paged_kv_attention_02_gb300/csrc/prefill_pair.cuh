// Prefill-chunk attention on the 5th-generation tensor cores for bf16 KV pools
// with head_dim 128: two query tiles of one KV head per work item.
//
// The arithmetic of a row is that of prefill_tc05.cuh (S = Q K^T in TMEM, a
// lazily rescaled running max in log2 units, P written back over S as bf16
// hi + lo, O += P V in TMEM, O / l at the end), over 64-key tiles (128-key tiles
// with one S buffer per query tile measured slower).  What
// changes is the work item: (sequence g, KV head kvh, query tiles 2qp and
// 2qp + 1), so every K and V tile that lands in shared memory serves 256
// query rows.  Per 128 query rows and key that halves the TMA page boxes (two
// 2 KB boxes per 16-slot page and 64-column block: their issue rate bounded
// the one-tile kernel) and it runs two softmax warpgroups side by side, one
// per query tile (the per-tile softmax on four warps bounded it as well).
//
// Tensor memory (512 columns): O_k at 128 k, and S/P buffers b of query tile
// k at 256 + 128 k + BN b (k in {0, 1}; b < NSB: two buffers of 64 keys, or
// one of 128).
//
// Warp roles (one CTA per SM, persistent over items, heavier items first):
//   warps 0-3   softmax of query tile 0 (thread t: its row t, TMEM lane t)
//   warp 4      QK: per key tile j, once K_j landed, issues S_0 = Q_0 K_j^T into
//               S buffer (0, j mod NSB) once PV_0(j-NSB) is done, then S_1
//               likewise
//   warp 5      PV: per key tile j, once V_j landed, issues O_0 += P_0 V_j once
//               P_0(j) is written, then O_1; it first zeroes V rows past the
//               sequence's end (and below the item's first visible key in the
//               first live page of a window): P is 0 there, V must not be NaN
//   warp 6      K producer: the item's two query tiles (4-D boxes) and, per
//               tile, one 3-D box per page and 64-column block of K
//   warp 7      V producer: the same for V
//   warps 8-11  softmax of query tile 1
// Waits on the per-tile barriers follow prefill_tc05.cuh (PV of tile t
// completes a phase of pv_done[k][t mod NSB]; a thread that has seen S_k(t)
// knows PV_k(t-NSB) is done).  Every wait is bounded; on a time-out the CTA sets
// RAD_ERRW_TIMEOUT and unwinds, waiting (bounded) for its copies and MMAs
// before freeing TMEM.
#pragma once
#include <cuda.h>

#include "attn_tile.cuh"
#include "prefill_tc05.cuh"
#include "tc05.cuh"

namespace rad {

struct PrefPairCfg {
    static constexpr int D = 128;
    static constexpr int BM = 128;                  // query rows per query tile
    static constexpr int BN = 64;                   // keys per tile
    static constexpr int NSB = 2;                   // S/P buffers per query tile
    static constexpr int NSK = 4;                   // K stages
    static constexpr int NSV = 4;                   // V stages
    static constexpr int HB_BYTES = BN * 128;       // one 64-column block of a K/V tile: [key][128 B]
    static constexpr int QHB_BYTES = BM * 128;      // one 64-column block of a query tile
    static constexpr int TILE_BYTES = BN * D * 2;   // K or V tile
    static constexpr int QTILE_BYTES = BM * D * 2;  // one query tile
    static constexpr int OFF_Q = 0;                 // [query tile][64-column block][row][128 B]
    static constexpr int OFF_K = 2 * QTILE_BYTES;
    static constexpr int OFF_V = OFF_K + NSK * TILE_BYTES;
    static constexpr int OFF_BARS = OFF_V + NSV * TILE_BYTES;
    // q_full, q_empty, k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV], s_full[2][2],
    // p_full[2][2], pv_done[2][2], o_free[2], final[2]
    static constexpr int NBARS = 2 + 2 * NSK + 2 * NSV + 4 + 4 + 4 + 2 + 2;
    static constexpr int OFF_MISC = OFF_BARS + NBARS * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr int NTHREADS = 12 * 32;
    static constexpr int W_QK = 4, W_PV = 5, W_PROD_K = 6, W_PROD_V = 7, W_SM1 = 8;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr float RESCALE_LOG2 = 8.f;   // rescale O when the max grows past 2^8
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && TILE_BYTES % 1024 == 0, "1 KB tiles");
};

// A pair item: its two query tiles' plans (tile 1 may hold no row: the last
// pair of an odd tile count) and the key tiles the pair runs over.
struct PairItem {
    PrefItem q[2];
    int g, kvh, L;
    bool seq_ok;
    int kt0;   // first key tile: that of query tile 0 (its window starts first)
    int T;     // key tiles kt0 .. kt0+T-1: up to query tile 1's last
};

// item order: pair rank first (later pairs see more keys: heaviest first),
// then sequence, then KV head.  p.n_qtiles counts query tiles of 128 rows.
template <bool GEN>
__device__ __forceinline__ PairItem plan_pair(int item, const AttnParams& p) {
    using C = PrefPairCfg;
    PairItem pi;
    const int n_pairs = (p.n_qtiles + 1) / 2;
    const int per_rank = p.groups * p.n_head_kv;
    const int rank = item / per_rank;
    const int rem = item - rank * per_rank;
    pi.g = rem / p.n_head_kv;
    pi.kvh = rem - pi.g * p.n_head_kv;
    const int qp = n_pairs - 1 - rank;
    pi.L = __ldg(p.seq_lens + pi.g);
    pi.seq_ok = pi.L >= p.rows && (long long)pi.L <= (long long)p.pages_per_seq * p.page_size;
    int kend = 0;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        PrefItem& it = pi.q[k];
        it.g = pi.g;
        it.kvh = pi.kvh;
        it.qt = 2 * qp + k;
        it.L = pi.L;
        it.seq_ok = pi.seq_ok;
        it.m0 = it.qt * C::BM;
        it.m_end = min(p.M, it.m0 + C::BM);
        const bool rows = it.m_end > it.m0;
        it.kmax = (it.seq_ok && rows) ? it.L - p.rows + (it.m_end - 1) / p.ratio + 1 : 0;
        it.klo = (GEN && it.seq_ok && rows) ? first_visible_key(it.L, p.rows, it.m0 / p.ratio, p.window) : 0;
        it.kt0 = it.klo / C::BN;
        it.T = rows ? (it.kmax + C::BN - 1) / C::BN - it.kt0 : 0;
        if (rows) kend = max(kend, (it.kmax + C::BN - 1) / C::BN);
    }
    pi.kt0 = pi.q[0].kt0;
    pi.T = kend - pi.kt0;
    return pi;
}

template <bool GEN>
__global__ void __launch_bounds__(PrefPairCfg::NTHREADS, 1)
    attn_prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ AttnParams p) {
    using C = PrefPairCfg;
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
    const uint32_t bar_s_full = bar_v_empty + 8 * C::NSV;   // [k][b]
    const uint32_t bar_p_full = bar_s_full + 32;            // [k][b]
    const uint32_t bar_pv_done = bar_p_full + 32;           // [k][b]
    const uint32_t bar_o_free = bar_pv_done + 32;           // [k]
    const uint32_t bar_final = bar_o_free + 16;             // [2]: QK warp, PV warp
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);  // [0] tmem, [1] abort

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar_q_full, 1);
        mbar_init(bar_q_empty, 1);
        for (int i = 0; i < C::NSK; ++i) {
            mbar_init(bar_k_full + 8 * i, 1);
            mbar_init(bar_k_empty + 8 * i, 1);
        }
        for (int i = 0; i < C::NSV; ++i) {
            mbar_init(bar_v_full + 8 * i, 1);
            mbar_init(bar_v_empty + 8 * i, 1);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(bar_s_full + 8 * i, 1);
            mbar_init(bar_p_full + 8 * i, 4);
            mbar_init(bar_pv_done + 8 * i, 1);
        }
        mbar_init(bar_o_free, 4);
        mbar_init(bar_o_free + 8, 4);
        mbar_init(bar_final, 1);
        mbar_init(bar_final + 8, 1);
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
    const auto t_o = [&](int k) { return tmem + 128u * (uint32_t)k; };
    const auto t_s = [&](int k, uint32_t b) { return tmem + 256u + 128u * (uint32_t)k + (uint32_t)C::BN * b; };

    const int n_items = p.n_items;
    bool abort = false;

    if (warp == C::W_PROD_K || warp == C::W_PROD_V) {
        // ===================================================== producers: K (and the query tiles), V
        const bool is_k = warp == C::W_PROD_K;
        const int NSX = is_k ? C::NSK : C::NSV;
        const uint32_t bar_full = is_k ? bar_k_full : bar_v_full;
        const uint32_t bar_empty = is_k ? bar_k_empty : bar_v_empty;
        const uint32_t ring = base + (is_k ? C::OFF_K : C::OFF_V);
        const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
        const uint64_t pol = policy_evict_last();   // K/V tiles are re-read by every query tile pair
        const int P = p.page_size;
        const int ppt = C::BN / P;
        const int oob_tok = p.num_pages * P;
        uint32_t sc = 0, ic = 0;
        if (lane == 0) {
            if (is_k) prefetch_tmap(&tm_q);
            prefetch_tmap(tm);
        }
        for (int rd = 0; rd * (int)gridDim.x < n_items && !abort; ++rd) {
            const int item = prefill_item_of<true>(rd, blockIdx.x, gridDim.x);
            if (item >= n_items) break;
            const PairItem pi = plan_pair<GEN>(item, p);
            if (!pi.seq_ok) continue;
            if (is_k) {
                if (ic >= 1 && !mbar_wait_bounded(bar_q_empty, (ic - 1) & 1u, p.wait_ns)) {
                    abort = true;
                    break;
                }
                if (lane == 0) {
                    // both query tiles (rows past the call's load as zeros)
                    mbar_arrive_expect_tx(bar_q_full, 2 * C::QTILE_BYTES);
#pragma unroll
                    for (int k = 0; k < 2; ++k)
#pragma unroll
                        for (int hb = 0; hb < 2; ++hb)
                            tma_load_4d(base + C::OFF_Q + k * C::QTILE_BYTES + hb * C::QHB_BYTES, &tm_q, bar_q_full,
                                        hb * 64, pi.kvh * p.ratio, pi.q[k].m0 / p.ratio, pi.g, pol);
                }
                ++ic;
            }
            const int kmax = max(pi.q[0].kmax, pi.q[1].kmax);
            const int page_hi = (kmax + P - 1) / P;
            const int page_lo = GEN ? pi.q[0].klo / P : 0;   // pages below hold no visible key: never read
            const int32_t* trow = p.page_table + (long long)pi.g * p.pages_per_seq;
            int batch0 = -1 << 30, my_pg = 0;
            for (int j = 0; j < pi.T; ++j) {
                const uint32_t st = sc % (uint32_t)NSX, use = sc / (uint32_t)NSX;
                if (use >= 1 && !mbar_wait_bounded(bar_empty + 8 * st, (use - 1) & 1u, p.wait_ns)) {
                    abort = true;
                    break;
                }
                const int pstart = (pi.kt0 + j) * ppt;
                if (pstart + ppt > batch0 + 32) {
                    batch0 = pstart;
                    const int pgi = batch0 + lane;
                    my_pg = 0;
                    if ((!GEN || pgi >= page_lo) && pgi < page_hi) {
                        const int pg = __ldg(trow + pgi);
                        my_pg = (pg < 0 || pg >= p.num_pages) ? 0 : pg;
                    }
                }
                const uint32_t dst = ring + st * C::TILE_BYTES;
                if (lane == 0) mbar_arrive_expect_tx(bar_full + 8 * st, C::TILE_BYTES);
                for (int i = 0; i < ppt; ++i) {
                    const int pgi = pstart + i;
                    const int pg = __shfl_sync(0xffffffffu, my_pg, (pgi - batch0) & 31);
                    const int tok = ((!GEN || pgi >= page_lo) && pgi < page_hi) ? pg * P : oob_tok;
                    if (lane == 0) {
#pragma unroll
                        for (int hb = 0; hb < 2; ++hb)
                            tma_load_3d(dst + hb * C::HB_BYTES + i * P * 128, tm, bar_full + 8 * st, hb * 64, pi.kvh,
                                        tok, pol);
                    }
                }
                ++sc;
            }
            if (misc[1]) abort = true;
        }
        // drain: nothing may still be landing in shared memory at exit
        if (lane == 0) {
            const uint32_t first = sc > (uint32_t)NSX ? sc - NSX : 0u;
            for (uint32_t c = first; c < sc; ++c)
                mbar_wait_bounded(bar_full + 8 * (c % NSX), (c / NSX) & 1u, p.wait_ns);
            if (is_k && ic >= 1) mbar_wait_bounded(bar_q_full, (ic - 1) & 1u, p.wait_ns);
        }
    } else if (warp == C::W_QK) {
        // ===================================================== QK issue
        constexpr uint32_t idesc_qk = umma_idesc_bf16(C::BM, C::BN, 0, 0);
        uint32_t sc = 0, tc = 0, ic = 0;
        bool issued = false;
        for (int rd = 0; rd * (int)gridDim.x < n_items && !abort; ++rd) {
            const int item = prefill_item_of<true>(rd, blockIdx.x, gridDim.x);
            if (item >= n_items) break;
            const PairItem pi = plan_pair<GEN>(item, p);
            if (!pi.seq_ok) continue;
            if (!mbar_wait_bounded(bar_q_full, ic & 1u, p.wait_ns)) {
                abort = true;
                break;
            }
            tc_fence_after();
            for (int j = 0; j < pi.T; ++j) {
                const uint32_t s_ = sc + j, st = s_ % C::NSK, tcj = tc + j, b = tcj % C::NSB;
                if (!mbar_wait_bounded(bar_k_full + 8 * st, (s_ / C::NSK) & 1u, p.wait_ns)) {
                    abort = true;
                    break;
                }
                const uint32_t kb = base + C::OFF_K + st * C::TILE_BYTES;
                for (int k = 0; k < 2 && !abort; ++k) {
                    // S buffer (k, b) is free: PV_k(tcj - NSB) read the P it held
                    if (tcj >= (uint32_t)C::NSB &&
                        !mbar_wait_bounded(bar_pv_done + 8 * (2 * k + b), ((tcj - C::NSB) / C::NSB) & 1u, p.wait_ns)) {
                        abort = true;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t qb = base + C::OFF_Q + k * C::QTILE_BYTES;
#pragma unroll
                        for (int kk = 0; kk < C::D / 16; ++kk) {
                            const uint32_t qoff = (kk >> 2) * C::QHB_BYTES + (kk & 3) * 32;
                            const uint32_t koff = (kk >> 2) * C::HB_BYTES + (kk & 3) * 32;
                            tc_mma_ss(t_s(k, b), umma_desc_sw128(qb + qoff, 16, 1024), umma_desc_sw128(kb + koff, 16, 1024),
                                      idesc_qk, kk > 0 ? 1u : 0u);
                        }
                        tc_commit(bar_s_full + 8 * (2 * k + b));
                        issued = true;
                    }
                    __syncwarp();
                }
                if (abort) break;
                if (lane == 0) tc_commit(bar_k_empty + 8 * st);   // the K tile is read once both QKs are done
                __syncwarp();
            }
            // the query tiles are read once the item's QKs are done
            if (lane == 0 && !abort) tc_commit(bar_q_empty);
            __syncwarp();
            sc += pi.T;
            tc += pi.T;
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
        constexpr uint32_t idesc_pv = umma_idesc_bf16(C::BM, C::D, 0, 1);
        uint32_t sc = 0, tc = 0, ic = 0;
        bool issued = false;
        for (int rd = 0; rd * (int)gridDim.x < n_items && !abort; ++rd) {
            const int item = prefill_item_of<true>(rd, blockIdx.x, gridDim.x);
            if (item >= n_items) break;
            const PairItem pi = plan_pair<GEN>(item, p);
            if (!pi.seq_ok) continue;
            // V rows to zero: slots past the sequence's end in its last page,
            // and slots of the first live page below the pair's first visible key
            const int P = p.page_size;
            const int zero_lo = pi.L, zero_hi = ((pi.L + P - 1) / P) * P;
            const int head_lo = (pi.q[0].klo / P) * P, head_hi = pi.q[0].klo;
            for (int jj = 0; jj < pi.T; ++jj) {
                const uint32_t tcj = tc + jj, b = tcj % C::NSB;
                const uint32_t s_ = sc + jj, st = s_ % C::NSV;
                if (!mbar_wait_bounded(bar_v_full + 8 * st, (s_ / C::NSV) & 1u, p.wait_ns)) {
                    abort = true;
                    break;
                }
                const uint32_t vb = base + C::OFF_V + st * C::TILE_BYTES;
                // zero V rows of keys past the sequence's end held by this tile
                const int key0 = (pi.kt0 + jj) * C::BN;
                const int z0 = max(zero_lo, key0) - key0, z1 = min(zero_hi, key0 + C::BN) - key0;
                const int h0 = max(head_lo, key0) - key0, h1 = min(head_hi, key0 + C::BN) - key0;
                const int nz = max(z1 - z0, 0), nh = GEN ? max(h1 - h0, 0) : 0;
                if (nz + nh > 0) {
                    for (int idx = lane; idx < (nz + nh) * 16; idx += 32) {
                        const int rr = idx / 16, c16 = idx % 16;
                        const int row = rr < nz ? z0 + rr : h0 + (rr - nz);
                        const uint32_t a = vb + (c16 >> 3) * C::HB_BYTES + row * 128 + (((c16 & 7) ^ (row & 7)) << 4);
                        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                for (int k = 0; k < 2 && !abort; ++k) {
                    // P_k(j) written, and at an item's first tile O_k read out
                    bool ok = mbar_wait_bounded(bar_p_full + 8 * (2 * k + b), (tcj / C::NSB) & 1u, p.wait_ns);
                    if (ok && jj == 0 && ic >= 1) ok = mbar_wait_bounded(bar_o_free + 8 * k, (ic - 1) & 1u, p.wait_ns);
                    if (!__all_sync(0xffffffffu, ok)) {
                        abort = true;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t sp = t_s(k, b);
#pragma unroll
                        for (int kk = 0; kk < C::BN / 16; ++kk) {
                            const uint64_t bd = umma_desc_sw128(vb + kk * 16 * 128, C::HB_BYTES, 1024);
                            tc_mma_ts(t_o(k), sp + kk * 8, bd, idesc_pv, (jj > 0 || kk > 0) ? 1u : 0u);
                            tc_mma_ts(t_o(k), sp + C::BN / 2 + kk * 8, bd, idesc_pv, 1u);
                        }
                        tc_commit(bar_pv_done + 8 * (2 * k + b));
                        issued = true;
                    }
                    __syncwarp();
                }
                if (abort) break;
                if (lane == 0) tc_commit(bar_v_empty + 8 * st);   // the V tile is read once both PVs are done
                __syncwarp();
            }
            sc += pi.T;
            tc += pi.T;
            ++ic;
            if (misc[1]) abort = true;
        }
        if (lane == 0 && issued) {
            tc_commit(bar_final + 8);
            mbar_wait_bounded(bar_final + 8, 0, p.wait_ns);
        }
        __syncwarp();
    } else {
        // ===================================================== softmax (warps 0-3: query tile 0, 8-11: 1)
        const int k = warp >= C::W_SM1 ? 1 : 0;
        const int t = threadIdx.x - (k ? C::W_SM1 * 32 : 0);   // query row of the tile
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;   // this warp's TMEM lanes
        const uint32_t nb = 1 + (uint32_t)k;                       // named barrier of this warpgroup
        const float c = p.scale_log2;
        uint32_t tc = 0;
        for (int rd = 0; rd * (int)gridDim.x < n_items && !abort; ++rd) {
            const int item = prefill_item_of<true>(rd, blockIdx.x, gridDim.x);
            if (item >= n_items) break;
            const PairItem pi = plan_pair<GEN>(item, p);
            const PrefItem it = k ? pi.q[1] : pi.q[0];   // (a copy: no runtime index into the pair)
            const int m = it.m0 + t;
            const bool valid = m < it.m_end;
            const int r = m / p.ratio, hl = m - r * p.ratio;
            __nv_bfloat16* orow =
                p.out + (((long long)it.g * p.rows + r) * p.n_head + it.kvh * p.ratio + hl) * C::D;
            if (!pi.seq_ok) {
                if (valid)
                    for (int i = 0; i < C::D / 8; ++i) reinterpret_cast<uint4*>(orow)[i] = make_uint4(0, 0, 0, 0);
                if (k == 0 && t == 0 && p.err_word) atomicOr(p.err_word, kErrSeqLen);
                continue;
            }
            // every page id the sequence's rows need must be valid, or all its
            // rows are zero
            bool bad = false;
            const int npg = (it.L + p.page_size - 1) / p.page_size;
            const int pg0 = GEN ? first_visible_key(it.L, p.rows, 0, p.window) / p.page_size : 0;
            const int32_t* trow = p.page_table + (long long)it.g * p.pages_per_seq;
            for (int i = pg0 + t; i < npg; i += 128) {
                const int pg = __ldg(trow + i);
                bad |= (pg < 0 || pg >= p.num_pages);
            }
            bad = named_barrier_or(nb, 128, bad);
            const int nk = valid ? it.L - p.rows + r + 1 : 0;
            const int nlo = (GEN && valid) ? first_visible_key(it.L, p.rows, r, p.window) : 0;   // row sees nlo .. nk-1
            float m_run = -CUDART_INF_F, l_run = 0.f;
            for (int j = 0; j < pi.T; ++j) {
                const uint32_t tcj = tc + j, b = tcj % C::NSB;
                // (every exit from here is taken by the whole warp: the tcgen05
                // loads and stores below are warp-collective)
                if (!__all_sync(0xffffffffu,
                                mbar_wait_bounded(bar_s_full + 8 * (2 * k + b), (tcj / C::NSB) & 1u, p.wait_ns))) {
                    abort = true;
                    break;
                }
                tc_fence_after();
                const uint32_t sc_ = t_s(k, b) + lane_off;
                uint32_t sv[C::BN];
                tmem_ld64(sc_, sv);
                // Logits are scaled by c after the max; a scale <= 0 would turn
                // that order around (and -inf * 0 into NaN), so then the tile is
                // scaled first and c taken as 1.
                float cs = c;
                if (GEN && c <= 0.f) {
#pragma unroll
                    for (int e = 0; e < C::BN; ++e) sv[e] = __float_as_uint(__uint_as_float(sv[e]) * c);
                    cs = 1.f;
                }
                const int key0 = (pi.kt0 + j) * C::BN;
                const int lim = nk - key0, lim_lo = nlo - key0;   // columns outside [lim_lo, lim) are masked
                if (lim < C::BN || (GEN && lim_lo > 0)) {
#pragma unroll
                    for (int e = 0; e < C::BN; ++e)
                        if (e >= lim || (GEN && e < lim_lo)) sv[e] = __float_as_uint(-CUDART_INF_F);
                }
                // row max as 8 independent chains
                float mx8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = __uint_as_float(sv[i]);
#pragma unroll
                for (int e = 8; e < C::BN; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], __uint_as_float(sv[e]));
                const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
                // A row whose max grew past 2^8 rescales its O row, warp-wide
                // (the others multiply by exactly 1).
                bool need = false;
                float alpha = 1.f, m_new = m_run;
                if (mx != -CUDART_INF_F) {
                    const float mx_s = mx * cs;
                    if (m_run == -CUDART_INF_F) {
                        m_run = mx_s;   // first keys of the row: nothing accumulated yet
                    } else if (mx_s > m_run + C::RESCALE_LOG2) {
                        need = true;
                        alpha = exp2f(m_run - mx_s);
                        m_new = mx_s;
                    }
                }
                if (__any_sync(0xffffffffu, need)) {
                    // PV of the previous tile must have landed before O is rescaled
                    const uint32_t tp = tcj - 1;
                    const bool ok = j == 0 || mbar_wait_bounded(bar_pv_done + 8 * (2 * k + tp % C::NSB),
                                                                 (tp / C::NSB) & 1u, p.wait_ns);
                    if (!__all_sync(0xffffffffu, ok)) {
                        abort = true;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t ov[32];
                        tmem_ld32(t_o(k) + lane_off + 32 * q, ov);
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                        tmem_st32(t_o(k) + lane_off + 32 * q, ov);
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
                for (int q = 0; q < C::BN / 32; ++q) {
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float p0 = exp2f(__uint_as_float(sv[32 * q + 2 * e]) * cs - m_use);
                        const float p1 = exp2f(__uint_as_float(sv[32 * q + 2 * e + 1]) * cs - m_use);
                        ps8[e & 7] += p0 + p1;
                        const uint32_t h = pack_bf16x2(p0, p1);
                        hi[e] = h;
                        lo[e] = pack_bf16x2(p0 - bf16_lo(h), p1 - bf16_hi(h));
                    }
                    tmem_st16(sc_ + 16 * q, hi);
                    tmem_st16(sc_ + C::BN / 2 + 16 * q, lo);
                }
                l_run += ((ps8[0] + ps8[1]) + (ps8[2] + ps8[3])) + ((ps8[4] + ps8[5]) + (ps8[6] + ps8[7]));
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_p_full + 8 * (2 * k + b));
                if (__any_sync(0xffffffffu, misc[1] != 0)) {
                    abort = true;
                    break;
                }
            }
            if (named_barrier_or(nb, 128, abort)) {
                abort = true;
                break;
            }
            // ---- epilogue: O / l -> bf16
            const uint32_t tcl = tc + pi.T - 1;
            if (!mbar_wait_bounded(bar_pv_done + 8 * (2 * k + tcl % C::NSB), (tcl / C::NSB) & 1u, p.wait_ns))
                abort = true;
            tc_fence_after();
            const float inv = (bad || l_run == 0.f) ? 0.f : 1.f / l_run;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t ov[32];
                tmem_ld32(t_o(k) + lane_off + 32 * q, ov);
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
            if (bad && k == 0 && t == 0 && p.err_word) atomicOr(p.err_word, kErrPage);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_o_free + 8 * k);
            tc += pi.T;
            if (named_barrier_or(nb, 128, abort)) {
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

// The launch: one CTA per SM, persistent over the pair items (p.n_items
// counts pairs); the general build for a sliding window or a scale <= 0.
inline cudaError_t launch_prefill_pair(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                       const AttnParams& p, int sms, cudaStream_t st) {
    using C = PrefPairCfg;
    auto kern = (p.window > 0 || p.scale_log2 <= 0.f) ? attn_prefill_pair_kernel<true>
                                                      : attn_prefill_pair_kernel<false>;
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
    return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p);
}

}  // namespace rad
