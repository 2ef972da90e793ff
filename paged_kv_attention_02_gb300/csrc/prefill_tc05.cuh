// Prefill-chunk attention on the 5th-generation tensor cores (tcgen05, TMEM).
//
// A work item is (sequence g, KV head kvh, query tile qt): 128 query rows of
// one KV head -- rows m = r*ratio + hl, the chunk's tokens r times the query
// heads hl that share the KV head ("Radiance architecture plugins", section
// "Declare: the metadata": n_head over n_head_kv) -- against keys
// 0 .. kmax-1 of the sequence, causal per row: row r sees keys 0 .. L-R+r
// ("kern manifest v7", $defs.Fill `seq_len`; $defs.Batch `context`: a
// prefill's expansion of the cached rows), or with a sliding window W only
// the last W of them ("Radiance architecture plugins", section "Declare:
// buffers and KV groups", RAD_KV_WINDOW); key tiles wholly below the tile's
// first row's window are skipped.
//
// Warp roles (one CTA per SM, persistent over items, heavier query tiles first):
//   warp 6      K producer: TMA loads of the item's query rows (one 4-D box per
//               128-byte column block) and, per 128-key tile, of every page's
//               K rows (one 3-D box per page and column block) into a ring of
//               K tiles, each free again once its QK is done; pages past the
//               tile's range load from an out-of-range coordinate (zero fill).
//   warp 7      V producer: the same for V rows, into a ring of V tiles, each
//               free again once its PV is done.  (With one ring of K+V stages
//               a tile's K waited for its PV too, and a stage's ~1.8 us load
//               could not hide behind three stages.)
//   warp 4      QK issue: lane 0 issues S_j = Q K_j^T (M 128, N 128, K =
//               head_dim; both operands in shared memory, K-major, 128-byte
//               swizzle) into TMEM buffer j & 1 once K_j landed and PV_{j-2}
//               (which read the P held there) is done.
//   warp 5      PV issue: once the softmax has written P_j, lane 0 issues
//               O += P_j V_j (A = P from TMEM, B = V MN-major from shared
//               memory).  The warp also zeroes V rows past the sequence's end
//               in the tile that holds its last page, and the rows below the
//               tile's first visible key in the first live page of a window
//               (P is 0 there, V must not be NaN).  Separate issuing warps keep
//               a late K tile from holding up the PV of a finished P.
//   warps 0-3   softmax: thread t owns query row t (TMEM lane t); per tile it
//               reads S_j with tcgen05.ld, masks, keeps the running max in
//               log2 units and rescales O in TMEM only when the max grew by
//               more than 2^8 (the row's arithmetic never depends on other
//               rows), writes P as bf16 hi + lo (hi = bf16(p), lo = bf16(p-hi))
//               back over S_j, and at the end reads O, divides by the sum and
//               stores the bf16 row.
// Every wait is bounded; on a time-out the CTA sets RAD_ERRW_TIMEOUT and
// unwinds, waiting (bounded) for its copies and MMAs before freeing TMEM.
#pragma once
#include <cuda.h>

#include "attn_tile.cuh"
#include "tc05.cuh"
#include "tile_configs.cuh"

namespace rad {

// D: head_dim 128 or 256.  At 256 a key tile holds 64 keys (a K or V tile is
// 32 KB, as a 128-key tile is at 128) and the query tile takes 64 KB.
template <int D_>
struct PrefillCfgD {
    static constexpr int D = D_;
    static constexpr int BM = 128;   // query rows per item
    static constexpr int BN = D == 128 ? RAD_PREFILL_BN : 64;   // keys per tile (64 or 128)
    static constexpr int NSK = RAD_PREFILL_NSK;   // K stages: a K tile is free once its QK is done
    static constexpr int NSV = RAD_PREFILL_NSV;   // V stages: a V tile is free once its PV is done
    static constexpr int CTAS = RAD_PREFILL_CTAS; // CTAs sharing an SM
    static constexpr int HB_BYTES = BN * 128;             // one 128-byte column block of a K/V tile
    static constexpr int QHB_BYTES = BM * 128;            // one 128-byte column block of the query tile
    static constexpr int TILE_BYTES = BN * D * 2;         // K or V tile
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = Q_BYTES;                    // NSK K tiles
    static constexpr int OFF_V = OFF_K + NSK * TILE_BYTES;   // NSV V tiles
    static constexpr int OFF_BARS = OFF_V + NSV * TILE_BYTES;
    // q_full, q_empty, k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV], s_full[2], p_full[2],
    // pv_done[2], o_free, final[2] (one per issuing warp)
    static constexpr int NBARS = 2 + 2 * NSK + 2 * NSV + 2 + 2 + 2 + 1 + 2;
    static constexpr int OFF_MISC = OFF_BARS + NBARS * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr int NTHREADS = 8 * 32;   // 4 softmax, QK issue, PV issue, K (+Q) and V producers
    static constexpr int W_QK = 4, W_PV = 5, W_PROD_K = 6, W_PROD_V = 7;
    // tensor memory: O in columns [0,D), S buffer b in [D + b*BN, D + (b+1)*BN);
    // P of a tile is written over its S buffer as bf16 pairs: hi in the first
    // BN/2 columns, lo in the next BN/2
    static constexpr uint32_t TMEM_COLS = D + 2 * BN <= 256 ? 256 : 512;
    static constexpr float RESCALE_LOG2 = 8.f;            // rescale O when the max grows past 2^8
    static_assert(BN == 64 || BN == 128, "key tile");
    static_assert(D == 128 || D == 256, "head_dim 128 or 256");
    static_assert(CTAS * (SMEM_BYTES + 1024) <= 233472, "shared memory budget");
    static_assert(CTAS * TMEM_COLS <= 512, "tensor memory budget");
};
using PrefillCfg = PrefillCfgD<128>;

struct PrefItem {
    int g, kvh, qt, L;
    bool seq_ok;
    int m0, m_end, kmax;
    int klo;    // first key some row of the tile sees
    int kt0;    // first key tile processed: klo / BN
    int T;      // key tiles processed: kt0 .. kt0+T-1
};

// The item a persistent CTA b of G takes in its round r.  SNAKE: rounds deal
// the heavy-first item order out in alternating directions, so the CTAs'
// key-tile totals stay close where a plain stride gives the first CTAs a
// heavier item in every round (on the 1 x 2048-row chunk over 8192 keys, the
// busiest CTA's 229 key tiles become 220, against a mean of 190); without it,
// a plain stride.  Past n_items in the last round: no item.
template <bool SNAKE>
__device__ __forceinline__ int prefill_item_of(int r, int b, int G) {
    return r * G + ((SNAKE && (r & 1)) ? G - 1 - b : b);
}

// GEN: the call has a sliding window or a scale <= 0; without either, those
// terms fold away at compile time.
template <bool GEN, int BM = PrefillCfg::BM, int BN = PrefillCfg::BN>
__device__ __forceinline__ PrefItem plan_prefill(int item, const AttnParams& p) {
    // item order: query tile rank first (later tiles see more keys, so they come
    // first), then sequence, then KV head
    PrefItem it;
    const int per_rank = p.groups * p.n_head_kv;
    const int rank = item / per_rank;
    const int rem = item - rank * per_rank;
    it.g = rem / p.n_head_kv;
    it.kvh = rem - it.g * p.n_head_kv;
    it.qt = p.n_qtiles - 1 - rank;
    it.L = __ldg(p.seq_lens + it.g);
    it.seq_ok = it.L >= p.rows && (long long)it.L <= (long long)p.pages_per_seq * p.page_size;
    it.m0 = it.qt * BM;
    it.m_end = min(p.M, it.m0 + BM);
    it.kmax = it.seq_ok ? it.L - p.rows + (it.m_end - 1) / p.ratio + 1 : 0;
    it.klo = (GEN && it.seq_ok) ? first_visible_key(it.L, p.rows, it.m0 / p.ratio, p.window) : 0;
    it.kt0 = it.klo / BN;
    it.T = (it.kmax + BN - 1) / BN - it.kt0;
    return it;
}

template <bool GEN, int D = 128>
__global__ void __launch_bounds__(PrefillCfgD<D>::NTHREADS, PrefillCfgD<D>::CTAS)
    attn_prefill_tc05_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ AttnParams p) {
    using C = PrefillCfgD<D>;
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
    const uint32_t bar_s_full = bar_v_empty + 8 * C::NSV;
    const uint32_t bar_p_full = bar_s_full + 16;
    // PV of tile t completes a phase of pv_done[t & 1].  A thread that has seen
    // S of tile t knows PV(t-2) is done (the MMA warp issues QK(t) after
    // PV(t-2), and a commit tracks every earlier operation of its thread), so
    // its waits for PV(t-1) or PV(t) are never more than one phase ahead of a
    // barrier: a single barrier would let a wait for PV(t) pass on the parity
    // of a still-pending PV(t-1).
    const uint32_t bar_pv_done = bar_p_full + 16;   // [2]
    const uint32_t bar_o_free = bar_pv_done + 16;
    const uint32_t bar_final = bar_o_free + 8;
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
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_s_full + 8 * i, 1);
            mbar_init(bar_p_full + 8 * i, 4);
        }
        mbar_init(bar_pv_done, 1);
        mbar_init(bar_pv_done + 8, 1);
        mbar_init(bar_o_free, 4);
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
    const uint32_t t_o = tmem;
    const uint32_t t_s = tmem + C::D;   // S buffer b at t_s + BN*b

    const int n_items = p.n_items;
    bool abort = false;

    if (warp == C::W_PROD_K || warp == C::W_PROD_V) {
        // ===================================================== producers: K (and the query tile), V
        const bool is_k = warp == C::W_PROD_K;
        const int NSX = is_k ? C::NSK : C::NSV;
        const uint32_t bar_full = is_k ? bar_k_full : bar_v_full;
        const uint32_t bar_empty = is_k ? bar_k_empty : bar_v_empty;
        const uint32_t ring = base + (is_k ? C::OFF_K : C::OFF_V);
        const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
        const uint64_t pol = policy_evict_last();   // K/V tiles are re-read by every query tile
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
            const PrefItem it = plan_prefill<GEN, C::BM, C::BN>(item, p);
            if (!it.seq_ok) continue;
            if (is_k) {
                if (ic >= 1 && !mbar_wait_bounded(bar_q_empty, (ic - 1) & 1u, p.wait_ns)) {
                    abort = true;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar_q_full, C::Q_BYTES);
#pragma unroll
                    for (int hb = 0; hb < C::D / 64; ++hb)
                        tma_load_4d(base + C::OFF_Q + hb * C::QHB_BYTES, &tm_q, bar_q_full, hb * 64, it.kvh * p.ratio,
                                    it.m0 / p.ratio, it.g, pol);
                }
                ++ic;
            }
            const int page_hi = (it.kmax + P - 1) / P;
            const int page_lo = GEN ? it.klo / P : 0;   // pages below hold no visible key: never read
            const int32_t* trow = p.page_table + (long long)it.g * p.pages_per_seq;
            int batch0 = -1 << 30, my_pg = 0;
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
                    if ((!GEN || pi >= page_lo) && pi < page_hi) {
                        const int pg = __ldg(trow + pi);
                        my_pg = (pg < 0 || pg >= p.num_pages) ? 0 : pg;
                    }
                }
                const uint32_t dst = ring + st * C::TILE_BYTES;
                if (lane == 0) mbar_arrive_expect_tx(bar_full + 8 * st, C::TILE_BYTES);
                for (int i = 0; i < ppt; ++i) {
                    const int pi = pstart + i;
                    const int pg = __shfl_sync(0xffffffffu, my_pg, (pi - batch0) & 31);
                    const int tok = ((!GEN || pi >= page_lo) && pi < page_hi) ? pg * P : oob_tok;
                    if (lane == 0) {
#pragma unroll
                        for (int hb = 0; hb < C::D / 64; ++hb)
                            tma_load_3d(dst + hb * C::HB_BYTES + i * P * 128, tm, bar_full + 8 * st, hb * 64, it.kvh,
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
            const PrefItem it = plan_prefill<GEN, C::BM, C::BN>(item, p);
            if (!it.seq_ok) continue;
            if (!mbar_wait_bounded(bar_q_full, ic & 1u, p.wait_ns)) {
                abort = true;
                break;
            }
            tc_fence_after();
            for (int j = 0; j < it.T; ++j) {
                const uint32_t s_ = sc + j, st = s_ % C::NSK, tcj = tc + j, b = tcj & 1u;
                // K landed, and S buffer b is free: PV(tcj - 2) read the P it held
                if (!mbar_wait_bounded(bar_k_full + 8 * st, (s_ / C::NSK) & 1u, p.wait_ns) ||
                    (tcj >= 2 && !mbar_wait_bounded(bar_pv_done + 8 * b, ((tcj - 2) >> 1) & 1u, p.wait_ns))) {
                    abort = true;
                    break;
                }
                tc_fence_after();
                const uint32_t kb = base + C::OFF_K + st * C::TILE_BYTES;
                if (lane == 0) {
#pragma unroll
                    for (int kk = 0; kk < C::D / 16; ++kk) {
                        const uint32_t qoff = (kk >> 2) * C::QHB_BYTES + (kk & 3) * 32;
                        const uint32_t koff = (kk >> 2) * C::HB_BYTES + (kk & 3) * 32;
                        tc_mma_ss(t_s + C::BN * b, umma_desc_sw128(base + C::OFF_Q + qoff, 16, 1024),
                                  umma_desc_sw128(kb + koff, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(bar_s_full + 8 * b);
                    tc_commit(bar_k_empty + 8 * st);   // the K tile is read once QK is done
                    issued = true;
                }
                __syncwarp();
            }
            // the query tile is read once the item's QKs are done
            if (lane == 0 && !abort) tc_commit(bar_q_empty);
            __syncwarp();
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
    } else if (warp == C::W_PV) {
        // ===================================================== PV issue
        constexpr uint32_t idesc_pv = umma_idesc_bf16(C::BM, C::D, 0, 1);
        uint32_t sc = 0, tc = 0, ic = 0;
        bool issued = false;
        for (int rd = 0; rd * (int)gridDim.x < n_items && !abort; ++rd) {
            const int item = prefill_item_of<true>(rd, blockIdx.x, gridDim.x);
            if (item >= n_items) break;
            const PrefItem it = plan_prefill<GEN, C::BM, C::BN>(item, p);
            if (!it.seq_ok) continue;
            // V rows to zero: slots past the sequence's end in its last page,
            // and slots of the first live page below the tile's first visible key
            const int P = p.page_size;
            const int zero_lo = it.L, zero_hi = ((it.L + P - 1) / P) * P;
            const int head_lo = (it.klo / P) * P, head_hi = it.klo;
            for (int jj = 0; jj < it.T; ++jj) {
                const uint32_t tcj = tc + jj, b = tcj & 1u;
                const uint32_t s_ = sc + jj, st = s_ % C::NSV;
                if (!mbar_wait_bounded(bar_p_full + 8 * b, (tcj >> 1) & 1u, p.wait_ns) ||
                    !mbar_wait_bounded(bar_v_full + 8 * st, (s_ / C::NSV) & 1u, p.wait_ns) ||
                    (jj == 0 && ic >= 1 && !mbar_wait_bounded(bar_o_free, (ic - 1) & 1u, p.wait_ns))) {
                    abort = true;
                    break;
                }
                const uint32_t vb = base + C::OFF_V + st * C::TILE_BYTES;
                // zero V rows of keys past the sequence's end held by this tile
                const int key0 = (it.kt0 + jj) * C::BN;
                const int z0 = max(zero_lo, key0) - key0, z1 = min(zero_hi, key0 + C::BN) - key0;
                const int h0 = max(head_lo, key0) - key0, h1 = min(head_hi, key0 + C::BN) - key0;
                const int nz = max(z1 - z0, 0), nh = GEN ? max(h1 - h0, 0) : 0;
                if (nz + nh > 0) {
                    constexpr int CPR = C::D / 8;   // 16-byte chunks of a row
                    for (int idx = lane; idx < (nz + nh) * CPR; idx += 32) {
                        const int rr = idx / CPR, c16 = idx % CPR;
                        const int row = rr < nz ? z0 + rr : h0 + (rr - nz);
                        const uint32_t a = vb + (c16 >> 3) * C::HB_BYTES + row * 128 + (((c16 & 7) ^ (row & 7)) << 4);
                        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sp = t_s + C::BN * b;
#pragma unroll
                    for (int kk = 0; kk < C::BN / 16; ++kk) {
                        const uint64_t bd = umma_desc_sw128(vb + kk * 16 * 128, C::HB_BYTES, 1024);
                        tc_mma_ts(t_o, sp + kk * 8, bd, idesc_pv, (jj > 0 || kk > 0) ? 1u : 0u);
                        tc_mma_ts(t_o, sp + C::BN / 2 + kk * 8, bd, idesc_pv, 1u);
                    }
                    tc_commit(bar_pv_done + 8 * b);
                    tc_commit(bar_v_empty + 8 * st);   // the V tile is read once PV is done
                    issued = true;
                }
                __syncwarp();
            }
            sc += it.T;
            tc += it.T;
            ++ic;
            if (misc[1]) abort = true;
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
        const float c = p.scale_log2;
        uint32_t tc = 0;
        for (int rd = 0; rd * (int)gridDim.x < n_items && !abort; ++rd) {
            const int item = prefill_item_of<true>(rd, blockIdx.x, gridDim.x);
            if (item >= n_items) break;
            const PrefItem it = plan_prefill<GEN, C::BM, C::BN>(item, p);
            const int m = it.m0 + t;
            const bool valid = m < it.m_end;
            const int r = m / p.ratio, hl = m - r * p.ratio;
            __nv_bfloat16* orow =
                p.out + (((long long)it.g * p.rows + r) * p.n_head + it.kvh * p.ratio + hl) * C::D;
            if (!it.seq_ok) {
                if (valid)
                    for (int i = 0; i < C::D / 8; ++i) reinterpret_cast<uint4*>(orow)[i] = make_uint4(0, 0, 0, 0);
                if (t == 0 && p.err_word) atomicOr(p.err_word, kErrSeqLen);
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
            bad = named_barrier_or(1, 128, bad);
            const int nk = valid ? it.L - p.rows + r + 1 : it.L;
            const int nlo = (GEN && valid) ? first_visible_key(it.L, p.rows, r, p.window) : 0;   // row sees nlo .. nk-1
            float m_run = -CUDART_INF_F, l_run = 0.f;
            for (int j = 0; j < it.T; ++j) {
                const uint32_t tcj = tc + j, b = tcj & 1u;
                // (every exit from here is taken by the whole warp: the tcgen05
                // loads and stores below are warp-collective)
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar_s_full + 8 * b, (tcj >> 1) & 1u, p.wait_ns))) {
                    abort = true;
                    break;
                }
                tc_fence_after();
                const uint32_t sc_ = t_s + C::BN * b + lane_off;
                uint32_t sv[C::BN];
                if constexpr (C::BN == 128) {
                    tmem_ld128(sc_, *reinterpret_cast<uint32_t(*)[128]>(sv));
                } else {
                    tmem_ld64(sc_, *reinterpret_cast<uint32_t(*)[64]>(sv));
                }
                // Logits are scaled by c after the max; a scale <= 0 would turn
                // that order around (and -inf * 0 into NaN), so then the tile is
                // scaled first and c taken as 1.
                float cs = c;
                if (GEN && c <= 0.f) {
#pragma unroll
                    for (int e = 0; e < C::BN; ++e) sv[e] = __float_as_uint(__uint_as_float(sv[e]) * c);
                    cs = 1.f;
                }
                const int key0 = (it.kt0 + j) * C::BN;
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
                // A row whose max grew past 2^8 rescales its O row.  tcgen05.ld/st
                // are warp-collective, so the warp rescales together when any of
                // its rows needs it; the others multiply by exactly 1.
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
                    const uint32_t tp = tcj - 1;   // the previous tile
                    const bool ok = mbar_wait_bounded(bar_pv_done + 8 * (tp & 1u), (tp >> 1) & 1u, p.wait_ns);
                    if (!__all_sync(0xffffffffu, ok)) {
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

// The launch: one CTA per SM (shared memory, TMEM), persistent over the items;
// the general build for a sliding window or a scale <= 0, else the lean one.
template <int D>
cudaError_t launch_prefill_tc05_dim(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                    const AttnParams& p, int sms, cudaStream_t st) {
    using C = PrefillCfgD<D>;
    auto kern = (p.window > 0 || p.scale_log2 <= 0.f) ? attn_prefill_tc05_kernel<true, D>
                                                      : attn_prefill_tc05_kernel<false, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    long long grid = (long long)sms * C::CTAS;
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
