// Split-call attention on the 5th-generation tensor cores (tcgen05, TMEM) for
// fp8-e4m3 KV pools with head_dim 128, the query rows on the MMA's M: the
// decode and speculative-verify call shapes ("kern manifest v7", $defs.Batch)
// of the `attn_paged` op.
//
// Work items and partial results are those of attn_tile.cuh: (split s,
// sequence g, KV head kvh, query tile of up to 32 rows -- the rows x
// n_head/n_head_kv query heads sharing the KV head), splits whose count
// depends only on the sequence length, and the same combine kernel.
//
// The item's (up to) 32 query rows are copied into the four 32-lane quarters
// of the MMA's M = 128, and a tile's 128 keys are shared out among the
// quarters: softmax warp w owns TMEM lanes 32w .. 32w+31 (lane 32w + r =
// query row r) and keys 32w .. 32w+31 of every tile.
//   S  = Q K^T   kind::f8f6f4, M 128 (four copies of the rows), N 128 keys,
//                K = head_dim: K straight from the TMA-staged e4m3 rows, each
//                query row as two exact e4m3 terms (q * 2^k = hi + lo, as in
//                prefill_fp8.cuh)
//   O += P V     kind::f16, A = P from TMEM (f16, p times the key's page V
//                scale; in lane 32w + r only keys 32w .. 32w+31 are non-zero),
//                B = V converted e4m3 -> f16 (exact), MN-major
// so quarter w of O accumulates row r over its own keys only, with its own
// running max and sum: no warp waits for another within an item, and the four
// partial results of a row are merged once per item, in warp order (a row's
// bits depend only on its sequence).  The tensor core does four times the
// rows' work, which it has time for.
//
// Warp roles (one CTA per SM, persistent):
//   warps 0-3    softmax (quarter w, thread = query row r): per tile, read its
//                32 logits, scale (row 2^-k, call scale, page K scale), mask,
//                keep the lazy running max (O quarter rescaled past 2^8,
//                warp-wide), write p x page V scale as f16 to TMEM; per item,
//                merge the four quarters' (max, sum, O) of each row and store
//                the row or the split's partial.
//   warp 4       QK: once K_j landed and PV_{j-NSP} is done (S/P buffer
//                j % NSP free), lane 0 issues QK_j (2 terms x 4 K-steps).
//   warp 5       PV: once P_j is written and V_j converted, lane 0 issues PV_j.
//   warps 6, 7   K and V producers: page ids, the per-page K/V scales (into the
//                K stage's meta block), one TMA box per page (page_size rows x
//                128 bytes of the KV head, issued by lanes 0-7); pages outside
//                the item's range load zeros.  The K producer also takes the
//                CTA's items from the counter shared by all CTAs and hands them
//                to the other warps (sched.cuh), each after issuing the previous
//                item's last tile.
//   warps 8-11   converters, one per scheduler partition: converter c turns key
//                rows 32c .. 32c+31 of every staged e4m3 V tile into f16 (a
//                quarter-rate instruction: on the MMA or softmax warps it set
//                the pace), and at each item's start splits a quarter of every
//                query row into the two e4m3 terms, written to the row's four
//                copies (overlapping the previous item's last tiles and merge);
//                each loads only its quarter of the rows, the row's scale coming
//                from the four quarters' largest exponents, exchanged through
//                shared memory.  At the start they pull the call's query rows
//                into L2: behind the K/V stream a row load from HBM at an item
//                boundary took ~3 us.
// TMEM holds O and NSP S/P buffers: the decode form and the head_dim-256 build
// two S buffers and two P buffers of their own (a quarter's lanes zero outside
// its columns for good), the head_dim-128 verify form three S buffers with P
// written over the first half of its S (zeros over the other quarters' columns
// at every tile).  PV of tile t completes a phase of pv_done[t % NSP]; a thread
// that has seen S(t) knows PV(t-NSP) is done (QK(t) waited for it), and every
// wait on pv_done is for a PV whose barrier cannot complete again before the
// waiter itself has acted (see prefill_tc05.cuh); the converters wait for
// PV(t-NV16) at every tile, in order, before they write f16 buffer t % NV16.
// Every wait is bounded; a time-out sets RAD_ERRW_TIMEOUT and the roles
// unwind.
#pragma once
#include <cuda.h>

#include "attn_tile.cuh"
#include "sched.cuh"
#include "tc05.cuh"

#ifndef RAD_SPLITTC_NSK
#define RAD_SPLITTC_NSK 4
#endif
// Stages of the form for calls with at most 8 query rows per KV head.
#ifndef RAD_SPLITTC_FEW_NSK
#define RAD_SPLITTC_FEW_NSK 4
#endif
#ifndef RAD_SPLITTC_FEW_NSV
#define RAD_SPLITTC_FEW_NSV 2
#endif
#ifndef RAD_SPLITTC_NSV
#define RAD_SPLITTC_NSV 3
#endif
// S/P buffers in TMEM (QK of tile t waits for PV of tile t - NSP) and f16 V
// buffers (the converters' rows of tile t wait for PV of tile t - NV16) of the
// head_dim-128 verify form; the decode form and the head_dim-256 build (one
// form for decode and verify calls) keep two and two.
#ifndef RAD_SPLITTC_NSP
#define RAD_SPLITTC_NSP 3
#endif
#ifndef RAD_SPLITTC_NV16
#define RAD_SPLITTC_NV16 2
#endif
// head_dim 256: the four query copies take 64 KB.
#ifndef RAD_SPLITTC256_NSK
#define RAD_SPLITTC256_NSK 3
#endif
#ifndef RAD_SPLITTC256_NSV
#define RAD_SPLITTC256_NSV 2
#endif

// The converters pull the call's query rows into L2 at the start (uniform calls).
#ifndef RAD_SPLITTC_Q_L2
#define RAD_SPLITTC_Q_L2 1
#endif

namespace rad {

// FEW: calls with at most 8 query rows per KV head (decode steps) take their
// own stage counts (same-box: four K and two V stages suit them, four and three
// the verify calls).  Nothing else changes, so a row's bits are those of the
// other form.  (Holding a decode item's 8 rows once, with a zero 8-row group
// stride in the QK descriptor as the bf16 kernel does, made this kernel's
// decode slower.)
template <bool FEW, int D_ = 128>
struct SplitTcCfg {
    static constexpr int D = D_;                    // head dim: 128 or 256
    static constexpr int BK = D == 128 ? 128 : 64;  // keys per tile (16 KB of e4m3 K rows either way)
    static constexpr int NKB = D / 128;             // 128-byte column blocks of an e4m3 row
    static constexpr int KW = BK / 4;               // keys of a tile per softmax warp
    static constexpr int QT = 32;                   // (item planner) query rows per item
    static constexpr int KS = BK;                   // (item planner) keys per stage
    static constexpr int NSK = D == 128 ? (FEW ? RAD_SPLITTC_FEW_NSK : RAD_SPLITTC_NSK)
                                        : RAD_SPLITTC256_NSK;   // K stages (with the page scales)
    static constexpr int NSV = D == 128 ? (FEW ? RAD_SPLITTC_FEW_NSV : RAD_SPLITTC_NSV)
                                        : RAD_SPLITTC256_NSV;   // V stages
    static constexpr int NSP = (FEW || D != 128) ? 2 : RAD_SPLITTC_NSP;   // S/P buffers in TMEM
    static constexpr bool P_OVER_S = NSP > 2;       // three S buffers leave no columns for P buffers of its own
    static constexpr int P_STRIDE = P_OVER_S ? BK : BK / 2;   // TMEM columns from P buffer b to b + 1
    static constexpr int NV16 = (FEW || D != 128) ? 2 : RAD_SPLITTC_NV16;   // f16 V buffers
    static constexpr int ROW = D;                   // bytes of one e4m3 key row
    static constexpr int KBLK = BK * 128;           // one 128-byte column block of a K or V tile
    static constexpr int KV_TILE = NKB * KBLK;      // e4m3 K or V rows of one tile
    static constexpr int ATOM = BK * 128;           // one 64-column block of the f16 V tile
    static constexpr int V16_BYTES = (D / 64) * ATOM;
    static constexpr int Q8_BLK = 128 * 128;        // one 128-byte column block of the four copies of the rows
    static constexpr int Q8_TERM = NKB * Q8_BLK;    // one e4m3 term of the four copies
    static constexpr int MAXPG = BK / 16;           // pages per tile
    static constexpr int META_STRIDE = 80;          // ks[8], vs[8], bad
    static constexpr int SCR_BYTES = 4 * 32 * 128;  // the merge: [warp][row][32 floats], chunks swizzled
    static constexpr int OFF_Q8 = 0;
    static constexpr int OFF_K = OFF_Q8 + 2 * Q8_TERM;
    static constexpr int OFF_V = OFF_K + NSK * KV_TILE;
    static constexpr int OFF_V16 = OFF_V + NSV * KV_TILE;
    static constexpr int OFF_SCR = OFF_V16 + NV16 * V16_BYTES;
    static constexpr int OFF_ML = OFF_SCR + SCR_BYTES;      // [2][4][32]: the quarters' row max, sum
    // [2][4][32] bytes, by item parity: the exponent field of each row's largest magnitude
    // within each quarter of its elements (the row's scale 2^k follows from their max)
    static constexpr int OFF_QEXP = OFF_ML + 2 * 4 * 32 * 4;
    static constexpr int OFF_META = OFF_QEXP + 2 * 4 * 32;
    static constexpr int OFF_BARS = OFF_META + NSK * META_STRIDE;
    // q8_full, q8_empty, k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV], s_full[NSP], p_full[NSP],
    // pv_done[NSP], v16_full[NV16], o_free, final[2], amax[2]
    static constexpr int NBARS = 2 + 2 * NSK + 2 * NSV + 3 * NSP + NV16 + 1 + 2 + 2;
    static constexpr int OFF_RING = OFF_BARS + NBARS * 8;     // the item ring (sched.cuh)
    static constexpr int OFF_MISC = OFF_RING + kRingBytesNoTaken;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;   // 1 KB alignment of the swizzled tiles
    static constexpr int NTHREADS = 12 * 32;
    static constexpr int RING_CONSUMERS = 11;                 // every warp but the K producer, which fills it
    static constexpr int W_QK = 4, W_PV = 5, W_PROD_K = 6, W_PROD_V = 7, W_CONV = 8;
    static constexpr int K_FULL_ARRIVALS = MAXPG;             // expect-tx arrive + the other page lanes' meta arrives
    static constexpr int K_EMPTY_ARRIVALS = 1 + 4;            // the QK commit + the softmax warps' scale reads
    // O [0, D), S_b [D + BK b, ...), P_b (f16 pairs) [D + NSP BK + (BK/2) b, ...) or, with three
    // S buffers, over the first BK/2 columns of S_b
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(D == 128 || D == 256, "head_dim 128 or 256");
    static_assert(D + NSP * BK + (P_OVER_S ? 0 : NSP * (BK / 2)) <= (int)TMEM_COLS, "tensor memory budget");
    // the converters wait on pv_done for PV(t - NV16) before their rows of tile t; that barrier's
    // next phase is PV(t - NV16 + NSP), which must need those rows too: NSP >= NV16
    static_assert(NSP >= NV16, "f16 V buffers");
    static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && OFF_V16 % 1024 == 0 && KV_TILE % 1024 == 0,
                  "1 KB tiles");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// One 128-code column block of key row `row` of a staged e4m3 V tile (`stage`:
// the block's [key][128 B] rows) -> the f16 MN-major tile PV reads (128-byte
// swizzle; `v16`: the block's pair of 64-column blocks, ATOM bytes apart);
// `zero` writes zeros (keys outside the item: P is 0 there, the staged row
// may hold anything).  The row's loads come before its stores, which may alias
// them as far as the compiler knows.
template <int ATOM>
__device__ __forceinline__ void convert_v_row(const uint8_t* stage, uint8_t* v16, int row, bool zero) {
    const uint32_t sw = (uint32_t)(row & 7);
    const uint8_t* src = stage + row * 128;
    uint8_t* dst = v16 + row * 128;
    uint4 in[8];
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
        in[ch] = zero ? make_uint4(0u, 0u, 0u, 0u) : *reinterpret_cast<const uint4*>(src + (((uint32_t)ch ^ sw) << 4));
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
        uint8_t* blk = dst + (ch >> 2) * ATOM;
        const uint32_t c2 = (uint32_t)((ch & 3) * 2);
        *reinterpret_cast<uint4*>(blk + ((c2 ^ sw) << 4)) = make_uint4(h0, h1, h2, h3);
        *reinterpret_cast<uint4*>(blk + (((c2 + 1) ^ sw) << 4)) = make_uint4(h4, h5, h6, h7);
    }
}

// k of a query row's scale 2^k: the largest magnitude a of the row times 2^k lies
// in [128, 256), k = 7 - floor(log2 a) kept to a normal float's range; from the
// exponent fields of the row's four quarter maxima (`qexp`: [quarter][32 rows]).
// (An all-zero row gets k = 127: every product with it is 0 whatever k is.)
__device__ __forceinline__ int row_scale_exp(const uint8_t* qexp, int r) {
    const int e = max(max((int)qexp[r], (int)qexp[32 + r]), max((int)qexp[64 + r], (int)qexp[96 + r]));
    return max(-126, min(127, 7 - (e - 127)));
}

// MODE: kModeCausal, kModeWindow or kModeTree (draft-tree rows, uniform row
// counts: bit i of a row's mask word lets it see the call's key i).
template <int MODE, bool FEW, int D = 128>
__global__ void __launch_bounds__(SplitTcCfg<FEW, D>::NTHREADS, 1)
    attn_split_tc05_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                                const __grid_constant__ AttnParams p) {
    using C = SplitTcCfg<FEW, D>;
    constexpr bool WIN = MODE == kModeWindow;
    constexpr bool TREE = MODE == kModeTree;
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
    const uint32_t bar_s_full = bar_v_empty + 8 * C::NSV;   // [NSP], by tile % NSP
    const uint32_t bar_p_full = bar_s_full + 8 * C::NSP;    // [NSP]
    const uint32_t bar_pv_done = bar_p_full + 8 * C::NSP;   // [NSP]
    const uint32_t bar_v16_full = bar_pv_done + 8 * C::NSP; // [NV16], by tile % NV16: the converters' rows
    const uint32_t bar_o_free = bar_v16_full + 8 * C::NV16;
    const uint32_t bar_final = bar_o_free + 8;              // [2]: QK warp, PV warp
    const uint32_t bar_amax = bar_final + 16;               // [2], by item parity: the converters' quarter maxima
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);  // [0] tmem, [1] abort
    const ItemRing iring(smem + C::OFF_RING, base + C::OFF_RING);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar_q8_full, 4);    // the converters
        mbar_init(bar_q8_empty, 1 + 4);   // the item's last QK commit + the softmax warps' 2^-k reads
        for (int i = 0; i < C::NSK; ++i) {
            mbar_init(bar_k_full + 8 * i, C::K_FULL_ARRIVALS);
            mbar_init(bar_k_empty + 8 * i, C::K_EMPTY_ARRIVALS);
        }
        for (int i = 0; i < C::NSV; ++i) {
            mbar_init(bar_v_full + 8 * i, 1);
            mbar_init(bar_v_empty + 8 * i, 4);   // the converters
        }
        for (int i = 0; i < C::NSP; ++i) {
            mbar_init(bar_s_full + 8 * i, 1);
            mbar_init(bar_p_full + 8 * i, 4);
            mbar_init(bar_pv_done + 8 * i, 1);
        }
        for (int i = 0; i < C::NV16; ++i) mbar_init(bar_v16_full + 8 * i, 4);
        mbar_init(bar_o_free, 4);
        mbar_init(bar_final, 1);
        mbar_init(bar_final + 8, 1);
        mbar_init(bar_amax, 4);
        mbar_init(bar_amax + 8, 4);
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
    const uint32_t t_s = tmem + C::D;                // S buffer b at t_s + BK b
    const uint32_t t_p = C::P_OVER_S ? t_s : tmem + C::D + C::NSP * C::BK;   // P buffer b at t_p + P_STRIDE b
    bool abort = false;

    // items that run the pipeline: active, a valid sequence length, keys to see
    const auto real = [&](const ItemPlan& it) { return it.active && it.seq_ok && it.n_stages > 0; };

    if (warp == C::W_PROD_K || warp == C::W_PROD_V) {
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
        ItemRing::Cursor cur;
        for (uint32_t n = 0; !abort; ++n) {
            int item = -1;
            if (is_k) {
                // the next item, fetched and handed out while the stages still
                // hold the previous item's last tiles
                bool ok = true;
                if (lane == 0) {
                    item = iring.fetch<C, WIN>(p, cur, misc + 1);
                    ok = iring.publish(n, item, p.wait_ns);
                }
                item = __shfl_sync(0xffffffffu, item, 0);
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    abort = true;
                    break;
                }
            } else if (!iring.take(n, item, p.wait_ns, false)) {
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
            float my_ks = 1.f, my_vs = 1.f;
            bool my_bad = false;
            for (int j = 0; j < it.n_stages; ++j) {
                const int pstart = (it.k0 + j * C::BK) / P;
                if (pstart + ppt > batch0 + 32) {
                    batch0 = pstart;
                    const int pi = batch0 + lane;
                    my_bad = false;
                    my_pg = 0;
                    my_ks = my_vs = 1.f;
                    if ((!WIN || pi >= page_lo) && pi < page_hi) {
                        const int pg = __ldg(trow + pi);
                        my_bad = (pg < 0 || pg >= p.num_pages);
                        my_pg = my_bad ? 0 : pg;
                        if (is_k) {
                            my_ks = __ldg(p.k_scales + my_pg);
                            my_vs = __ldg(p.v_scales + my_pg);
                        }
                    }
                }
                const uint32_t st = sc % (uint32_t)NSX, use = sc / (uint32_t)NSX;
                if (use >= 1 && !mbar_wait_bounded(bar_empty + 8 * st, (use - 1) & 1u, p.wait_ns)) {
                    abort = true;
                    break;
                }
                // lane i < ppt: page i of the tile (its id, scales and flag in one shuffle each)
                const int pi = pstart + lane;
                const int srcl = (pstart - batch0 + lane) & 31;
                const int pg = __shfl_sync(0xffffffffu, my_pg, srcl);
                const bool mine = lane < ppt;
                if (is_k) {
                    // each of lanes 0 .. MAXPG-1 releases its own meta entries with its arrive
                    const float ksl = __shfl_sync(0xffffffffu, my_ks, srcl);
                    const float vsl = __shfl_sync(0xffffffffu, my_vs, srcl);
                    const bool badl = __shfl_sync(0xffffffffu, (uint32_t)my_bad, srcl) != 0u;
                    const bool bad_any = __any_sync(0xffffffffu, mine && pi < page_hi && badl);
                    float* meta = reinterpret_cast<float*>(smem + C::OFF_META + st * C::META_STRIDE);
                    if (lane < C::MAXPG) {
                        meta[lane] = ksl;
                        meta[8 + lane] = vsl;
                    }
                    if (lane == 0) reinterpret_cast<uint32_t*>(meta)[16] = bad_any ? kErrPage : 0u;
                    if (lane > 0 && lane < C::MAXPG) mbar_arrive(bar_full + 8 * st);
                }
                // one 3-D box per page and 128-byte column block (P rows x 128 bytes of this
                // KV head, 128-byte swizzle), issued by lanes 0 .. NKB * ppt - 1: lane i
                // loads page i % ppt, block i / ppt
                if (lane == 0) mbar_arrive_expect_tx(bar_full + 8 * st, (uint32_t)C::KV_TILE);
                __syncwarp();
                if constexpr (C::NKB == 1) {
                    const bool live = mine && (!WIN || pi >= page_lo) && pi < page_hi;
                    if (mine)
                        tma_load_3d(ring + st * C::KV_TILE + (uint32_t)(lane * P * 128), tm, bar_full + 8 * st, 0,
                                    it.kvh, live ? pg * P : oob_tok, pol_kv);
                } else {
                    const int pl = lane % ppt, kb = lane / ppt;
                    const int pib = pstart + pl;
                    const int pgb = __shfl_sync(0xffffffffu, my_pg, (pstart - batch0 + pl) & 31);
                    const bool boxl = lane < C::NKB * ppt;
                    const bool liveb = boxl && (!WIN || pib >= page_lo) && pib < page_hi;
                    if (boxl)
                        tma_load_3d(ring + st * C::KV_TILE + (uint32_t)(kb * C::KBLK + pl * P * 128), tm,
                                    bar_full + 8 * st, kb * 128, it.kvh, liveb ? pgb * P : oob_tok, pol_kv);
                }
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
    } else if (warp >= C::W_CONV) {
        // ===================================================== converters
        const int cv = warp - C::W_CONV;   // (row, block) pairs 32cv .. 32cv+31 of every V tile; query-row quarter cv
        if (RAD_SPLITTC_Q_L2 && !p.cu_seqlens) {
            // The call's query rows (a few MB) into L2, a slice per CTA: they are read again
            // at every item boundary, where a load from HBM behind the K/V stream took ~3 us
            const size_t qbytes = (size_t)p.groups * p.rows * p.n_head * C::D * 2;
            const size_t per = ((qbytes + gridDim.x - 1) / gridDim.x + 127) & ~(size_t)127;
            const size_t lo = per * blockIdx.x, hi = min(qbytes, lo + per);
            for (size_t off = lo + 128 * (size_t)(cv * 32 + lane); off < hi; off += 128 * 128)
                prefetch_l2(reinterpret_cast<const char*>(p.q) + off);
        }
        uint32_t tc = 0, ic = 0;
        for (uint32_t n = 0; !abort; ++n) {
            int item;
            if (!iring.take(n, item, p.wait_ns, false)) {
                abort = true;
                break;
            }
            if (item < 0) break;
            const ItemPlan it = plan_item<C, WIN>(item, p);
            if (!real(it)) continue;
            // ---- the item's query rows as two e4m3 terms (this converter a quarter of
            // every row, into all four copies), once the previous item's QKs are done and
            // the softmax warps have read its 2^-k; each row's scale is found before that
            // wait
            const auto q8_free = [&]() {
                return ic == 0 || __all_sync(0xffffffffu, mbar_wait_bounded(bar_q8_empty, (ic - 1) & 1u, p.wait_ns));
            };
            {
                const int r = lane;
                const int nrows = it.m_end - it.m0;
                const bool valid = r < nrows;
                const int m = it.m0 + r;
                const int tok = m / p.ratio, hl = m - tok * p.ratio;
                // this converter's quarter of the row (16-element chunks CH cv .. CH cv + CH-1),
                // its largest magnitude shared with the other converters: the row's scale
                constexpr int CH = C::D / 64;
                const uint4* qrow =
                    reinterpret_cast<const uint4*>(p.q + ((it.qrow0 + tok) * p.n_head + it.kvh * p.ratio + hl) * C::D);
                uint4 qq[2 * CH];
#pragma unroll
                for (int i = 0; i < 2 * CH; ++i)
                    qq[i] = valid ? __ldg(qrow + 2 * CH * cv + i) : make_uint4(0u, 0u, 0u, 0u);
                float amq = 0.f;
#pragma unroll
                for (int i = 0; i < 2 * CH; ++i) {
                    const uint32_t x[4] = {qq[i].x, qq[i].y, qq[i].z, qq[i].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) amq = fmaxf(amq, fmaxf(fabsf(bf16_lo(x[e])), fabsf(bf16_hi(x[e]))));
                }
                uint8_t* const qexp = smem + C::OFF_QEXP + (ic & 1u) * 128;
                qexp[cv * 32 + r] = (uint8_t)((__float_as_uint(amq) >> 23) & 0xFFu);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_amax + 8 * (ic & 1u));
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar_amax + 8 * (ic & 1u), (ic >> 1) & 1u, p.wait_ns))) {
                    abort = true;
                    break;
                }
                const int kx = row_scale_exp(qexp, r);
                const float sq = __uint_as_float((uint32_t)(kx + 127) << 23);
                if (!q8_free()) {
                    abort = true;
                    break;
                }
                // the quarter as the two terms, written to all four copies of the row
#pragma unroll
                for (int ii = 0; ii < CH; ++ii) {
                    const int i = CH * cv + ii;   // chunk i % 8 of column block i / 8 of each term's row
                    uint32_t wt[2][4];
                    const uint4 qa = qq[2 * ii], qb = qq[2 * ii + 1];
                    const uint32_t words[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t x0 = words[2 * e], x1 = words[2 * e + 1];
                        const float v0 = bf16_lo(x0) * sq, v1 = bf16_hi(x0) * sq;
                        const float v2 = bf16_lo(x1) * sq, v3 = bf16_hi(x1) * sq;
                        const uint32_t h01 = f32x2_to_e4m3x2(v0, v1), h23 = f32x2_to_e4m3x2(v2, v3);
                        const float2 a01 = e4m3x2_to_f32x2(h01), a23 = e4m3x2_to_f32x2(h23);
                        const uint32_t l01 = f32x2_to_e4m3x2(v0 - a01.x, v1 - a01.y);
                        const uint32_t l23 = f32x2_to_e4m3x2(v2 - a23.x, v3 - a23.y);
                        wt[0][e] = h01 | (h23 << 16);
                        wt[1][e] = l01 | (l23 << 16);
                    }
                    // row 32 copy + r of the M = 128 operand; (32 copy + r) & 7 = r & 7
                    uint8_t* q8 = smem + C::OFF_Q8 + (i >> 3) * C::Q8_BLK + r * 128 +
                                  ((((uint32_t)i & 7u) ^ (uint32_t)(r & 7)) << 4);
#pragma unroll
                    for (int copy = 0; copy < 4; ++copy)
#pragma unroll
                        for (int term = 0; term < 2; ++term)
                            *reinterpret_cast<uint4*>(q8 + copy * 32 * 128 + term * C::Q8_TERM) =
                                make_uint4(wt[term][0], wt[term][1], wt[term][2], wt[term][3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_q8_full);   // also releases the rows' 2^-k
            }
            // ---- this converter's rows of every V tile of the item
            for (int j = 0; j < it.n_stages; ++j) {
                const uint32_t tcj = tc + j, b = tcj % C::NV16, sv = tcj % C::NSV;
                bool ok = mbar_wait_bounded(bar_v_full + 8 * sv, (tcj / C::NSV) & 1u, p.wait_ns);
                // f16 buffer b was last read by PV(tcj - NV16) (waited at every tile, in order; the
                // barrier's next phase needs PV(tcj - NV16 + NSP), after this warp's rows of tile tcj)
                if (ok && tcj >= (uint32_t)C::NV16)
                    ok = mbar_wait_bounded(bar_pv_done + 8 * ((tcj - C::NV16) % C::NSP), ((tcj - C::NV16) / C::NSP) & 1u,
                                           p.wait_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    abort = true;
                    break;
                }
                // (row, 128-code block) pairs 32cv .. 32cv+31 of the tile's BK x NKB
                const int pr = 32 * cv + lane;
                const int row = C::NKB == 1 ? pr : pr % C::BK, kb = C::NKB == 1 ? 0 : pr / C::BK;
                const int key = it.k0 + j * C::BK + row;
                convert_v_row<C::ATOM>(smem + C::OFF_V + sv * C::KV_TILE + kb * C::KBLK,
                                       smem + C::OFF_V16 + b * C::V16_BYTES + 2 * kb * C::ATOM, row,
                                       key < it.klo || key >= it.k1);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar_v16_full + 8 * b);
                    mbar_arrive(bar_v_empty + 8 * sv);
                }
            }
            tc += it.n_stages;
            ++ic;
            if (__any_sync(0xffffffffu, misc[1] != 0)) abort = true;
        }
    } else if (warp == C::W_QK) {
        // ===================================================== QK issue
        constexpr uint32_t idesc_qk = umma_idesc_e4m3(128, C::BK);
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
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar_q8_full, ic & 1u, p.wait_ns))) {
                abort = true;
                break;
            }
            tc_fence_after();
            for (int j = 0; j < T; ++j) {
                const uint32_t tcj = tc + j, b = tcj % C::NSP, sk = tcj % C::NSK;
                // K landed, and S/P buffer b is free: PV(tcj - NSP) is done
                bool ok = mbar_wait_bounded(bar_k_full + 8 * sk, (tcj / C::NSK) & 1u, p.wait_ns);
                if (ok && tcj >= (uint32_t)C::NSP)
                    ok = mbar_wait_bounded(bar_pv_done + 8 * b, (tcj / C::NSP - 1) & 1u, p.wait_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    abort = true;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t kb = base + C::OFF_K + sk * C::KV_TILE;
#pragma unroll
                    for (int term = 0; term < 2; ++term)
#pragma unroll
                        for (int kk = 0; kk < C::D / 32; ++kk)
                            tc_mma_ss_f8(t_s + C::BK * b,
                                         umma_desc_sw128(base + C::OFF_Q8 + term * C::Q8_TERM + (kk >> 2) * C::Q8_BLK +
                                                             (kk & 3) * 32,
                                                         16, 1024),
                                         umma_desc_sw128(kb + (kk >> 2) * C::KBLK + (kk & 3) * 32, 16, 1024), idesc_qk,
                                         (term > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(bar_s_full + 8 * b);
                    tc_commit(bar_k_empty + 8 * sk);
                    if (j == T - 1) tc_commit(bar_q8_empty);   // the item's query terms are read
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
        constexpr uint32_t idesc_pv = umma_idesc_f16(128, C::D, 0, 1);
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
                const uint32_t tcj = tc + j, b = tcj % C::NSP, b16 = tcj % C::NV16;
                // P_j written, V_j converted, and at an item's first tile the previous item's O read out
                bool ok = mbar_wait_bounded(bar_p_full + 8 * b, (tcj / C::NSP) & 1u, p.wait_ns);
                if (ok) ok = mbar_wait_bounded(bar_v16_full + 8 * b16, (tcj / C::NV16) & 1u, p.wait_ns);
                if (ok && j == 0 && ic >= 1) ok = mbar_wait_bounded(bar_o_free, (ic - 1) & 1u, p.wait_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    abort = true;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t vb = base + C::OFF_V16 + b16 * C::V16_BYTES;
#pragma unroll
                    for (int kk = 0; kk < C::BK / 16; ++kk)
                        tc_mma_ts(t_o, t_p + C::P_STRIDE * b + kk * 8, umma_desc_sw128(vb + kk * 16 * 128, C::ATOM, 1024),
                                  idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(bar_pv_done + 8 * b);
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
    } else {
        // ===================================================== softmax (warps 0-3)
        const int w = warp;                                     // quarter: keys 32w .. 32w+31 of a tile
        const int r = lane;                                     // query row r of the item
        const uint32_t lane_off = (uint32_t)(w * 32) << 16;     // this warp's TMEM lanes
        const int t = threadIdx.x;                              // 0 .. 127
        float* const ml = reinterpret_cast<float*>(smem + C::OFF_ML);
        uint8_t* const scr = smem + C::OFF_SCR;
        if constexpr (!C::P_OVER_S) {
            // this quarter's lanes of the P buffers hold zeros outside its own columns for good
            uint32_t z[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) z[e] = 0u;
#pragma unroll
            for (int q = 0; q < C::NSP * C::BK / 64; ++q) tmem_st32(t_p + lane_off + 32 * q, z);
            tmem_wait_st();
        }
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
            // the rows' 2^-k, from the converters' split of this item's query rows
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar_q8_full, ic & 1u, p.wait_ns))) abort = true;
            if (named_barrier_or(1, 128, abort)) {   // all four warps leave together
                abort = true;
                break;
            }
            const float isq = __uint_as_float((uint32_t)(127 - row_scale_exp(smem + C::OFF_QEXP + (ic & 1u) * 128, r)) << 23);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_q8_empty);
            // keys row r sees: [nlo, nk) (tree rows: every cached key, of the call's
            // keys only their paths), within the item's [klo, k1)
            const int nk = valid ? min(it.L - it.qlen + tok + 1, it.k1) : 0;
            const int nlo = max(it.klo, (WIN && valid) ? first_visible_key(it.L, it.qlen, tok, p.window) : 0);
            const int n_full = TREE ? it.L - it.qlen : nk;   // keys below: no tree bit to test
            const float crow = p.scale_log2 * isq;
            const int lp = (p.page_size == 16) ? 4 : 5;
            float m_run = -CUDART_INF_F, l_run = 0.f;
            for (int j = 0; j < T; ++j) {
                const uint32_t tcj = tc + j, b = tcj % C::NSP, sk = tcj % C::NSK;
                // S_j landed, and the K stage's scales are visible (QK waited for its K-full
                // phase); the stage is released after the reads
                bool ok = mbar_wait_bounded(bar_s_full + 8 * b, (tcj / C::NSP) & 1u, p.wait_ns);
                if (ok) ok = mbar_wait_bounded(bar_k_full + 8 * sk, (tcj / C::NSK) & 1u, p.wait_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    abort = true;
                    break;
                }
                const float* meta = reinterpret_cast<const float*>(smem + C::OFF_META + sk * C::META_STRIDE);
                // this quarter's keys KW w .. KW w + KW-1, in runs of 16 within one page
                constexpr int KW = C::KW;
                float kf[KW / 16], vf[KW / 16];
#pragma unroll
                for (int g = 0; g < KW / 16; ++g) {
                    kf[g] = crow * meta[(KW * w + 16 * g) >> lp];
                    vf[g] = meta[8 + ((KW * w + 16 * g) >> lp)];
                }
                bad |= reinterpret_cast<const uint32_t*>(meta)[16];
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_k_empty + 8 * sk);
                tc_fence_after();
                uint32_t sv[KW];
                tmem_ld_cols<KW>(t_s + C::BK * b + KW * w + lane_off, sv);
#pragma unroll
                for (int e = 0; e < KW; ++e) sv[e] = __float_as_uint(__uint_as_float(sv[e]) * kf[e / 16]);
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
                    const bool okw =
                        j == 0 || mbar_wait_bounded(bar_pv_done + 8 * (tp % C::NSP), (tp / C::NSP) & 1u, p.wait_ns);
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
                uint32_t pk[KW / 2];
#pragma unroll
                for (int e = 0; e < KW / 2; ++e) {
                    const float p0 = exp2f(X(2 * e) - m_use), p1 = exp2f(X(2 * e + 1) - m_use);
                    ps8[e & 7] += p0 + p1;
                    pk[e] = pack_f16x2(p0 * vf[e / 8], p1 * vf[e / 8]);
                }
#undef X
                // this quarter's KW/2 columns of P buffer b; over S, zeros over the other
                // quarters' columns too (in these lanes PV must see only this quarter's keys,
                // and the S values there are not this warp's)
                const uint32_t pb = t_p + C::P_STRIDE * b + lane_off;
                if constexpr (C::P_OVER_S) {
                    uint32_t zk[KW / 2];
#pragma unroll
                    for (int e = 0; e < KW / 2; ++e) zk[e] = 0u;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (q == w) tmem_st_cols<KW / 2>(pb + (KW / 2) * q, pk);
                        else tmem_st_cols<KW / 2>(pb + (KW / 2) * q, zk);
                    }
                } else {
                    tmem_st_cols<KW / 2>(pb + (KW / 2) * w, pk);
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
            // ---- epilogue: the four quarters' (max, sum, O) of row r, merged in warp order
            const uint32_t tcl = tc + T - 1;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar_pv_done + 8 * (tcl % C::NSP), (tcl / C::NSP) & 1u, p.wait_ns)))
                abort = true;
            tc_fence_after();
            if (named_barrier_or(1, 128, abort)) {   // all four warps leave together
                abort = true;
                break;
            }
            ml[w * 32 + r] = m_run;
            ml[128 + w * 32 + r] = l_run;
            const bool page_bad = named_barrier_or(1, 128, (bad & kErrPage) != 0);
            const bool mask_bad = TREE && named_barrier_or(1, 128, (bad & kErrMask) != 0);
            const bool item_bad = page_bad || mask_bad;
            const uint32_t bad_bits = (page_bad ? kErrPage : 0u) | (mask_bad ? kErrMask : 0u);
            float mq[4], M = -CUDART_INF_F;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                mq[q] = ml[q * 32 + r];
                M = fmaxf(M, mq[q]);
            }
            const float mu = (M == -CUDART_INF_F) ? 0.f : M;
            float L = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) L += exp2f(mq[q] - mu) * ml[128 + q * 32 + r];
            const float f_me = exp2f(m_run - mu);
            const bool final_write = it.n_splits - it.s_first == 1;
            const float inv = L == 0.f ? 0.f : 1.f / L;
            float* pacc = p.part_acc + slot_idx * p.qtv * C::D;
            for (int c = 0; c < C::D / 32; ++c) {
                // quarter w's scaled O of row r, columns 32c .. 32c+31, 16-byte chunks
                // swizzled by the row
                uint32_t ov[32];
                tmem_ld32(t_o + lane_off + 32 * c, ov);
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
                    if (lane == 0) mbar_arrive(bar_o_free);
                }
                named_barrier_sync(1, 128);
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
                named_barrier_sync(1, 128);   // the scratch is free for the next chunk
            }
            if (final_write) {
                if (item_bad && t == 0 && p.err_word) atomicOr(p.err_word, bad_bits);
            } else {
                float* pml = p.part_ml + slot_idx * p.qtv * 2;
                if (w == 0 && valid) __stcg(reinterpret_cast<float2*>(pml) + r, make_float2(L == 0.f ? -CUDART_INF_F : M, L));
                if (t == 0) __stcg(p.part_flag + slot_idx, bad_bits);
            }
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

// Launch of one form: one CTA per SM (shared memory, all of TMEM), persistent
// over the items; calls with a sliding window run the window build, calls
// with tree masks the tree build, others the causal one.
template <bool FEW, int D>
cudaError_t launch_split_tc05_form(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, int sms,
                                   cudaStream_t st) {
    using C = SplitTcCfg<FEW, D>;
    auto kern = p.window > 0  ? attn_split_tc05_kernel<kModeWindow, FEW, D>
                : p.tree_mask ? attn_split_tc05_kernel<kModeTree, FEW, D>
                              : attn_split_tc05_kernel<kModeCausal, FEW, D>;
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
