// Paged-KV attention tile kernel (sm_103a).
//
// One CTA is persistent and walks a list of work items.  A work item is
// (split s, sequence g, KV head kvh, query tile qt): the query rows of one KV
// head -- the `rows` rows times the n_head/n_head_kv query heads that share it
// ("Radiance architecture plugins", section "Declare: the metadata": n_head over
// n_head_kv) -- against one contiguous range of the sequence's keys.
//
// Warp roles.  The last two warps are producers: they read page ids from the
// page table ("kern manifest v7", $defs.Domain: `stride` token slots per
// entry) and copy the item's K rows (one warp) and V rows (the other) into a
// ring of shared-memory stages with 16-byte cp.async copies, straight into a
// 128-byte-swizzled layout; the first producer also bulk-copies the item's
// query rows.  (Each page row of one KV head is only head_dim*elem bytes, and
// tensor-map boxes that small are issue-bound well below HBM speed on this
// part; 16-byte copies of the same rows are not.)  The other warps consume
// stages:
//
//   S^T[key][q] = K[key][:] . Q[q][:]          mma.m16n8k16, keys as M, query
//                                              rows as N (8 per n-tile)
//   online softmax over keys, per query row    fp32, exp2, warp shuffles
//   O^T[d][q]  += V^T[d][key] P^T[key][q]      mma.m16n8k16, P^T re-laid out
//                                              from the S^T accumulator with
//                                              movmatrix
//
// Keys as the M dimension keeps a decode step (a handful of query rows per KV
// head) at no worse than half-used n-tiles.
//
// Splits.  With split_len > 0 a sequence's keys are cut into ceil(L/split_len)
// ranges whose count and boundaries depend only on L.  A sequence with one
// range writes its output rows directly; otherwise each range writes a partial
// (running max, sum, unnormalised accumulator) to the workspace and the
// combine kernel merges the partials in split order 0..n-1.  Every output row
// is therefore the same function of its own sequence whatever else is in the
// call ("Adding a model", step 4: verified rows must equal decode rows bit
// for bit).
//
// bf16 pools: the softmax weights P enter the PV product as two bf16 terms,
// hi = bf16(p) and lo = bf16(p - hi), so the product sees p to ~2^-17; a single
// bf16 P (2^-9) would put errors of ~1e-3 on short-context rows.
//
// fp8 pools (e4m3 codes, one fp32 scale per page and pool): codes are turned
// into f16 pairs with cvt.rn.f16x2.e4m3x2 (exact), Q is rounded bf16->f16
// (exact inside the f16 range; elements past it raise RAD_ERRW_QRANGE), the
// page's K scale multiplies the logits and its V scale multiplies P before
// P is rounded to f16 for the PV product.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include <cstdint>

#include "ptx.cuh"

namespace rad {

// Device error bits (mirror of RAD_ERRW_* in include/rad_attn.h).
constexpr uint32_t kErrSeqLen = 1u;
constexpr uint32_t kErrPage = 2u;
constexpr uint32_t kErrQRange = 4u;
constexpr uint32_t kErrTimeout = 8u;
constexpr uint32_t kErrCuSeq = 16u;
constexpr uint32_t kErrMask = 32u;

// Row-visibility modes of the tile kernel: causal rows, causal rows with a
// sliding window, or draft-tree rows (a per-row mask over the call's keys).
constexpr int kModeCausal = 0;
constexpr int kModeWindow = 1;
constexpr int kModeTree = 2;

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // default limit of each bounded wait: 2 s

// Test-only fault injection (AttnParams::fault): the K producer of the tcgen05
// bf16 split kernel in CTA 0 leaves its first tile's copy unissued, so the
// waits on that tile run out and the kernel unwinds with kErrTimeout.
constexpr int kFaultNone = 0;
constexpr int kFaultSkipFirstKTile = 1;

// The running max of a row moves (and its accumulator is rescaled) only when
// new logits exceed it by more than this many powers of two.
#ifndef RAD_LAZY_RESCALE_LOG2
#define RAD_LAZY_RESCALE_LOG2 8.f
#endif
constexpr float kLazyRescaleLog2 = RAD_LAZY_RESCALE_LOG2;

// The most sequences of a call whose split items are sorted heaviest first
// (sched.cuh: their lengths are staged in shared memory).
constexpr int kOrderMaxGroups = 8192;

struct AttnParams {
    const __nv_bfloat16* q;
    const uint8_t* k_pool;
    const uint8_t* v_pool;
    const int32_t* page_table;
    const int32_t* seq_lens;
    const float* k_scales;
    const float* v_scales;
    __nv_bfloat16* out;
    float* part_acc;       // [slots][qtv][D]
    float* part_ml;        // [slots][qtv][2]  (max in log2 units, sum)
    uint32_t* part_flag;   // [slots]         page-id error seen by the split
    uint32_t* err_word;    // optional
    const int32_t* cu_seqlens;   // [groups + 1] absolute q row offsets, or null: `rows` rows per group
    const uint32_t* tree_mask;   // one word per q row (bit i: sees the call's key i), or null: causal
    // Ragged calls (cu_seqlens given): (sequence, query tile) of each of the
    // call's query tiles in sequence order, (-1, 0) past the last; n_qtiles
    // is then the bound on the call's tiles, not a per-sequence count.
    const int2* tile_map;
    int groups, rows, n_head, n_head_kv, ratio, page_size, pages_per_seq, num_pages;   // rows: max per group
    int M;                 // rows * ratio: query rows per KV head (the most of any group)
    int n_qtiles;          // ceil(M / QT) per sequence; ragged calls: tiles of the whole call (a bound)
    int qtv;               // query rows stored per partial slot: min(M, QT)
    int qt_rows;           // QT of the split kernel's tile
    int max_splits;        // 1 without splitting
    int split_len;         // keys per split; 0 = one range over the whole context
    int n_items;           // max_splits * groups * n_head_kv * n_qtiles
    int window;            // > 0: each row sees only its last `window` keys; 0: no window
    float scale_log2;      // scale * log2(e)
    uint64_t wait_ns;      // limit of each bounded wait (kWaitLimitNs unless a test lowers it)
    int fault;             // kFaultNone, or a test's injected fault
    uint32_t* sched_ctr;   // tcgen05 split kernels: the shared item counter (zero at launch), or null
    int32_t* item_order;   // tcgen05 split kernels: (split, sequence) pairs heaviest first (sched.cuh), or null
                           // (uniform calls of at most kOrderMaxGroups sequences)
};

// First key that query row r of a call with `rows` rows over a sequence of
// length L may see: 0, or with a sliding window W (a RAD_KV_WINDOW group,
// "Radiance architecture plugins", section "Declare: buffers and KV groups")
// the first of the row's last W keys.
__device__ __forceinline__ int first_visible_key(int L, int rows, int r, int window) {
    const int n = L - rows + r + 1;   // keys 0 .. n-1 are causal for row r
    return (window > 0 && n > window) ? n - window : 0;
}

// Rows of group g and the q/output row of its row 0.  Without cu_seqlens every
// group has `rows` rows at g*rows; with it ("kern manifest v7", $defs.Fill
// `cu_seqlens`: exclusive prefix sums of rows per sequence, absolute offsets)
// group g has cu[g+1] - cu[g].  Returns false for entries that name no valid
// row range (a negative offset or count, or more rows than the call's most).
struct GroupRows {
    long long row0;
    int n;
};
__device__ __forceinline__ bool group_rows(const AttnParams& p, int g, GroupRows& gr) {
    if (!p.cu_seqlens) {
        gr.row0 = (long long)g * p.rows;
        gr.n = p.rows;
        return true;
    }
    const int a = __ldg(p.cu_seqlens + g), b = __ldg(p.cu_seqlens + g + 1);
    gr.row0 = a;
    gr.n = b - a;
    return a >= 0 && b >= a && b - a <= p.rows;
}

template <int D_, bool FP8_, int WQ_, int NQW_, int WK_, int KS_, int NS_, int MINB_ = 1>
struct TileCfg {
    static constexpr int D = D_;
    static constexpr bool FP8 = FP8_;
    static constexpr int WQ = WQ_;      // consumer warps along query rows
    static constexpr int NQW = NQW_;    // 8-row query n-tiles per warp
    static constexpr int WK = WK_;      // consumer warps along keys
    static constexpr int KS = KS_;      // keys per stage
    static constexpr int NS = NS_;      // stages
    static constexpr int MINB = MINB_;  // CTAs meant to share an SM
    static constexpr int E = FP8 ? 1 : 2;
    static constexpr int QT = WQ * NQW * 8;
    static constexpr int NCW = WQ * WK;
    static constexpr int NCT = NCW * 32;
    static constexpr int NTHREADS = NCT + 64;   // + K and V producer warps
    static constexpr int FULL_ARRIVALS = 64 + 1; // 64 async lane arrivals + stage meta
    static constexpr int SUBS = KS / 16;
    static constexpr int ROW_BYTES = D * E;
    static constexpr int TILE_BYTES = KS * ROW_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int MAX_PAGES_STAGE = KS / 16;
    // A page of one KV head lands as D/BOXW blocks of [page_size][128 bytes]
    // (one 128-byte column block each), so 8 consecutive keys hit 8 different
    // swizzle phases.
    static constexpr int BOXW = 128 / E;          // elements per 128-byte row
    static constexpr int NBOX = D / BOXW;
    static constexpr int Q_SLOT_BYTES = QT * D * 2;
    static constexpr int OFF_Q = NS * STAGE_BYTES;
    static constexpr int OFF_MERGE = OFF_Q + 2 * Q_SLOT_BYTES;
    // merge: one warp state [query column][head dim] (each of two key warps
    // publishes half of its own), every key warp's (max, sum) per query
    // column, and the merged (max, sum)
    static constexpr int MSTRIDE = D + 4;   // floats per merge row (bank spread)
    static constexpr int MERGE_BYTES = QT * MSTRIDE * 4;
    static constexpr int ML_BYTES = WK > 1 ? WQ * WK * NQW * 4 * 16 : 0;
    static constexpr int OFF_ML = OFF_MERGE + MERGE_BYTES;
    static constexpr int OFF_MLF = OFF_ML + ML_BYTES;
    static constexpr int OFF_META = OFF_MLF + QT * 8;
    static constexpr int META_STRIDE = 64;  // ks[4], vs[4], bad, pad
    static constexpr int OFF_BARS = OFF_META + NS * META_STRIDE;
    static constexpr int OFF_MISC = OFF_BARS + (2 * NS + 4) * 8;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    // The swizzle is applied to offsets in software (not by address bits), so
    // 128-byte alignment of the base is all the copies and ldmatrix need.
    static constexpr int SMEM_BYTES = SMEM_USED + 128;    // base alignment slack
    static_assert(KS % 32 == 0, "a stage holds whole pages of either page size (16 or 32 slots)");
    static_assert(SUBS % WK == 0, "stage keys must split evenly over key warps");
    static_assert(WK == 1 || WK == 2, "the merge pairs at most two key warps");
    static_assert(MAX_PAGES_STAGE <= 4, "stage meta holds 4 pages");
    static_assert(D % 32 == 0, "head_dim multiple of 32");
    static_assert(SMEM_BYTES * MINB <= 233472 - 1024 * MINB, "shared memory budget");
};

// Byte offset, inside a stage tile, of element d of key `key` (both relative to
// the stage); P is the page size (16 or 32), lp = log2(P).
template <class C>
__device__ __forceinline__ uint32_t kv_off(int key, int d, int lp) {
    const int P = 1 << lp;
    return (uint32_t)(((key >> lp) * P * C::ROW_BYTES) + (d / C::BOXW) * P * 128 + (key & (P - 1)) * 128 +
                      (d % C::BOXW) * C::E);
}

struct ItemPlan {
    int s, g, kvh, qt;
    long long gq;      // partial-slot group of the item: (sequence, KV head, query tile)
    int L;
    long long qrow0;   // q/output row of the group's row 0
    int qlen;          // the group's rows
    bool cu_ok;        // the group's cu_seqlens entries are valid
    bool seq_ok;
    bool active;
    int n_splits;      // splits of the sequence, ceil(L / split_len)
    int s_first;       // first split holding a key some row of the tile sees
    int klo;           // first key some row of the tile sees
    int kmax;          // keys 0 .. kmax-1 hold every key some row of the tile sees
    int k0, k1;        // key range of the item (k0 a multiple of KS)
    int m0, m_end;     // query rows [m0, m_end) of the KV head
    int n_stages;
};

// WIN: the call has a sliding window (p.window > 0); without one, every
// window term folds away at compile time.
// Sequence index of a work item (items are split-major).
__device__ __forceinline__ int item_group(int item, const AttnParams& p) {
    const int per_split = p.groups * p.n_head_kv * p.n_qtiles;
    return (item % per_split) / (p.n_head_kv * p.n_qtiles);
}

// The plan of a work item given its sequence length (L < 0: load it).
template <class C, bool WIN>
__device__ __forceinline__ ItemPlan plan_item(int item, const AttnParams& p, int L_known = -1) {
    ItemPlan it;
    if (p.tile_map) {
        // ragged: items are (split, tile of the call, KV head)
        const int per_split = p.n_qtiles * p.n_head_kv;
        it.s = item / per_split;
        const int rem = item - it.s * per_split;
        const int t = rem / p.n_head_kv;
        it.kvh = rem - t * p.n_head_kv;
        it.gq = (long long)t * p.n_head_kv + it.kvh;
        const int2 gm = __ldg(p.tile_map + t);
        if (gm.x < 0) {   // past the call's last tile
            it.g = it.qt = it.L = it.qlen = 0;
            it.qrow0 = 0;
            it.active = it.seq_ok = it.cu_ok = false;
            it.m0 = it.m_end = it.k0 = it.k1 = it.klo = it.kmax = 0;
            it.n_stages = it.s_first = 0;
            it.n_splits = 1;
            return it;
        }
        it.g = gm.x;
        it.qt = gm.y;
    } else {
        const int per_split = p.groups * p.n_head_kv * p.n_qtiles;
        it.s = item / per_split;
        const int rem = item - it.s * per_split;
        const int per_g = p.n_head_kv * p.n_qtiles;
        it.g = rem / per_g;
        const int rem2 = rem - it.g * per_g;
        it.kvh = rem2 / p.n_qtiles;
        it.qt = rem2 - it.kvh * p.n_qtiles;
        if (p.split_len == 0) it.qt = p.n_qtiles - 1 - it.qt;   // causal: later tiles see more keys
        it.gq = ((long long)it.g * p.n_head_kv + it.kvh) * p.n_qtiles + it.qt;
    }
    GroupRows gr;
    it.cu_ok = group_rows(p, it.g, gr);
    it.qrow0 = gr.row0;
    it.qlen = gr.n;
    it.L = L_known >= 0 ? L_known : __ldg(p.seq_lens + it.g);
    it.seq_ok = it.cu_ok && it.L >= it.qlen && (long long)it.L <= (long long)p.pages_per_seq * p.page_size;
    it.m0 = it.qt * C::QT;
    it.m_end = it.cu_ok ? min(it.qlen * p.ratio, it.m0 + C::QT) : it.m0;
    it.k0 = it.k1 = 0;
    it.n_stages = 0;
    it.n_splits = 1;
    it.s_first = 0;
    it.klo = it.kmax = 0;
    if (!it.cu_ok) {
        // malformed offsets: one item of the group raises the error bit, no row is written
        it.active = (it.s == 0 && it.kvh == 0 && it.qt == 0);
        return it;
    }
    if (it.m_end <= it.m0) {   // no row of the group in this query tile
        it.active = false;
        return it;
    }
    if (!it.seq_ok) {
        it.active = (it.s == 0);
        return it;
    }
    const int r_last = (it.m_end - 1) / p.ratio;
    it.kmax = it.L - it.qlen + r_last + 1;
    it.klo = WIN ? first_visible_key(it.L, it.qlen, it.m0 / p.ratio, p.window) : 0;
    // Stages start on absolute multiples of KS (split_len is one too), so a
    // key falls in the same sub-tile, and goes to the same key warp, whatever
    // the tile's first visible key: rows of different calls at one position
    // see the same schedule.
    const int klo_stage = (it.klo / C::KS) * C::KS;
    if (p.split_len > 0) {
        it.n_splits = (it.L + p.split_len - 1) / p.split_len;
        it.s_first = it.klo / p.split_len;
        it.active = it.s >= it.s_first && it.s < it.n_splits;
        it.k0 = max(it.s * p.split_len, klo_stage);
        it.k1 = min(it.s * p.split_len + p.split_len, it.kmax);
    } else {
        it.active = (it.s == 0);
        it.k0 = klo_stage;
        it.k1 = it.kmax;
    }
    if (it.k1 < it.k0) it.k1 = it.k0;
    it.n_stages = (it.k1 - it.k0 + C::KS - 1) / C::KS;
    return it;
}

// Column (query row index within the KV head) held by this lane.
template <class C>
__device__ __forceinline__ int lane_col(int wq, int j, int t4, int c) {
    return (wq * C::NQW + j) * 8 + 2 * t4 + c;
}

// Head-dim index of accumulator row `row16` (0..15) of d-tile `mt`.
template <class C>
__device__ __forceinline__ int d_of(int mt, int row16) {
    if constexpr (C::FP8) {
        // fp8 V fragments are built so that m-tile 2b+hb, row g holds
        // d = 32b + 4g + 2hb and row g+8 holds d = 32b + 4g + 2hb + 1.
        const int b = mt >> 1, hb = mt & 1;
        const int g = row16 & 7, hi = row16 >> 3;
        return 32 * b + 4 * g + 2 * hb + hi;
    } else {
        return 16 * mt + row16;
    }
}

template <class C, int MODE>
__global__ void __launch_bounds__(C::NTHREADS, C::MINB) attn_tile_kernel(const __grid_constant__ AttnParams p) {
    constexpr bool WIN = MODE == kModeWindow;
    constexpr bool TREE = MODE == kModeTree;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base = (raw_addr + 127u) & ~127u;
    uint8_t* smem = smem_raw + (base - raw_addr);

    const uint32_t bar_full = base + C::OFF_BARS;
    const uint32_t bar_empty = bar_full + 8 * C::NS;
    const uint32_t bar_qfull = bar_empty + 8 * C::NS;
    const uint32_t bar_qempty = bar_qfull + 16;
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NS; ++i) {
            mbar_init(bar_full + 8 * i, C::FULL_ARRIVALS);
            mbar_init(bar_empty + 8 * i, C::NCW);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_qfull + 8 * i, 1);
            mbar_init(bar_qempty + 8 * i, C::NCW);
        }
        misc[0] = 0;  // abort flag (set by any warp that timed out)
        misc[1] = 0;  // error bits of the current item (RAD_ERRW_* values)
        fence_mbarrier_init();
    }
    __syncthreads();

    if (warp >= C::NCW) {
        // ===================================================== producer warps
        const int pw = warp - C::NCW;   // 0: K rows (+ query rows, stage meta), 1: V rows
        const uint8_t* pool = pw == 0 ? p.k_pool : p.v_pool;
        const uint64_t pol_kv = policy_evict_first();
        // Lane -> (row within a group of rows, 16-byte chunk within the row).
        constexpr int CPR = C::ROW_BYTES / 16;          // chunks per row: 8, 16 or 32
        constexpr int RPI = 32 / CPR;                   // rows per warp-wide copy
        const int lrow = lane / CPR, lc = lane % CPR;
        uint32_t scount = 0, qcount = 0;
        bool abort = false;
        for (int item = blockIdx.x; item < p.n_items && !abort; item += gridDim.x) {
            const ItemPlan it = plan_item<C, WIN>(item, p);
            if (!it.active || !it.seq_ok) continue;
            // ---- query rows of the item
            if (pw == 0) {
                const uint32_t slot = qcount & 1u, use = qcount >> 1;
                if (use >= 1 && !mbar_wait_bounded(bar_qempty + 8 * slot, (use - 1) & 1u, p.wait_ns)) {
                    abort = true;
                    break;
                }
                const int nrows = it.m_end - it.m0;
                if (lane == 0) mbar_arrive_expect_tx(bar_qfull + 8 * slot, (uint32_t)(nrows * C::D * 2));
                __syncwarp();
                const uint32_t qdst = base + C::OFF_Q + slot * C::Q_SLOT_BYTES;
                for (int i = lane; i < nrows; i += 32) {
                    const int m = it.m0 + i;
                    const int r = m / p.ratio, hl = m - r * p.ratio;
                    const __nv_bfloat16* src =
                        p.q + ((it.qrow0 + r) * p.n_head + it.kvh * p.ratio + hl) * C::D;
                    bulk_load(qdst + i * C::D * 2, src, C::D * 2, bar_qfull + 8 * slot);
                }
                ++qcount;
            }
            // ---- KV pages of the item, page ids fetched 32 at a time
            const int P = p.page_size;
            const int page_hi = (it.k1 + P - 1) / P;   // exclusive
            const int page_lo = WIN ? it.klo / P : 0;  // pages below hold no visible key: never read
            const uint32_t lsmem = (uint32_t)((lc >> 3) * P * 128);   // this lane's 128-byte column block
            const int32_t* trow = p.page_table + (long long)it.g * p.pages_per_seq;
            const long long row_stride = (long long)p.n_head_kv * C::ROW_BYTES;   // bytes between token slots
            const uint8_t* head_base = pool + (long long)it.kvh * C::ROW_BYTES + (long long)lrow * row_stride + lc * 16;
            int batch0 = -1 << 30;
            int my_pg = 0;
            float my_ks = 1.f, my_vs = 1.f;
            bool my_bad = false;
            for (int st = 0; st < it.n_stages; ++st) {
                const int key0 = it.k0 + st * C::KS;
                const int pstart = key0 / P;
                const int npages = min(C::KS / P, page_hi - pstart);
                if (pstart + npages > batch0 + 32) {
                    batch0 = pstart;
                    const int pi = batch0 + lane;
                    my_bad = false;
                    my_pg = 0;
                    my_ks = my_vs = 1.f;
                    if ((!WIN || pi >= page_lo) && pi < page_hi) {
                        const int pg = __ldg(trow + pi);
                        my_bad = (pg < 0 || pg >= p.num_pages);
                        my_pg = my_bad ? 0 : pg;
                        if (C::FP8 && pw == 0) {
                            my_ks = __ldg(p.k_scales + my_pg);
                            my_vs = __ldg(p.v_scales + my_pg);
                        }
                    }
                }
                const uint32_t slot = scount % C::NS, use = scount / C::NS;
                if (use >= 1 && !mbar_wait_bounded(bar_empty + 8 * slot, (use - 1) & 1u, p.wait_ns)) {
                    abort = true;
                    break;
                }
                const uint32_t tile = base + slot * C::STAGE_BYTES + pw * C::TILE_BYTES;
                for (int i = 0; i < npages; ++i) {
                    if (WIN && pstart + i < page_lo) continue;   // slots stay stale: masked in S and V
                    const int pg = __shfl_sync(0xffffffffu, my_pg, (pstart - batch0 + i) & 31);
                    const uint8_t* src = head_base + (long long)pg * P * row_stride;
                    const uint32_t dst = tile + (uint32_t)(i * P * C::ROW_BYTES) + lsmem;
#pragma unroll 4
                    for (int t0 = 0; t0 < P; t0 += RPI) {
                        const int t = t0 + lrow;
                        cp_async_16(dst + t * 128 + (((lc & 7) ^ (t & 7)) << 4), src + (long long)t0 * row_stride,
                                    pol_kv);
                    }
                }
                cp_async_arrive_noinc(bar_full + 8 * slot);
                if (pw == 0) {
                    uint32_t bad_any = 0;
                    float kss[C::MAX_PAGES_STAGE], vss[C::MAX_PAGES_STAGE];
#pragma unroll
                    for (int i = 0; i < C::MAX_PAGES_STAGE; ++i) {
                        const int src = (pstart - batch0 + i) & 31;
                        kss[i] = __shfl_sync(0xffffffffu, my_ks, src);
                        vss[i] = __shfl_sync(0xffffffffu, my_vs, src);
                        const uint32_t b = __shfl_sync(0xffffffffu, (uint32_t)my_bad, src);
                        if (i < npages) bad_any |= b;
                    }
                    if (lane == 0) {
                        float* meta = reinterpret_cast<float*>(smem + C::OFF_META + slot * C::META_STRIDE);
#pragma unroll
                        for (int i = 0; i < C::MAX_PAGES_STAGE; ++i) {
                            meta[i] = kss[i];
                            meta[4 + i] = vss[i];
                        }
                        reinterpret_cast<uint32_t*>(meta)[8] = bad_any ? kErrPage : 0u;
                        mbar_arrive(bar_full + 8 * slot);
                    }
                }
                ++scount;
            }
            if (misc[0]) abort = true;
        }
        if (abort) {
            misc[0] = 1;
            if (lane == 0 && p.err_word) atomicOr(p.err_word, kErrTimeout);
        }
        // Drain: no copy into shared memory may still be in flight at exit.
        cp_async_wait_all();
        if (pw == 0 && lane == 0) {
            const uint32_t qfirst = qcount > 2u ? qcount - 2u : 0u;
            for (uint32_t c = qfirst; c < qcount; ++c)
                mbar_wait_bounded(bar_qfull + 8 * (c & 1u), (c >> 1) & 1u, p.wait_ns);
        }
        return;
    }

    // ========================================================= consumer warps
    const int wq = warp / C::WK;
    const int wk = warp - wq * C::WK;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int tid = threadIdx.x;   // 0 .. NCT-1
    uint32_t scount = 0, qcount = 0;
    bool abort = false;

    for (int item = blockIdx.x; item < p.n_items && !abort; item += gridDim.x) {
        const ItemPlan it = plan_item<C, WIN>(item, p);
        if (!it.active) continue;
        if (!it.seq_ok) {
            // Invalid length: this group's rows become zeros (the split-0 items
            // of every query tile write them).  Malformed cu_seqlens entries
            // name no rows: only the error bit.
            for (int idx = tid; idx < (it.m_end - it.m0) * C::D; idx += C::NCT) {
                const int m = it.m0 + idx / C::D, d = idx % C::D;
                const int r = m / p.ratio, hl = m - r * p.ratio;
                p.out[((it.qrow0 + r) * p.n_head + it.kvh * p.ratio + hl) * C::D + d] = __float2bfloat16_rn(0.f);
            }
            if (tid == 0 && p.err_word) atomicOr(p.err_word, it.cu_ok ? kErrSeqLen : kErrCuSeq);
            continue;
        }

        // ---- query fragments (B operand of S^T = K Q^T), one per n-tile and k-step
        uint32_t qb[C::NQW][C::D / 16][2];
        int nk[C::NQW][2];   // a column sees keys nk - wlim .. nk - 1 (and none below 0)
        // tree rows: bit i set iff the column sees key nk - 1 - i (its own path
        // among the call's keys, every cached key below them)
        uint32_t amask[C::NQW][2];
        {
            const uint32_t slot = qcount & 1u, use = qcount >> 1;
            if (!mbar_wait_bounded(bar_qfull + 8 * slot, use & 1u, p.wait_ns)) abort = true;
            const uint8_t* qs = smem + C::OFF_Q + slot * C::Q_SLOT_BYTES;
            bool qrange_bad = false;
#pragma unroll
            for (int j = 0; j < C::NQW; ++j) {
                const int colb = (wq * C::NQW + j) * 8 + g8;      // this lane's B column
                const bool valid = it.m0 + colb < it.m_end;
                const uint32_t* qrow = reinterpret_cast<const uint32_t*>(qs + colb * C::D * 2);
#pragma unroll
                for (int ks = 0; ks < C::D / 16; ++ks) {
                    uint32_t b0 = 0, b1 = 0;
                    if (valid) {
                        if constexpr (C::FP8) {
                            const int b = ks >> 1, hh = ks & 1;
                            const int d0 = 32 * b + 8 * t4 + 4 * hh;
                            const uint32_t x0 = qrow[d0 / 2], x1 = qrow[d0 / 2 + 1];
                            const float f0 = bf16_lo(x0), f1 = bf16_hi(x0), f2 = bf16_lo(x1), f3 = bf16_hi(x1);
                            qrange_bad |= fabsf(f0) > 65504.f || fabsf(f1) > 65504.f ||
                                          fabsf(f2) > 65504.f || fabsf(f3) > 65504.f;
                            b0 = pack_f16x2(f0, f1);
                            b1 = pack_f16x2(f2, f3);
                        } else {
                            b0 = qrow[(16 * ks + 2 * t4) / 2];
                            b1 = qrow[(16 * ks + 8 + 2 * t4) / 2];
                        }
                    }
                    qb[j][ks][0] = b0;
                    qb[j][ks][1] = b1;
                }
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int m = it.m0 + lane_col<C>(wq, j, t4, c);
                    const int r = m / p.ratio;
                    nk[j][c] = (m < it.m_end) ? it.L - it.qlen + r + 1 : 0;
                    amask[j][c] = 0u;
                    if (TREE && m < it.m_end) {
                        // word bit i (the call's key i) -> bit r - i; bits past r are cached keys
                        const uint32_t w = __ldg(p.tree_mask + it.qrow0 + r);
                        amask[j][c] = (__brev(w) >> (31 - r)) | (r < 31 ? ~0u << (r + 1) : 0u);
                    }
                }
            }
            if (C::FP8 && qrange_bad && p.err_word) atomicOr(p.err_word, kErrQRange);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_qempty + 8 * slot);
            ++qcount;
        }

        float m_run[C::NQW][2], l_run[C::NQW][2];
        float oacc[C::NQW][C::D / 16][4];
#pragma unroll
        for (int j = 0; j < C::NQW; ++j) {
            m_run[j][0] = m_run[j][1] = -CUDART_INF_F;
            l_run[j][0] = l_run[j][1] = 0.f;
#pragma unroll
            for (int mt = 0; mt < C::D / 16; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) oacc[j][mt][e] = 0.f;
        }
        uint32_t bad = 0;   // RAD_ERRW_* bits seen by this thread
        // Every item checks all mask words of its group (at most 32), so every
        // row of a group with a malformed word is zero: a word must hold its
        // own row's bit and no later row's.
        if (TREE && tid < it.qlen) {
            const uint32_t w = __ldg(p.tree_mask + it.qrow0 + tid);
            if ((w >> tid) != 1u) bad |= kErrMask;
        }
        // Pages the group needs that no item of this tile loads (below the
        // tile's window, or past its last row's keys) are checked by the
        // tile's first item, so every row of a group with a bad page is zero.
        if (it.s == it.s_first) {
            const int P_ = p.page_size;
            const int glo = WIN ? first_visible_key(it.L, it.qlen, 0, p.window) / P_ : 0;
            const int tlo = it.klo / P_, thi = (it.kmax + P_ - 1) / P_, ghi = (it.L + P_ - 1) / P_;
            const int32_t* trow = p.page_table + (long long)it.g * p.pages_per_seq;
            const int n_below = tlo - glo;
            for (int i = tid; i < n_below + (ghi - thi); i += C::NCT) {
                const int pi = i < n_below ? glo + i : thi + (i - n_below);
                const int pg = __ldg(trow + pi);
                bad |= (pg < 0 || pg >= p.num_pages) ? kErrPage : 0u;
            }
        }
        const int P = p.page_size;
        const int lp = (P == 16) ? 4 : 5;
        // key is visible to a column iff 0 <= nk - 1 - key < wlim
        const uint32_t wlim = p.window > 0 ? (uint32_t)p.window : 0x7FFFFFFFu;

        for (int st = 0; st < it.n_stages && !abort; ++st) {
            const uint32_t slot = scount % C::NS, use = scount / C::NS;
            if (!mbar_wait_bounded(bar_full + 8 * slot, use & 1u, p.wait_ns)) {
                abort = true;
                break;
            }
            const uint32_t kbase = base + slot * C::STAGE_BYTES;
            const uint32_t vbase = kbase + C::TILE_BYTES;
            const float* meta = reinterpret_cast<const float*>(smem + C::OFF_META + slot * C::META_STRIDE);
            bad |= reinterpret_cast<const uint32_t*>(meta)[8];
            const int skey0 = it.k0 + st * C::KS;

#pragma unroll 1
            for (int kt = wk; kt < C::SUBS; kt += C::WK) {
                const int key0 = skey0 + kt * 16;
                if (key0 >= it.k1) break;
                float kfac = p.scale_log2, vfac = 1.f;
                if constexpr (C::FP8) {
                    const int pi = (kt * 16) / P;   // page of this 16-key sub-tile within the stage
                    kfac *= meta[pi];
                    vfac = meta[4 + pi];
                }
                // ---------------- S^T = K Q^T
                float sacc[C::NQW][4];
#pragma unroll
                for (int j = 0; j < C::NQW; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sacc[j][e] = 0.f;
                if constexpr (!C::FP8) {
                    const int mi = lane >> 3, ri = lane & 7;
                    const int row = kt * 16 + ri + 8 * (mi & 1);
#pragma unroll
                    for (int ks = 0; ks < C::D / 16; ++ks) {
                        const uint32_t off = kv_off<C>(row, 16 * ks + 8 * (mi >> 1), lp);
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4(kbase + swz128(off), a0, a1, a2, a3);
#pragma unroll
                        for (int j = 0; j < C::NQW; ++j) mma_bf16(sacc[j], a0, a1, a2, a3, qb[j][ks][0], qb[j][ks][1]);
                    }
                } else {
#pragma unroll
                    for (int b = 0; b < C::D / 32; ++b) {
                        const int col = 32 * b + 8 * t4;
                        uint32_t lo0, lo1, hi0, hi1;
                        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(lo0), "=r"(lo1) : "r"(kbase + swz128(kv_off<C>(kt * 16 + g8, col, lp))));
                        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(hi0), "=r"(hi1) : "r"(kbase + swz128(kv_off<C>(kt * 16 + g8 + 8, col, lp))));
                        // k-step 2b: bytes 0..3 ; k-step 2b+1: bytes 4..7
                        const uint32_t a0 = e4m3x2_to_f16x2((uint16_t)(lo0 & 0xFFFF));
                        const uint32_t a1 = e4m3x2_to_f16x2((uint16_t)(hi0 & 0xFFFF));
                        const uint32_t a2 = e4m3x2_to_f16x2((uint16_t)(lo0 >> 16));
                        const uint32_t a3 = e4m3x2_to_f16x2((uint16_t)(hi0 >> 16));
                        const uint32_t c0 = e4m3x2_to_f16x2((uint16_t)(lo1 & 0xFFFF));
                        const uint32_t c1 = e4m3x2_to_f16x2((uint16_t)(hi1 & 0xFFFF));
                        const uint32_t c2 = e4m3x2_to_f16x2((uint16_t)(lo1 >> 16));
                        const uint32_t c3 = e4m3x2_to_f16x2((uint16_t)(hi1 >> 16));
#pragma unroll
                        for (int j = 0; j < C::NQW; ++j) {
                            mma_f16(sacc[j], a0, a1, a2, a3, qb[j][2 * b][0], qb[j][2 * b][1]);
                            mma_f16(sacc[j], c0, c1, c2, c3, qb[j][2 * b + 1][0], qb[j][2 * b + 1][1]);
                        }
                    }
                }
                // ---------------- mask, online softmax
                // bf16 pools carry P as a bf16 pair hi + lo (hi = bf16(p), lo =
                // bf16(p - hi)), so the PV product sees p to ~2^-17 relative;
                // fp8 pools carry P (times the page's V scale) in f16.
                uint32_t pb[C::NQW][2];
                uint32_t pl[C::NQW][2];
#pragma unroll
                for (int j = 0; j < C::NQW; ++j) {
                    float x[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int key = key0 + g8 + ((e >> 1) << 3);
                        bool in;
                        if constexpr (TREE) {
                            const uint32_t du = (uint32_t)(nk[j][e & 1] - 1 - key);   // distance back from the row
                            in = du < 32u ? ((amask[j][e & 1] >> du) & 1u) != 0u : du < 0x80000000u;
                        } else {
                            in = WIN ? (uint32_t)(nk[j][e & 1] - 1 - key) < wlim : key < nk[j][e & 1];
                        }
                        x[e] = in ? sacc[j][e] * kfac : -CUDART_INF_F;
                    }
                    // The running max moves only when a sub-tile's max exceeds it by
                    // more than 2^8 (or on the first keys); weights up to 2^8 are exact
                    // to carry, and the accumulators are rescaled only then.
                    float alpha[2];
                    bool moved = false;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        float mx = fmaxf(x[c], x[c + 2]);
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                        alpha[c] = 1.f;
                        if (mx > m_run[j][c] + kLazyRescaleLog2 || (m_run[j][c] == -CUDART_INF_F && mx != -CUDART_INF_F)) {
                            alpha[c] = exp2f(m_run[j][c] - mx);
                            m_run[j][c] = mx;
                            moved = true;
                        }
                        const float m_use = (m_run[j][c] == -CUDART_INF_F) ? 0.f : m_run[j][c];
                        x[c] = exp2f(x[c] - m_use);
                        x[c + 2] = exp2f(x[c + 2] - m_use);
                        l_run[j][c] = l_run[j][c] * alpha[c] + (x[c] + x[c + 2]);
                    }
                    if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
                        for (int mt = 0; mt < C::D / 16; ++mt) {
                            oacc[j][mt][0] *= alpha[0];
                            oacc[j][mt][1] *= alpha[1];
                            oacc[j][mt][2] *= alpha[0];
                            oacc[j][mt][3] *= alpha[1];
                        }
                    }
                    if constexpr (C::FP8) {
                        pb[j][0] = movmatrix_trans(pack_f16x2(x[0] * vfac, x[1] * vfac));
                        pb[j][1] = movmatrix_trans(pack_f16x2(x[2] * vfac, x[3] * vfac));
                    } else {
                        const uint32_t h01 = pack_bf16x2(x[0], x[1]);
                        const uint32_t h23 = pack_bf16x2(x[2], x[3]);
                        const uint32_t l01 = pack_bf16x2(x[0] - bf16_lo(h01), x[1] - bf16_hi(h01));
                        const uint32_t l23 = pack_bf16x2(x[2] - bf16_lo(h23), x[3] - bf16_hi(h23));
                        pb[j][0] = movmatrix_trans(h01);
                        pb[j][1] = movmatrix_trans(h23);
                        pl[j][0] = movmatrix_trans(l01);
                        pl[j][1] = movmatrix_trans(l23);
                    }
                }
                // ---------------- O^T += V^T P^T
                // keys outside [klo, k1) are zeroed in V: past the item's range
                // the slots may hold anything, below klo they may be stale
                const bool edge = key0 + 16 > it.k1 || (WIN && key0 < it.klo);
                const auto vis = [&](int k) { return (!WIN || k >= it.klo) && k < it.k1; };
                if constexpr (!C::FP8) {
                    const int mi = lane >> 3, ri = lane & 7;
                    const int row = kt * 16 + ri + 8 * (mi >> 1);
                    const int ke = key0 + 2 * t4;
                    const uint32_t m_lo = (edge ? ((vis(ke) ? 0x0000FFFFu : 0u) | (vis(ke + 1) ? 0xFFFF0000u : 0u)) : 0xFFFFFFFFu);
                    const uint32_t m_hi = (edge ? ((vis(ke + 8) ? 0x0000FFFFu : 0u) | (vis(ke + 9) ? 0xFFFF0000u : 0u)) : 0xFFFFFFFFu);
#pragma unroll
                    for (int dt = 0; dt < C::D / 16; ++dt) {
                        const uint32_t off = kv_off<C>(row, 16 * dt + 8 * (mi & 1), lp);
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4_trans(vbase + swz128(off), a0, a1, a2, a3);
                        a0 &= m_lo;
                        a1 &= m_lo;
                        a2 &= m_hi;
                        a3 &= m_hi;
#pragma unroll
                        for (int j = 0; j < C::NQW; ++j) {
                            mma_bf16(oacc[j][dt], a0, a1, a2, a3, pb[j][0], pb[j][1]);
                            mma_bf16(oacc[j][dt], a0, a1, a2, a3, pl[j][0], pl[j][1]);
                        }
                    }
                } else {
                    const int kr = kt * 16 + 2 * t4;
                    const int ke = key0 + 2 * t4;
                    const bool z0 = edge && !vis(ke), z1 = edge && !vis(ke + 1);
                    const bool z2 = edge && !vis(ke + 8), z3 = edge && !vis(ke + 9);
#pragma unroll
                    for (int b = 0; b < C::D / 32; ++b) {
                        const int col = 32 * b + 4 * g8;
                        uint32_t w0, w1, w2, w3;
                        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w0) : "r"(vbase + swz128(kv_off<C>(kr, col, lp))));
                        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w1) : "r"(vbase + swz128(kv_off<C>(kr + 1, col, lp))));
                        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w2) : "r"(vbase + swz128(kv_off<C>(kr + 8, col, lp))));
                        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w3) : "r"(vbase + swz128(kv_off<C>(kr + 9, col, lp))));
                        if (z0) w0 = 0;
                        if (z1) w1 = 0;
                        if (z2) w2 = 0;
                        if (z3) w3 = 0;
                        // pairs (key 2t, key 2t+1) and (key 2t+8, key 2t+9) at one d
                        const uint32_t p01_lo = __byte_perm(w0, w1, 0x5140);   // d+0 | d+1
                        const uint32_t p01_hi = __byte_perm(w0, w1, 0x7362);   // d+2 | d+3
                        const uint32_t p89_lo = __byte_perm(w2, w3, 0x5140);
                        const uint32_t p89_hi = __byte_perm(w2, w3, 0x7362);
                        // m-tile 2b: rows g (d+0), g+8 (d+1); m-tile 2b+1: rows g (d+2), g+8 (d+3)
                        const uint32_t e0 = e4m3x2_to_f16x2((uint16_t)(p01_lo & 0xFFFF));
                        const uint32_t e1 = e4m3x2_to_f16x2((uint16_t)(p01_lo >> 16));
                        const uint32_t e2 = e4m3x2_to_f16x2((uint16_t)(p89_lo & 0xFFFF));
                        const uint32_t e3 = e4m3x2_to_f16x2((uint16_t)(p89_lo >> 16));
                        const uint32_t f0 = e4m3x2_to_f16x2((uint16_t)(p01_hi & 0xFFFF));
                        const uint32_t f1 = e4m3x2_to_f16x2((uint16_t)(p01_hi >> 16));
                        const uint32_t f2 = e4m3x2_to_f16x2((uint16_t)(p89_hi & 0xFFFF));
                        const uint32_t f3 = e4m3x2_to_f16x2((uint16_t)(p89_hi >> 16));
#pragma unroll
                        for (int j = 0; j < C::NQW; ++j) {
                            mma_f16(oacc[j][2 * b], e0, e1, e2, e3, pb[j][0], pb[j][1]);
                            mma_f16(oacc[j][2 * b + 1], f0, f1, f2, f3, pb[j][0], pb[j][1]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
            ++scount;
            if (misc[0]) abort = true;
        }
        // Every consumer warp reaches this barrier once per item, whatever
        // happened above, so a time-out never strands the others.
        if (named_barrier_or(1, C::NCT, abort)) {
            abort = true;
            break;
        }

        // ---------------- per-warp sums over the 8 key lanes
#pragma unroll
        for (int j = 0; j < C::NQW; ++j)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float l = l_run[j][c];
                l += __shfl_xor_sync(0xffffffffu, l, 4);
                l += __shfl_xor_sync(0xffffffffu, l, 8);
                l += __shfl_xor_sync(0xffffffffu, l, 16);
                l_run[j][c] = l;
            }
        // ---------------- merge the key warps' states
        // One [query column][head dim] buffer holds a single warp state.  With
        // two key warps per query group each owns half of the d-tiles: it
        // publishes the other half into the buffer, then merges its own half
        // from its registers and the published values and writes the result
        // back in place (every element is published, read and rewritten by
        // fixed lanes, ordered by the barriers).  The merge sums in key-warp
        // order 0, 1 whichever warp performs it.  All consumer threads then
        // write the tile out with coalesced 16-byte reads.
        constexpr int MT = C::D / 16;
        constexpr int MTW = MT / C::WK;   // d-tiles owned per key warp
        const int own0 = wk * MTW;
        float* mrg = reinterpret_cast<float*>(smem + C::OFF_MERGE);       // [QT][MSTRIDE]
        float4* mlpub = reinterpret_cast<float4*>(smem + C::OFF_ML);      // [wq][wk][j][t4]
        float2* mlfin = reinterpret_cast<float2*>(smem + C::OFF_MLF);     // [QT] merged (max, sum)
        if constexpr (C::WK > 1) {
#pragma unroll
            for (int j = 0; j < C::NQW; ++j) {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    if (mt >= own0 && mt < own0 + MTW) continue;
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        mrg[lane_col<C>(wq, j, t4, e & 1) * C::MSTRIDE + d_of<C>(mt, g8 + ((e >> 1) << 3))] =
                            oacc[j][mt][e];
                }
                if (g8 == 0)
                    mlpub[((wq * C::WK + wk) * C::NQW + j) * 4 + t4] =
                        make_float4(m_run[j][0], l_run[j][0], m_run[j][1], l_run[j][1]);
            }
        }
        // Stage-meta `bad` words were OR-ed per warp; make them CTA-wide (this
        // barrier also orders the published states before their reads).
        if (bad) atomicOr(const_cast<uint32_t*>(misc + 1), bad);
        const bool item_bad = named_barrier_or(1, C::NCT, bad != 0);
        const uint32_t bad_bits = item_bad ? misc[1] : 0u;

        // one split holding visible keys: the row is written here, else partials
        const bool final_write = (p.split_len == 0) || it.n_splits - it.s_first == 1;
#pragma unroll
        for (int j = 0; j < C::NQW; ++j) {
            float fw[2][C::WK], scale_out[2];   // scale_out: 1/l per column
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float mv[C::WK], lv[C::WK];
#pragma unroll
                for (int w = 0; w < C::WK; ++w) {
                    if (C::WK == 1) {
                        mv[w] = m_run[j][c];
                        lv[w] = l_run[j][c];
                    } else {
                        const float4 o = mlpub[((wq * C::WK + w) * C::NQW + j) * 4 + t4];
                        mv[w] = c ? o.z : o.x;
                        lv[w] = c ? o.w : o.y;
                    }
                }
                float mx = mv[0];
#pragma unroll
                for (int w = 1; w < C::WK; ++w) mx = fmaxf(mx, mv[w]);
                const float m_use = (mx == -CUDART_INF_F) ? 0.f : mx;
#pragma unroll
                for (int w = 0; w < C::WK; ++w) fw[c][w] = exp2f(mv[w] - m_use);
                float l = fw[c][0] * lv[0];
#pragma unroll
                for (int w = 1; w < C::WK; ++w) l = fmaf(fw[c][w], lv[w], l);
                // acc * (1/l), the combine kernel's form, so a row written here
                // and the same row merged from splits round identically
                scale_out[c] = 1.f / l;
                const int col = lane_col<C>(wq, j, t4, c);
                if (!final_write && wk == 0 && g8 == 0) mlfin[col] = make_float2(mx, l);
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                if (mt < own0 || mt >= own0 + MTW) continue;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = e & 1;
                    float* slot = mrg + lane_col<C>(wq, j, t4, c) * C::MSTRIDE + d_of<C>(mt, g8 + ((e >> 1) << 3));
                    float acc;
                    if constexpr (C::WK == 1) {
                        acc = fw[c][0] * oacc[j][mt][e];
                    } else {
                        const float other = *slot;
                        const float a0 = wk == 0 ? oacc[j][mt][e] : other;
                        const float a1 = wk == 0 ? other : oacc[j][mt][e];
                        acc = fmaf(fw[c][1], a1, fw[c][0] * a0);
                    }
                    *slot = final_write ? (item_bad ? 0.f : acc * scale_out[c]) : acc;
                }
            }
        }
        named_barrier_sync(1, C::NCT);
        {
            const int ncols = it.m_end - it.m0;
            constexpr int D4 = C::D / 4;
            if (final_write) {
                for (int idx = tid; idx < ncols * D4; idx += C::NCT) {
                    const int col = idx / D4, d4 = idx - col * D4;
                    const float4 v = *reinterpret_cast<const float4*>(mrg + col * C::MSTRIDE + 4 * d4);
                    const int m = it.m0 + col;
                    const int r = m / p.ratio, hl = m - r * p.ratio;
                    __nv_bfloat16* o = p.out + ((it.qrow0 + r) * p.n_head + it.kvh * p.ratio + hl) * C::D + 4 * d4;
                    uint2 w;
                    w.x = pack_bf16x2(v.x, v.y);
                    w.y = pack_bf16x2(v.z, v.w);
                    *reinterpret_cast<uint2*>(o) = w;
                }
                if (item_bad && tid == 0 && p.err_word) atomicOr(p.err_word, bad_bits);
            } else {
                const long long slot_idx = it.gq * p.max_splits + it.s;
                float* pacc = p.part_acc + slot_idx * p.qtv * C::D;
                float* pml = p.part_ml + slot_idx * p.qtv * 2;
                for (int idx = tid; idx < ncols * D4; idx += C::NCT) {
                    const int col = idx / D4, d4 = idx - col * D4;
                    __stcg(reinterpret_cast<float4*>(pacc + col * C::D) + d4,
                           *reinterpret_cast<const float4*>(mrg + col * C::MSTRIDE + 4 * d4));
                }
                for (int col = tid; col < ncols; col += C::NCT)
                    __stcg(reinterpret_cast<float2*>(pml) + col, mlfin[col]);
                if (tid == 0) __stcg(p.part_flag + slot_idx, bad_bits);
            }
        }
        // the merge buffers (and the error word) are rewritten by the next item
        named_barrier_sync(1, C::NCT);
        if (tid == 0 && item_bad) misc[1] = 0u;
    }
    if (abort) {
        misc[0] = 1;
        if (lane == 0 && p.err_word) atomicOr(p.err_word, kErrTimeout);
    }
}

}  // namespace rad
