// Split-call attention on the 5th-generation tensor cores (tcgen05, TMEM) for
// fp8-e4m3 KV pools with head_dim 128: the decode and speculative-verify call
// shapes ("kern manifest v7", $defs.Batch) of the `attn_paged` op.
//
// Work items and partial results are those of attn_tile.cuh: (split s,
// sequence g, KV head kvh, query tile qt) with N query rows per tile (the
// rows x n_head/n_head_kv query heads sharing the KV head), splits of
// split_len keys whose count depends only on the sequence length, and the
// same combine kernel.
//
// Keys are the MMA's M dimension (128 per tile) and the query rows its N:
//   S^T[key][q] = K[key][:] . Q[q][:]        kind::f8f6f4, M 128, N, K = head_dim:
//                                            K straight from the staged e4m3 rows,
//                                            Q as two e4m3 terms (below)
//   O^T[d][q]  += V^T[d][key] . P^T[key][q]   kind::f16, M = head_dim 128, N, K = 128
//                                            keys: V converted to f16, P in f16
// Q row q is split as q * 2^k = hi + lo, each term e4m3 (k per row puts the
// row's largest |q| in [128, 256)): hi is q * 2^k rounded to 4 significant
// bits, and the remainder of a bf16 value (8 significant bits) then has at
// most 4, so lo holds it exactly -- the two terms are q itself, except where
// lo falls into e4m3's subnormal range (elements below 2^-8 of the row's
// largest).  The tensor core forms the products exactly in fp32 and the
// logits are scaled back by 2^-k.
// so a decode step's few query rows per KV head cost a narrow N instead of
// an idle M.  Warp roles (one CTA per SM, persistent):
//   last two    producers: page ids from the page table ("kern manifest v7",
//               $defs.Domain), one TMA box per page (page_size rows x 128
//               bytes of the KV head) of each tile's e4m3 K rows and V rows
//               (one warp each, one issuing lane) into the staging ring, the
//               per-page scales, and a 1-D bulk copy of the query rows.
//               (16-byte cp.async copies took the producer ~2300 cycles per
//               tile to issue, which then set the tile period.)
//   warp 4G     QK MMA: one lane issues the tcgen05.mma of S^T per tile as
//               soon as its K stage has landed and its TMEM S buffer is free
//               (up to NSB tiles ahead of the softmax, across items); then the
//               warp converts key rows 0-63 of the previous tile's staged e4m3
//               V rows to f16 (exact) in the 128-byte-swizzled layout the MMA
//               reads, into f16 buffer (t-1) & 1 once PV of tile t-3 has read
//               it (at an item's last tile, also tile t's rows).
//   warp 4G+1   PV MMA: converts key rows 64-127 of tile t the same way, then
//               one lane issues O^T += V^T P^T once the workers published P
//               and the QK warp's rows are converted.
//   warps 0 .. 4G-1  workers; thread t serves key slot k = t % 128 (TMEM
//               lane k) and group h = t / 128 of the query rows (warps w,
//               w+4, .. share TMEM lanes 32(w%4)..): split the item's query
//               rows into e4m3 terms, run the online softmax of key k against
//               its group of query rows, write P^T, and in the epilogue read
//               O^T (lane k = head-dim element k) and store its rows.
//               (The V conversion ran on the workers before: 800 of the 3200
//               cycles of a tile's chain through them, in a globaltimer /
//               clock64 trace of one CTA.)
// Per query row, the running max moves (and O and the sums are rescaled)
// only when a tile's logits exceed it by more than 2^8; the per-row sums are
// kept per key slot and reduced once per item in a fixed order, so a row's
// arithmetic depends only on its own sequence and on its position, never on
// the other rows of the call.
//
// Every mbarrier wait is bounded; a time-out sets RAD_ERRW_TIMEOUT and the
// roles unwind (the workers only at a barrier all four reach), waiting
// (bounded) for their copies and MMAs before TMEM is freed.
#pragma once
#include <cuda.h>

#include "attn_tile.cuh"
#include "tc05.cuh"

#ifndef RAD_SPLITTC_NS
#define RAD_SPLITTC_NS 3
#endif
// Groups G the query rows of an item are split into among the workers (4G
// worker warps, G per TMEM lane quarter).
#ifndef RAD_SPLITTC_GROUPS
#define RAD_SPLITTC_GROUPS 2
#endif

namespace rad {

template <int N_>
struct SplitTcCfg {
    static constexpr int D = 128;      // head dim
    static constexpr int BK = 128;     // keys per tile: the MMA's M
    static constexpr int N = N_;       // query rows per item: the MMA's N
    static constexpr int NSB = 3;      // S buffers: QK runs up to two tiles ahead of PV
    static constexpr int G = RAD_SPLITTC_GROUPS;
    static constexpr int V = N / G;    // query rows per worker thread
    static constexpr int QT = N;       // (item planner) query rows per tile
    static constexpr int KS = BK;      // (item planner) keys per stage
    static constexpr int NS = RAD_SPLITTC_NS;
    static constexpr int ROW = 128;                  // bytes of one e4m3 key row
    static constexpr int STG_TILE = BK * ROW;        // 16 KB: K or V of one tile
    static constexpr int STG_BYTES = 2 * STG_TILE;
    static constexpr int ATOM = BK * 128;            // f16 tile: stride between 64-column blocks
    static constexpr int F16_TILE = 2 * ATOM;        // [column block 2][key 128][128 B]
    static constexpr int Q8_TERM = N * 128;          // one e4m3 term of the query rows: [q N][128 B]
    static constexpr int QTERMS = 2;                 // e4m3 terms per query row (hi, lo)
    static constexpr int Q8_BYTES = QTERMS * Q8_TERM;
    static constexpr int QSTG_BYTES = N * D * 2;     // bf16 query rows, one slot
    static constexpr int PATOM = N * 128;
    static constexpr int P_BYTES = 2 * PATOM;        // [key block 2][q N][128 B]
    static constexpr int MAXPG = BK / 16;            // pages per tile
    static constexpr int META_STRIDE = 128;          // ks[8], vs[8], bad
    // K and V staging rings (NS stages each; a staged K tile is the QK MMA's A
    // operand as it lands), two f16 V tiles, the query terms, two P tiles
    static constexpr int OFF_STG = 0;            // stage i: K at i*STG_BYTES, V at +STG_TILE
    static constexpr int OFF_V16 = OFF_STG + NS * STG_BYTES;    // two buffers
    static constexpr int OFF_Q8 = OFF_V16 + 2 * F16_TILE;
    static constexpr int OFF_P = OFF_Q8 + Q8_BYTES;
    static constexpr int OFF_QSTG = OFF_P + 2 * P_BYTES;        // one slot
    static constexpr int OFF_META = OFF_QSTG + QSTG_BYTES;
    static constexpr int OFF_RED = OFF_META + NS * META_STRIDE;
    static constexpr int OFF_ISQ = OFF_RED + 5 * N * 4;    // red: [G][4][V] partials + [G][V] totals
    static constexpr int OFF_TMW = OFF_ISQ + N * 4;        // isq: 2^-k of each query row
    static constexpr int OFF_BARS = OFF_TMW + N * 4;       // tmw: tree-mask word of each query row
    // k_full[NS], k_empty[NS], v_full[NS], v_empty[NS], qstg_full, qstg_empty,
    // q8_full, (unused), v16_full[2], p_full[2], s_full[NSB], s_empty[NSB], pv_done[2],
    // o_free, final_qk, final_pv
    static constexpr int NBARS = 4 * NS + 2 + 2 + 2 + 2 + 2 * NSB + 2 + 3;
    static constexpr int OFF_MISC = OFF_BARS + NBARS * 8;          // [0] tmem, [1] abort, [2] worker abort
    static constexpr int SMEM_USED = OFF_MISC + 16;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;   // 1 KB alignment of the swizzled operand tiles
    static constexpr int NWORK = 4 * G;                  // worker warps
    static constexpr int NWT = NWORK * 32;               // worker threads
    static constexpr int W_QK = NWORK, W_PV = NWORK + 1, W_PROD = NWORK + 2;
    static constexpr int NTHREADS = (NWORK + 4) * 32;
    static constexpr int K_ARRIVALS = MAXPG;   // the producer's expect-tx arrive + 7 lanes' meta arrives
    static constexpr int V_ARRIVALS = 1;       // the producer's expect-tx arrive
    static constexpr uint32_t TMEM_COLS = (NSB + 1) * N <= 64 ? 64 : 128;   // S[NSB] and O
    static_assert(N == 16 || N == 32, "query rows per item");
    static_assert((G == 2 || G == 4) && V >= 4, "query-row groups");
    static_assert(STG_BYTES % 1024 == 0 && OFF_V16 % 1024 == 0 && OFF_Q8 % 1024 == 0 && OFF_P % 1024 == 0 &&
                      Q8_TERM % 1024 == 0,
                  "swizzled operand tiles on 1 KB boundaries");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};


// Converts key row t of a staged tile (128 e4m3 codes, 16-byte chunks
// swizzled by t & 7) to f16 in an f16 tile [column block][key][128 B] with the
// same 128-byte swizzle; `zero` writes zeros instead.  The row's loads come
// first: the stores after them may alias them as far as the compiler knows.
template <class C>
__device__ __forceinline__ void convert_key_row(const uint8_t* src, uint8_t* dst, int t, bool zero) {
    const uint32_t sw = (uint32_t)(t & 7);
    uint4 in[8];
#pragma unroll
    for (int c = 0; c < 8; ++c)
        in[c] = zero ? make_uint4(0u, 0u, 0u, 0u) : *reinterpret_cast<const uint4*>(src + t * 128 + ((c ^ sw) << 4));
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 v = in[c];
        const uint32_t h0 = e4m3x2_to_f16x2((uint16_t)(v.x & 0xFFFFu)), h1 = e4m3x2_to_f16x2((uint16_t)(v.x >> 16));
        const uint32_t h2 = e4m3x2_to_f16x2((uint16_t)(v.y & 0xFFFFu)), h3 = e4m3x2_to_f16x2((uint16_t)(v.y >> 16));
        const uint32_t h4 = e4m3x2_to_f16x2((uint16_t)(v.z & 0xFFFFu)), h5 = e4m3x2_to_f16x2((uint16_t)(v.z >> 16));
        const uint32_t h6 = e4m3x2_to_f16x2((uint16_t)(v.w & 0xFFFFu)), h7 = e4m3x2_to_f16x2((uint16_t)(v.w >> 16));
        // codes 16c .. 16c+15 -> f16 chunks 2c, 2c+1 of the row (8 values each)
        uint8_t* row = dst + (c >> 2) * C::ATOM + t * 128;
        const uint32_t ch = (uint32_t)((c & 3) * 2);
        *reinterpret_cast<uint4*>(row + ((ch ^ sw) << 4)) = make_uint4(h0, h1, h2, h3);
        *reinterpret_cast<uint4*>(row + (((ch + 1) ^ sw) << 4)) = make_uint4(h4, h5, h6, h7);
    }
}

// Key rows lane + 32 r, r = r0 .. r0 + 1, of staged V tile `slot` -> f16 V
// buffer vb, zeros outside the item's keys [klo, k1) (P is 0 there; those
// slots may hold anything).  Called by the QK warp (r0 = 0) and the PV warp
// (r0 = 2) once per tile.
template <class C>
__device__ __forceinline__ void convert_v_half(uint8_t* smem, uint32_t slot, uint32_t vb, int r0, int key0, int klo,
                                               int k1, int lane) {
    const uint8_t* src = smem + C::OFF_STG + slot * C::STG_BYTES + C::STG_TILE;
    uint8_t* dst = smem + C::OFF_V16 + vb * C::F16_TILE;
#pragma unroll 1
    for (int r = r0; r < r0 + 2; ++r) {
        const int t = lane + 32 * r;
        const int key = key0 + t;
        convert_key_row<C>(src, dst, t, key < klo || key >= k1);
    }
}

// Reduces v over the 32 lanes of the warp so that lane l returns the result
// for column l & (V-1) (max or sum); the combination tree is fixed by lane
// bits (16, 8, 4, 2, 1), whatever V.
template <int V, bool MAX>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[V], int lane) {
#pragma unroll
    for (int o = 16; o >= V; o >>= 1) {
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const float x = __shfl_xor_sync(0xffffffffu, v[k], o);
            v[k] = MAX ? fmaxf(v[k], x) : v[k] + x;
        }
    }
#pragma unroll
    for (int o = V / 2; o >= 1; o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int k = 0; k < o; ++k) {
            const float send = upper ? v[k] : v[k + o];
            const float keep = upper ? v[k + o] : v[k];
            const float recv = __shfl_xor_sync(0xffffffffu, send, o);
            v[k] = MAX ? fmaxf(keep, recv) : keep + recv;
        }
    }
    return v[0];
}

// All worker warps: for each group h of the query rows, totals of v over the
// 128 key slots, per row, into tot[V] of every thread of that group (the
// partials of the four warps of a group combined in warp order).
template <int V, int NWT, bool MAX>
__device__ __forceinline__ void workers_reduce(float (&v)[V], float (&tot)[V], float* red, int wq, int h, int lane,
                                               int k) {
    constexpr int TOT = NWT / 32 * V;   // offset of the totals: [G][4][V] partials first
    const float mine = warp_transpose_reduce<V, MAX>(v, lane);
    if (lane < V) red[(h * 4 + wq) * V + lane] = mine;
    named_barrier_sync(2, NWT);
    if (k < V) {
        float a = red[(h * 4) * V + k];
#pragma unroll
        for (int w = 1; w < 4; ++w) a = MAX ? fmaxf(a, red[(h * 4 + w) * V + k]) : a + red[(h * 4 + w) * V + k];
        red[TOT + h * V + k] = a;
    }
    named_barrier_sync(2, NWT);
#pragma unroll
    for (int q = 0; q < V; q += 4) {
        const float4 f = *reinterpret_cast<const float4*>(red + TOT + h * V + q);
        tot[q] = f.x;
        tot[q + 1] = f.y;
        tot[q + 2] = f.z;
        tot[q + 3] = f.w;
    }
}

template <int V>
__device__ __forceinline__ void tmem_ldV(uint32_t taddr, uint32_t (&r)[V]) {
    if constexpr (V == 4) tmem_ld4(taddr, r);
    else if constexpr (V == 8) tmem_ld8(taddr, r);
    else tmem_ld16(taddr, r);
}
template <int V>
__device__ __forceinline__ void tmem_stV(uint32_t taddr, const uint32_t (&r)[V]) {
    if constexpr (V == 4) tmem_st4(taddr, r);
    else if constexpr (V == 8) tmem_st8(taddr, r);
    else tmem_st16(taddr, r);
}

// MODE: kModeCausal, kModeWindow or kModeTree (draft-tree rows, uniform row
// counts: bit i of a row's mask word lets it see the call's key i).
template <int N, int MODE>
__global__ void __launch_bounds__(SplitTcCfg<N>::NTHREADS, 1)
    attn_split_tc05_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ AttnParams p) {
    using C = SplitTcCfg<N>;
    constexpr bool WIN = MODE == kModeWindow;
    constexpr bool TREE = MODE == kModeTree;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_addr);

    const uint32_t bar_k_full = base + C::OFF_BARS;
    const uint32_t bar_k_empty = bar_k_full + 8 * C::NS;
    const uint32_t bar_v_full = bar_k_empty + 8 * C::NS;
    const uint32_t bar_v_empty = bar_v_full + 8 * C::NS;
    const uint32_t bar_qstg_full = bar_v_empty + 8 * C::NS;
    const uint32_t bar_qstg_empty = bar_qstg_full + 8;
    const uint32_t bar_q8_full = bar_qstg_empty + 8;
    const uint32_t bar_v16_full = bar_q8_full + 16;     // [2], per f16 V buffer: the QK warp's half converted
    const uint32_t bar_p_full = bar_v16_full + 16;      // [2], per P buffer
    const uint32_t bar_s_full = bar_p_full + 16;        // [NSB], per S buffer
    const uint32_t bar_s_empty = bar_s_full + 8 * C::NSB;   // [NSB], S read by the workers
    const uint32_t bar_pv_done = bar_s_empty + 8 * C::NSB;  // [2], PV of tiles of each parity
    const uint32_t bar_o_free = bar_pv_done + 16;
    const uint32_t bar_final = bar_o_free + 8;          // [2]: QK warp, PV warp
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NS; ++i) {
            mbar_init(bar_k_full + 8 * i, C::K_ARRIVALS);
            mbar_init(bar_k_empty + 8 * i, 1 + C::NWORK);   // the QK MMA's commit + the workers' scale reads
            mbar_init(bar_v_full + 8 * i, C::V_ARRIVALS);
            mbar_init(bar_v_empty + 8 * i, 2);   // converted: the QK warp's and the PV warp's rows
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_v16_full + 8 * i, 1);   // the QK warp's rows of the tile
            mbar_init(bar_p_full + 8 * i, C::NWORK);
            mbar_init(bar_pv_done + 8 * i, 1);
        }
        for (int i = 0; i < C::NSB; ++i) {
            mbar_init(bar_s_full + 8 * i, 1);
            mbar_init(bar_s_empty + 8 * i, C::NWORK);
        }
        mbar_init(bar_qstg_full, 1);
        mbar_init(bar_qstg_empty, C::NWORK);
        mbar_init(bar_q8_full, C::NWORK);
        mbar_init(bar_o_free, C::NWORK);
        mbar_init(bar_final, 1);
        mbar_init(bar_final + 8, 1);
        misc[1] = 0;
        misc[2] = 0;
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
    const uint32_t t_s = tmem;                  // S buffer b: columns [b*N, b*N + N)
    const uint32_t t_o = tmem + C::NSB * N;     // O^T: columns [NSB*N, NSB*N + N)
    bool abort = false;

    if (warp >= C::W_PROD) {
        // ===================================================== producers
        const int pw = warp - C::W_PROD;   // 0: K rows (also the query rows and the stage meta); 1: V rows
        const CUtensorMap* tm = pw == 0 ? &tm_k : &tm_v;
        const uint64_t pol_kv = policy_evict_first();
        const uint32_t bar_full = pw == 0 ? bar_k_full : bar_v_full;
        const uint32_t bar_empty = pw == 0 ? bar_k_empty : bar_v_empty;
        const int oob_tok = p.num_pages * p.page_size;   // a row past the pool: TMA fills the box with zeros
        uint32_t scount = 0, qcount = 0;
        if (lane == 0) prefetch_tmap(tm);
        for (int item = blockIdx.x; item < p.n_items && !abort; item += gridDim.x) {
            const ItemPlan it = plan_item<C, WIN>(item, p);
            if (!it.active || !it.seq_ok || it.n_stages == 0) continue;
            if (pw == 0) {
                if (qcount >= 1 && !mbar_wait_bounded(bar_qstg_empty, (qcount - 1) & 1u, kWaitLimitNs)) {
                    abort = true;
                    break;
                }
                const int nrows = it.m_end - it.m0;
                if (lane == 0) mbar_arrive_expect_tx(bar_qstg_full, (uint32_t)(nrows * C::D * 2));
                __syncwarp();
                const uint32_t qdst = base + C::OFF_QSTG;
                for (int i = lane; i < nrows; i += 32) {
                    const int m = it.m0 + i;
                    const int r = m / p.ratio, hl = m - r * p.ratio;
                    const __nv_bfloat16* src =
                        p.q + (((long long)it.g * p.rows + r) * p.n_head + it.kvh * p.ratio + hl) * C::D;
                    bulk_load(qdst + i * C::D * 2, src, C::D * 2, bar_qstg_full);
                }
                ++qcount;
            }
            const int P = p.page_size;
            const int ppt = C::BK / P;    // pages per tile
            const int page_hi = (it.k1 + P - 1) / P;
            const int page_lo = WIN ? it.klo / P : 0;
            const int32_t* trow = p.page_table + (long long)it.g * p.pages_per_seq;
            int batch0 = -1 << 30;
            int my_pg = 0;
            float my_ks = 1.f, my_vs = 1.f;
            bool my_bad = false;
            for (int st = 0; st < it.n_stages; ++st) {
                const int key0 = it.k0 + st * C::BK;
                const int pstart = key0 / P;
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
                        if (pw == 0) {
                            my_ks = __ldg(p.k_scales + my_pg);
                            my_vs = __ldg(p.v_scales + my_pg);
                        }
                    }
                }
                const uint32_t slot = scount % C::NS, use = scount / C::NS;
                if (use >= 1 && !mbar_wait_bounded(bar_empty + 8 * slot, (use - 1) & 1u, kWaitLimitNs)) {
                    abort = true;
                    break;
                }
                const uint32_t tile = base + C::OFF_STG + slot * C::STG_BYTES + pw * C::STG_TILE;
                // lane i < ppt: page i of the tile (its id, scales and flag in one shuffle each)
                const int pi = pstart + lane;
                const int srcl = (pstart - batch0 + lane) & 31;
                const int pg = __shfl_sync(0xffffffffu, my_pg, srcl);
                const bool mine = lane < ppt;
                const bool live = mine && (!WIN || pi >= page_lo) && pi < page_hi;
                if (pw == 0) {
                    // the tile's page scales and page-id flag, released by the arrive below
                    const float ksl = __shfl_sync(0xffffffffu, my_ks, srcl);
                    const float vsl = __shfl_sync(0xffffffffu, my_vs, srcl);
                    const bool badl = __shfl_sync(0xffffffffu, (uint32_t)my_bad, srcl) != 0u;
                    const bool bad_any = __any_sync(0xffffffffu, mine && pi < page_hi && badl);
                    // each of lanes 0 .. MAXPG-1 releases its own entries with its arrive
                    float* meta = reinterpret_cast<float*>(smem + C::OFF_META + slot * C::META_STRIDE);
                    if (lane < C::MAXPG) {
                        meta[lane] = ksl;
                        meta[8 + lane] = vsl;
                    }
                    if (lane == 0) reinterpret_cast<uint32_t*>(meta)[16] = bad_any ? kErrPage : 0u;
                    if (lane > 0 && lane < C::MAXPG) mbar_arrive(bar_full + 8 * slot);
                }
                // one 3-D box per page (P rows x 128 bytes of this KV head, 128-byte swizzle,
                // the layout the MMA and the conversion read), issued by lanes 0 .. ppt-1;
                // pages outside the item's range (past the sequence, or below the window)
                // load zeros
                if (lane == 0) mbar_arrive_expect_tx(bar_full + 8 * slot, (uint32_t)C::STG_TILE);
                __syncwarp();
                if (mine)
                    tma_load_3d(tile + (uint32_t)(lane * P * C::ROW), tm, bar_full + 8 * slot, 0, it.kvh,
                                live ? pg * P : oob_tok, pol_kv);
                __syncwarp();
                ++scount;
            }
            if (misc[1]) abort = true;
        }
        // drain: nothing may still be landing in shared memory at exit
        if (lane == 0) {
            const uint32_t first = scount > (uint32_t)C::NS ? scount - C::NS : 0u;
            for (uint32_t c = first; c < scount; ++c)
                mbar_wait_bounded(bar_full + 8 * (c % C::NS), (c / C::NS) & 1u, kWaitLimitNs);
            if (pw == 0 && qcount >= 1) mbar_wait_bounded(bar_qstg_full, (qcount - 1) & 1u, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == C::W_QK) {
        // ===================================================== QK MMA issue
        constexpr uint32_t idesc_qk = umma_idesc_e4m3(128, N);        // A = K, B = Q terms (both K-major)
        const uint32_t q8 = base + C::OFF_Q8;
        uint32_t tcnt = 0, scnt = 0, icnt = 0;
        bool issued = false;
        // Key rows 0 .. 63 of tile tt (an index over all tiles of this CTA; its
        // stage is tt % NS) -> f16 buffer tt & 1, last read by PV(tt - 2).
        const auto convert_qk_half = [&](uint32_t tt, int key0, const ItemPlan& it) -> bool {
            const uint32_t slot = tt % C::NS, vb = tt & 1u;
            bool ok = mbar_wait_bounded(bar_v_full + 8 * slot, (tt / C::NS) & 1u, kWaitLimitNs);
            if (ok && tt >= 2) ok = mbar_wait_bounded(bar_pv_done + 8 * vb, ((tt - 2) >> 1) & 1u, kWaitLimitNs);
            if (!__all_sync(0xffffffffu, ok)) return false;
            convert_v_half<C>(smem, slot, vb, 0, key0, it.klo, it.k1, lane);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar_v16_full + 8 * vb);
                mbar_arrive(bar_v_empty + 8 * slot);
            }
            return true;
        };
        for (int item = blockIdx.x; item < p.n_items && !abort; item += gridDim.x) {
            const ItemPlan it = plan_item<C, WIN>(item, p);
            if (!it.active || !it.seq_ok || it.n_stages == 0) continue;
            const int T = it.n_stages;
            if (!mbar_wait_bounded(bar_q8_full, icnt & 1u, kWaitLimitNs)) {
                abort = true;
                break;
            }
            for (int i = 0; i < T; ++i) {
                const uint32_t tt = tcnt + i, sb = tt % C::NSB;
                const uint32_t slot = (scnt + i) % C::NS, use = (scnt + i) / C::NS;
                // the S buffer was read by the workers NSB tiles ago; the K stage has landed
                if ((tt >= (uint32_t)C::NSB &&
                     !mbar_wait_bounded(bar_s_empty + 8 * sb, ((tt / C::NSB) - 1) & 1u, kWaitLimitNs)) ||
                    !mbar_wait_bounded(bar_k_full + 8 * slot, use & 1u, kWaitLimitNs)) {
                    abort = true;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t kt = base + C::OFF_STG + slot * C::STG_BYTES;
#pragma unroll
                    for (int term = 0; term < C::QTERMS; ++term)
#pragma unroll
                        for (int kk = 0; kk < C::D / 32; ++kk)
                            tc_mma_ss_f8(t_s + N * sb, umma_desc_sw128(kt + kk * 32, 16, 1024),
                                         umma_desc_sw128(q8 + term * C::Q8_TERM + kk * 32, 16, 1024), idesc_qk,
                                         (term > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(bar_s_full + 8 * sb);
                    tc_commit(bar_k_empty + 8 * slot);
                    issued = true;
                }
                __syncwarp();
                // key rows 0 .. 63 of the previous tile of the item (its f16 buffer was
                // freed by PV(tt - 3)), and at the item's last tile of this one too (freed
                // by PV(tt - 2)), so no PV waits for the next item's first QK; converting
                // tile tt itself here would hold QK(tt + 1) until PV(tt - 2) is done
                if ((i >= 1 && !convert_qk_half(tt - 1, it.k0 + (i - 1) * C::BK, it)) ||
                    (i == T - 1 && !convert_qk_half(tt, it.k0 + i * C::BK, it))) {
                    abort = true;
                    break;
                }
            }
            tcnt += T;
            scnt += T;
            ++icnt;
            if (misc[1]) abort = true;
        }
        // every MMA this thread issued is complete before TMEM is released
        if (lane == 0 && issued) {
            tc_commit(bar_final);
            mbar_wait_bounded(bar_final, 0, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == C::W_PV) {
        // ===================================================== PV MMA issue
        constexpr uint32_t idesc_pv = umma_idesc_f16(128, N, 1, 0);   // A = V^T (MN-major), B = P^T (K-major)
        uint32_t tcnt = 0, icnt = 0;
        bool issued = false;
        for (int item = blockIdx.x; item < p.n_items && !abort; item += gridDim.x) {
            const ItemPlan it = plan_item<C, WIN>(item, p);
            if (!it.active || !it.seq_ok || it.n_stages == 0) continue;
            const int T = it.n_stages;
            for (int j = 0; j < T; ++j) {
                const uint32_t tt = tcnt + j, b = tt & 1u;
                // key rows 64 .. 127 of V_j -> f16 buffer b (last read by PV(tt - 2)) while
                // the workers run the softmax of tile j
                const uint32_t slot = tt % C::NS, use = tt / C::NS;
                bool ok = mbar_wait_bounded(bar_v_full + 8 * slot, use & 1u, kWaitLimitNs);
                if (ok && tt >= 2) ok = mbar_wait_bounded(bar_pv_done + 8 * b, ((tt - 2) >> 1) & 1u, kWaitLimitNs);
                if (!__all_sync(0xffffffffu, ok)) {
                    abort = true;
                    break;
                }
                convert_v_half<C>(smem, slot, b, 2, it.k0 + j * C::BK, it.klo, it.k1, lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_v_empty + 8 * slot);
                if (!mbar_wait_bounded(bar_p_full + 8 * b, (tt >> 1) & 1u, kWaitLimitNs) ||
                    !mbar_wait_bounded(bar_v16_full + 8 * b, (tt >> 1) & 1u, kWaitLimitNs) ||
                    (j == 0 && icnt >= 1 && !mbar_wait_bounded(bar_o_free, (icnt - 1) & 1u, kWaitLimitNs))) {
                    abort = true;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t pt = base + C::OFF_P + b * C::P_BYTES;
                    const uint32_t vt = base + C::OFF_V16 + b * C::F16_TILE;
#pragma unroll
                    for (int kk = 0; kk < C::BK / 16; ++kk) {
                        const uint64_t ad = umma_desc_sw128(vt + kk * 16 * 128, C::ATOM, 1024);
                        const uint64_t bd = umma_desc_sw128(pt + (kk >> 2) * C::PATOM + (kk & 3) * 32, 16, 1024);
                        tc_mma_ss(t_o, ad, bd, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(bar_pv_done + 8 * b);
                    issued = true;
                }
                __syncwarp();
            }
            if (abort) break;
            tcnt += T;
            ++icnt;
            if (misc[1]) abort = true;
        }
        if (lane == 0 && issued) {
            tc_commit(bar_final + 8);
            mbar_wait_bounded(bar_final + 8, 0, kWaitLimitNs);
        }
        __syncwarp();
    } else {
        // ===================================================== workers
        constexpr int V = C::V;
        constexpr int NWT = C::NWT;
        const int t = threadIdx.x;                 // 0 .. NWT-1
        const int k = t & 127;                     // key slot / TMEM lane / head-dim element
        const int h = t >> 7;                      // group of the query rows: rows h*V .. h*V+V-1
        const int wq = warp & 3;                   // TMEM lane quarter
        const int col0 = h * V;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        uint8_t* const q8p = smem + C::OFF_Q8;
        float* const isq = reinterpret_cast<float*>(smem + C::OFF_ISQ);
        uint32_t* const tmw = reinterpret_cast<uint32_t*>(smem + C::OFF_TMW);
        float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
        // P^T store offsets of key slot k for the 8 swizzle phases of a row q
        uint32_t poff[8];
#pragma unroll
        for (int qq = 0; qq < 8; ++qq)
            poff[qq] = (uint32_t)((k >> 6) * C::PATOM + ((((k & 63) >> 3) ^ qq) << 4) + (k & 7) * 2);
        uint32_t scount = 0, qcount = 0, tcnt = 0;
        // A time-out seen by this thread; published to the other workers at the
        // next barrier they all reach, where all worker warps leave together.
        bool lab = false;
        uint32_t icnt = 0;
        // Items that need no pipeline (an invalid sequence length: zero rows; a
        // later split none of whose keys the tile's rows see: an empty partial)
        // are written as they are met; returns the next item that does need it.
        const auto next_real = [&](int item, int L_first) -> int {
            for (; item < p.n_items; item += gridDim.x, L_first = -1) {
                const ItemPlan it = plan_item<C, WIN>(item, p, L_first);
                if (!it.active) continue;
                if (!it.seq_ok) {
                    for (int idx = t; idx < (it.m_end - it.m0) * C::D; idx += NWT) {
                        const int m = it.m0 + idx / C::D, d = idx % C::D;
                        const int r = m / p.ratio, hl = m - r * p.ratio;
                        p.out[(((long long)it.g * p.rows + r) * p.n_head + it.kvh * p.ratio + hl) * C::D + d] =
                            __float2bfloat16_rn(0.f);
                    }
                    if (t == 0 && p.err_word) atomicOr(p.err_word, kErrSeqLen);
                    continue;
                }
                const int nrows = it.m_end - it.m0;
                if (it.n_stages == 0) {
                    // A later split none of whose keys this query tile's rows see
                    // (never the tile's first split): an empty partial.
                    const long long gq = ((long long)it.g * p.n_head_kv + it.kvh) * p.n_qtiles + it.qt;
                    const long long slot_idx = gq * p.max_splits + it.s;
                    float* pacc = p.part_acc + slot_idx * p.qtv * C::D;
                    float* pml = p.part_ml + slot_idx * p.qtv * 2;
                    for (int q = h; q < nrows; q += C::G) __stcg(pacc + q * C::D + k, 0.f);
                    if (t < nrows) __stcg(reinterpret_cast<float2*>(pml) + t, make_float2(-CUDART_INF_F, 0.f));
                    if (t == 0) __stcg(p.part_flag + slot_idx, 0u);
                    continue;
                }
                return item;
            }
            return p.n_items;
        };
        // The query rows of an item, split into e4m3 terms for its QK MMAs
        // (the previous item's QKs are all done: its S tiles were read).
        const auto convert_q = [&](const ItemPlan& it) {
            const int nrows = it.m_end - it.m0;
            {
                if (!lab && !mbar_wait_bounded(bar_qstg_full, qcount & 1u, kWaitLimitNs)) lab = true;
                const uint8_t* qs = smem + C::OFF_QSTG;
                // 16 threads (a half-warp) per row, 8 head-dim elements each
                for (int i = t; i < N * 16; i += NWT) {
                    const int row = i >> 4, ch = i & 15;
                    float f[8];
                    float amax = 0.f;
                    if (row < nrows && !lab) {
                        const uint4 v = *reinterpret_cast<const uint4*>(qs + row * (C::D * 2) + ch * 16);
                        const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            f[2 * e] = bf16_lo(x[e]);
                            f[2 * e + 1] = bf16_hi(x[e]);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = 0.f;
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
#pragma unroll
                    for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                    // 2^k with amax * 2^k in [128, 256): k = 7 - floor(log2 amax), kept a normal float
                    const int ex = amax > 0.f ? (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127 : 7;
                    const int kx = max(-126, min(127, 7 - ex));
                    const float sq = __uint_as_float((uint32_t)(kx + 127) << 23);
                    uint32_t w[2][2];
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        const float v0 = f[e] * sq, v1 = f[e + 1] * sq;
                        const uint32_t hi = f32x2_to_e4m3x2(v0, v1);
                        const float2 hv = e4m3x2_to_f32x2(hi);
                        const uint32_t lo = f32x2_to_e4m3x2(v0 - hv.x, v1 - hv.y);
                        const int wi = e >> 2, sh = (e & 3) * 8;
                        if (sh == 0) {
                            w[0][wi] = hi;
                            w[1][wi] = lo;
                        } else {
                            w[0][wi] |= hi << sh;
                            w[1][wi] |= lo << sh;
                        }
                    }
                    // element 8ch of the row: 16-byte chunk ch/2 (swizzled by row & 7), byte 8 (ch & 1)
                    const uint32_t off = row * 128 + ((((uint32_t)ch >> 1) ^ (row & 7)) << 4) + (ch & 1) * 8;
#pragma unroll
                    for (int term = 0; term < C::QTERMS; ++term)
                        *reinterpret_cast<uint2*>(q8p + term * C::Q8_TERM + off) = make_uint2(w[term][0], w[term][1]);
                    if (ch == 0) isq[row] = __uint_as_float((uint32_t)(127 - kx) << 23);
                    if (TREE && ch == 0)
                        tmw[row] = row < nrows ? __ldg(p.tree_mask + (long long)it.g * p.rows + (it.m0 + row) / p.ratio)
                                               : 0u;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar_q8_full);
                    mbar_arrive(bar_qstg_empty);
                }
                ++qcount;
                named_barrier_sync(2, NWT);   // every row's 2^-k visible to all workers
            }
        };
        int cur = next_real(blockIdx.x, -1);
        if (cur < p.n_items) convert_q(plan_item<C, WIN>(cur, p));
        if (lab) misc[2] = 1u;
        named_barrier_sync(2, NWT);
        if (misc[2]) abort = true;
        while (cur < p.n_items && !abort) {
            const ItemPlan it = plan_item<C, WIN>(cur, p);
            const int T = it.n_stages;
            const int nrows = it.m_end - it.m0;
            // the next candidate item's sequence length, loaded now and used after
            // this item's tiles (a dependent load there stalls the item boundary)
            const int cand = cur + gridDim.x;
            const int L_cand = cand < p.n_items ? __ldg(p.seq_lens + item_group(cand, p)) : -1;
            uint32_t bad = 0;
            // pages the group needs that no item of this query tile loads
            if (it.s == it.s_first) {
                const int P_ = p.page_size;
                const int glo = WIN ? first_visible_key(it.L, p.rows, 0, p.window) / P_ : 0;
                const int tlo = it.klo / P_, thi = (it.kmax + P_ - 1) / P_, ghi = (it.L + P_ - 1) / P_;
                const int32_t* trow = p.page_table + (long long)it.g * p.pages_per_seq;
                const int n_below = tlo - glo;
                for (int i = t; i < n_below + (ghi - thi); i += NWT) {
                    const int pi = i < n_below ? glo + i : thi + (i - n_below);
                    const int pg = __ldg(trow + pi);
                    bad |= (pg < 0 || pg >= p.num_pages) ? kErrPage : 0u;
                }
            }
            // every item checks all mask words of its group, so a malformed word
            // zeroes every row of the group: a word holds its own row's bit and
            // no later row's
            if (TREE && t < p.rows) {
                const uint32_t w = __ldg(p.tree_mask + (long long)it.g * p.rows + t);
                if ((w >> t) != 1u) bad |= kErrMask;
            }
            // ---- per query row state of this thread's half (identical across its key slots)
            float mu[V], thr[V], lsum[V];
#pragma unroll
            for (int q = 0; q < V; ++q) {
                mu[q] = 0.f;                 // running max in log2 units (0 while no key was seen)
                thr[q] = -CUDART_INF_F;      // logits above this move the max
                lsum[q] = 0.f;               // this key slot's share of the row sum
            }
            const int nk0 = it.L - p.rows + it.m0 / p.ratio + 1;                    // keys row q=0 sees
            const int klo_last = WIN ? first_visible_key(it.L, p.rows, (it.m_end - 1) / p.ratio, p.window) : 0;
            // Key k's page scales of tile i and the stage's page-id flag, read
            // before the K stage goes back to the producer (which also waits for
            // the QK MMA that reads it).
            float kc_cur = 0.f, vs_cur = 0.f;
            const auto read_scales = [&](int i) {
                const uint32_t slot = (scount + i) % C::NS, use = (scount + i) / C::NS;
                if (!lab && !mbar_wait_bounded(bar_k_full + 8 * slot, use & 1u, kWaitLimitNs)) lab = true;
                const float* meta = reinterpret_cast<const float*>(smem + C::OFF_META + slot * C::META_STRIDE);
                kc_cur = p.scale_log2 * meta[k / p.page_size];
                vs_cur = meta[8 + k / p.page_size];
                bad |= reinterpret_cast<const uint32_t*>(meta)[16];
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_k_empty + 8 * slot);
            };
            // Waits until PV of tile tt (an index over all tiles of this CTA) is done.
            const auto wait_pv = [&](uint32_t tt) {
                if (!lab && !mbar_wait_bounded(bar_pv_done + 8 * (tt & 1u), (tt >> 1) & 1u, kWaitLimitNs)) lab = true;
                tc_fence_after();
            };
            for (int j = 0; j < T; ++j) {
                const uint32_t tt = tcnt + j, b = tt & 1u, sb = tt % C::NSB;
                const int kbase = it.k0 + j * C::BK;
                // S(j) = QK(j) done
                if (!lab && !mbar_wait_bounded(bar_s_full + 8 * sb, (tt / C::NSB) & 1u, kWaitLimitNs)) lab = true;
                tc_fence_after();
                read_scales(j);
                // ---- softmax of key kbase + k against this half's query rows
                uint32_t sv[V];
                tmem_ldV<V>(t_s + N * sb + col0 + lane_off, sv);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_s_empty + 8 * sb);
                const float c_t = kc_cur, vs_t = vs_cur;
                float sc[V];   // logit scale of each of this half's rows: page K scale x scale x 2^-k_row
#pragma unroll
                for (int q = 0; q < V; q += 4) {
                    const float4 f = *reinterpret_cast<const float4*>(isq + col0 + q);
                    sc[q] = c_t * f.x;
                    sc[q + 1] = c_t * f.y;
                    sc[q + 2] = c_t * f.z;
                    sc[q + 3] = c_t * f.w;
                }
                float xs[V];
                // tree rows see every cached key but, of the call's keys, only their paths
                const int n_full = TREE ? it.L - p.rows : nk0;
                const bool full = kbase + C::BK <= it.k1 && kbase + C::BK <= n_full && kbase >= klo_last;
                if (full) {
#pragma unroll
                    for (int q = 0; q < V; ++q) xs[q] = __uint_as_float(sv[q]) * sc[q];
                } else if (TREE) {
                    const int key = kbase + k;
                    const int i = key - (it.L - p.rows);   // the call's key i, or a cached key (< 0)
                    const bool in_item = key >= it.klo && key < it.k1;
#pragma unroll
                    for (int q = 0; q < V; ++q) {
                        const bool vis = in_item && (i < 0 || ((tmw[col0 + q] >> i) & 1u));
                        xs[q] = vis ? __uint_as_float(sv[q]) * sc[q] : -CUDART_INF_F;
                    }
                } else {
                    // key is visible to row q (query row m0+q at position L-R+(m0+q)/ratio)
                    // iff qc <= q < qw; thresholds clamped to [-1, N]
                    const int key = kbase + k;
                    const long long dk = (long long)key - (it.L - p.rows + 1);
                    long long qc = (dk + 1) * p.ratio - it.m0;
                    long long qw = WIN ? (dk + p.window + 1) * p.ratio - it.m0 : (long long)N;
                    qc = qc < -1 ? -1 : (qc > N ? N : qc);
                    qw = qw < -1 ? -1 : (qw > N ? N : qw);
                    const bool in_item = key >= it.klo && key < it.k1;
                    const int qci = in_item ? (int)qc - col0 : V, qwi = (int)qw - col0;
#pragma unroll
                    for (int q = 0; q < V; ++q)
                        xs[q] = (q >= qci && q < qwi) ? __uint_as_float(sv[q]) * sc[q] : -CUDART_INF_F;
                }
                bool trig = false;
#pragma unroll
                for (int q = 0; q < V; ++q) trig |= xs[q] > thr[q];
                if (lab) misc[2] = 1u;
                const bool any_trig = named_barrier_or(2, NWT, trig);
                if (misc[2]) {
                    abort = true;
                    break;
                }
                if (any_trig) {
                    // tile max per row; a row's max moves only past 2^8 (or on its first keys)
                    float v[V], mx[V];
#pragma unroll
                    for (int q = 0; q < V; ++q) v[q] = xs[q];
                    workers_reduce<V, NWT, true>(v, mx, red, wq, h, lane, k);
                    float alpha[V];
                    bool moved_any = false;
#pragma unroll
                    for (int q = 0; q < V; ++q) {
                        const bool first = thr[q] == -CUDART_INF_F;
                        const bool mv = first ? mx[q] != -CUDART_INF_F : mx[q] > thr[q];
                        alpha[q] = 1.f;
                        if (mv) {
                            alpha[q] = first ? 0.f : exp2f(mu[q] - mx[q]);
                            mu[q] = mx[q];
                            thr[q] = mx[q] + kLazyRescaleLog2;
                            lsum[q] *= alpha[q];
                            moved_any = true;
                        }
                    }
                    if (moved_any && j > 0) {
                        // O must hold PV(0 .. j-1) complete before it is rescaled
                        wait_pv(tt - 1);
                        uint32_t ov[V];
                        tmem_ldV<V>(t_o + col0 + lane_off, ov);
#pragma unroll
                        for (int q = 0; q < V; ++q) ov[q] = __float_as_uint(__uint_as_float(ov[q]) * alpha[q]);
                        tmem_stV<V>(t_o + col0 + lane_off, ov);
                        tmem_wait_st();
                    }
                }
                // ---- P^T[key][q] = f16(2^(x - max) * V scale), sums without the V scale;
                // the P buffer was last read by PV(j-2)
                if (j >= 2) wait_pv(tt - 2);
                uint8_t* const pt = smem + C::OFF_P + b * C::P_BYTES;
#pragma unroll
                for (int q = 0; q < V; ++q) {
                    const float pr = exp2f(xs[q] - mu[q]);
                    lsum[q] += pr;
                    *reinterpret_cast<__half*>(pt + poff[q & 7] + (col0 + q) * 128) = __float2half_rn(pr * vs_t);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_p_full + 8 * b);
            }
            if (abort) break;
            // ---- the next item's query rows now, so its QKs run during this epilogue
            const int nxt = next_real(cand, L_cand);
            if (nxt < p.n_items) convert_q(plan_item<C, WIN>(nxt, p, nxt == cand ? L_cand : -1));
            // ---- epilogue: row sums over the 128 key slots, O^T (lane k = head-dim element k)
            wait_pv(tcnt + T - 1);
            float ltot[V];
            workers_reduce<V, NWT, false>(lsum, ltot, red, wq, h, lane, k);
            if (lab) misc[2] = 1u;
            const bool page_bad = named_barrier_or(2, NWT, (bad & kErrPage) != 0);
            if (misc[2]) {
                abort = true;
                break;
            }
            const bool mask_bad = TREE && named_barrier_or(2, NWT, (bad & kErrMask) != 0);
            const bool item_bad = page_bad || mask_bad;
            const uint32_t bad_bits = (page_bad ? kErrPage : 0u) | (mask_bad ? kErrMask : 0u);
            uint32_t ov[V];
            tmem_ldV<V>(t_o + col0 + lane_off, ov);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_o_free);
            const bool final_write = it.n_splits - it.s_first == 1;
            if (final_write) {
                int r = (it.m0 + col0) / p.ratio, hl = (it.m0 + col0) - r * p.ratio;
#pragma unroll
                for (int q = 0; q < V; ++q) {
                    if (col0 + q < nrows) {
                        // acc * (1/l), the combine kernel's form
                        const float o = item_bad ? 0.f : __uint_as_float(ov[q]) * (1.f / ltot[q]);
                        p.out[(((long long)it.g * p.rows + r) * p.n_head + it.kvh * p.ratio + hl) * C::D + k] =
                            __float2bfloat16_rn(o);
                    }
                    if (++hl == p.ratio) {
                        hl = 0;
                        ++r;
                    }
                }
                if (item_bad && t == 0 && p.err_word) atomicOr(p.err_word, bad_bits);
            } else {
                const long long gq = ((long long)it.g * p.n_head_kv + it.kvh) * p.n_qtiles + it.qt;
                const long long slot_idx = gq * p.max_splits + it.s;
                float* pacc = p.part_acc + slot_idx * p.qtv * C::D;
                float* pml = p.part_ml + slot_idx * p.qtv * 2;
#pragma unroll
                for (int q = 0; q < V; ++q) {
                    if (col0 + q < nrows) {
                        __stcg(pacc + (col0 + q) * C::D + k, __uint_as_float(ov[q]));
                        if (k == q)
                            __stcg(reinterpret_cast<float2*>(pml) + col0 + q,
                                   make_float2(ltot[q] == 0.f ? -CUDART_INF_F : mu[q], ltot[q]));
                    }
                }
                if (t == 0) __stcg(p.part_flag + slot_idx, bad_bits);
            }
            scount += T;
            tcnt += T;
            ++icnt;
            cur = nxt;
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

}  // namespace rad
