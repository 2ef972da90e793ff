// Work-item queue of a persistent CTA: a scheduler warp hands the CTA's work
// items to every warp role through a small ring in shared memory.
//
// Items are taken from a counter shared by all CTAs (atomicAdd on a word of
// the workspace, zeroed before the launch), so a CTA that finishes early takes
// more: with a fixed stride over the items, the sequences' different lengths
// leave some CTAs with far more key tiles than others.  The CTA's first item
// is its block index; counter value c names item gridDim.x + c.  Without a
// counter (AttnParams::sched_ctr null) the items are the fixed stride
// blockIdx.x, blockIdx.x + gridDim.x, ...
//
// Only active items (plan_item's `active`) enter the ring; -1 ends it.  Which
// CTA runs an item does not change the item's arithmetic, so every output bit
// is the same either way.
//
// The e4m3 split kernel and the head_dim-256 bf16 build take the items of a
// uniform call with more than two items per SM heaviest first (the host
// decides; the head_dim-128 bf16 build measured slower so):
// item_order_kernel, run just before them, sorts the (split, sequence) pairs
// by the keys of the split (most first) into AttnParams::item_order, and the
// fetch maps position c to item c % (KV heads x query tiles) of pair
// item_order[c / (KV heads x query tiles)] (skipping inactive ones as before).
// Taken in split order instead, the last items handed out were random-length
// last splits of the longest sequences, and the CTAs that drew long ones set
// the kernel's end.
//
// Barriers per ring slot: full (the scheduler's write), empty (every consumer
// warp has read it) and taken (the first consumer, the K producer, has read
// it).  A kernel with a scheduler warp (run) fetches entry m once entry
// m - kRingLead is taken, so the CTA holds at most kRingLead items beyond the
// one its producer loads; a kernel without one lets its K producer fetch and
// publish each entry itself (fetch, publish) after issuing the previous
// item's last tile, while its stages still hold tiles for the consumers.  An
// entry is written once entry m - kRingSlots is empty.  All waits are
// bounded.
#pragma once
#include "attn_tile.cuh"

namespace rad {

constexpr int kRingSlots = 8;
constexpr int kRingLead = 2;
// int32 items[kRingSlots], then full, empty and taken barriers [kRingSlots] each;
// a ring filled by the K producer itself has no taken barriers
constexpr int kRingBytes = kRingSlots * 4 + 3 * kRingSlots * 8;
constexpr int kRingBytesNoTaken = kRingSlots * 4 + 2 * kRingSlots * 8;

struct ItemRing {
    volatile int* items;
    uint32_t full, empty, taken;   // shared-memory addresses of the barrier arrays

    // `at` / `at_addr`: kRingBytes of shared memory, 8-byte aligned
    __device__ ItemRing(uint8_t* at, uint32_t at_addr)
        : items(reinterpret_cast<volatile int*>(at)),
          full(at_addr + kRingSlots * 4),
          empty(at_addr + kRingSlots * 4 + kRingSlots * 8),
          taken(at_addr + kRingSlots * 4 + 2 * kRingSlots * 8) {}

    // One thread, before fence_mbarrier_init: `consumers` warps read every entry;
    // `with_taken`: the ring has its taken barriers (kRingBytes).
    __device__ void init(uint32_t consumers, bool with_taken) const {
        for (int s = 0; s < kRingSlots; ++s) {
            mbar_init(full + 8 * s, 1);
            mbar_init(empty + 8 * s, consumers);
            if (with_taken) mbar_init(taken + 8 * s, 1);
        }
    }

    // A consumer warp (all lanes): entry n of the ring into `item` (-1: no more).
    // `first`: the warp is the K producer, whose reads pace the scheduler.
    // Returns false on a time-out.
    __device__ bool take(uint32_t n, int& item, uint64_t wait_ns, bool first) const {
        const uint32_t s = n % kRingSlots;
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(full + 8 * s, (n / kRingSlots) & 1u, wait_ns));
        if (!ok) return false;
        item = items[s];
        __syncwarp();
        if ((threadIdx.x & 31) == 0) {
            mbar_arrive(empty + 8 * s);
            if (first) mbar_arrive(taken + 8 * s);
        }
        return true;
    }

    // Where a CTA's next item comes from: its first item, then the shared
    // counter (or, without one, the fixed stride).
    struct Cursor {
        bool first = true;
        unsigned next_static = blockIdx.x;
    };

    // One thread: the CTA's next item for which keep(item) holds, or -1 once
    // the items run out (or `abort_flag` is set).
    template <class Keep>
    __device__ int fetch_if(const AttnParams& p, Cursor& cur, const volatile uint32_t* abort_flag,
                            const Keep& keep) const {
        while (!*abort_flag) {
            unsigned cand;
            if (!p.sched_ctr) {
                cand = cur.next_static;
                cur.next_static += gridDim.x;
            } else if (cur.first) {
                cand = blockIdx.x;
            } else {
                cand = atomicAdd(p.sched_ctr, 1u) + gridDim.x;
            }
            cur.first = false;
            if (cand >= (unsigned)p.n_items) return -1;
            if (p.item_order) {
                // position cand: item j of the k-th heaviest (split, sequence) pair
                const unsigned per_g = (unsigned)(p.n_head_kv * p.n_qtiles);
                const unsigned k = cand / per_g, j = cand - k * per_g;
                const unsigned pr = (unsigned)__ldg(p.item_order + k);
                const unsigned sp = pr / (unsigned)p.groups, g = pr - sp * (unsigned)p.groups;
                cand = sp * (unsigned)p.groups * per_g + g * per_g + j;
            }
            if (keep((int)cand)) return (int)cand;
        }
        return -1;
    }

    // The split kernels: the CTA's next active item (plan_item's `active`).
    template <class C, bool WIN>
    __device__ int fetch(const AttnParams& p, Cursor& cur, const volatile uint32_t* abort_flag) const {
        return fetch_if(p, cur, abort_flag, [&](int item) { return plan_item<C, WIN>(item, p).active; });
    }

    // One thread: writes entry m once entry m - kRingSlots has been read by
    // every consumer.  Returns false on a time-out.
    __device__ bool publish(uint32_t m, int item, uint64_t wait_ns) const {
        if (m >= (uint32_t)kRingSlots &&
            !mbar_wait_bounded(empty + 8 * (m % kRingSlots), (m / kRingSlots - 1) & 1u, wait_ns))
            return false;
        items[m % kRingSlots] = item;
        mbar_arrive(full + 8 * (m % kRingSlots));
        return true;
    }

    // A scheduler warp's one thread: fills the ring, each entry once entry
    // m - kRingLead has been taken by the first consumer, until the items run
    // out (or `abort_flag` is set), then writes -1.  Returns false on a
    // time-out.
    template <class C, bool WIN>
    __device__ bool run(const AttnParams& p, const volatile uint32_t* abort_flag) const {
        Cursor cur;
        for (uint32_t m = 0;; ++m) {
            if (m >= (uint32_t)kRingLead &&
                !mbar_wait_bounded(taken + 8 * ((m - kRingLead) % kRingSlots),
                                   ((m - kRingLead) / kRingSlots) & 1u, p.wait_ns))
                return false;
            const int item = fetch<C, WIN>(p, cur, abort_flag);
            if (!publish(m, item, p.wait_ns)) return false;
            if (item < 0) return true;
        }
    }
};

constexpr int kOrderThreads = 1024;
constexpr int kOrderBuckets = 64;   // by key tiles: 0 .. 62, and 63 or more

// One CTA, in the stream just before a split kernel of a uniform call (no row
// offsets, no tile map): zeroes the shared item counter and sorts the call's
// (split s, sequence g) pairs heaviest first into p.item_order, as pair ids
// s * groups + g.  A pair's weight is the keys of its split: min(split_len,
// L - s split_len) for a sequence of L keys (0 past its last split), in
// buckets of KS keys; pairs of one bucket come in no particular order.  The
// fetch hands out each pair's items (its KV heads and query tiles) one after
// another, as the split order did, so items reading the same pages still run
// side by side; it still skips inactive items, so the set of items run is the
// same in any order.  The lengths are staged in shared memory and each warp
// makes one shared atomic per bucket its pairs fall in.
template <class C>
__global__ void __launch_bounds__(kOrderThreads) item_order_kernel(const __grid_constant__ AttnParams p) {
    __shared__ uint32_t at[kOrderBuckets];   // counts, then each bucket's next position
    __shared__ int lens[kOrderMaxGroups];
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid < kOrderBuckets) at[tid] = 0u;
    for (int g = tid; g < p.groups; g += kOrderThreads) lens[g] = __ldg(p.seq_lens + g);
    __syncthreads();
    const int n_pairs = p.max_splits * p.groups;
    // bucket 0 holds the heaviest pairs; -1: past the last pair
    const auto bucket_of = [&](int pr) {
        if (pr >= n_pairs) return -1;
        const int sp = pr / p.groups, g = pr - sp * p.groups;
        const int keys = min(p.split_len, max(0, lens[g] - sp * p.split_len));
        return kOrderBuckets - 1 - min((keys + C::KS - 1) / C::KS, kOrderBuckets - 1);
    };
    for (int i0 = 0; i0 < n_pairs; i0 += kOrderThreads) {
        const int b = bucket_of(i0 + tid);
        const unsigned peers = __match_any_sync(0xffffffffu, b);
        if (b >= 0 && lane == __ffs(peers) - 1) atomicAdd(&at[b], (uint32_t)__popc(peers));
    }
    __syncthreads();
    if (tid == 0) {
        uint32_t sum = 0;
        for (int b = 0; b < kOrderBuckets; ++b) {
            const uint32_t n = at[b];
            at[b] = sum;
            sum += n;
        }
        p.sched_ctr[0] = 0u;
    }
    __syncthreads();
    for (int i0 = 0; i0 < n_pairs; i0 += kOrderThreads) {
        const int pr = i0 + tid;
        const int b = bucket_of(pr);
        const unsigned peers = __match_any_sync(0xffffffffu, b);
        const int leader = __ffs(peers) - 1;
        uint32_t pos = 0;
        if (b >= 0 && lane == leader) pos = atomicAdd(&at[b], (uint32_t)__popc(peers));
        pos = __shfl_sync(0xffffffffu, pos, leader);
        if (b >= 0) p.item_order[pos + __popc(peers & ((1u << lane) - 1u))] = pr;
    }
}

// The order kernel of a split kernel's launch (C: its config, for KS).
template <class C>
cudaError_t launch_item_order(const AttnParams& p, cudaStream_t st) {
    if (!p.item_order) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(kOrderThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, item_order_kernel<C>, p);
}

}  // namespace rad
