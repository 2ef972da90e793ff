// Host side of the C ABI declared in include/rad_attn.h: argument checks, the
// kernel choice, workspace layout, TMA descriptors and the launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstddef>
#include <cmath>
#include <cstdio>
#include <cstring>

#include "rad_attn.h"
#include "tile_configs.cuh"

namespace {

using rad::AttnParams;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    std::atomic<int> ready{0};
    int sms = 0;
    int cc_major = 0, cc_minor = 0;
};
DeviceInfo g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<int> g_encode_ready{0};

bool is_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------------ call plan
struct Plan {
    int family;
    int split_len;
    int ratio, M, n_qtiles, qtv, max_splits;
    bool ragged;       // items and partial slots run over the call's query tiles (a tile map)
    rad::TileInfo tile;
    long long n_items;
    size_t sched_bytes, map_bytes, flags_bytes, ml_bytes, acc_bytes, total_bytes;
    // A ragged call whose family is the verify or wide tile runs its
    // decode-shaped sequences (at most the decode tile's rows per KV head) on
    // the decode tile instead, as a second tile list: `dec`.  The two tiles
    // share one key schedule, so a row's bits do not depend on which runs it.
    bool dual;
    struct Part {
        rad::TileInfo tile;
        int n_qtiles, qtv;
        long long n_items;
        size_t map_bytes, flags_bytes, ml_bytes, acc_bytes;
    } dec;
};

int check_scalars(int32_t groups, int32_t rows, int32_t n_head, int32_t n_head_kv, int32_t head_dim,
                  int32_t page_size, int32_t pages_per_seq, int32_t kv_dtype) {
    if (groups <= 0 || rows <= 0) return RAD_E_SHAPE;
    if (n_head <= 0 || n_head_kv <= 0 || n_head % n_head_kv != 0) return RAD_E_SHAPE;
    if (pages_per_seq <= 0) return RAD_E_SHAPE;
    if (head_dim != 128 && head_dim != 256) return RAD_E_DTYPE;
    if (page_size != 16 && page_size != 32) return RAD_E_DTYPE;
    if (kv_dtype != RAD_KV_BF16 && kv_dtype != RAD_KV_FP8_E4M3) return RAD_E_DTYPE;
    const long long M = (long long)rows * (n_head / n_head_kv);
    if (M > (1ll << 30) || (long long)groups * rows * n_head > (1ll << 40)) return RAD_E_SHAPE;
    return RAD_OK;
}

rad::TileInfo tile_for(int head_dim, int kv_dtype, int family) {
    const bool fp8 = kv_dtype == RAD_KV_FP8_E4M3;
    if (head_dim == 128) return fp8 ? rad::tile_info<128, true>(family) : rad::tile_info<128, false>(family);
    return fp8 ? rad::tile_info<256, true>(family) : rad::tile_info<256, false>(family);
}

// Prefill chunks (no split) run on the tcgen05 prefill kernels when whole
// query heads tile their 128-row blocks: head_dim 128 or 256, bf16 or fp8 pools.
bool use_prefill_tc(int32_t rows, int32_t ratio, int32_t head_dim, int32_t kv_dtype) {
    const bool dim_ok = head_dim == 128 ||
                        (head_dim == 256 && (kv_dtype == RAD_KV_BF16 ? RAD_PREFILL_TC05_D256 : RAD_PREFILL_FP8_D256));
    return rows > rad::kSplitMaxRows && dim_ok && ratio <= 128 && 128 % ratio == 0;
}

// `general`: a call with ragged rows (cu_seqlens) or tree masks.  Split calls
// (both head dims, both pool types) run on the tcgen05 split kernels whether
// ragged or not, with or without tree masks; longer calls that the prefill
// kernels do not take, on the tile kernels.  `ragged_rows`
// >= 0 marks a ragged call: its work and workspace run
// over the call's query tiles, bounded with the caller's total of rows when
// it gives one (> 0), else with `rows` rows per sequence.
Plan make_plan(int32_t groups, int32_t rows, int32_t n_head, int32_t n_head_kv, int32_t head_dim,
               int32_t page_size, int32_t pages_per_seq, int32_t kv_dtype, bool general = false,
               long long ragged_rows = -1) {
    Plan pl{};
    pl.ratio = n_head / n_head_kv;
    pl.M = rows * pl.ratio;
    // Split calls: the decode tile for <= 8 query rows per KV head, else the
    // verify tile (32 rows per query tile, as many tiles as needed); both
    // share one key schedule.  Longer calls: the tcgen05 prefill kernel where
    // it applies, else the wide tile.
    pl.split_len = rows <= rad::kSplitMaxRows ? rad::kSplitLen : 0;
    const bool ragged = ragged_rows >= 0;
    if (pl.split_len > 0 && kv_dtype == RAD_KV_FP8_E4M3 && (head_dim == 128 ? RAD_SPLIT_TC05 : RAD_SPLIT_TC05_D256)) {
        pl.family = rad::kFamSplitTC;
        pl.split_len = head_dim == 128 ? rad::kSplitLenTC : rad::kSplitLenTC_E4M3_256;
    }
    else if (pl.split_len > 0 && kv_dtype == RAD_KV_BF16 &&
             (head_dim == 128 ? RAD_SPLIT_BF16_TC05 : RAD_SPLIT_BF16_TC05_D256)) {
        pl.family = rad::kFamSplitBf;
        pl.split_len = head_dim == 128 ? rad::kSplitLenBf : rad::kSplitLenTC256;
    }
    else if (pl.split_len > 0)
        pl.family = pl.M <= 8 ? rad::kFamDecode : rad::kFamVerify;
    else
        pl.family = !general && use_prefill_tc(rows, pl.ratio, head_dim, kv_dtype) ? rad::kFamPrefillTC
                                                                                   : rad::kFamWide;
    if (pl.family == rad::kFamPrefillTC)
        pl.tile = rad::TileInfo{head_dim, kv_dtype == RAD_KV_FP8_E4M3 ? 1 : 0, 4, 0, 0,
                                kv_dtype == RAD_KV_FP8_E4M3 ? rad::prefill_fp8_tile_keys(head_dim)
                                                            : rad::prefill_tc05_tile_keys(head_dim),
                                RAD_PREFILL_NSK + RAD_PREFILL_NSV, 128, 256, 0, RAD_PREFILL_CTAS};
    else if (pl.family == rad::kFamSplitTC)
        pl.tile = rad::split_tc05_info(pl.M <= 8, head_dim);
    else if (pl.family == rad::kFamSplitBf)
        pl.tile = rad::split_bf16_tc05_info(pl.M <= 8, head_dim);
    else
        pl.tile = tile_for(head_dim, kv_dtype, pl.family);
    pl.n_qtiles = (pl.M + pl.tile.QT - 1) / pl.tile.QT;
    pl.qtv = pl.M < pl.tile.QT ? pl.M : pl.tile.QT;
    const long long cap_keys = (long long)pages_per_seq * page_size;
    pl.max_splits = pl.split_len > 0 ? (int)((cap_keys + pl.split_len - 1) / pl.split_len) : 1;
    long long n_gq = (long long)groups * n_head_kv * pl.n_qtiles;
    pl.ragged = ragged;
    if (pl.ragged) {
        // sum over sequences of ceil(R_g * ratio / QT) <= ceil(total * ratio / QT) + groups
        long long tiles = (long long)groups * pl.n_qtiles;
        if (ragged_rows > 0) {
            const long long b = (ragged_rows * pl.ratio + pl.tile.QT - 1) / pl.tile.QT + groups;
            if (b < tiles) tiles = b;
        }
        if (tiles > 0x7FFFFFFFll) tiles = 0x7FFFFFFFll;
        pl.n_qtiles = (int)tiles;
        n_gq = tiles * n_head_kv;
        pl.map_bytes = round_up((size_t)tiles * 8, 256);
    }
    pl.n_items = n_gq * pl.max_splits;
    if (pl.split_len > 0) {
        const long long slots = n_gq * pl.max_splits;
        pl.flags_bytes = round_up((size_t)slots * 4, 256);
        pl.ml_bytes = round_up((size_t)slots * pl.qtv * 2 * 4, 256);
        pl.acc_bytes = round_up((size_t)slots * pl.qtv * head_dim * 4, 256);
    }
    // the tcgen05 kernels' shared item counter (zeroed before each launch that uses it); the
    // bf16 prefill kernel deals its items in a fixed snake order instead
    if (pl.family == rad::kFamSplitBf || pl.family == rad::kFamSplitTC ||
        (pl.family == rad::kFamPrefillTC && kv_dtype == RAD_KV_FP8_E4M3))
        pl.sched_bytes = 256;
    // the split kernels' items heaviest first: one int32 an item after the counter
    if (RAD_ITEM_ORDER && (pl.family == rad::kFamSplitBf || pl.family == rad::kFamSplitTC))
        pl.sched_bytes += round_up((size_t)pl.n_items * 4, 256);
    pl.total_bytes = pl.sched_bytes + pl.map_bytes + pl.flags_bytes + pl.ml_bytes + pl.acc_bytes;
    pl.dual = pl.ragged && (pl.family == rad::kFamVerify || pl.family == rad::kFamWide);
    if (pl.dual) {
        Plan::Part& d = pl.dec;
        d.tile = tile_for(head_dim, kv_dtype, rad::kFamDecode);
        // a decode-shaped sequence has one tile of at most QT rows, and at least one row
        long long tiles = groups;
        if (ragged_rows > 0 && ragged_rows < tiles) tiles = ragged_rows;
        d.n_qtiles = (int)tiles;
        d.qtv = d.tile.QT;
        d.n_items = tiles * n_head_kv * pl.max_splits;
        d.map_bytes = round_up((size_t)tiles * 8, 256);
        if (pl.split_len > 0) {
            const long long slots = tiles * n_head_kv * pl.max_splits;
            d.flags_bytes = round_up((size_t)slots * 4, 256);
            d.ml_bytes = round_up((size_t)slots * d.qtv * 2 * 4, 256);
            d.acc_bytes = round_up((size_t)slots * d.qtv * head_dim * 4, 256);
        }
        pl.total_bytes += d.map_bytes + d.flags_bytes + d.ml_bytes + d.acc_bytes;
    }
    return pl;
}

const char* family_name(int f) {
    switch (f) {
        case rad::kFamDecode: return "decode";
        case rad::kFamVerify: return "verify";
        case rad::kFamWide: return "wide";
        case rad::kFamPrefillTC: return "prefill_tc05";
        case rad::kFamSplitBf: return "split_bf16_tc05";
        default: return "split_tc05";
    }
}

int get_encoder() {
    if (g_encode_ready.load(std::memory_order_acquire)) return RAD_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return RAD_E_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    g_encode_ready.store(1, std::memory_order_release);
    return RAD_OK;
}

// Tiled TMA descriptor with 128-byte swizzle over a bf16 or byte (e4m3 code)
// tensor (dims and box innermost first, strides in bytes for dims 1..rank-1).
int encode_map(CUtensorMap* m, CUtensorMapDataType type, const void* ptr, int rank, const cuuint64_t* dims,
               const cuuint64_t* strides, const cuuint32_t* box) {
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(m, type, rank, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? RAD_OK : RAD_E_CUDA;
}
int encode_bf16_map(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                    const cuuint32_t* box) {
    return encode_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr, rank, dims, strides, box);
}

// ------------------------------------------------------------------ device facts
int device_info(int* dev_out, int* sms_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RAD_E_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return RAD_E_DEVICE;
    DeviceInfo& d = g_dev[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        int sms = 0, ma = 0, mi = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&ma, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return RAD_E_CUDA;
        d.sms = sms;
        d.cc_major = ma;
        d.cc_minor = mi;
        d.ready.store(1, std::memory_order_release);
    }
    if (d.cc_major != 10 || d.cc_minor != 3) return RAD_E_DEVICE;
    *dev_out = dev;
    *sms_out = d.sms;
    return RAD_OK;
}

int attn_paged_impl(const void* q, const void* k_pool, const void* v_pool, const int32_t* page_table,
                    const int32_t* seq_lens, int32_t groups, int32_t rows, int32_t n_head, int32_t n_head_kv,
                    int32_t head_dim, int32_t page_size, int32_t pages_per_seq, int32_t num_pages, float scale,
                    int32_t kv_dtype, const float* k_scales, const float* v_scales, int32_t window,
                    const int32_t* cu_seqlens, const uint32_t* tree_mask, int32_t total_rows, void* out,
                    void* workspace, size_t workspace_bytes, uint32_t* err_word, rad_stream_t stream,
                    uint64_t wait_ns = rad::kWaitLimitNs, int fault = rad::kFaultNone);

// Fields of a RadAttnPagedArgs that an older caller's struct_size leaves out read as zero.
template <class T>
T ex_field(const RadAttnPagedArgs* a, const T RadAttnPagedArgs::*field, size_t offset) {
    return a->struct_size >= offset + sizeof(T) ? a->*field : T{};
}

// Common struct_size rules of the ex entry points: RAD_OK, or RAD_E_ARG.
int check_ex_struct(const RadAttnPagedArgs* a) {
    if (!a) return RAD_E_ARG;
    const size_t base = offsetof(RadAttnPagedArgs, err_word) + sizeof(a->err_word);
    if (a->struct_size < base) return RAD_E_ARG;
    if (a->struct_size > sizeof(RadAttnPagedArgs)) {
        // a newer caller: the fields this library does not know must be zero
        const unsigned char* tail = reinterpret_cast<const unsigned char*>(a) + sizeof(RadAttnPagedArgs);
        for (size_t i = 0; i < a->struct_size - sizeof(RadAttnPagedArgs); ++i)
            if (tail[i] != 0) return RAD_E_ARG;
    }
    return RAD_OK;
}

}  // namespace

extern "C" {

size_t rad_attn_paged_workspace_bytes(int32_t groups, int32_t rows, int32_t n_head,
                                      int32_t n_head_kv, int32_t head_dim, int32_t page_size,
                                      int32_t pages_per_seq, int32_t kv_dtype) {
    if (check_scalars(groups, rows, n_head, n_head_kv, head_dim, page_size, pages_per_seq, kv_dtype) !=
        RAD_OK)
        return 0;
    return make_plan(groups, rows, n_head, n_head_kv, head_dim, page_size, pages_per_seq, kv_dtype)
        .total_bytes;
}

int rad_attn_paged(const void* q, const void* k_pool, const void* v_pool, const int32_t* page_table,
                   const int32_t* seq_lens, int32_t groups, int32_t rows, int32_t n_head,
                   int32_t n_head_kv, int32_t head_dim, int32_t page_size, int32_t pages_per_seq,
                   int32_t num_pages, float scale, int32_t kv_dtype, const float* k_scales,
                   const float* v_scales, void* out, void* workspace, size_t workspace_bytes,
                   uint32_t* err_word, rad_stream_t stream) {
    return attn_paged_impl(q, k_pool, v_pool, page_table, seq_lens, groups, rows, n_head, n_head_kv, head_dim,
                           page_size, pages_per_seq, num_pages, scale, kv_dtype, k_scales, v_scales, 0, nullptr,
                           nullptr, 0, out, workspace, workspace_bytes, err_word, stream);
}

int rad_attn_paged_window(const void* q, const void* k_pool, const void* v_pool, const int32_t* page_table,
                          const int32_t* seq_lens, int32_t groups, int32_t rows, int32_t n_head,
                          int32_t n_head_kv, int32_t head_dim, int32_t page_size, int32_t pages_per_seq,
                          int32_t num_pages, float scale, int32_t kv_dtype, const float* k_scales,
                          const float* v_scales, int32_t window, void* out, void* workspace,
                          size_t workspace_bytes, uint32_t* err_word, rad_stream_t stream) {
    return attn_paged_impl(q, k_pool, v_pool, page_table, seq_lens, groups, rows, n_head, n_head_kv, head_dim,
                           page_size, pages_per_seq, num_pages, scale, kv_dtype, k_scales, v_scales, window,
                           nullptr, nullptr, 0, out, workspace, workspace_bytes, err_word, stream);
}

int rad_attn_paged_ex(const RadAttnPagedArgs* a, rad_stream_t stream) {
    const int rc = check_ex_struct(a);
    if (rc != RAD_OK) return rc;
    const int32_t window = ex_field(a, &RadAttnPagedArgs::window, offsetof(RadAttnPagedArgs, window));
    const int32_t* cu = ex_field(a, &RadAttnPagedArgs::cu_seqlens, offsetof(RadAttnPagedArgs, cu_seqlens));
    const uint32_t* tm = ex_field(a, &RadAttnPagedArgs::tree_mask, offsetof(RadAttnPagedArgs, tree_mask));
    const int32_t total = ex_field(a, &RadAttnPagedArgs::total_rows, offsetof(RadAttnPagedArgs, total_rows));
    return attn_paged_impl(a->q, a->k_pool, a->v_pool, a->page_table, a->seq_lens, a->groups, a->rows, a->n_head,
                           a->n_head_kv, a->head_dim, a->page_size, a->pages_per_seq, a->num_pages, a->scale,
                           a->kv_dtype, a->k_scales, a->v_scales, window, cu, tm, total, a->out, a->workspace,
                           a->workspace_bytes, a->err_word, stream);
}

size_t rad_attn_paged_ex_workspace_bytes(const RadAttnPagedArgs* a) {
    if (check_ex_struct(a) != RAD_OK) return 0;
    if (check_scalars(a->groups, a->rows, a->n_head, a->n_head_kv, a->head_dim, a->page_size, a->pages_per_seq,
                      a->kv_dtype) != RAD_OK)
        return 0;
    const bool ragged = ex_field(a, &RadAttnPagedArgs::cu_seqlens, offsetof(RadAttnPagedArgs, cu_seqlens));
    const bool general = ragged || ex_field(a, &RadAttnPagedArgs::tree_mask, offsetof(RadAttnPagedArgs, tree_mask));
    const int32_t total = ex_field(a, &RadAttnPagedArgs::total_rows, offsetof(RadAttnPagedArgs, total_rows));
    if (total < 0) return 0;
    return make_plan(a->groups, a->rows, a->n_head, a->n_head_kv, a->head_dim, a->page_size, a->pages_per_seq,
                     a->kv_dtype, general, ragged ? total : -1)
        .total_bytes;
}

int rad_attn_paged_fault_test(const RadAttnPagedArgs* a, uint64_t wait_limit_ns, int32_t fault,
                              rad_stream_t stream) {
    const int rc = check_ex_struct(a);
    if (rc != RAD_OK) return rc;
    if (wait_limit_ns != 0 && (wait_limit_ns < 1000000ull || wait_limit_ns > rad::kWaitLimitNs)) return RAD_E_ARG;
    if (fault != RAD_FAULT_NONE && fault != RAD_FAULT_SKIP_FIRST_K_TILE) return RAD_E_ARG;
    const int32_t window = ex_field(a, &RadAttnPagedArgs::window, offsetof(RadAttnPagedArgs, window));
    const int32_t* cu = ex_field(a, &RadAttnPagedArgs::cu_seqlens, offsetof(RadAttnPagedArgs, cu_seqlens));
    const uint32_t* tm = ex_field(a, &RadAttnPagedArgs::tree_mask, offsetof(RadAttnPagedArgs, tree_mask));
    const int32_t total = ex_field(a, &RadAttnPagedArgs::total_rows, offsetof(RadAttnPagedArgs, total_rows));
    return attn_paged_impl(a->q, a->k_pool, a->v_pool, a->page_table, a->seq_lens, a->groups, a->rows, a->n_head,
                           a->n_head_kv, a->head_dim, a->page_size, a->pages_per_seq, a->num_pages, a->scale,
                           a->kv_dtype, a->k_scales, a->v_scales, window, cu, tm, total, a->out, a->workspace,
                           a->workspace_bytes, a->err_word, stream, wait_limit_ns ? wait_limit_ns : rad::kWaitLimitNs,
                           fault == RAD_FAULT_SKIP_FIRST_K_TILE ? rad::kFaultSkipFirstKTile : rad::kFaultNone);
}

}  // extern "C"

namespace {

int attn_paged_impl(const void* q, const void* k_pool, const void* v_pool, const int32_t* page_table,
                    const int32_t* seq_lens, int32_t groups, int32_t rows, int32_t n_head, int32_t n_head_kv,
                    int32_t head_dim, int32_t page_size, int32_t pages_per_seq, int32_t num_pages, float scale,
                    int32_t kv_dtype, const float* k_scales, const float* v_scales, int32_t window,
                    const int32_t* cu_seqlens, const uint32_t* tree_mask, int32_t total_rows, void* out,
                    void* workspace, size_t workspace_bytes, uint32_t* err_word, rad_stream_t stream,
                    uint64_t wait_ns, int fault) {
    int rc = check_scalars(groups, rows, n_head, n_head_kv, head_dim, page_size, pages_per_seq, kv_dtype);
    if (rc != RAD_OK) return rc;
    if (num_pages <= 0 || (long long)num_pages * page_size > 0x7FFFFFFFll) return RAD_E_SHAPE;
    if (tree_mask && rows > 32) return RAD_E_SHAPE;   // a mask word covers 32 nodes
    if (total_rows < 0) return RAD_E_ARG;
    const bool general = cu_seqlens || tree_mask;
    const Plan pl = make_plan(groups, rows, n_head, n_head_kv, head_dim, page_size, pages_per_seq, kv_dtype, general,
                              cu_seqlens ? total_rows : -1);
    if (pl.n_items > 0x7FFFFFFFll || (pl.dual && pl.dec.n_items > 0x7FFFFFFFll)) return RAD_E_SHAPE;
    if (!q || !k_pool || !v_pool || !page_table || !seq_lens || !out) return RAD_E_ARG;
    if (!is_aligned(q, 16) || !is_aligned(k_pool, 16) || !is_aligned(v_pool, 16) || !is_aligned(out, 16) ||
        !is_aligned(page_table, 4) || !is_aligned(seq_lens, 4) || !is_aligned(err_word, 4) ||
        !is_aligned(cu_seqlens, 4) || !is_aligned(tree_mask, 4))
        return RAD_E_ARG;
    const bool fp8 = kv_dtype == RAD_KV_FP8_E4M3;
    if (fp8 && (!k_scales || !v_scales || !is_aligned(k_scales, 4) || !is_aligned(v_scales, 4)))
        return RAD_E_ARG;
    if (!std::isfinite(scale) || window < 0) return RAD_E_ARG;
    if (tree_mask && window > 0) return RAD_E_ARG;    // tree rows take no sliding window
    if (pl.total_bytes > 0 && (!workspace || workspace_bytes < pl.total_bytes || !is_aligned(workspace, 256)))
        return RAD_E_WORKSPACE;
    // an injected fault is honoured by the bf16 tcgen05 split kernel only
    if (fault != rad::kFaultNone && (fault != rad::kFaultSkipFirstKTile || pl.family != rad::kFamSplitBf))
        return RAD_E_ARG;

    int dev = 0, sms = 0;
    rc = device_info(&dev, &sms);
    if (rc != RAD_OK) return rc;

    AttnParams p{};
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k_pool = static_cast<const uint8_t*>(k_pool);
    p.v_pool = static_cast<const uint8_t*>(v_pool);
    p.page_table = page_table;
    p.seq_lens = seq_lens;
    p.k_scales = fp8 ? k_scales : nullptr;
    p.v_scales = fp8 ? v_scales : nullptr;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.err_word = err_word;
    p.cu_seqlens = cu_seqlens;
    p.tree_mask = tree_mask;
    p.groups = groups;
    p.rows = rows;
    p.n_head = n_head;
    p.n_head_kv = n_head_kv;
    p.ratio = pl.ratio;
    p.page_size = page_size;
    p.pages_per_seq = pages_per_seq;
    p.num_pages = num_pages;
    p.M = pl.M;
    p.n_qtiles = pl.n_qtiles;
    p.qtv = pl.qtv;
    p.qt_rows = pl.tile.QT;
    p.max_splits = pl.max_splits;
    p.split_len = pl.split_len;
    p.n_items = (int)pl.n_items;
    p.window = window;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.wait_ns = wait_ns;
    p.fault = fault;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // decode-shaped sequences of a dual ragged call: the decode tile's own
    // tile list and partials
    AttnParams pd = p;
    // a kernel with more items than CTAs takes them from a shared counter
    const bool dynamic = RAD_SPLIT_DYNAMIC && pl.sched_bytes > 0 && pl.n_items > sms;
    // ... heaviest first, sorted by an order kernel that also zeroes the counter
    // (uniform calls: the order kernel weighs items by the sequence lengths alone).  Measured
    // same box: the e4m3 kernel gains at both head dims (64 x 8 verify -3 %, 24-sequence decode
    // -10 %) and so does the head_dim-256 bf16 build (-3 %), whose one O buffer makes item
    // boundaries dear; the head_dim-128 bf16 build, with two O buffers, lost ~2 %.  With at
    // most two items per CTA there is no tail to even out, and the order kernel only costs.
    const bool ordered = dynamic && RAD_ITEM_ORDER && !pl.ragged && !cu_seqlens &&
                         groups <= rad::kOrderMaxGroups && pl.n_items > 2LL * sms &&
                         (pl.family == rad::kFamSplitTC || (pl.family == rad::kFamSplitBf && head_dim == 256));
    if (pl.total_bytes > 0) {
        char* ws = static_cast<char*>(workspace);
        if (dynamic) p.sched_ctr = reinterpret_cast<uint32_t*>(ws);
        if (ordered) p.item_order = reinterpret_cast<int32_t*>(ws + 256);
        ws += pl.sched_bytes;
        if (pl.ragged) p.tile_map = reinterpret_cast<const int2*>(ws);
        ws += pl.map_bytes;
        if (pl.split_len > 0) {
            p.part_flag = reinterpret_cast<uint32_t*>(ws);
            p.part_ml = reinterpret_cast<float*>(ws + pl.flags_bytes);
            p.part_acc = reinterpret_cast<float*>(ws + pl.flags_bytes + pl.ml_bytes);
        }
        ws += pl.flags_bytes + pl.ml_bytes + pl.acc_bytes;
        if (pl.dual) {
            const Plan::Part& d = pl.dec;
            pd = p;
            pd.tile_map = reinterpret_cast<const int2*>(ws);
            ws += d.map_bytes;
            if (pl.split_len > 0) {
                pd.part_flag = reinterpret_cast<uint32_t*>(ws);
                pd.part_ml = reinterpret_cast<float*>(ws + d.flags_bytes);
                pd.part_acc = reinterpret_cast<float*>(ws + d.flags_bytes + d.ml_bytes);
            }
            pd.n_qtiles = d.n_qtiles;
            pd.qtv = d.qtv;
            pd.qt_rows = d.tile.QT;
            pd.n_items = (int)d.n_items;
        }
    }
    cudaError_t e;
    if (dynamic && !ordered && cudaMemsetAsync(p.sched_ctr, 0, sizeof(uint32_t), st) != cudaSuccess) return RAD_E_CUDA;
    if (pl.ragged) {
        // the tile lists of the call's sequence classes, on the device
        rad::RaggedMaps m{};
        m.map[0] = const_cast<int2*>(pl.dual ? pd.tile_map : p.tile_map);
        m.qt[0] = pl.dual ? pd.qt_rows : p.qt_rows;
        m.bound[0] = pl.dual ? pd.n_qtiles : p.n_qtiles;
        m.map[1] = pl.dual ? const_cast<int2*>(p.tile_map) : nullptr;
        m.qt[1] = p.qt_rows;
        m.bound[1] = p.n_qtiles;
        m.split_m = pd.qt_rows;
        e = rad::launch_ragged_tile_map(p, m, st);
        if (e != cudaSuccess) return RAD_E_CUDA;
    }
    if (pl.dual) {
        e = head_dim == 128 ? (fp8 ? rad::launch_d128_fp8(rad::kFamDecode, pd, sms, st)
                                   : rad::launch_d128_bf16(rad::kFamDecode, pd, sms, st))
                            : (fp8 ? rad::launch_d256_fp8(rad::kFamDecode, pd, sms, st)
                                   : rad::launch_d256_bf16(rad::kFamDecode, pd, sms, st));
        if (e != cudaSuccess) return RAD_E_CUDA;
    }
    if ((pl.family == rad::kFamPrefillTC && fp8) || pl.family == rad::kFamSplitTC) {
        rc = get_encoder();
        if (rc != RAD_OK) return rc;
        // e4m3 pools viewed as [tokens][n_head_kv][head_dim bytes]: one box = one page of one
        // KV head x 128 bytes (the 128-byte swizzle's span: two boxes a page at head_dim 256)
        const cuuint64_t kd[3] = {(cuuint64_t)head_dim, (cuuint64_t)n_head_kv,
                                  (cuuint64_t)num_pages * (cuuint64_t)page_size};
        const cuuint64_t ks[2] = {(cuuint64_t)head_dim, (cuuint64_t)n_head_kv * head_dim};
        const cuuint32_t kb[3] = {128, 1, (cuuint32_t)page_size};
        CUtensorMap tk, tv;
        if (encode_map(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, k_pool, 3, kd, ks, kb) != RAD_OK ||
            encode_map(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, v_pool, 3, kd, ks, kb) != RAD_OK)
            return RAD_E_CUDA;
        if (pl.family == rad::kFamSplitTC)
            e = head_dim == 128 ? rad::launch_split_tc05(tk, tv, p, sms, st, pl.M <= 8)
                                : rad::launch_split_tc05_d256(tk, tv, p, sms, st);
        else
            e = head_dim == 128 ? rad::launch_prefill_fp8(tk, tv, p, sms, st)
                                : rad::launch_prefill_fp8_d256(tk, tv, p, sms, st);
    } else if (pl.family == rad::kFamSplitBf) {
        rc = get_encoder();
        if (rc != RAD_OK) return rc;
        // pools viewed as [tokens][n_head_kv][head_dim]: one box = one page of one KV head x 64 columns
        const cuuint64_t kd[3] = {(cuuint64_t)head_dim, (cuuint64_t)n_head_kv,
                                  (cuuint64_t)num_pages * (cuuint64_t)page_size};
        const cuuint64_t ks[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)n_head_kv * head_dim * 2};
        const cuuint32_t kb[3] = {64, 1, (cuuint32_t)page_size};
        CUtensorMap tk, tv;
        if (encode_bf16_map(&tk, k_pool, 3, kd, ks, kb) != RAD_OK || encode_bf16_map(&tv, v_pool, 3, kd, ks, kb) != RAD_OK)
            return RAD_E_CUDA;
        e = head_dim == 128 ? rad::launch_split_bf16_tc05(tk, tv, p, sms, st, pl.M <= 8)
                            : rad::launch_split_bf16_tc05_d256(tk, tv, p, sms, st, pl.M <= 8);
    } else if (pl.family == rad::kFamPrefillTC) {
        rc = get_encoder();
        if (rc != RAD_OK) return rc;
        // q viewed as [groups][rows][n_head][head_dim]: one box = 128 query rows
        // (128/ratio tokens x the ratio heads of one KV head) x 64 columns
        const cuuint64_t qd[4] = {(cuuint64_t)head_dim, (cuuint64_t)n_head, (cuuint64_t)rows, (cuuint64_t)groups};
        const cuuint64_t qs[3] = {(cuuint64_t)head_dim * 2, (cuuint64_t)n_head * head_dim * 2,
                                  (cuuint64_t)rows * n_head * head_dim * 2};
        const cuuint32_t qb[4] = {64, (cuuint32_t)pl.ratio, (cuuint32_t)(128 / pl.ratio), 1};
        // pools viewed as [tokens][n_head_kv][head_dim]: one box = one page of one KV head x 64 columns
        const cuuint64_t kd[3] = {(cuuint64_t)head_dim, (cuuint64_t)n_head_kv,
                                  (cuuint64_t)num_pages * (cuuint64_t)page_size};
        const cuuint64_t ks[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)n_head_kv * head_dim * 2};
        const cuuint32_t kb[3] = {64, 1, (cuuint32_t)page_size};
        CUtensorMap tq, tk, tv;
        if (encode_bf16_map(&tq, q, 4, qd, qs, qb) != RAD_OK || encode_bf16_map(&tk, k_pool, 3, kd, ks, kb) != RAD_OK ||
            encode_bf16_map(&tv, v_pool, 3, kd, ks, kb) != RAD_OK)
            return RAD_E_CUDA;
        e = head_dim == 256  ? rad::launch_prefill_tc05_d256(tq, tk, tv, p, sms, st)
            : RAD_PREFILL_PAIR ? rad::launch_prefill_tc05_pair(tq, tk, tv, p, sms, st)
                               : rad::launch_prefill_tc05(tq, tk, tv, p, sms, st);
    } else if (head_dim == 128)
        e = fp8 ? rad::launch_d128_fp8(pl.family, p, sms, st) : rad::launch_d128_bf16(pl.family, p, sms, st);
    else
        e = fp8 ? rad::launch_d256_fp8(pl.family, p, sms, st) : rad::launch_d256_bf16(pl.family, p, sms, st);
    return e == cudaSuccess ? RAD_OK : RAD_E_CUDA;
}

int describe_call(int32_t rows, int32_t n_head, int32_t n_head_kv, int32_t head_dim, int32_t page_size,
                  int32_t kv_dtype, bool general, bool ragged, char* buf, size_t buf_len) {
    const int rc = check_scalars(1, rows, n_head, n_head_kv, head_dim, page_size, 1, kv_dtype);
    if (!buf || buf_len == 0) return rc != RAD_OK ? rc : RAD_E_ARG;
    if (rc != RAD_OK) {
        snprintf(buf, buf_len, "refused: %s", rad_attn_status_string(rc));
        return rc;
    }
    const Plan pl = make_plan(1, rows, n_head, n_head_kv, head_dim, page_size, 1, kv_dtype, general, ragged ? 0 : -1);
    const rad::TileInfo& t = pl.tile;
    // a ragged call first maps its query tiles (one small kernel)
    const char* pre = ragged ? "ragged_tile_map + " : "";
    if (pl.family == rad::kFamSplitTC) {
        snprintf(buf, buf_len,
                 "%sattn_split_tc05 family=%s head_dim=%d kv=fp8e4m3 query_rows_per_kv_head=%d tile_rows=%d "
                 "keys_per_tile=%d stages=%d ctas_per_sm=1 warps=12 4 softmax (a quarter of each tile's keys "
                 "each)+1 qk+1 pv+2 tma producers+4 v converters mma=tcgen05 (query rows as M, four copies; keys "
                 "as N; QK kind::f8f6f4 on the staged e4m3 K with Q as two e4m3 terms, PV kind::f16 with P from "
                 "TMEM and V e4m3 -> f16 once per tile) "
                 "split_len=%d + attn_combine (split order)%s",
                 pre, family_name(pl.family), head_dim, pl.M, t.QT, t.KS, t.NS, pl.split_len,
                 ragged ? "" : "; uniform calls of more than two items per CTA first run item_order (one CTA)");
        return RAD_OK;
    }
    if (pl.family == rad::kFamSplitBf) {
        snprintf(buf, buf_len,
                 "%sattn_split_bf16_tc05 family=%s head_dim=%d kv=bf16 query_rows_per_kv_head=%d tile_rows=%d "
                 "keys_per_tile=%d stages=%d ctas_per_sm=1 warps=13 4 softmax (a quarter of each tile's keys "
                 "each)+1 qk+1 pv+2 tma producers+1 query rows+4 epilogue (%s) mma=tcgen05 (query rows as M, four copies; keys as "
                 "N; QK kind::f16 bf16, PV kind::f16 with P from TMEM as bf16 hi+lo over S) "
                 "split_len=%d + attn_combine (split order)%s",
                 pre, family_name(pl.family), head_dim, pl.M, t.QT, t.KS, t.NS,
                 head_dim == 128 ? "two O buffers" : "one O buffer", pl.split_len,
                 (head_dim == 256 && !ragged)
                     ? "; uniform calls of more than two items per CTA first run item_order (one CTA)"
                     : "");
        return RAD_OK;
    }
    if (pl.family == rad::kFamPrefillTC && kv_dtype == RAD_KV_FP8_E4M3) {
        snprintf(buf, buf_len,
                 "attn_prefill_tc05 family=%s head_dim=%d kv=fp8e4m3 query_rows_per_kv_head=%d tile_rows=128 "
                 "keys_per_tile=%d k_stages=%d v_stages=%d ctas_per_sm=1 warps=4 softmax+1 qk (+ half the v "
                 "convert)+1 pv (+ half the v convert)+2 producers mma=tcgen05 (QK kind::f8f6f4 on the staged e4m3 "
                 "K with Q as two e4m3 terms, PV kind::f16 with V e4m3 -> f16 once per tile and P f16 from TMEM) "
                 "split_len=0",
                 family_name(pl.family), head_dim, pl.M, t.KS, head_dim == 128 ? RAD_PREFILL_FP8_NSK : 3,
                 head_dim == 128 ? RAD_PREFILL_FP8_NSV : 3);
        return RAD_OK;
    }
    if (pl.family == rad::kFamPrefillTC) {
        snprintf(buf, buf_len,
                 "attn_prefill_tc05 family=%s head_dim=%d kv=bf16 query_rows_per_kv_head=%d tile_rows=128 "
                 "keys_per_tile=%d k_stages=%d v_stages=%d ctas_per_sm=%d warps=4 softmax+1 qk+1 pv+2 producers "
                 "mma=tcgen05.kind::f16 (S and O in TMEM, P bf16 hi+lo from TMEM) split_len=0",
                 family_name(pl.family), head_dim, pl.M, pl.tile.KS, RAD_PREFILL_NSK, RAD_PREFILL_NSV,
                 pl.tile.minb);
        return RAD_OK;
    }
    const auto tile_desc = [&](char* b, size_t n, int family, const rad::TileInfo& ti, int rows_kv) {
        return snprintf(b, n,
                        "attn_tile family=%s head_dim=%d kv=%s query_rows_per_kv_head=%d tile_rows=%d "
                        "warps(q=%d,k=%d)+2 producers n_tiles_per_warp=%d keys_per_stage=%d stages=%d split_len=%d "
                        "threads=%d smem=%d ctas_per_sm=%d mma=m16n8k16.%s%s",
                        family_name(family), head_dim, kv_dtype == RAD_KV_FP8_E4M3 ? "fp8e4m3" : "bf16", rows_kv,
                        ti.QT, ti.WQ, ti.WK, ti.NQW, ti.KS, ti.NS, pl.split_len, ti.threads, ti.smem, ti.minb,
                        kv_dtype == RAD_KV_FP8_E4M3 ? "f16" : "bf16",
                        pl.split_len > 0 ? " + attn_combine (split order)" : "");
    };
    int used = snprintf(buf, buf_len, "%s", pre);
    if (pl.dual && used >= 0 && (size_t)used < buf_len) {
        // sequences with at most the decode tile's rows per KV head run on it
        const int k = tile_desc(buf + used, buf_len - used, rad::kFamDecode, pl.dec.tile, pl.dec.tile.QT);
        if (k > 0) used += k;
        if ((size_t)used < buf_len) {
            const int k2 = snprintf(buf + used, buf_len - used, " + ");
            if (k2 > 0) used += k2;
        }
    }
    if (used >= 0 && (size_t)used < buf_len) tile_desc(buf + used, buf_len - used, pl.family, t, pl.M);
    return RAD_OK;
}

}  // namespace

extern "C" {

int rad_attn_paged_describe(int32_t rows, int32_t n_head, int32_t n_head_kv, int32_t head_dim,
                            int32_t page_size, int32_t kv_dtype, char* buf, size_t buf_len) {
    return describe_call(rows, n_head, n_head_kv, head_dim, page_size, kv_dtype, false, false, buf, buf_len);
}

int rad_attn_paged_ex_describe(const RadAttnPagedArgs* a, char* buf, size_t buf_len) {
    const int rc = check_ex_struct(a);
    if (rc != RAD_OK) {
        if (buf && buf_len) snprintf(buf, buf_len, "refused: %s", rad_attn_status_string(rc));
        return rc;
    }
    const bool ragged = ex_field(a, &RadAttnPagedArgs::cu_seqlens, offsetof(RadAttnPagedArgs, cu_seqlens));
    const bool general = ragged || ex_field(a, &RadAttnPagedArgs::tree_mask, offsetof(RadAttnPagedArgs, tree_mask));
    return describe_call(a->rows, a->n_head, a->n_head_kv, a->head_dim, a->page_size, a->kv_dtype, general, ragged,
                         buf, buf_len);
}

const char* rad_attn_status_string(int status) {
    switch (status) {
        case RAD_OK: return "RAD_OK";
        case RAD_E_SHAPE: return "RAD_E_SHAPE";
        case RAD_E_DTYPE: return "RAD_E_DTYPE";
        case RAD_E_ARG: return "RAD_E_ARG";
        case RAD_E_WORKSPACE: return "RAD_E_WORKSPACE";
        case RAD_E_CUDA: return "RAD_E_CUDA";
        case RAD_E_DEVICE: return "RAD_E_DEVICE";
        default: return "RAD_E_UNKNOWN";
    }
}

const char* rad_attn_version(void) { return "rad_attn 0.1.0 sm_103a"; }

}  // extern "C"
