/*
 * rad_attn.h -- C ABI of the paged-KV attention library (GB300, sm_103a).
 *
 * One operation: attention of a batch of query rows against a paged KV cache,
 * the `attn_paged` op of "Radiance architecture plugins -- declaring a model"
 * (section "Declare: the metadata", RadBuildCtx `attn_prefill_fp8`: "pass as
 * attn_paged's prefill_fp8").  The call shapes are those of "kern manifest v7",
 * $defs.Batch: a decode step (`groups` sequences x `rows` = 1), a speculative
 * verify round (`rows` = 8, causal within the round) and a prefill chunk
 * (`groups` = 1, `rows` = the chunk's tokens, over the cached context).
 *
 * Definition (for each group g, row r < rows, query head h < n_head):
 *   kv    = h / (n_head / n_head_kv)                 (grouped-query heads)
 *   n     = seq_lens[g] - rows + r + 1               (keys row r may see)
 *   key j < n is token slot j % page_size of physical page
 *           page_table[g * pages_per_seq + j / page_size]
 *   out[g][r][h][:] = sum_j softmax_j(scale * q[g][r][h][:] . K_j) * V_j
 * with K_j = K[page][slot][kv][:] (times k_scales[page] for fp8) and likewise
 * V.  seq_lens is "each sequence's length after this call (rows already in the
 * state plus this call's)" (kern manifest v7, $defs.Fill `seq_len`), so the
 * K/V rows of this call's own tokens must already be in the pool: writing
 * them (the `slot` fill of $defs.Fill) is the caller's job.
 *
 * Layouts (all row-major, innermost dimension contiguous):
 *   q, out      bf16 [groups][rows][n_head][head_dim]
 *   k_pool      [num_pages][page_size][n_head_kv][head_dim], bf16 or e4m3
 *   v_pool      same layout and dtype as k_pool
 *   page_table  int32 [groups][pages_per_seq]; entries past a sequence's
 *               last page are never read
 *   seq_lens    int32 [groups]
 *   k_scales, v_scales  fp32 [num_pages], fp8 pools only: element value =
 *               e4m3 code * scale of its physical page (one scale per page
 *               and pool, shared by every slot and KV head of the page)
 * The pool layout is the host-allocated paged state of kern manifest v7
 * ($defs.HostTensor / $defs.State `host`: a strided tensor whose outermost
 * extent is the host's page count), with the page table as the input whose
 * domain indexes it with `stride` = page_size token slots per entry
 * ($defs.Domain).
 *
 * Ownership: every pointer is caller-owned device memory (except where a
 * comment says otherwise).  The library allocates nothing, keeps no per-call
 * state, never synchronises the stream and never reads seq_lens or the page
 * table on the host, so a call can be captured in a CUDA graph (kern
 * manifest v7, $defs.Program `graph`: decode and verify programs are
 * replayed from a captured graph).  Work is ordered on `stream`.
 *
 * Row invariance: each output row is a function of its own sequence's data,
 * seq_len and the call's shape scalars (rows, head counts, head_dim,
 * page_size, kv dtype) only -- never of `groups`, of the other sequences or of
 * their order ("Adding a model", step 4: every verified row must equal the
 * decode step's row bit for bit, or speculation is not lossless).
 */
#ifndef RAD_ATTN_H
#define RAD_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's cudaStream_t is `struct CUstream_st *`; NULL is the
 * legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* rad_stream_t;

/* Synchronous status codes.  On any nonzero code nothing was written and
 * nothing was launched, except RAD_E_CUDA (a launch was attempted and the
 * runtime refused it). */
enum {
    RAD_OK = 0,
    RAD_E_SHAPE = 1,     /* groups or rows == 0 ("zero rows is not a call":
                            Radiance architecture plugins, section "Step:
                            issuing the graph"); n_head not a multiple of
                            n_head_kv; a size < 1; num_pages*page_size
                            beyond 2^31-1 */
    RAD_E_DTYPE = 2,     /* head_dim not 128/256, page_size not 16/32, or an
                            unknown kv_dtype: refused by name, never
                            substituted (Radiance architecture plugins,
                            section "Probe": a switch that cannot be honoured
                            is an error, never a silent substitution) */
    RAD_E_ARG = 3,       /* a required pointer is NULL, a pool, q or out
                            pointer is not 16-byte aligned, a non-finite
                            scale, or fp8 without scale arrays */
    RAD_E_WORKSPACE = 4, /* workspace NULL, not 256-byte aligned, or smaller
                            than rad_attn_paged_workspace_bytes() */
    RAD_E_CUDA = 5,      /* the CUDA runtime refused a launch or a query */
    RAD_E_DEVICE = 6     /* the current device is not sm_103 (GB300) */
};

/* KV cache element types ("kern manifest v7", $defs.DType: bf16, fp8e4m3). */
enum { RAD_KV_BF16 = 0, RAD_KV_FP8_E4M3 = 1 };

/* Device-side error bits, OR-ed into *err_word by the kernel ("kern manifest
 * v7", $defs.Fill `error`: a one-word error flag read after every call;
 * nonzero is a failed step).  A group that raises RAD_ERRW_SEQLEN,
 * RAD_ERRW_PAGE or RAD_ERRW_MASK gets all-zero output rows; one that raises
 * RAD_ERRW_CUSEQ gets none written (its rows are unknown); the other groups
 * are unaffected.  No out-of-bounds access happens in any case. */
enum {
    RAD_ERRW_SEQLEN = 1u,  /* seq_lens[g] < rows or > pages_per_seq*page_size */
    RAD_ERRW_PAGE = 2u,    /* a page id the group needs is outside [0, num_pages) */
    RAD_ERRW_QRANGE = 4u,  /* fp8 pools with head_dim 256, calls of more than
                              256 rows whose n_head/n_head_kv does not divide
                              128 (the mma.sync wide tile, which rounds q to
                              f16): a q element beyond the f16 range
                              (|q| > 65504) -- that row's output is not
                              meaningful.  Every other call carries q exactly
                              and never raises it. */
    RAD_ERRW_TIMEOUT = 8u, /* an internal wait ran past its time limit (2 s
                              by default); the kernel unwinds and returns,
                              the affected outputs are not meaningful, and
                              later calls on the stream are unaffected */
    RAD_ERRW_CUSEQ = 16u,  /* ragged rows: cu_seqlens[g] < 0, cu_seqlens[g+1] <
                              cu_seqlens[g], or more rows than `rows` */
    RAD_ERRW_MASK = 32u    /* tree rows: a mask word without its own row's bit,
                              or with the bit of a later row */
};

/*
 * Bytes of scratch memory `rad_attn_paged` needs for a call of this shape
 * (0 is possible).  A pure function of its arguments; no device access.
 * Returns 0 as well for shapes rad_attn_paged would refuse.  The workspace
 * holds per-split partial results ("kern manifest v7", $defs.Impl `scratch`:
 * implementation-private buffers) and, for the tcgen05 split kernels and the
 * fp8 prefill kernel, a work counter that the call zeroes on its stream before
 * the kernel: a 4-byte cudaMemsetAsync, or, where the split kernel takes its
 * items heaviest first, a one-CTA kernel that also writes the item order (one
 * int32 an item, after the counter).  Both are stream-ordered, so they are
 * captured with the call in a CUDA graph.  It is dead between calls; calls
 * that may run concurrently need separate workspaces.
 */
size_t rad_attn_paged_workspace_bytes(int32_t groups, int32_t rows, int32_t n_head,
                                      int32_t n_head_kv, int32_t head_dim, int32_t page_size,
                                      int32_t pages_per_seq, int32_t kv_dtype);

/*
 * Launches the op on `stream`.  Arguments:
 *   q, k_pool, v_pool, page_table, seq_lens, out: device pointers, layouts above
 *   groups        sequences in the call (>= 1)
 *   rows          query rows per sequence (>= 1): 1 decode, 8 verify, the
 *                 chunk length for a prefill
 *   n_head, n_head_kv  query and KV heads (n_head % n_head_kv == 0)
 *   head_dim      128 or 256, as read from the model metadata -- never derived
 *                 from hidden size / heads (Radiance architecture plugins,
 *                 section "Declare: the metadata")
 *   page_size     token slots per page: 16 or 32
 *   pages_per_seq page-table row stride (entries per sequence, >= 1)
 *   num_pages     pages in each pool (bounds for page ids)
 *   scale         logit scale (usually 1/sqrt(head_dim))
 *   kv_dtype      RAD_KV_BF16 or RAD_KV_FP8_E4M3
 *   k_scales, v_scales  fp8: device fp32 [num_pages]; bf16: ignored (may be NULL)
 *   workspace, workspace_bytes  device scratch of at least
 *                 rad_attn_paged_workspace_bytes(...) bytes (may be NULL when
 *                 that is 0); its contents need no initialisation
 *   err_word      optional device uint32 the kernel ORs RAD_ERRW_* bits into
 *                 (the caller zeroes it); NULL disables reporting
 *   stream        CUDA stream (cudaStream_t)
 * Returns RAD_OK or a status code above.
 */
int rad_attn_paged(const void* q, const void* k_pool, const void* v_pool,
                   const int32_t* page_table, const int32_t* seq_lens, int32_t groups,
                   int32_t rows, int32_t n_head, int32_t n_head_kv, int32_t head_dim,
                   int32_t page_size, int32_t pages_per_seq, int32_t num_pages, float scale,
                   int32_t kv_dtype, const float* k_scales, const float* v_scales, void* out,
                   void* workspace, size_t workspace_bytes, uint32_t* err_word,
                   rad_stream_t stream);

/*
 * rad_attn_paged_window -- the op over a sliding-window KV group.
 *
 * A RAD_KV_WINDOW group ("Radiance architecture plugins", section "Declare:
 * buffers and KV groups": a KV state bounded by a window) keeps only the last
 * `window` keys of each sequence live.  Row r then sees keys
 *   max(0, n - window) .. n - 1,   n = seq_lens[g] - rows + r + 1
 * instead of 0 .. n - 1; `window` = 0 means no window (exactly rad_attn_paged).
 * Every other argument, layout, status and error bit is that of
 * rad_attn_paged, with two differences that follow from the bound:
 *   - page ids of pages wholly below row 0's window are never read, so the
 *     caller may leave stale or invalid ids there (a recycled page);
 *     RAD_ERRW_PAGE covers only the pages from row 0's first visible key on;
 *   - K/V slots of the first live page below a row's window are never used.
 * The workspace need is rad_attn_paged_workspace_bytes() of the same shape
 * (an upper bound: splits wholly below the window are skipped).
 * A window < 0 returns RAD_E_ARG.  Rows of one position give the same bits
 * in every call shape that shares its window, as rad_attn_paged's rows do.
 */
int rad_attn_paged_window(const void* q, const void* k_pool, const void* v_pool,
                          const int32_t* page_table, const int32_t* seq_lens, int32_t groups,
                          int32_t rows, int32_t n_head, int32_t n_head_kv, int32_t head_dim,
                          int32_t page_size, int32_t pages_per_seq, int32_t num_pages, float scale,
                          int32_t kv_dtype, const float* k_scales, const float* v_scales,
                          int32_t window, void* out, void* workspace, size_t workspace_bytes,
                          uint32_t* err_word, rad_stream_t stream);

/*
 * rad_attn_paged_ex -- every argument of the op in one struct that grows only
 * at its end behind `struct_size` (the ABI rule of "Radiance architecture
 * plugins", section "Declare: drafters, encoders, generators": adding a field
 * does not move the ABI).
 *
 *   struct_size  sizeof(RadAttnPagedArgs) as the caller compiled it.  It must
 *                cover at least the fields up to err_word (the base call);
 *                fields past it take their defaults (window = 0, no
 *                cu_seqlens, no tree_mask).  A struct larger than this
 *                library's is accepted only when the bytes past the fields
 *                it knows are all zero, since a non-zero field it does not
 *                know is a switch it cannot honour (RAD_E_ARG, nothing
 *                launched).
 *   the fields   as in rad_attn_paged / rad_attn_paged_window, and:
 *
 *   cu_seqlens   ragged rows ("kern manifest v7", $defs.Fill `cu_seqlens`:
 *                exclusive prefix sums of rows per sequence, groups + 1
 *                entries; "Radiance architecture plugins", section "Step:
 *                issuing the graph": `q_lens`, `max_q_len`, and the offsets
 *                are absolute into the token operands).  Device int32
 *                [groups + 1], or NULL for `rows` rows per group.  Group g
 *                then has R_g = cu[g+1] - cu[g] rows; its row r is row
 *                cu[g] + r of q and of out (both [*][n_head][head_dim]), sits
 *                at position seq_lens[g] - R_g + r and sees keys up to it.
 *                `rows` is the call's largest R_g (max_q_len): it picks the
 *                kernel and sizes the workspace.  A group with R_g = 0 is
 *                skipped; out rows that no group names are not written.
 *                Entries with cu[g] < 0, R_g < 0 or R_g > rows raise
 *                RAD_ERRW_CUSEQ for the group.  Offsets are read on the
 *                device; the caller guarantees that q and out hold every row
 *                they name.
 *   tree_mask    tree verify ("Adding a model", step 4: forward_tree;
 *                "Radiance architecture plugins", section "Declare:
 *                drafters, encoders, generators": a tree over the
 *                proposals).  Device uint32, one word per q row (indexed like
 *                q's rows), or NULL for causal rows.  A group's R_g rows are
 *                the nodes of a draft tree flattened parents-first, node r's
 *                K/V written at position seq_lens[g] - R_g + r; bit i of node
 *                r's word is set iff node i is r or one of its ancestors.
 *                Row r sees every key below the call's first position plus
 *                the call's keys whose bits are set: a decode over its path.
 *                A chain (bits 0..r) gives the causal call's bits exactly.
 *                Words must hold their own bit and no later node's
 *                (RAD_ERRW_MASK otherwise).  Requires rows <= 32
 *                (RAD_E_SHAPE) and window == 0 (RAD_E_ARG).
 *   total_rows   ragged rows: an upper bound on the call's rows, cu[groups]
 *                - cu[0] (RadBatch `n_tok`, "Radiance architecture plugins",
 *                section "Step: issuing the graph"), known to the host that
 *                built the batch.  The work and the workspace of a ragged
 *                call run over its query tiles, at most
 *                ceil(total_rows * n_head/n_head_kv / tile rows) + groups
 *                of them; 0 sizes them for `rows` rows per sequence
 *                instead.  A call whose offsets hold more rows than the
 *                bound raises RAD_ERRW_CUSEQ and leaves the rows past it
 *                unwritten.  Negative: RAD_E_ARG.  A ragged call first runs a
 *                small kernel that maps its query tiles into the workspace.
 *
 * Calls with cu_seqlens or tree_mask run on the same kernel family as a
 * uniform call of their shape when head_dim is 128 or the pools are bf16 (the
 * tcgen05 split kernels for calls of at most 256 rows), else on the mma.sync
 * tile kernels, so their rows keep the uniform call's bits; their workspace need is
 * rad_attn_paged_ex_workspace_bytes(args), which may differ from
 * rad_attn_paged_workspace_bytes() of the same shape.
 * Returns the status rad_attn_paged_window returns for the same arguments,
 * RAD_E_ARG for a cu_seqlens or tree_mask pointer not 4-byte aligned.
 */
typedef struct RadAttnPagedArgs {
    size_t struct_size;
    const void* q;
    const void* k_pool;
    const void* v_pool;
    const int32_t* page_table;
    const int32_t* seq_lens;
    int32_t groups, rows, n_head, n_head_kv, head_dim, page_size, pages_per_seq, num_pages;
    float scale;
    int32_t kv_dtype;
    const float* k_scales;
    const float* v_scales;
    void* out;
    void* workspace;
    size_t workspace_bytes;
    uint32_t* err_word;
    /* ---- fields added after the base call (defaults when struct_size ends before them) */
    int32_t window;                /* sliding window: each row sees its last `window` keys; 0 = none */
    const int32_t* cu_seqlens;     /* ragged rows: [groups + 1] absolute row offsets; NULL = `rows` each */
    const uint32_t* tree_mask;     /* tree rows: one word per q row; NULL = causal */
    int32_t total_rows;            /* ragged rows: bound on cu[groups] - cu[0]; 0 = unknown */
} RadAttnPagedArgs;

int rad_attn_paged_ex(const RadAttnPagedArgs* args, rad_stream_t stream);

/* Bytes of workspace rad_attn_paged_ex needs for these arguments (pointers
 * are not read; only their presence counts).  0 for arguments it would
 * refuse on shape, dtype or struct_size. */
size_t rad_attn_paged_ex_workspace_bytes(const RadAttnPagedArgs* args);

/* rad_attn_paged_describe for the call these arguments make (the kernels of
 * a ragged or tree call differ from the uniform call's).  Pointers are not
 * read; only their presence counts.  Same buffer rules and results. */
int rad_attn_paged_ex_describe(const RadAttnPagedArgs* args, char* buf, size_t buf_len);

/*
 * rad_attn_paged_fault_test -- a test hook for the time-out path of the
 * device error word ("kern manifest v7", $defs.Fill `error`: a one-word
 * error flag the host reads after the call).
 *
 * Runs the call described by `args` exactly as rad_attn_paged_ex does, with
 * two test-only settings:
 *   wait_limit_ns  the limit of every bounded wait inside the kernels, in
 *                  [1e6, 2e9] ns; 0 keeps the default (2 s).
 *   fault          RAD_FAULT_NONE, or RAD_FAULT_SKIP_FIRST_K_TILE: the K
 *                  producer of the first CTA leaves its first K tile's copy
 *                  unissued, so the waits on that tile run out; the kernel
 *                  then sets RAD_ERRW_TIMEOUT in err_word, unwinds its warp
 *                  roles (copies in flight drained, tensor memory freed) and
 *                  returns, leaving that CTA's rows unwritten.
 * The fault is honoured only by calls that run on the bf16 tcgen05 split
 * kernel (split calls over bf16 pools, either head_dim); any other call
 * with a fault, an unknown fault or a limit outside the range returns
 * RAD_E_ARG and launches nothing.  Nothing here is meant for production use.
 */
enum { RAD_FAULT_NONE = 0, RAD_FAULT_SKIP_FIRST_K_TILE = 1 };

int rad_attn_paged_fault_test(const RadAttnPagedArgs* args, uint64_t wait_limit_ns, int32_t fault,
                              rad_stream_t stream);

/*
 * rad_attn_paged_noalloc -- the same op for callers that cannot allocate.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot obtain device memory at call time: a runtime that plans all of
 * its device memory once, at load time (its own arena, or a framework's
 * caching allocator that owns the device), and code handed only the tensors
 * of the call (a plugin given inputs and outputs but no scratch buffer).
 * For them a per-call cudaMalloc either fails once the arena has reserved
 * the device or breaks the one-time memory plan.
 *
 * Arguments and results are those of rad_attn_paged without `workspace` and
 * `workspace_bytes`: the scratch lives in a library-owned device array of
 * RAD_NOALLOC_SCRATCH_BYTES, which every GPU that loads the library holds
 * until the process exits.  The call allocates nothing (no cudaMalloc, no
 * cudaFree, no allocating library routine).
 *   - A call whose scratch need (rad_attn_paged_workspace_bytes) exceeds
 *     RAD_NOALLOC_SCRATCH_BYTES returns RAD_E_WORKSPACE and launches nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first
 *     call before any stream capture on the device.  The address is kept
 *     per device together with the context it was found in; after a device
 *     reset (or a new primary context) the next call looks it up again, so
 *     that call too should come before any capture.
 *   - Every call shares the one array and leaves its contents behind; no
 *     part of it needs to start at zero (a call reads only what it wrote
 *     earlier in the same call).  Calls
 *     whose executions overlap on the GPU (different streams, or different
 *     host threads without ordering) race on the array and give undefined
 *     results: order them on one stream.
 */
#define RAD_NOALLOC_SCRATCH_BYTES (16u << 20)

int rad_attn_paged_noalloc(const void* q, const void* k_pool, const void* v_pool,
                           const int32_t* page_table, const int32_t* seq_lens, int32_t groups,
                           int32_t rows, int32_t n_head, int32_t n_head_kv, int32_t head_dim,
                           int32_t page_size, int32_t pages_per_seq, int32_t num_pages,
                           float scale, int32_t kv_dtype, const float* k_scales,
                           const float* v_scales, void* out, uint32_t* err_word,
                           rad_stream_t stream);

/*
 * Writes a one-line, NUL-terminated description of the kernel a call of this
 * shape would launch (family, tile, split length, stages) into buf (host
 * memory, buf_len bytes) -- the pattern of "Radiance architecture plugins",
 * section "Verifying a new plugin" (`--debug-graph`: every op, its resolved
 * kernel, and why).  Returns the same status a call of this shape would get
 * from its scalar checks.  No device access.
 */
int rad_attn_paged_describe(int32_t rows, int32_t n_head, int32_t n_head_kv, int32_t head_dim,
                            int32_t page_size, int32_t kv_dtype, char* buf, size_t buf_len);

/* Static, NUL-terminated name of a status code ("RAD_E_SHAPE", ...). */
const char* rad_attn_status_string(int status);

/* Static, NUL-terminated library version string. */
const char* rad_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RAD_ATTN_H */
