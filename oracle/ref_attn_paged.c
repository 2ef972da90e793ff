/*
 * Oracle for paged-KV attention (the `attn_paged` op) -- TEST INFRASTRUCTURE.
 *
 * This file is the plain, slow, obviously-correct CPU definition that the CUDA
 * path is checked against.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may build, load or call it.  It shares no code,
 * header, table or constant with the CUDA library, and the library never calls
 * it: there is no CPU fallback anywhere in the product.
 *
 * What it computes, for every selected (group g, row r, query head h):
 *
 *   kv   = h / (n_head / n_head_kv)          grouped-query heads: "Radiance
 *                                            architecture plugins", section
 *                                            "Declare: the metadata" (n_head,
 *                                            n_head_kv read from the metadata)
 *   pos  = seq_len[g] - rows + r             "kern manifest v7", $defs.Fill
 *                                            `seq_len`: each sequence's length
 *                                            after this call, i.e. the rows
 *                                            already in the state plus this
 *                                            call's rows; row r is the r-th of
 *                                            the call's rows
 *   n    = pos + 1                           causal within the call: a row sees
 *                                            the cached keys and the call's
 *                                            rows up to itself ("Adding a
 *                                            model", step 4: every verified row
 *                                            equals the decode step's row)
 *   key j (0 <= j < n) lives in physical page page_table[g][j / page_size],
 *   token slot j % page_size             "kern manifest v7", $defs.Domain
 *                                            `stride` (token slots per page-
 *                                            table entry) and $defs.State
 *                                            `host` (a paged KV cache)
 *   k_j  = dec(K[page][slot][kv][:]) * k_scale[page]   (scale 1 for bf16)
 *   v_j  = dec(V[page][slot][kv][:]) * v_scale[page]
 *   s_j  = scale * <dec(q[g][r][h][:]), k_j>
 *   out  = sum_j softmax(s)_j * v_j
 *
 * With a sliding window W > 0 (a windowed KV group: "Radiance architecture
 * plugins", section "Declare: buffers and KV groups", RAD_KV_WINDOW, state
 * bounded by a window) row r sees only the last W of those keys,
 * j = max(0, pos - W + 1) .. pos; W = 0 means no window.
 *
 * Ragged rows ("kern manifest v7", $defs.Fill `cu_seqlens`: exclusive prefix
 * sums of rows per sequence, groups + 1 entries; "Radiance architecture
 * plugins", section "Step: issuing the graph": `q_lens`, `max_q_len`, and
 * `cu_seqlens` holds absolute offsets into the token operands).  With
 * cu_seqlens given, group g has R_g = cu[g+1] - cu[g] rows, its row r is row
 * cu[g] + r of q (and of the output), and `rows` is the call's max_q_len.
 * Everything above holds with R_g in place of rows.  A group with R_g == 0 has
 * no rows and no error.  An entry with cu[g] < 0, R_g < 0 or R_g > rows makes
 * the group's rows unknowable: error bit CUSEQ, nothing is computed for it.
 *
 * Tree verify ("Adding a model", step 4: forward_tree; "Radiance architecture
 * plugins", section "Declare: drafters, encoders, generators":
 * rad_drafter_tree, a tree over the proposals).  The call's R_g rows are the
 * nodes of a draft tree flattened parents-first; node r's key was written at
 * position L - R_g + r.  With tree_mask given, word tree_mask[row of node r]
 * has bit i set iff node i is node r itself or one of its ancestors, and row
 * r sees the cached keys 0 .. L - R_g - 1 plus the call's keys whose bit is
 * set.  This is a decode over the path from the root to the node: the same
 * keys, in the same order.  A chain (bits 0..r) is the causal case above.
 * A word without bit r, or with a bit above r (a descendant), is an error:
 * bit MASK, the group's rows are zero.  Trees hold at most 32 nodes
 * (rows <= 32) and take no sliding window.
 *
 * everything in IEEE double.  The softmax is the textbook one: subtract the
 * maximum, exponentiate, divide by the sum.  No tiling, no splitting, no
 * reordering beyond that definition.
 *
 * Pool layout: [num_pages][page_size][n_head_kv][head_dim], innermost
 * contiguous, one pool for K and one for V ("kern manifest v7", $defs.HostTensor:
 * a strided host tensor whose outermost extent is the host's page count).
 *
 * Error behaviour (mirrors the op's contract): a group whose seq_len is below
 * its row count or above pages_per_seq*page_size (SEQLEN), whose visible keys
 * name a page outside [0, num_pages) (PAGE), or whose tree mask is malformed
 * (MASK) gets all-zero output rows and sets a bit in the returned error word;
 * a group whose cu_seqlens entries are malformed sets CUSEQ.  "Zero rows is not a call" ("Radiance architecture
 * plugins", section "Step: issuing the graph"): rows == 0 or groups == 0
 * returns ORACLE_E_SHAPE and writes nothing.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

#define ORACLE_KV_BF16 0
#define ORACLE_KV_FP8_E4M3 1

#define ORACLE_OK 0
#define ORACLE_E_SHAPE 1
#define ORACLE_E_DTYPE 2
#define ORACLE_E_ARG 3

#define ORACLE_ERRW_SEQLEN 1u
#define ORACLE_ERRW_PAGE 2u
#define ORACLE_ERRW_CUSEQ 16u
#define ORACLE_ERRW_MASK 32u

/* bfloat16: the upper 16 bits of an IEEE binary32.  Placing the bits there
 * gives the float exactly; widening to double is exact. */
double oracle_bf16_to_f64(uint16_t bits) {
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3 ("fn" variant): 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits.  Exponent field 0 encodes subnormals m * 2^-9.
 * Exponent 15 with mantissa 7 (S.1111.111) is NaN; there is no infinity, so
 * exponent 15 with mantissa 0..6 are ordinary normals up to 448. */
double oracle_e4m3_to_f64(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);             /* m/8 * 2^(1-7) */
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

int oracle_max_threads(void);

typedef struct {
    const uint16_t* q;
    const void* k_pool;
    const void* v_pool;
    const int32_t* page_table;
    const int32_t* seq_lens;
    int32_t groups, rows, n_head, n_head_kv, head_dim, page_size, pages_per_seq, num_pages;
    double scale;
    int32_t kv_dtype;
    const float* k_scales;
    const float* v_scales;
    int32_t window;
    const int32_t* cu_seqlens;   /* NULL: group g has `rows` rows, q row g*rows + r */
    const uint32_t* tree_mask;   /* NULL: causal rows */
} oracle_call;

/* Rows of group g, and the q/output row of its row 0. */
static int64_t group_rows(const oracle_call* c, int32_t g) {
    return c->cu_seqlens ? (int64_t)c->cu_seqlens[g + 1] - c->cu_seqlens[g] : (int64_t)c->rows;
}
static int64_t group_row0(const oracle_call* c, int32_t g) {
    return c->cu_seqlens ? (int64_t)c->cu_seqlens[g] : (int64_t)g * c->rows;
}
static int cu_entry_ok(const oracle_call* c, int32_t g) {
    if (!c->cu_seqlens) return 1;
    const int64_t R = group_rows(c, g);
    return c->cu_seqlens[g] >= 0 && R >= 0 && R <= c->rows;
}

static double pool_elem(const oracle_call* c, const void* pool, int64_t idx) {
    if (c->kv_dtype == ORACLE_KV_BF16) return oracle_bf16_to_f64(((const uint16_t*)pool)[idx]);
    return oracle_e4m3_to_f64(((const uint8_t*)pool)[idx]);
}

/* Checks one group; returns its error bits (0 when the group is valid).  The
 * pages checked are those holding a key some row of the call may see. */
static uint32_t group_error(const oracle_call* c, int32_t g) {
    if (!cu_entry_ok(c, g)) return ORACLE_ERRW_CUSEQ;
    const int64_t R = group_rows(c, g);
    if (R == 0) return 0;                                         /* no rows: nothing to check */
    int64_t L = c->seq_lens[g];
    if (L < R || L > (int64_t)c->pages_per_seq * c->page_size) return ORACLE_ERRW_SEQLEN;
    uint32_t e = 0;
    if (c->tree_mask)
        for (int64_t r = 0; r < R; ++r)
            if ((c->tree_mask[group_row0(c, g) + r] >> r) != 1u) e |= ORACLE_ERRW_MASK;
    int64_t pages = (L + c->page_size - 1) / c->page_size;
    const int64_t n0 = L - R + 1;                                 /* keys seen by row 0 */
    const int64_t lo = (c->window > 0 && n0 > c->window) ? n0 - c->window : 0;
    for (int64_t p = lo / c->page_size; p < pages; ++p) {
        int32_t pg = c->page_table[(int64_t)g * c->pages_per_seq + p];
        if (pg < 0 || pg >= c->num_pages) {
            e |= ORACLE_ERRW_PAGE;
            break;
        }
    }
    return e;
}

/* One output row.  `w` (optional, length >= n) receives the softmax weights. */
static void one_row(const oracle_call* c, int32_t g, int32_t r, int32_t h, double* out, double* w,
                    int64_t* n_keys_out) {
    const int32_t D = c->head_dim;
    const int32_t ratio = c->n_head / c->n_head_kv;
    const int32_t kv = h / ratio;
    const int64_t L = c->seq_lens[g];
    const int64_t R = group_rows(c, g);
    const int64_t n = L - R + r + 1;                             /* keys 0 .. pos */
    const int64_t lo = (c->window > 0 && n > c->window) ? n - c->window : 0;   /* first visible key */
    const int64_t c0 = L - R;                                    /* key of the call's row 0 */
    const uint32_t tm = c->tree_mask ? c->tree_mask[group_row0(c, g) + r] : 0u;
#define VISIBLE(j) ((j) >= lo && (!c->tree_mask || (j) < c0 || ((tm >> ((j) - c0)) & 1u)))
    const uint16_t* qrow = c->q + ((group_row0(c, g) + r) * c->n_head + h) * D;

    double* qd = (double*)malloc(sizeof(double) * (size_t)D);
    double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    for (int32_t d = 0; d < D; ++d) qd[d] = oracle_bf16_to_f64(qrow[d]);

    double m = -INFINITY;
    for (int64_t j = lo; j < n; ++j) {
        if (!VISIBLE(j)) continue;
        int32_t pg = c->page_table[(int64_t)g * c->pages_per_seq + j / c->page_size];
        int64_t slot = j % c->page_size;
        int64_t base = (((int64_t)pg * c->page_size + slot) * c->n_head_kv + kv) * D;
        double ks = (c->kv_dtype == ORACLE_KV_FP8_E4M3) ? (double)c->k_scales[pg] : 1.0;
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d) dot += qd[d] * (pool_elem(c, c->k_pool, base + d) * ks);
        s[j] = c->scale * dot;
        if (s[j] > m) m = s[j];
    }
    double Z = 0.0;
    for (int64_t j = lo; j < n; ++j) {
        if (!VISIBLE(j)) continue;
        s[j] = exp(s[j] - m);
        Z += s[j];
    }
    for (int32_t d = 0; d < D; ++d) out[d] = 0.0;
    for (int64_t j = 0; j < n; ++j)
        if (w) w[j] = 0.0;
    for (int64_t j = lo; j < n; ++j) {
        if (!VISIBLE(j)) continue;
        double wj = s[j] / Z;
        if (w) w[j] = wj;
        int32_t pg = c->page_table[(int64_t)g * c->pages_per_seq + j / c->page_size];
        int64_t slot = j % c->page_size;
        int64_t base = (((int64_t)pg * c->page_size + slot) * c->n_head_kv + kv) * D;
        double vs = (c->kv_dtype == ORACLE_KV_FP8_E4M3) ? (double)c->v_scales[pg] : 1.0;
        for (int32_t d = 0; d < D; ++d) out[d] += wj * (pool_elem(c, c->v_pool, base + d) * vs);
    }
    if (n_keys_out) *n_keys_out = n;
    free(qd);
    free(s);
#undef VISIBLE
}

static int check_call(const oracle_call* c) {
    if (c->groups <= 0 || c->rows <= 0) return ORACLE_E_SHAPE;
    if (c->n_head <= 0 || c->n_head_kv <= 0 || c->n_head % c->n_head_kv != 0) return ORACLE_E_SHAPE;
    if (c->head_dim <= 0 || c->page_size <= 0 || c->pages_per_seq <= 0 || c->num_pages <= 0)
        return ORACLE_E_SHAPE;
    if (c->kv_dtype != ORACLE_KV_BF16 && c->kv_dtype != ORACLE_KV_FP8_E4M3) return ORACLE_E_DTYPE;
    if (!c->q || !c->k_pool || !c->v_pool || !c->page_table || !c->seq_lens) return ORACLE_E_ARG;
    if (c->kv_dtype == ORACLE_KV_FP8_E4M3 && (!c->k_scales || !c->v_scales)) return ORACLE_E_ARG;
    if (c->window < 0) return ORACLE_E_ARG;
    if (c->tree_mask && c->rows > 32) return ORACLE_E_SHAPE;
    if (c->tree_mask && c->window > 0) return ORACLE_E_ARG;
    return ORACLE_OK;
}

/*
 * Computes the selected output rows.  `sel` holds n_sel triples (g, r, h);
 * out is [n_sel][head_dim].  If `weights` is non-null, row i's softmax weights
 * go to weights[i*weights_stride + j] for its visible keys j, and n_keys[i]
 * receives their count.  *err_word receives the OR of the error bits of every
 * group the selection touches.  Rows of an invalid group are zero.
 */
int oracle_attn_paged_rows(const uint16_t* q, const void* k_pool, const void* v_pool,
                           const int32_t* page_table, const int32_t* seq_lens, int32_t groups,
                           int32_t rows, int32_t n_head, int32_t n_head_kv, int32_t head_dim,
                           int32_t page_size, int32_t pages_per_seq, int32_t num_pages, double scale,
                           int32_t kv_dtype, const float* k_scales, const float* v_scales,
                           const int32_t* sel, int64_t n_sel, double* out, double* weights,
                           int64_t weights_stride, int64_t* n_keys, uint32_t* err_word,
                           int32_t n_threads, int32_t window, const int32_t* cu_seqlens,
                           const uint32_t* tree_mask) {
    oracle_call c = {q, k_pool, v_pool, page_table, seq_lens, groups, rows, n_head, n_head_kv,
                     head_dim, page_size, pages_per_seq, num_pages, scale, kv_dtype, k_scales,
                     v_scales, window, cu_seqlens, tree_mask};
    int rc = check_call(&c);
    if (rc != ORACLE_OK) return rc;
    if (!sel || !out) return ORACLE_E_ARG;
    for (int64_t i = 0; i < n_sel; ++i) {
        const int32_t* t = sel + 3 * i;
        if (t[0] < 0 || t[0] >= groups || t[1] < 0 || t[1] >= rows || t[2] < 0 || t[2] >= n_head)
            return ORACLE_E_ARG;
        /* a row past its group's count (the group's entries being valid) names nothing */
        if (cu_entry_ok(&c, t[0]) && t[1] >= group_rows(&c, t[0])) return ORACLE_E_ARG;
    }
    uint32_t* gerr = (uint32_t*)calloc((size_t)groups, sizeof(uint32_t));
    for (int32_t g = 0; g < groups; ++g) gerr[g] = group_error(&c, g);
    uint32_t acc = 0;
    for (int64_t i = 0; i < n_sel; ++i) acc |= gerr[sel[3 * i]];
    if (err_word) *err_word = acc;

    const int nt = n_threads > 0 ? n_threads : oracle_max_threads();
    (void)nt;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int64_t i = 0; i < n_sel; ++i) {
        const int32_t g = sel[3 * i], r = sel[3 * i + 1], h = sel[3 * i + 2];
        double* o = out + i * head_dim;
        double* w = weights ? weights + i * weights_stride : NULL;
        if (gerr[g]) {
            for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
            if (n_keys) n_keys[i] = 0;
            continue;
        }
        int64_t nk = 0;
        one_row(&c, g, r, h, o, w, &nk);
        if (n_keys) n_keys[i] = nk;
    }
    free(gerr);
    return ORACLE_OK;
}

/* Number of OpenMP threads a parallel region would use with n_threads <= 0
 * meaning "all"; reported with the CPU baseline. */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
