// Split combine kernel (sm_103a): merges the per-split partials the tile
// kernel wrote for every (sequence, KV head, query tile) whose context was cut
// into more than one split, and writes the bf16 output rows.
//
// For one output row with partials (m_s, l_s, acc_s), s = s0..n-1 (m in log2
// units, acc unnormalised; s0 > 0 only with a sliding window, when the query
// tile's rows see no key of splits below s0):
//     M = max_s m_s,  out = (sum_s 2^(m_s - M) acc_s) / (sum_s 2^(m_s - M) l_s)
// Sums run in split order, in chunks of CH splits aligned to multiples of CH,
// so a row's bits depend only on its own sequence -- never on the batch
// around it.  A split none of whose keys a row sees has m = -inf, l = 0,
// acc = 0 and adds exact zeros.
#pragma once
#include <cuda_bf16.h>
#include <math_constants.h>

#include <cstdint>

#include "attn_tile.cuh"

namespace rad {

constexpr int kCombineThreads = 128;
constexpr int kCombineCols = 8;     // output rows per CTA
constexpr int kCombineChunk = 128;  // splits staged in shared memory at a time

// One CTA per (sequence, KV head, query tile, group of kCombineCols rows).
template <int D>
__global__ void __launch_bounds__(kCombineThreads) attn_combine_kernel(const __grid_constant__ AttnParams p) {
    constexpr int NT = kCombineThreads, CG = kCombineCols, CH = kCombineChunk, D4 = D / 4;
    constexpr int OWN = (CG * D4 + NT - 1) / NT;
    __shared__ float ml_s[CH * CG * 2];
    __shared__ float w_s[CH * CG];
    __shared__ float st_m[CG], st_l[CG], st_a[CG];
    __shared__ uint32_t bad_bits;

    const int n_cg = (p.qt_rows + CG - 1) / CG;
    const int cgi = blockIdx.x % n_cg;
    const int gq = blockIdx.x / n_cg;                 // (g, kvh, qt), ragged calls (tile, kvh)
    int g, kvh, qt;
    if (p.tile_map) {
        kvh = gq % p.n_head_kv;
        const int2 gm = __ldg(p.tile_map + gq / p.n_head_kv);
        if (gm.x < 0) return;                                                         // past the last tile
        g = gm.x;
        qt = gm.y;
    } else {
        qt = gq % p.n_qtiles;
        kvh = (gq / p.n_qtiles) % p.n_head_kv;
        g = gq / (p.n_qtiles * p.n_head_kv);
    }
    GroupRows gr;
    if (!group_rows(p, g, gr)) return;                                                // no rows named
    const int L = __ldg(p.seq_lens + g);
    if (L < gr.n || (long long)L > (long long)p.pages_per_seq * p.page_size) return;  // zeros already written
    const int ns = (L + p.split_len - 1) / p.split_len;
    const int t_m0 = qt * p.qt_rows;
    const int g_m = gr.n * p.ratio;                                                   // the group's query rows
    if (t_m0 >= g_m) return;
    const int s_first = first_visible_key(L, gr.n, t_m0 / p.ratio, p.window) / p.split_len;
    if (ns - s_first <= 1) return;                                                    // written directly
    const int t_ncol = min(g_m, t_m0 + p.qt_rows) - t_m0;
    const int c0 = cgi * CG;
    const int ncol = min(CG, t_ncol - c0);
    if (ncol <= 0) return;
    const int tid = threadIdx.x;
    const long long slot0 = (long long)gq * p.max_splits;

    if (tid < ncol) {
        st_m[tid] = -CUDART_INF_F;
        st_l[tid] = 0.f;
    }
    if (tid == 0) bad_bits = 0u;
    float4 acc[OWN];
#pragma unroll
    for (int k = 0; k < OWN; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    uint32_t any_bad = 0;
    for (int s0 = s_first; s0 < ns; s0 = (s0 / CH + 1) * CH) {
        const int cn = min((s0 / CH + 1) * CH, ns) - s0;
        __syncthreads();
        for (int i = tid; i < cn * ncol; i += NT) {
            const int s = i / ncol, col = i - s * ncol;
            const float2 v =
                __ldcg(reinterpret_cast<const float2*>(p.part_ml + (slot0 + s0 + s) * p.qtv * 2) + c0 + col);
            ml_s[2 * i] = v.x;
            ml_s[2 * i + 1] = v.y;
        }
        for (int i = tid; i < cn; i += NT) any_bad |= __ldcg(p.part_flag + slot0 + s0 + i);
        __syncthreads();
        if (tid < ncol) {
            const int col = tid;
            float mx = st_m[col];
            for (int s = 0; s < cn; ++s) mx = fmaxf(mx, ml_s[2 * (s * ncol + col)]);
            const float m_use = (mx == -CUDART_INF_F) ? 0.f : mx;
            const float alpha = exp2f(st_m[col] - m_use);
            float l = st_l[col] * alpha;
            for (int s = 0; s < cn; ++s) {
                const float w = exp2f(ml_s[2 * (s * ncol + col)] - m_use);
                w_s[s * ncol + col] = w;
                l += w * ml_s[2 * (s * ncol + col) + 1];
            }
            st_m[col] = mx;
            st_l[col] = l;
            st_a[col] = alpha;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < OWN; ++k) {
            const int e = tid + k * NT;
            if (e < ncol * D4) {
                const int col = e / D4, d4 = e - col * D4;
                const float a = st_a[col];
                float4 r = acc[k];
                r.x *= a;
                r.y *= a;
                r.z *= a;
                r.w *= a;
                const float4* src =
                    reinterpret_cast<const float4*>(p.part_acc + (slot0 + s0) * p.qtv * D) + (c0 + col) * D4 + d4;
                const long long sstride = (long long)p.qtv * D4;
                for (int s = 0; s < cn; s += 8) {
                    float4 v[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        v[i] = (s + i < cn) ? __ldcg(src + (s + i) * sstride) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (s + i < cn) {
                            const float w = w_s[(s + i) * ncol + col];
                            r.x += w * v[i].x;
                            r.y += w * v[i].y;
                            r.z += w * v[i].z;
                            r.w += w * v[i].w;
                        }
                    }
                }
                acc[k] = r;
            }
        }
    }
    if (any_bad) atomicOr(&bad_bits, any_bad);
    const bool bad = __syncthreads_or(any_bad != 0);
#pragma unroll
    for (int k = 0; k < OWN; ++k) {
        const int e = tid + k * NT;
        if (e < ncol * D4) {
            const int col = e / D4, d4 = e - col * D4;
            const float inv = bad ? 0.f : 1.f / st_l[col];
            const int m = t_m0 + c0 + col;
            const int r = m / p.ratio, hl = m - r * p.ratio;
            __nv_bfloat16* o = p.out + ((gr.row0 + r) * p.n_head + kvh * p.ratio + hl) * D + 4 * d4;
            const float4 a = bad ? make_float4(0.f, 0.f, 0.f, 0.f) : acc[k];
            *reinterpret_cast<__nv_bfloat162*>(o) = __floats2bfloat162_rn(a.x * inv, a.y * inv);
            *reinterpret_cast<__nv_bfloat162*>(o + 2) = __floats2bfloat162_rn(a.z * inv, a.w * inv);
        }
    }
    // the partials' flags hold the RAD_ERRW_* bits their items saw
    if (bad && tid == 0 && cgi == 0 && p.err_word) atomicOr(p.err_word, bad_bits);
}

}  // namespace rad
