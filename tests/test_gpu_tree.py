"""GPU tests of ragged rows (cu_seqlens) and draft-tree rows (tree_mask)
through rad_attn_paged_ex.

Ragged rows: "kern manifest v7", $defs.Fill `cu_seqlens` and "Radiance
architecture plugins", section "Step: issuing the graph" (a mixed step holds
decode rows, verify rounds and prefill chunks side by side; the offsets are
absolute).  Tree rows: "Adding a model", step 4 (forward_tree; every verified
row equals the decode step's row bit for bit).  Expected values come from the
fp64 oracle on the same inputs.  Q rows that no group names are NaN, and the
output starts as a sentinel: rows no group names must stay untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import DevWorkload, as_f64, assert_parity, bf16_tensor, bits
from paged_kv_attention_02_gb300 import binding as b
from paged_kv_attention_02_gb300 import workloads as wl
from paged_kv_attention_02_gb300.workloads import chain, mask_words, random_parents

pytestmark = pytest.mark.gpu

SENTINEL = 0x4242   # bf16 bits of 48.5: never a result of these inputs


def cfg(name, G, R, H, Hkv, D, P, dt, seed, lens, pps):
    return wl.Config(name, G, R, H, Hkv, D, P, dt, seed, lens, pages_per_seq=pps)


# (config, q_lens): every tile family (decode, verify, wide), both head dims
# and pool types, empty sequences, single rows beside full rounds, contexts
# spanning several splits, and chunks past the split limit (no splitting).
RAGGED = {
    "d128_bf16": (cfg("d128_bf16", 6, 8, 32, 8, 128, 16, wl.KV_BF16, 301, "fixed:8,1,700,2100,5000,64", 320),
                  [8, 1, 0, 3, 8, 5]),
    "d128_fp8": (cfg("d128_fp8", 6, 8, 32, 8, 128, 16, wl.KV_FP8_E4M3, 302, "fixed:9,2,3000,1100,16,4100", 260),
                 [7, 2, 8, 1, 0, 8]),
    "d128_bf16_dec": (cfg("d128_bf16_dec", 5, 2, 8, 2, 128, 32, wl.KV_BF16, 303, "fixed:1,2,1500,3300,9", 110),
                      [1, 2, 0, 1, 2]),
    "d256_bf16": (cfg("d256_bf16", 5, 8, 16, 2, 256, 32, wl.KV_BF16, 304, "fixed:9,1200,3000,40,8", 100),
                  [2, 8, 1, 0, 8]),
    "d256_fp8": (cfg("d256_fp8", 4, 6, 16, 2, 256, 16, wl.KV_FP8_E4M3, 305, "fixed:6,2500,33,1000", 160),
                 [6, 1, 5, 3]),
    "chunk_d128": (cfg("chunk_d128", 4, 300, 8, 2, 128, 16, wl.KV_BF16, 306, "fixed:300,1,2000,900", 130),
                   [300, 1, 40, 0]),
    "chunk_fp8_d256": (cfg("chunk_fp8_d256", 3, 260, 4, 1, 256, 32, wl.KV_FP8_E4M3, 307, "fixed:260,1000,3", 40),
                       [260, 17, 3]),
}

# (config, forests?): draft trees of 8, 16 and 32 nodes.
TREES = {
    "t8_d128_bf16": (cfg("t8_d128_bf16", 5, 8, 32, 8, 128, 16, wl.KV_BF16, 311, "fixed:8,40,1100,2500,4000", 260),
                     True),
    "t8_d128_fp8": (cfg("t8_d128_fp8", 5, 8, 32, 8, 128, 16, wl.KV_FP8_E4M3, 312, "fixed:8,900,1030,3000,20", 200),
                    True),
    "t16_d128_bf16_r1": (cfg("t16_d128_bf16_r1", 3, 16, 4, 4, 128, 32, wl.KV_BF16, 313, "fixed:16,600,2100", 70),
                         False),
    "t32_d256_bf16": (cfg("t32_d256_bf16", 3, 32, 8, 2, 256, 32, wl.KV_BF16, 314, "fixed:32,1500,64", 50), True),
    "t16_d256_fp8": (cfg("t16_d256_fp8", 4, 16, 16, 2, 256, 16, wl.KV_FP8_E4M3, 315, "fixed:16,17,2000,700", 130),
                     True),
    "t32_d128_fp8_r8": (cfg("t32_d128_fp8_r8", 3, 32, 64, 8, 128, 16, wl.KV_FP8_E4M3, 316, "fixed:32,800,3000", 190),
                        False),
    # the e4m3 tcgen05 split kernel's 4096-key split boundaries
    "t8_d128_fp8_splits": (cfg("t8_d128_fp8_splits", 4, 8, 32, 8, 128, 16, wl.KV_FP8_E4M3, 317,
                               "fixed:4096,4100,8192,8199", 520), True),
}


@pytest.fixture(scope="module")
def wls():
    cache = {}

    def get(table, name):
        if (table, name) not in cache:
            c = (RAGGED if table == "ragged" else TREES)[name][0]
            w = wl.make_workload(c, poison=True)
            cache[(table, name)] = (w, DevWorkload(w))
        return cache[(table, name)]
    return get


def ragged_q(w, q_lens, base=0, tail=0):
    """Group g's first q_lens[g] query rows packed at base + sum(q_lens[:g]);
    rows no group names hold NaN."""
    c = w.cfg
    cu = (base + np.concatenate([[0], np.cumsum(q_lens)])).astype(np.int32)
    q = np.full((int(cu[-1]) + tail, c.n_head, c.head_dim), wl.BF16_NAN, dtype=np.uint16)
    for g, ql in enumerate(q_lens):
        q[cu[g]:cu[g] + ql] = w.q[g, :ql]
    return q, cu


def tree_masks(w, parents):
    return np.stack([mask_words(pa) for pa in parents]).astype(np.uint32)


def run_general(dw, q_bits, rows, cu=None, mask=None, window=0, lens=None, total_rows=None):
    """One rad_attn_paged_ex call; returns (out bits, err word)."""
    c = dw.w.cfg
    q = bf16_tensor(q_bits)
    out = torch.full(q.shape, 0, dtype=torch.int16, device="cuda")
    out.fill_(SENTINEL)
    out = out.view(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cu_t = None if cu is None else torch.from_numpy(np.asarray(cu, dtype=np.int32)).cuda()
    mask_t = None if mask is None else torch.from_numpy(np.asarray(mask, dtype=np.uint32).view(np.int32)).cuda()
    b.attn_paged_general(q, dw.k, dw.v, dw.table, dw.lens if lens is None else lens, rows=rows,
                         n_head=c.n_head, n_head_kv=c.n_head_kv, head_dim=c.head_dim, page_size=c.page_size,
                         scale=c.scale, kv_dtype=c.kv_dtype, k_scales=dw.ks, v_scales=dw.vs, cu_seqlens=cu_t,
                         tree_mask=mask_t, window=window, total_rows=total_rows, out=out, err_word=err)
    torch.cuda.synchronize()
    return bits(out), int(err.item())


def oracle_general(w, q_bits, rows, cu=None, mask=None, window=0, seq_lens=None):
    args = w.call_args()
    args["rows"] = rows
    return oracle.attn_paged(q_bits, w.k_pool, w.v_pool, w.page_table,
                             w.seq_lens if seq_lens is None else seq_lens, k_scales=w.k_scales,
                             v_scales=w.v_scales, window=window, cu_seqlens=cu, tree_mask=mask, **args)


def as_float(bits_arr):
    return as_f64(torch.from_numpy(bits_arr).view(torch.bfloat16))


def named_rows(cu, n_rows):
    named = np.zeros(n_rows, dtype=bool)
    for g in range(len(cu) - 1):
        named[cu[g]:cu[g + 1]] = True
    return named


# ----------------------------------------------------------------------------- ragged rows

@pytest.mark.parametrize("name", list(RAGGED))
def test_ragged_matches_oracle_and_writes_only_named_rows(wls, name):
    w, dw = wls("ragged", name)
    q_lens = RAGGED[name][1]
    q, cu = ragged_q(w, q_lens, base=3, tail=2)
    got, err = run_general(dw, q, max(q_lens), cu=cu)
    assert err == 0
    ref = oracle_general(w, q, max(q_lens), cu=cu)
    assert ref.err_word == 0
    named = named_rows(cu, q.shape[0])
    assert np.all(got[~named] == np.int16(SENTINEL)), "a row no group names was written"
    assert_parity(as_float(got[named]), ref.out[named], dw.fp8, name)


@pytest.mark.parametrize("name", ["d128_bf16", "d256_fp8", "chunk_d128"])
def test_ragged_windowed_matches_oracle(wls, name):
    w, dw = wls("ragged", name)
    q_lens = RAGGED[name][1]
    q, cu = ragged_q(w, q_lens)
    for W in (1, 37, 1000):
        got, err = run_general(dw, q, max(q_lens), cu=cu, window=W)
        assert err == 0
        ref = oracle_general(w, q, max(q_lens), cu=cu, window=W)
        named = named_rows(cu, q.shape[0])
        assert_parity(as_float(got[named]), ref.out[named], dw.fp8, f"{name} window {W}")


@pytest.mark.parametrize("name", ["d128_bf16", "d128_fp8", "chunk_fp8_d256"])
def test_ragged_rows_are_bit_identical_alone_and_batched(wls, name):
    w, dw = wls("ragged", name)
    q_lens = RAGGED[name][1]
    q, cu = ragged_q(w, q_lens)
    got, _ = run_general(dw, q, max(q_lens), cu=cu)
    rows = max(q_lens)   # the same call shape: the same kernel and key schedule
    for g, ql in enumerate(q_lens):
        if ql == 0:
            continue
        one = w.select_groups([g])
        dwo = DevWorkload(one)
        qo, cuo = ragged_q(one, [ql])
        alone, err = run_general(dwo, qo, rows, cu=cuo)
        assert err == 0
        assert np.array_equal(alone, got[cu[g]:cu[g] + ql]), f"{name}: group {g}"


@pytest.mark.parametrize("name", ["d128_bf16", "d128_bf16_dec", "d128_fp8", "d256_bf16", "d256_fp8"])
def test_ragged_rows_equal_the_uniform_call_bit_for_bit(wls, name):
    """Each group's rows equal a uniform call over that sequence with rows =
    its own count (both on the tile kernels, whose per-row arithmetic and key
    schedule do not depend on the call's width)."""
    w, dw = wls("ragged", name)
    q_lens = RAGGED[name][1]
    q, cu = ragged_q(w, q_lens)
    got, _ = run_general(dw, q, max(q_lens), cu=cu)
    c = w.cfg
    for g, ql in enumerate(q_lens):
        if ql == 0:
            continue
        one = w.select_groups([g])
        dwo = DevWorkload(one)
        out = b.attn_paged(dwo.q[:, :ql].contiguous(), dwo.k, dwo.v, dwo.table, dwo.lens, rows=ql,
                           n_head=c.n_head, n_head_kv=c.n_head_kv, head_dim=c.head_dim, page_size=c.page_size,
                           scale=c.scale, kv_dtype=c.kv_dtype, k_scales=dwo.ks, v_scales=dwo.vs)
        torch.cuda.synchronize()
        assert np.array_equal(bits(out)[0], got[cu[g]:cu[g] + ql]), f"{name}: group {g}"


def test_ragged_malformed_offsets_flag_their_group_and_write_nothing_of_it(wls):
    w, dw = wls("ragged", "d128_bf16")
    q_lens = RAGGED["d128_bf16"][1]
    q, cu = ragged_q(w, q_lens)
    good, _ = run_general(dw, q, 8, cu=cu)
    bad_cu = cu.copy()
    bad_cu[4] = bad_cu[3] - 1            # group 3 ends before it starts; group 4 claims 11 rows
    got, err = run_general(dw, q, 8, cu=bad_cu)
    assert err == b.RAD_ERRW_CUSEQ
    for g in (0, 1, 5):
        assert np.array_equal(got[cu[g]:cu[g + 1]], good[cu[g]:cu[g + 1]]), g
    assert np.all(got[cu[3]:cu[5]] == np.int16(SENTINEL))
    neg = cu.copy()
    neg[0] = -2
    got, err = run_general(dw, q, 8, cu=neg)
    assert err == b.RAD_ERRW_CUSEQ
    assert np.array_equal(got[cu[1]:], good[cu[1]:])


@pytest.mark.parametrize("name", ["d128_fp8", "chunk_d128"])
def test_ragged_row_total_bounds_the_work(wls, name):
    """The exact row total and no total (0: sized for `rows` per sequence)
    give the same bits as q's row count.  A total of one row bounds each tile
    list: the decode tile's (sequences of at most its rows per KV head) to one
    tile, the main tile's to ceil(ratio / tile rows) + groups; past a bound the
    call raises RAD_ERRW_CUSEQ and runs only the list's first tiles, in
    sequence order."""
    w, dw = wls("ragged", name)
    q_lens = RAGGED[name][1]
    q, cu = ragged_q(w, q_lens, base=2, tail=5)
    ref, _ = run_general(dw, q, max(q_lens), cu=cu)
    for total in (int(cu[-1] - cu[0]), 0):
        got, err = run_general(dw, q, max(q_lens), cu=cu, total_rows=total)
        assert err == 0 and np.array_equal(got, ref), total
    c = w.cfg
    ratio = c.n_head // c.n_head_kv
    desc = b.ex_describe(b.shape_args(w.groups, max(q_lens), c.n_head, c.n_head_kv, c.head_dim, c.page_size,
                                      w.pages_per_seq, c.kv_dtype, ragged=True))
    qts = [int(x.split()[0]) for x in desc.split("tile_rows=")[1:]]
    dual = len(qts) == 2
    qt_dec, qt_main = (qts[0], qts[1]) if dual else (None, qts[0])
    G = len(q_lens)
    bounds = {"dec": 1, "main": min(-(-ratio // qt_main) + G, G * -(-max(q_lens) * ratio // qt_main))}
    got, err = run_general(dw, q, max(q_lens), cu=cu, total_rows=1)
    done = {"dec": 0, "main": 0}
    over = False
    for g, ql in enumerate(q_lens):
        if ql == 0:
            continue
        cls = "dec" if dual and ql * ratio <= qt_dec else "main"
        qt = qt_dec if cls == "dec" else qt_main
        tiles = -(-ql * ratio // qt)
        run = max(0, min(tiles, bounds[cls] - done[cls]))
        over |= run < tiles
        rows_run = min(ql, run * qt // ratio)
        a = int(cu[g])
        assert np.array_equal(got[a:a + rows_run], ref[a:a + rows_run]), g
        assert np.all(got[a + rows_run:a + ql] == np.int16(SENTINEL)), g
        done[cls] += tiles
    assert err == (b.RAD_ERRW_CUSEQ if over else 0)


def test_ragged_sequence_shorter_than_its_rows_is_zero_and_flagged(wls):
    w, dw = wls("ragged", "d256_bf16")
    q_lens = RAGGED["d256_bf16"][1]
    q, cu = ragged_q(w, q_lens)
    good, _ = run_general(dw, q, 8, cu=cu)
    lens = dw.lens.clone()
    lens[1] = 7                            # 8 rows over 7 keys
    got, err = run_general(dw, q, 8, cu=cu, lens=lens)
    assert err == b.RAD_ERRW_SEQLEN
    assert np.all(got[cu[1]:cu[2]] == 0)
    keep = named_rows(cu, q.shape[0])
    keep[cu[1]:cu[2]] = False
    assert np.array_equal(got[keep], good[keep])


# ----------------------------------------------------------------------------- tree rows

def tree_inputs(w, forest, seed):
    rng = np.random.default_rng(seed)
    parents = [random_parents(rng, w.cfg.rows, forest=forest) for _ in range(w.groups)]
    return parents, tree_masks(w, parents)


@pytest.mark.parametrize("name", list(TREES))
def test_tree_matches_oracle(wls, name):
    w, dw = wls("tree", name)
    parents, mask = tree_inputs(w, TREES[name][1], 900)
    R = w.cfg.rows
    got, err = run_general(dw, w.q, R, mask=mask.reshape(-1))
    assert err == 0
    ref = oracle_general(w, w.q, R, mask=mask)
    assert ref.err_word == 0
    assert_parity(as_float(got), ref.out, dw.fp8, name)


@pytest.mark.parametrize("name", ["t8_d128_fp8", "t32_d256_bf16"])
def test_ragged_trees_match_oracle(wls, name):
    """Trees of different sizes (and single decode rows) in one call."""
    w, dw = wls("tree", name)
    R = w.cfg.rows
    rng = np.random.default_rng(901)
    q_lens = [int(x) for x in rng.integers(0, R + 1, size=w.groups)]
    q_lens[0] = R
    q, cu = ragged_q(w, q_lens, base=1, tail=1)
    mask = np.zeros(q.shape[0], dtype=np.uint32)
    for g, ql in enumerate(q_lens):
        if ql:
            mask[cu[g]:cu[g] + ql] = mask_words(random_parents(rng, ql))
    got, err = run_general(dw, q, R, cu=cu, mask=mask)
    assert err == 0
    ref = oracle_general(w, q, R, cu=cu, mask=mask)
    named = named_rows(cu, q.shape[0])
    assert np.all(got[~named] == np.int16(SENTINEL))
    assert_parity(as_float(got[named]), ref.out[named], dw.fp8, name)


@pytest.mark.parametrize("name", list(TREES))
def test_chain_mask_equals_the_causal_call_bit_for_bit(wls, name):
    w, dw = wls("tree", name)
    R, G = w.cfg.rows, w.groups
    mask = np.tile(mask_words(chain(R)), G)
    tree, err = run_general(dw, w.q, R, mask=mask)
    assert err == 0
    out, err = dw.run()   # the causal call through rad_attn_paged: the same kernel
    assert err == 0 and np.array_equal(tree, bits(out))


@pytest.mark.parametrize("name", ["t8_d128_bf16", "t32_d256_bf16", "t16_d256_fp8", "t8_d128_fp8",
                                  "t32_d128_fp8_r8"])
def test_chain_prefix_nodes_equal_the_decode_rows_bit_for_bit(wls, name):
    """A node whose ancestors are exactly the nodes before it sits where a
    decode step would, over the same keys: the rows are equal bit for bit."""
    w, dw = wls("tree", name)
    R = w.cfg.rows
    parents, mask = tree_inputs(w, TREES[name][1], 902)
    for pa in parents:   # make a chain prefix of a few nodes in every tree
        pa[1], pa[2], pa[3] = 0, 1, 2
    mask = tree_masks(w, parents)
    got, err = run_general(dw, w.q, R, mask=mask.reshape(-1))
    assert err == 0
    c = w.cfg
    for r in range(R):
        on_chain = [g for g in range(w.groups) if mask[g, r] == (1 << (r + 1)) - 1]
        if not on_chain:
            continue
        out = b.attn_paged(dw.q[:, r:r + 1].contiguous(), dw.k, dw.v, dw.table, dw.lens - R + r + 1, rows=1,
                           n_head=c.n_head, n_head_kv=c.n_head_kv, head_dim=c.head_dim, page_size=c.page_size,
                           scale=c.scale, kv_dtype=c.kv_dtype, k_scales=dw.ks, v_scales=dw.vs)
        torch.cuda.synchronize()
        dec = bits(out)[:, 0]
        for g in on_chain:
            assert np.array_equal(got[g, r], dec[g]), (name, g, r)


@pytest.mark.parametrize("name", ["t8_d128_bf16", "t8_d128_fp8"])
def test_rows_do_not_see_keys_off_their_path(wls, name):
    """Changing the K/V of one node changes no row whose path misses it, and
    changing other nodes' mask words changes no row at all but theirs."""
    w, dw = wls("tree", name)
    R, G, P = w.cfg.rows, w.groups, w.cfg.page_size
    parents, mask = tree_inputs(w, True, 903)
    base, _ = run_general(dw, w.q, R, mask=mask.reshape(-1))
    j = 3
    k2, v2 = dw.k.clone(), dw.v.clone()
    for g in range(G):
        pos = int(w.seq_lens[g]) - R + j
        pg = int(w.page_table[g, pos // P])
        if dw.fp8:   # other finite e4m3 codes: flip the sign bit, step the mantissa
            k2[pg, pos % P] ^= 0x80
            v2[pg, pos % P] = torch.where((v2[pg, pos % P] & 0x7F) < 0x70, v2[pg, pos % P] + 8, v2[pg, pos % P] - 8)
        else:
            k2[pg, pos % P] = -k2[pg, pos % P] * 3
            v2[pg, pos % P] = v2[pg, pos % P] + 5
    dw2 = DevWorkload(w)
    dw2.k, dw2.v = k2, v2
    got, _ = run_general(dw2, w.q, R, mask=mask.reshape(-1))
    for g in range(G):
        assert not np.array_equal(got[g, j], base[g, j]), g       # the node itself sees the change
        for r in range(R):
            if not (mask[g, r] >> j) & 1:
                assert np.array_equal(got[g, r], base[g, r]), (g, r)
    # re-hang node R-1 elsewhere: only its own row may move
    m2 = mask.copy()
    m2[:, R - 1] = (1 << (R - 1)) | 1
    got, _ = run_general(dw, w.q, R, mask=m2.reshape(-1))
    assert np.array_equal(got[:, :R - 1], base[:, :R - 1])


def test_malformed_mask_words_zero_their_group_only(wls):
    w, dw = wls("tree", "t8_d128_fp8")
    R, G = w.cfg.rows, w.groups
    parents, mask = tree_inputs(w, True, 904)
    good, _ = run_general(dw, w.q, R, mask=mask.reshape(-1))
    for g, r, word in ((1, 5, 0b0001), (3, 2, 0b1100), (2, 0, 0)):
        m = mask.copy()
        m[g, r] = word
        got, err = run_general(dw, w.q, R, mask=m.reshape(-1))
        assert err == b.RAD_ERRW_MASK, (g, r)
        assert np.all(got[g] == 0)
        others = [x for x in range(G) if x != g]
        assert np.array_equal(got[others], good[others])
