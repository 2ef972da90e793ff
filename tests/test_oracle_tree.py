"""Pins for the oracle's ragged rows (cu_seqlens) and tree-verify masks
(CPU only, no GPU).

Ragged rows: "kern manifest v7", $defs.Fill `cu_seqlens` (exclusive prefix
sums of rows per sequence, groups + 1 entries) and "Radiance architecture
plugins", section "Step: issuing the graph" (`q_lens`, `max_q_len`; the
offsets are absolute).  Tree verify: "Adding a model", step 4 (forward_tree,
every verified row equal to the decode step's row) and "Radiance architecture
plugins", section "Declare: drafters, encoders, generators" (a tree over the
proposals).  The pins tie the oracle to the brute force over explicit paths,
to plain decode calls over each node's path re-paged from scratch, and to the
causal case a chain reduces to.
"""
import math

import numpy as np
import pytest

import oracle
from brute import attend_sequence
from test_oracle import bf16_bits, bf16_values, e4m3_values, paged_from_logical, random_case, run_oracle
from paged_kv_attention_02_gb300.workloads import mask_words, path_of, random_parents


def logical_kv(c, g, P, fp8):
    """Decoded K/V values of sequence g in position order (fp64)."""
    L = c["seqs_k"][g].shape[0]
    if not fp8:
        return bf16_values(c["seqs_k"][g]), bf16_values(c["seqs_v"][g])
    pages = c["table"][g]
    ks = np.array([c["ks"][pages[j // P]] for j in range(L)], dtype=np.float64)
    vs = np.array([c["vs"][pages[j // P]] for j in range(L)], dtype=np.float64)
    return (e4m3_values(c["seqs_k"][g]) * ks[:, None, None],
            e4m3_values(c["seqs_v"][g]) * vs[:, None, None])


def ragged_case(rng, *, q_lens, extra, H, Hkv, D, P, base=0, tail=0, fp8=False):
    """A ragged call: group g has q_lens[g] rows and q_lens[g] + extra[g] keys.
    Its q rows sit at base + sum(q_lens[:g]) of a [T, H, D] array."""
    lens = [ql + ex for ql, ex in zip(q_lens, extra)]
    c = random_case(rng, G=len(lens), R=1, H=H, Hkv=Hkv, D=D, P=P, lens=lens, fp8=fp8)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32) + base
    T = int(cu[-1]) + tail
    c["q"] = bf16_bits(rng.standard_normal((T, H, D)))
    c["cu"] = cu
    return c


def run_ragged(c, *, rows, H, Hkv, D, P, scale, fp8=False, **kw):
    return oracle.attn_paged(c["q"], c["kp"], c["vp"], c["table"], c["lens"], rows=rows, n_head=H,
                             n_head_kv=Hkv, head_dim=D, page_size=P, scale=scale,
                             kv_dtype=oracle.KV_FP8_E4M3 if fp8 else oracle.KV_BF16,
                             k_scales=c["ks"], v_scales=c["vs"], cu_seqlens=c["cu"], **kw)


# ----------------------------------------------------------------------------- ragged rows

@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("shape", [
    dict(q_lens=[1, 8, 0, 5, 3], extra=[9, 0, 4, 13, 40], H=4, Hkv=2, D=8, P=4, base=0, W=0),
    dict(q_lens=[6, 1, 2], extra=[1, 30, 5], H=2, Hkv=1, D=16, P=8, base=5, W=0),
    dict(q_lens=[4, 0, 7, 1], extra=[20, 3, 2, 0], H=6, Hkv=2, D=8, P=4, base=2, W=5),
])
def test_ragged_matches_brute_force(shape, fp8):
    rng = np.random.default_rng(70 + len(shape["q_lens"]) + int(fp8))
    s = dict(shape)
    q_lens, extra, W, base = s.pop("q_lens"), s.pop("extra"), s.pop("W"), s.pop("base")
    H, Hkv, D, P = (s[k] for k in ("H", "Hkv", "D", "P"))
    c = ragged_case(rng, q_lens=q_lens, extra=extra, H=H, Hkv=Hkv, D=D, P=P, base=base, tail=3, fp8=fp8)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    res = run_ragged(c, rows=max(q_lens), H=H, Hkv=Hkv, D=D, P=P, scale=scale, fp8=fp8, window=W)
    assert res.err_word == 0
    assert res.out.shape == (c["q"].shape[0], H, D)
    qv = bf16_values(c["q"])
    named = np.zeros(c["q"].shape[0], dtype=bool)
    for g, ql in enumerate(q_lens):
        a = int(c["cu"][g])
        named[a:a + ql] = True
        if ql == 0:
            continue
        kf, vf = logical_kv(c, g, P, fp8)
        want = attend_sequence(qv[a:a + ql].tolist(), kf.tolist(), vf.tolist(), scale, Hkv, window=W)
        np.testing.assert_allclose(res.out[a:a + ql], np.array(want), rtol=1e-12, atol=1e-12)
    assert np.all(res.out[~named] == 0)


def test_ragged_row_equals_its_sequence_called_alone():
    """Each sequence of a ragged call, called alone with rows = its own count,
    gives the same bits."""
    rng = np.random.default_rng(80)
    q_lens, extra = [3, 1, 7, 2], [11, 0, 6, 25]
    H, Hkv, D, P = 4, 1, 8, 4
    c = ragged_case(rng, q_lens=q_lens, extra=extra, H=H, Hkv=Hkv, D=D, P=P, base=1)
    res = run_ragged(c, rows=7, H=H, Hkv=Hkv, D=D, P=P, scale=0.6)
    for g, ql in enumerate(q_lens):
        a = int(c["cu"][g])
        one = oracle.attn_paged(c["q"][None, a:a + ql], c["kp"], c["vp"], c["table"][g:g + 1],
                                c["lens"][g:g + 1], rows=ql, n_head=H, n_head_kv=Hkv, head_dim=D,
                                page_size=P, scale=0.6)
        assert np.array_equal(res.out[a:a + ql], one.out[0])


def test_uniform_offsets_equal_the_uniform_call():
    rng = np.random.default_rng(81)
    R, H, Hkv, D, P = 3, 2, 2, 8, 4
    c = random_case(rng, G=3, R=R, H=H, Hkv=Hkv, D=D, P=P, lens=[3, 9, 17])
    base = run_oracle(c, R=R, H=H, Hkv=Hkv, D=D, P=P, scale=0.9)
    cu = np.arange(4, dtype=np.int32) * R
    rag = oracle.attn_paged(c["q"].reshape(3 * R, H, D), c["kp"], c["vp"], c["table"], c["lens"], rows=R,
                            n_head=H, n_head_kv=Hkv, head_dim=D, page_size=P, scale=0.9, cu_seqlens=cu)
    assert np.array_equal(rag.out.reshape(base.out.shape), base.out)


def test_ragged_malformed_entries_flag_only_their_group():
    rng = np.random.default_rng(82)
    q_lens, extra = [2, 3, 1, 2], [5, 5, 5, 5]
    H, Hkv, D, P = 2, 1, 8, 4
    c = ragged_case(rng, q_lens=q_lens, extra=extra, H=H, Hkv=Hkv, D=D, P=P, base=0)
    good = run_ragged(c, rows=3, H=H, Hkv=Hkv, D=D, P=P, scale=0.5)
    assert good.err_word == 0
    # group 1 claims more rows than the call's largest count
    bad = oracle.attn_paged_rows(c["q"], c["kp"], c["vp"], c["table"], c["lens"], rows=2, n_head=H,
                                 n_head_kv=Hkv, head_dim=D, page_size=P, scale=0.5, cu_seqlens=c["cu"],
                                 sel=[(0, 0, 0), (0, 1, 1), (2, 0, 0)])
    assert bad.err_word == 0      # group 1 not touched
    full = oracle.attn_paged(c["q"], c["kp"], c["vp"], c["table"], c["lens"], rows=2, n_head=H,
                             n_head_kv=Hkv, head_dim=D, page_size=P, scale=0.5, cu_seqlens=c["cu"])
    assert full.err_word == oracle.ERRW_CUSEQ
    a1 = int(c["cu"][1])
    keep = np.ones(c["q"].shape[0], dtype=bool)
    keep[a1:a1 + 3] = False
    assert np.array_equal(full.out[keep], good.out[keep])
    assert np.all(full.out[a1:a1 + 3] == 0)
    # decreasing and negative offsets
    for cu in ([0, 2, 1, 6, 8], [-1, 2, 5, 6, 8]):
        r = oracle.attn_paged(c["q"], c["kp"], c["vp"], c["table"], c["lens"], rows=3, n_head=H,
                              n_head_kv=Hkv, head_dim=D, page_size=P, scale=0.5,
                              cu_seqlens=np.array(cu, dtype=np.int32))
        assert r.err_word == oracle.ERRW_CUSEQ
    # a sequence shorter than its rows
    lens = c["lens"].copy()
    lens[3] = 1
    r = oracle.attn_paged(c["q"], c["kp"], c["vp"], c["table"], lens, rows=3, n_head=H, n_head_kv=Hkv,
                          head_dim=D, page_size=P, scale=0.5, cu_seqlens=c["cu"])
    assert r.err_word == oracle.ERRW_SEQLEN
    a3 = int(c["cu"][3])
    assert np.all(r.out[a3:a3 + 2] == 0) and np.array_equal(r.out[:a3], good.out[:a3])


def test_empty_sequences_have_no_rows_and_no_error():
    rng = np.random.default_rng(83)
    c = ragged_case(rng, q_lens=[0, 2, 0], extra=[4, 4, 4], H=2, Hkv=1, D=8, P=4)
    c["lens"][0] = 1 << 20     # never looked at: the group has no rows
    res = run_ragged(c, rows=2, H=2, Hkv=1, D=8, P=4, scale=1.0)
    assert res.err_word == 0 and res.out.shape == (2, 2, 8)
    with pytest.raises(oracle.OracleError):   # a row past its group's count names nothing
        oracle.attn_paged_rows(c["q"], c["kp"], c["vp"], c["table"], c["lens"], rows=2, n_head=2,
                               n_head_kv=1, head_dim=8, page_size=4, scale=1.0, cu_seqlens=c["cu"],
                               sel=[(0, 0, 0)])


# ----------------------------------------------------------------------------- tree masks

@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("shape", [
    dict(R=8, H=4, Hkv=2, D=8, P=4, lens=[8, 19, 40]),
    dict(R=5, H=2, Hkv=1, D=16, P=8, lens=[30, 5]),
    dict(R=32, H=2, Hkv=2, D=4, P=16, lens=[32, 70]),
])
def test_tree_matches_brute_force(shape, fp8):
    rng = np.random.default_rng(90 + shape["R"] + int(fp8))
    R, H, Hkv, D, P, lens = (shape[k] for k in ("R", "H", "Hkv", "D", "P", "lens"))
    c = random_case(rng, G=len(lens), R=R, H=H, Hkv=Hkv, D=D, P=P, lens=lens, fp8=fp8)
    parents = [random_parents(rng, R) for _ in lens]
    mask = np.stack([mask_words(pa) for pa in parents])
    scale = float(np.float32(1.0 / math.sqrt(D)))
    res = run_oracle(c, R=R, H=H, Hkv=Hkv, D=D, P=P, scale=scale, fp8=fp8, tree_mask=mask)
    assert res.err_word == 0
    qv = bf16_values(c["q"])
    for g in range(len(lens)):
        kf, vf = logical_kv(c, g, P, fp8)
        want = attend_sequence(qv[g].tolist(), kf.tolist(), vf.tolist(), scale, Hkv, parents=parents[g])
        np.testing.assert_allclose(res.out[g], np.array(want), rtol=1e-12, atol=1e-12)


def test_tree_row_equals_a_decode_over_its_path():
    """Node r of a tree equals a one-row decode over the cached keys followed by
    the keys of its path, laid out contiguously and re-paged from scratch:
    the same keys in the same order give the same bits."""
    rng = np.random.default_rng(91)
    R, H, Hkv, D, P = 9, 4, 2, 8, 4
    lens = [9, 23]
    c = random_case(rng, G=2, R=R, H=H, Hkv=Hkv, D=D, P=P, lens=lens)
    parents = [[-1, 0, 0, 1, -1, 4, 3, 2, 6], random_parents(rng, R)]
    mask = np.stack([mask_words(pa) for pa in parents])
    res = run_oracle(c, R=R, H=H, Hkv=Hkv, D=D, P=P, scale=0.45, tree_mask=mask)
    for g, L in enumerate(lens):
        c0 = L - R
        for r in range(R):
            keep = list(range(c0)) + sorted(c0 + i for i in path_of(parents[g], r))
            kk = [c["seqs_k"][g][keep]]
            vv = [c["seqs_v"][g][keep]]
            kp, vp, table = paged_from_logical(kk, vv, P, (len(keep) + P - 1) // P + 2, rng)
            one = oracle.attn_paged(np.ascontiguousarray(c["q"][g:g + 1, r:r + 1]), kp, vp, table,
                                    np.array([len(keep)], dtype=np.int32), rows=1, n_head=H,
                                    n_head_kv=Hkv, head_dim=D, page_size=P, scale=0.45)
            assert np.array_equal(res.out[g, r], one.out[0, 0]), (g, r)


def test_chain_mask_is_the_causal_call():
    rng = np.random.default_rng(92)
    R, H, Hkv, D, P = 8, 4, 1, 8, 4
    c = random_case(rng, G=3, R=R, H=H, Hkv=Hkv, D=D, P=P, lens=[8, 12, 33], fp8=True)
    chain = np.tile(mask_words(list(range(-1, R - 1))), (3, 1))
    assert chain[0, 3] == 0b1111
    a = run_oracle(c, R=R, H=H, Hkv=Hkv, D=D, P=P, scale=0.3, fp8=True)
    b = run_oracle(c, R=R, H=H, Hkv=Hkv, D=D, P=P, scale=0.3, fp8=True, tree_mask=chain)
    assert np.array_equal(a.out, b.out)


def test_tree_weights_are_zero_off_the_path():
    rng = np.random.default_rng(93)
    R, L = 6, 14
    c = random_case(rng, G=1, R=R, H=2, Hkv=1, D=8, P=4, lens=[L])
    parents = [-1, 0, -1, 2, 0, 3]
    mask = mask_words(parents)[None]
    sel = [(0, r, h) for r in range(R) for h in range(2)]
    res = oracle.attn_paged_rows(c["q"], c["kp"], c["vp"], c["table"], c["lens"], rows=R, n_head=2,
                                 n_head_kv=1, head_dim=8, page_size=4, scale=1.2, sel=sel,
                                 want_weights=True, tree_mask=mask)
    for i, (g, r, h) in enumerate(sel):
        w = res.weights[i]
        on = set(range(L - R)) | {L - R + x for x in path_of(parents, r)}
        assert all((w[j] > 0) == (j in on) for j in range(L)), r
        assert abs(w.sum() - 1.0) < 1e-12


def test_malformed_mask_words_zero_their_group_only():
    rng = np.random.default_rng(94)
    R, H, Hkv, D, P = 4, 2, 1, 8, 4
    c = random_case(rng, G=3, R=R, H=H, Hkv=Hkv, D=D, P=P, lens=[6, 9, 12])
    mask = np.tile(mask_words([-1, 0, 1, 1]), (3, 1))
    good = run_oracle(c, R=R, H=H, Hkv=Hkv, D=D, P=P, scale=0.7, tree_mask=mask)
    assert good.err_word == 0
    for g, r, word in ((1, 2, 0b0011), (1, 1, 0b0110), (2, 0, 0b1001)):   # no self bit / a later node
        m = mask.copy()
        m[g, r] = word
        bad = run_oracle(c, R=R, H=H, Hkv=Hkv, D=D, P=P, scale=0.7, tree_mask=m)
        assert bad.err_word == oracle.ERRW_MASK
        assert np.all(bad.out[g] == 0)
        others = [x for x in range(3) if x != g]
        assert np.array_equal(bad.out[others], good.out[others])


def test_tree_refuses_a_window_and_more_than_32_nodes():
    rng = np.random.default_rng(95)
    c = random_case(rng, G=1, R=4, H=2, Hkv=1, D=8, P=4, lens=[10])
    mask = mask_words([-1, 0, 1, 2])[None]
    with pytest.raises(oracle.OracleError):
        run_oracle(c, R=4, H=2, Hkv=1, D=8, P=4, scale=1.0, tree_mask=mask, window=3)
    c33 = random_case(rng, G=1, R=33, H=1, Hkv=1, D=4, P=16, lens=[40])
    with pytest.raises(oracle.OracleError):
        run_oracle(c33, R=33, H=1, Hkv=1, D=4, P=16, scale=1.0, tree_mask=np.ones((1, 33), np.uint32))


def test_ragged_tree_matches_brute_force():
    """Trees of different sizes in one ragged call."""
    rng = np.random.default_rng(96)
    q_lens, extra = [5, 1, 0, 8], [7, 20, 3, 0]
    H, Hkv, D, P = 4, 2, 8, 4
    c = ragged_case(rng, q_lens=q_lens, extra=extra, H=H, Hkv=Hkv, D=D, P=P, base=2, tail=1)
    parents = [random_parents(rng, ql) if ql else [] for ql in q_lens]
    mask = np.zeros(c["q"].shape[0], dtype=np.uint32)
    for g, ql in enumerate(q_lens):
        a = int(c["cu"][g])
        mask[a:a + ql] = mask_words(parents[g]) if ql else []
    scale = float(np.float32(0.4))   # the op takes an fp32 scale
    res = run_ragged(c, rows=8, H=H, Hkv=Hkv, D=D, P=P, scale=scale, tree_mask=mask)
    assert res.err_word == 0
    qv = bf16_values(c["q"])
    for g, ql in enumerate(q_lens):
        if ql == 0:
            continue
        a = int(c["cu"][g])
        kf, vf = logical_kv(c, g, P, False)
        want = attend_sequence(qv[a:a + ql].tolist(), kf.tolist(), vf.tolist(), scale, Hkv, parents=parents[g])
        np.testing.assert_allclose(res.out[a:a + ql], np.array(want), rtol=1e-12, atol=1e-12)
