"""Pins for the oracle (CPU only, no GPU).

The oracle is trusted only after these tie it to things other than itself:
the number formats' definitions (and torch's independent converters), a
brute-force pure-Python attention on contiguous inputs, hand-derived closed
forms (tests/golden/), and invariants that the definition fixes (page
permutation, grouped-query replication, causal rows, weights summing to 1).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from brute import attend_sequence
from paged_kv_attention_02_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- helpers

def bf16_bits(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def bf16_values(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16) \
        .to(torch.float64).numpy()


def e4m3_values(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn) \
        .to(torch.float64).numpy()


def paged_from_logical(seqs_k, seqs_v, page_size, num_pages, rng, pages_per_seq=None, fill=0):
    """Scatter per-sequence contiguous K/V ([L][Hkv][D] code arrays) into a
    shuffled page pool; returns (k_pool, v_pool, page_table)."""
    G = len(seqs_k)
    Hkv, D = seqs_k[0].shape[1:]
    need = [(k.shape[0] + page_size - 1) // page_size for k in seqs_k]
    pps = pages_per_seq or max(need)
    perm = rng.permutation(num_pages)
    dt = seqs_k[0].dtype
    kp = np.full((num_pages, page_size, Hkv, D), fill, dtype=dt)
    vp = np.full((num_pages, page_size, Hkv, D), fill, dtype=dt)
    table = np.full((G, pps), -1, dtype=np.int32)
    off = 0
    for g in range(G):
        for p in range(need[g]):
            pg = int(perm[off])
            off += 1
            table[g, p] = pg
            sl = slice(p * page_size, min((p + 1) * page_size, seqs_k[g].shape[0]))
            n = sl.stop - sl.start
            kp[pg, :n] = seqs_k[g][sl]
            vp[pg, :n] = seqs_v[g][sl]
    return kp, vp, table


def random_case(rng, *, G, R, H, Hkv, D, P, lens, fp8=False, spare_pages=3):
    """Random codes for a tiny call plus the decoded values the brute force reads."""
    seqs_k, seqs_v, kvals, vvals = [], [], [], []
    for L in lens:
        if fp8:
            ck = rng.integers(0, 256, size=(L, Hkv, D)).astype(np.uint8)
            cv = rng.integers(0, 256, size=(L, Hkv, D)).astype(np.uint8)
            ck[(ck & 0x7F) == 0x7F] = 0x3C   # no NaN codes in live data
            cv[(cv & 0x7F) == 0x7F] = 0x41
        else:
            ck = bf16_bits(rng.standard_normal((L, Hkv, D)))
            cv = bf16_bits(rng.standard_normal((L, Hkv, D)))
        seqs_k.append(ck)
        seqs_v.append(cv)
    num_pages = sum((L + P - 1) // P for L in lens) + spare_pages
    kp, vp, table = paged_from_logical(seqs_k, seqs_v, P, num_pages, rng)
    q = bf16_bits(rng.standard_normal((G, R, H, D)))
    ks = vs = None
    if fp8:
        ks = (rng.uniform(0.01, 2.0, size=num_pages)).astype(np.float32)
        vs = (rng.uniform(0.01, 2.0, size=num_pages)).astype(np.float32)
    return dict(q=q, kp=kp, vp=vp, table=table, lens=np.array(lens, dtype=np.int32), ks=ks, vs=vs,
                seqs_k=seqs_k, seqs_v=seqs_v)


def run_oracle(c, *, R, H, Hkv, D, P, scale, fp8=False, **kw):
    return oracle.attn_paged(c["q"], c["kp"], c["vp"], c["table"], c["lens"], rows=R, n_head=H,
                             n_head_kv=Hkv, head_dim=D, page_size=P, scale=scale,
                             kv_dtype=oracle.KV_FP8_E4M3 if fp8 else oracle.KV_BF16,
                             k_scales=c["ks"], v_scales=c["vs"], **kw)


# ----------------------------------------------------------------------------- number formats

def test_bf16_decoder_matches_torch_on_every_code():
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bf16_values(codes)
    got = np.array([oracle.bf16_to_f64(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_decoder_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = e4m3_values(codes)
    got = np.array([oracle.e4m3_to_f64(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert nan.sum() == 2     # only S.1111.111
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_decoder_known_code_points():
    for line in open(os.path.join(GOLDEN, "e4m3_known_codes.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        code, val = line.split()
        got = oracle.e4m3_to_f64(int(code, 16))
        if val == "nan":
            assert math.isnan(got), code
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), code


# ----------------------------------------------------------------------------- closed forms

def test_closed_form_golden_cases():
    spec = json.load(open(os.path.join(GOLDEN, "closed_form_cases.json")))
    for case in spec["cases"]:
        R, H, Hkv, D, P = (case[k] for k in ("rows", "n_head", "n_head_kv", "head_dim", "page_size"))
        keys = bf16_bits(case["keys_logical"])
        vals = bf16_bits(case["values_logical"])
        table_l = case["page_table"]
        num_pages = len(table_l)
        kp = np.zeros((num_pages, P, Hkv, D), dtype=np.uint16)
        vp = np.zeros_like(kp)
        for j in range(case["seq_len"]):
            kp[table_l[j // P], j % P] = keys[j]
            vp[table_l[j // P], j % P] = vals[j]
        q = bf16_bits(case["q"]).reshape(1, R, H, D)
        res = oracle.attn_paged(q, kp, vp, np.array([table_l], dtype=np.int32),
                                np.array([case["seq_len"]], dtype=np.int32), rows=R, n_head=H,
                                n_head_kv=Hkv, head_dim=D, page_size=P, scale=case["scale"])
        np.testing.assert_allclose(res.out[0], np.array(case["expected"], dtype=np.float64),
                                   rtol=0, atol=1e-12, err_msg=case["name"])


def test_single_key_returns_that_value_row():
    rng = np.random.default_rng(1)
    c = random_case(rng, G=1, R=1, H=4, Hkv=2, D=16, P=4, lens=[1])
    res = run_oracle(c, R=1, H=4, Hkv=2, D=16, P=4, scale=0.3)
    v = bf16_values(c["seqs_v"][0][0])          # [Hkv][D]
    for h in range(4):
        assert np.array_equal(res.out[0, 0, h], v[h // 2])


def test_constant_values_give_that_constant():
    rng = np.random.default_rng(2)
    c = random_case(rng, G=2, R=3, H=4, Hkv=1, D=8, P=4, lens=[9, 17])
    c["vp"][:] = bf16_bits(-3.5)
    res = run_oracle(c, R=3, H=4, Hkv=1, D=8, P=4, scale=0.7)
    np.testing.assert_allclose(res.out, -3.5, rtol=1e-14, atol=0)


def test_scale_zero_gives_mean_of_visible_values():
    rng = np.random.default_rng(3)
    c = random_case(rng, G=2, R=2, H=2, Hkv=2, D=8, P=4, lens=[5, 11])
    res = run_oracle(c, R=2, H=2, Hkv=2, D=8, P=4, scale=0.0)
    for g, L in enumerate(c["lens"]):
        v = bf16_values(c["seqs_v"][g])       # [L][Hkv][D]
        for r in range(2):
            n = L - 2 + r + 1
            for h in range(2):
                np.testing.assert_allclose(res.out[g, r, h], np.mean(v[:n, h], axis=0), rtol=1e-13,
                                           atol=1e-15)


def test_peaked_softmax_selects_the_aligned_key_without_overflow():
    # keys are basis vectors; q points at key jstar with a logit of 30 (or
    # 3e4 / 1e38-range: the max subtraction must keep exp finite).
    D, L, jstar = 16, 12, 7
    keys = np.zeros((L, 1, D), dtype=np.float32)
    for j in range(L):
        keys[j, 0, j] = 1.0
    rng = np.random.default_rng(4)
    vals = rng.standard_normal((L, 1, D)).astype(np.float32)
    kbits, vbits = bf16_bits(keys), bf16_bits(vals)
    kp, vp, table = paged_from_logical([kbits], [vbits], 4, 5, rng)
    v = bf16_values(vbits)
    for big, tol in ((30.0, (L - 1) * math.exp(-30) * 10), (3.0e4, 0.0), (1.0e30, 0.0)):
        q = np.zeros((1, 1, 1, D), dtype=np.float32)
        q[0, 0, 0, jstar] = big
        res = oracle.attn_paged(bf16_bits(q), kp, vp, table, np.array([L], dtype=np.int32), rows=1,
                                n_head=1, n_head_kv=1, head_dim=D, page_size=4, scale=1.0)
        assert np.all(np.isfinite(res.out))
        np.testing.assert_allclose(res.out[0, 0, 0], v[jstar, 0], rtol=0, atol=tol + 1e-15)


# ----------------------------------------------------------------------------- brute force

@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("shape", [
    dict(G=3, R=1, H=4, Hkv=2, D=8, P=4, lens=[1, 13, 40]),
    dict(G=2, R=3, H=6, Hkv=2, D=4, P=2, lens=[3, 23]),
    dict(G=2, R=8, H=3, Hkv=3, D=8, P=16, lens=[8, 37]),
    dict(G=1, R=2, H=2, Hkv=1, D=128, P=16, lens=[19]),
])
def test_matches_brute_force(shape, fp8):
    rng = np.random.default_rng(10 + shape["D"] + shape["R"] + int(fp8))
    s = dict(shape)
    lens = s.pop("lens")
    G, R, H, Hkv, D, P = (s[k] for k in ("G", "R", "H", "Hkv", "D", "P"))
    c = random_case(rng, G=G, R=R, H=H, Hkv=Hkv, D=D, P=P, lens=lens, fp8=fp8)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    res = run_oracle(c, R=R, H=H, Hkv=Hkv, D=D, P=P, scale=scale, fp8=fp8, want_weights=True)
    assert res.err_word == 0
    qv = bf16_values(c["q"])
    for g, L in enumerate(lens):
        if fp8:
            pages = c["table"][g]
            ks = np.array([c["ks"][pages[j // P]] for j in range(L)], dtype=np.float64)
            vs = np.array([c["vs"][pages[j // P]] for j in range(L)], dtype=np.float64)
            kf = e4m3_values(c["seqs_k"][g]) * ks[:, None, None]
            vf = e4m3_values(c["seqs_v"][g]) * vs[:, None, None]
        else:
            kf, vf = bf16_values(c["seqs_k"][g]), bf16_values(c["seqs_v"][g])
        want = attend_sequence(qv[g].tolist(), kf.tolist(), vf.tolist(), scale, Hkv)
        np.testing.assert_allclose(res.out[g], np.array(want), rtol=1e-12, atol=1e-12)


def test_weights_are_a_distribution():
    rng = np.random.default_rng(5)
    c = random_case(rng, G=2, R=4, H=4, Hkv=2, D=16, P=4, lens=[6, 33])
    sel = [(g, r, h) for g in range(2) for r in range(4) for h in range(4)]
    res = oracle.attn_paged_rows(c["q"], c["kp"], c["vp"], c["table"], c["lens"], rows=4, n_head=4,
                                 n_head_kv=2, head_dim=16, page_size=4, scale=2.0, sel=sel,
                                 want_weights=True)
    for i, (g, r, h) in enumerate(sel):
        n = int(res.n_keys[i])
        assert n == c["lens"][g] - 4 + r + 1
        w = res.weights[i, :n]
        assert np.all(w >= 0)
        assert abs(w.sum() - 1.0) < 1e-12
        assert np.all(res.weights[i, n:] == 0)


# ----------------------------------------------------------------------------- invariants

def test_page_permutation_leaves_output_bit_identical():
    rng = np.random.default_rng(6)
    c = random_case(rng, G=3, R=2, H=4, Hkv=2, D=16, P=4, lens=[7, 16, 29], spare_pages=5)
    base = run_oracle(c, R=2, H=4, Hkv=2, D=16, P=4, scale=0.25)
    perm = rng.permutation(c["kp"].shape[0])      # new physical id of each old page
    kp2 = np.empty_like(c["kp"])
    vp2 = np.empty_like(c["vp"])
    kp2[perm] = c["kp"]
    vp2[perm] = c["vp"]
    table2 = np.where(c["table"] >= 0, perm[np.maximum(c["table"], 0)], -1).astype(np.int32)
    c2 = dict(c, kp=kp2, vp=vp2, table=table2)
    moved = run_oracle(c2, R=2, H=4, Hkv=2, D=16, P=4, scale=0.25)
    assert np.array_equal(base.out, moved.out)


def test_grouped_heads_equal_replicated_kv_heads():
    rng = np.random.default_rng(7)
    c = random_case(rng, G=2, R=2, H=8, Hkv=2, D=16, P=4, lens=[10, 21])
    base = run_oracle(c, R=2, H=8, Hkv=2, D=16, P=4, scale=0.3)
    rep = dict(c, kp=np.repeat(c["kp"], 4, axis=2), vp=np.repeat(c["vp"], 4, axis=2))
    full = run_oracle(rep, R=2, H=8, Hkv=8, D=16, P=4, scale=0.3)
    assert np.array_equal(base.out, full.out)


def test_causal_row_equals_decode_at_its_position():
    rng = np.random.default_rng(8)
    R = 8
    c = random_case(rng, G=2, R=R, H=4, Hkv=2, D=16, P=4, lens=[9, 30])
    verify = run_oracle(c, R=R, H=4, Hkv=2, D=16, P=4, scale=0.4)
    for r in range(R):
        dec = dict(c, q=np.ascontiguousarray(c["q"][:, r:r + 1]), lens=c["lens"] - R + r + 1)
        one = run_oracle(dec, R=1, H=4, Hkv=2, D=16, P=4, scale=0.4)
        assert np.array_equal(verify.out[:, r], one.out[:, 0])


def test_batch_composition_does_not_change_a_row():
    rng = np.random.default_rng(9)
    c = random_case(rng, G=3, R=2, H=4, Hkv=2, D=8, P=4, lens=[5, 12, 26])
    full = run_oracle(c, R=2, H=4, Hkv=2, D=8, P=4, scale=0.5)
    for g in range(3):
        alone = dict(c, q=c["q"][g:g + 1], table=c["table"][g:g + 1], lens=c["lens"][g:g + 1])
        one = run_oracle(alone, R=2, H=4, Hkv=2, D=8, P=4, scale=0.5)
        assert np.array_equal(full.out[g], one.out[0])


# ----------------------------------------------------------------------------- error contract

def test_invalid_groups_are_zero_and_flagged_others_unaffected():
    rng = np.random.default_rng(11)
    c = random_case(rng, G=3, R=2, H=2, Hkv=1, D=8, P=4, lens=[6, 10, 14])
    good = run_oracle(c, R=2, H=2, Hkv=1, D=8, P=4, scale=0.5)
    bad = dict(c, lens=c["lens"].copy(), table=c["table"].copy())
    bad["lens"][0] = 1                          # fewer than rows
    res = run_oracle(bad, R=2, H=2, Hkv=1, D=8, P=4, scale=0.5)
    assert res.err_word == oracle.ERRW_SEQLEN
    assert np.all(res.out[0] == 0) and np.array_equal(res.out[1:], good.out[1:])
    bad = dict(c, table=c["table"].copy())
    bad["table"][1, 1] = c["kp"].shape[0]      # page id past the pool
    res = run_oracle(bad, R=2, H=2, Hkv=1, D=8, P=4, scale=0.5)
    assert res.err_word == oracle.ERRW_PAGE
    assert np.all(res.out[1] == 0) and np.array_equal(res.out[[0, 2]], good.out[[0, 2]])
    bad = dict(c, lens=c["lens"].copy())
    bad["lens"][2] = c["table"].shape[1] * 4 + 1   # longer than the page table holds
    res = run_oracle(bad, R=2, H=2, Hkv=1, D=8, P=4, scale=0.5)
    assert res.err_word == oracle.ERRW_SEQLEN and np.all(res.out[2] == 0)


def test_zero_rows_is_not_a_call():
    rng = np.random.default_rng(12)
    c = random_case(rng, G=1, R=1, H=2, Hkv=1, D=8, P=4, lens=[5])
    with pytest.raises(oracle.OracleError):
        run_oracle(dict(c, q=c["q"][:, :0]), R=0, H=2, Hkv=1, D=8, P=4, scale=0.5)


# ----------------------------------------------------------------------------- sliding window
# A windowed KV group (RAD_KV_WINDOW, Radiance architecture plugins, "Declare:
# buffers and KV groups") bounds what a row sees to its last W keys.

@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("shape", [
    dict(G=3, R=1, H=4, Hkv=2, D=8, P=4, lens=[1, 13, 40], W=5),
    dict(G=2, R=3, H=6, Hkv=2, D=4, P=2, lens=[3, 23], W=1),
    dict(G=2, R=8, H=3, Hkv=3, D=8, P=16, lens=[8, 37], W=4),
    dict(G=2, R=8, H=2, Hkv=1, D=8, P=4, lens=[9, 50], W=16),
    dict(G=1, R=2, H=2, Hkv=1, D=128, P=16, lens=[40], W=100),
])
def test_window_matches_brute_force(shape, fp8):
    rng = np.random.default_rng(40 + shape["W"] + shape["R"] + int(fp8))
    s = dict(shape)
    lens, W = s.pop("lens"), s.pop("W")
    G, R, H, Hkv, D, P = (s[k] for k in ("G", "R", "H", "Hkv", "D", "P"))
    c = random_case(rng, G=G, R=R, H=H, Hkv=Hkv, D=D, P=P, lens=lens, fp8=fp8)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    res = run_oracle(c, R=R, H=H, Hkv=Hkv, D=D, P=P, scale=scale, fp8=fp8, window=W)
    assert res.err_word == 0
    qv = bf16_values(c["q"])
    for g, L in enumerate(lens):
        if fp8:
            pages = c["table"][g]
            ks = np.array([c["ks"][pages[j // P]] for j in range(L)], dtype=np.float64)
            vs = np.array([c["vs"][pages[j // P]] for j in range(L)], dtype=np.float64)
            kf = e4m3_values(c["seqs_k"][g]) * ks[:, None, None]
            vf = e4m3_values(c["seqs_v"][g]) * vs[:, None, None]
        else:
            kf, vf = bf16_values(c["seqs_k"][g]), bf16_values(c["seqs_v"][g])
        want = attend_sequence(qv[g].tolist(), kf.tolist(), vf.tolist(), scale, Hkv, window=W)
        np.testing.assert_allclose(res.out[g], np.array(want), rtol=1e-12, atol=1e-12)


def test_window_of_one_returns_the_current_value_row():
    rng = np.random.default_rng(41)
    R, H, Hkv, D, P = 4, 4, 2, 8, 4
    c = random_case(rng, G=2, R=R, H=H, Hkv=Hkv, D=D, P=P, lens=[4, 19])
    res = run_oracle(c, R=R, H=H, Hkv=Hkv, D=D, P=P, scale=3.0, window=1)
    for g, L in enumerate(c["lens"]):
        v = bf16_values(c["seqs_v"][g])
        for r in range(R):
            for h in range(H):
                assert np.array_equal(res.out[g, r, h], v[L - R + r, h // (H // Hkv)])


def test_window_row_equals_unwindowed_row_over_its_last_keys():
    """Row r of a windowed call is the plain op over a sequence that holds only
    the row's last W keys, re-paged from scratch (bit for bit: the same sums)."""
    rng = np.random.default_rng(42)
    R, H, Hkv, D, P, W = 5, 4, 2, 16, 4, 7
    lens = [5, 11, 30]
    c = random_case(rng, G=3, R=R, H=H, Hkv=Hkv, D=D, P=P, lens=lens)
    res = run_oracle(c, R=R, H=H, Hkv=Hkv, D=D, P=P, scale=0.35, window=W)
    for g, L in enumerate(lens):
        for r in range(R):
            pos = L - R + r
            lo = max(0, pos - W + 1)
            kk = [c["seqs_k"][g][lo:pos + 1]]
            vv = [c["seqs_v"][g][lo:pos + 1]]
            n_pages = (pos + 1 - lo + P - 1) // P + 2
            kp, vp, table = paged_from_logical(kk, vv, P, n_pages, rng)
            one = oracle.attn_paged(np.ascontiguousarray(c["q"][g:g + 1, r:r + 1]), kp, vp, table,
                                    np.array([pos + 1 - lo], dtype=np.int32), rows=1, n_head=H,
                                    n_head_kv=Hkv, head_dim=D, page_size=P, scale=0.35)
            assert np.array_equal(res.out[g, r], one.out[0, 0])


def test_window_covering_the_context_changes_nothing():
    rng = np.random.default_rng(43)
    c = random_case(rng, G=2, R=3, H=2, Hkv=1, D=8, P=4, lens=[3, 26])
    base = run_oracle(c, R=3, H=2, Hkv=1, D=8, P=4, scale=0.5)
    for W in (26, 27, 1 << 20):
        win = run_oracle(c, R=3, H=2, Hkv=1, D=8, P=4, scale=0.5, window=W)
        assert np.array_equal(base.out, win.out)
    with pytest.raises(oracle.OracleError):
        run_oracle(c, R=3, H=2, Hkv=1, D=8, P=4, scale=0.5, window=-1)


def test_window_weights_vanish_below_the_window():
    rng = np.random.default_rng(44)
    R, W = 4, 6
    c = random_case(rng, G=1, R=R, H=2, Hkv=1, D=8, P=4, lens=[21])
    sel = [(0, r, h) for r in range(R) for h in range(2)]
    res = oracle.attn_paged_rows(c["q"], c["kp"], c["vp"], c["table"], c["lens"], rows=R, n_head=2,
                                 n_head_kv=1, head_dim=8, page_size=4, scale=1.5, sel=sel,
                                 want_weights=True, window=W)
    for i, (g, r, h) in enumerate(sel):
        pos = 21 - R + r
        w = res.weights[i]
        assert np.all(w[:pos - W + 1] == 0) and np.all(w[pos + 1:] == 0)
        assert np.all(w[pos - W + 1:pos + 1] > 0)
        assert abs(w.sum() - 1.0) < 1e-12


def test_window_pages_below_every_rows_window_are_never_read():
    """Page ids wholly below row 0's window may be stale or invalid; the page
    holding row 0's first visible key must still be valid."""
    rng = np.random.default_rng(45)
    R, P, W = 3, 4, 6
    c = random_case(rng, G=2, R=R, H=2, Hkv=1, D=8, P=P, lens=[9, 30])
    good = run_oracle(c, R=R, H=2, Hkv=1, D=8, P=P, scale=0.5, window=W)
    lo0 = 30 - R + 0 - W + 1               # row 0's first visible key in group 1: 22
    table = c["table"].copy()
    table[1, :lo0 // P] = -7               # pages 0..4 lie below every row's window
    res = run_oracle(dict(c, table=table), R=R, H=2, Hkv=1, D=8, P=P, scale=0.5, window=W)
    assert res.err_word == 0 and np.array_equal(res.out, good.out)
    table[1, lo0 // P] = c["kp"].shape[0]  # the page holding key 22 is needed
    res = run_oracle(dict(c, table=table), R=R, H=2, Hkv=1, D=8, P=P, scale=0.5, window=W)
    assert res.err_word == oracle.ERRW_PAGE
    assert np.all(res.out[1] == 0) and np.array_equal(res.out[0], good.out[0])


# ----------------------------------------------------------------------------- generator sanity

def test_tiny_workload_matches_its_recipe():
    w = wl.make_workload("tiny_decode", poison=True)
    assert list(w.seq_lens) == [37, 64, 129, 300]
    assert w.num_pages == 64
    used = w.page_table[w.page_table >= 0]
    assert used.size == 35 and len(set(used.tolist())) == 35
    res = oracle.attn_paged(w.q, w.k_pool, w.v_pool, w.page_table, w.seq_lens, **w.call_args())
    assert res.err_word == 0 and np.all(np.isfinite(res.out))


def test_fp8_generator_codes_decode_within_half_an_ulp():
    cfg = wl.Config("t", 2, 8, 4, 2, 128, 16, wl.KV_FP8_E4M3, 3, "fixed:40,70", pages_per_seq=8)
    w = wl.make_workload(cfg)
    x = e4m3_values(w.k_pool) * w.k_scales[:, None, None, None]
    assert np.all(np.isfinite(x))
    amax = np.abs(e4m3_values(w.k_pool)).reshape(w.num_pages, -1).max(axis=1)
    assert np.all(amax == 448.0)


# ----------------------------------------------------------------------------- random tiny shapes

@pytest.mark.parametrize("seed", range(24))
def test_random_tiny_shapes_match_brute_force(seed):
    """Seeded random tiny calls -- rows, GQA grouping, page size, lengths from
    the row count up, fp8 or bf16 codes, with or without a window -- against
    the pure-Python brute force over the contiguous sequences."""
    r = np.random.default_rng(5000 + seed)
    G, R = int(r.integers(1, 4)), int(r.integers(1, 6))
    Hkv, ratio = int(r.integers(1, 4)), int(r.integers(1, 4))
    H, D, P = Hkv * ratio, int(r.choice([2, 4, 8])), int(r.choice([1, 2, 4, 8]))
    fp8 = bool(r.integers(0, 2))
    lens = [R + int(r.integers(0, 30)) for _ in range(G)]
    W = int(r.choice([0, 0, 1, 3, 10]))
    c = random_case(r, G=G, R=R, H=H, Hkv=Hkv, D=D, P=P, lens=lens, fp8=fp8)
    scale = float(np.float32(r.uniform(0.05, 1.5)))
    res = run_oracle(c, R=R, H=H, Hkv=Hkv, D=D, P=P, scale=scale, fp8=fp8, window=W)
    assert res.err_word == 0
    qv = bf16_values(c["q"])
    for g, L in enumerate(lens):
        if fp8:
            pages = c["table"][g]
            ks = np.array([c["ks"][pages[j // P]] for j in range(L)], dtype=np.float64)
            vs = np.array([c["vs"][pages[j // P]] for j in range(L)], dtype=np.float64)
            kf = e4m3_values(c["seqs_k"][g]) * ks[:, None, None]
            vf = e4m3_values(c["seqs_v"][g]) * vs[:, None, None]
        else:
            kf, vf = bf16_values(c["seqs_k"][g]), bf16_values(c["seqs_v"][g])
        want = attend_sequence(qv[g].tolist(), kf.tolist(), vf.tolist(), scale, Hkv, window=W)
        np.testing.assert_allclose(res.out[g], np.array(want), rtol=1e-12, atol=1e-12)
