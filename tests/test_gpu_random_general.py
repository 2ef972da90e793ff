"""Seeded random ragged and draft-tree calls (rad_attn_paged_ex) against the
oracle.

Each case draws a mix the fixed cases do not name: per-sequence row counts
from empty to a 40-row chunk (so the decode-shaped and the other tile lists
both fill, or one stays empty), uniform-row draft forests of 2 to 32 nodes,
ragged forests, both head dims, page sizes and pool types, GQA ratios 1 to 8,
and lengths at split and page boundaries.  Rows no sequence names must stay
untouched."""
import math
import random

import numpy as np
import pytest

from gpu_util import DevWorkload, assert_parity
from paged_kv_attention_02_gb300 import workloads as wl
from test_gpu_tree import SENTINEL, as_float, named_rows, oracle_general, ragged_q, run_general
from paged_kv_attention_02_gb300.workloads import mask_words, random_parents

pytestmark = pytest.mark.gpu

N_CASES = 32


def random_general(i: int):
    """(config, kind, q_lens or None): kind is 'ragged', 'tree' or 'ragged_tree'."""
    r = random.Random(11000 + i)
    kind = r.choice(["ragged", "ragged", "tree", "ragged_tree"])
    head_dim = r.choice([128, 128, 256])
    page = r.choice([16, 32])
    dtype = r.choice([wl.KV_BF16, wl.KV_FP8_E4M3])
    ratio = r.choice([1, 2, 4, 8])
    n_head_kv = r.choice([1, 2]) if ratio >= 4 else r.choice([1, 2, 4])
    groups = r.randint(2, 7)
    if kind == "ragged":
        q_lens = [r.choice([0, 1, 1, 2, 3, 8, 13, 40]) for _ in range(groups)]
    elif kind == "tree":
        q_lens = None
    else:
        q_lens = [r.choice([0, 1, 2, 5, 8, 16, 32]) for _ in range(groups)]
    rows = r.choice([2, 4, 8, 16, 32]) if q_lens is None else max(1, max(q_lens))
    lens = []
    for g in range(groups):
        need = rows if q_lens is None else max(q_lens[g], 1)
        L = r.choice([need, need + r.randint(1, 3000), r.choice([1023, 1024, 2048, 2049]) + need])
        lens.append(L)
    pages = math.ceil(max(lens) / page) + r.randint(0, 2)
    meta = {"head_dim": head_dim, "n_embd": 213 * ratio * n_head_kv} if head_dim == 256 else {}
    c = wl.Config(f"gen{i}", groups, rows, ratio * n_head_kv, n_head_kv, head_dim, page, dtype, 11000 + i,
                  "fixed:" + ",".join(map(str, lens)), pages_per_seq=pages, meta=meta)
    return c, kind, q_lens


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_general_call_matches_oracle(i):
    c, kind, q_lens = random_general(i)
    w = wl.make_workload(c, poison=True)
    dw = DevWorkload(w)
    rng = np.random.default_rng(12000 + i)
    R = c.rows
    if kind == "tree":
        parents = [random_parents(rng, R, forest=bool(rng.integers(0, 2))) for _ in range(c.groups)]
        mask = np.stack([mask_words(pa) for pa in parents]).astype(np.uint32)
        got, err = run_general(dw, w.q, R, mask=mask.reshape(-1))
        assert err == 0, (c, kind, err)
        ref = oracle_general(w, w.q, R, mask=mask)
        assert ref.err_word == 0
        assert_parity(as_float(got), ref.out, dw.fp8, f"{c.name} {kind}: {c}")
        return
    q, cu = ragged_q(w, q_lens, base=int(rng.integers(0, 3)), tail=int(rng.integers(0, 3)))
    mask = None
    if kind == "ragged_tree":
        mask = np.zeros(q.shape[0], dtype=np.uint32)
        for g, ql in enumerate(q_lens):
            if ql:
                mask[cu[g]:cu[g] + ql] = mask_words(random_parents(rng, ql))
    got, err = run_general(dw, q, R, cu=cu, mask=mask)
    assert err == 0, (c, kind, q_lens, err)
    ref = oracle_general(w, q, R, cu=cu, mask=mask)
    assert ref.err_word == 0
    named = named_rows(cu, q.shape[0])
    assert np.all(got[~named] == np.int16(SENTINEL)), "a row no group names was written"
    assert_parity(as_float(got[named]), ref.out[named], dw.fp8, f"{c.name} {kind} {q_lens}: {c}")
