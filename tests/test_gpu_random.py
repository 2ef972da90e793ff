"""Seeded random call shapes against the oracle, every row.

The fixed cases elsewhere pin each kernel family at chosen boundaries; these
draw the combinations they do not name -- odd row counts on the tensor-core
kernels (3 or 5 rows of 4 heads fill part of a query tile), GQA ratios from 1
to 16, both page sizes, head dims and pool types, lengths at split and page
boundaries or equal to the row count, and a sliding window on about a third
of the calls -- from a fixed seed per case, so a failure is reproducible by its
id."""
import math
import random

import pytest

from gpu_util import DevWorkload, as_f64, assert_parity, oracle_rows
from paged_kv_attention_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

N_CASES = 48


def random_window(i: int) -> int | None:
    """The case's sliding window (keys a row sees, itself included), or None."""
    r = random.Random(9000 + i)
    return r.choice([1, 7, 64, 300, 1000, 2100]) if r.random() < 0.35 else None


def random_config(i: int) -> wl.Config:
    r = random.Random(7000 + i)
    head_dim = r.choice([128, 128, 256])
    page = r.choice([16, 32])
    dtype = r.choice([wl.KV_BF16, wl.KV_FP8_E4M3])
    rows = r.choice([1, 1, 2, 3, 5, 8, 8, 13, 40, 300])
    ratio = r.choice([1, 2, 4, 8, 16])
    n_head_kv = r.choice([1, 2, 4]) if ratio <= 4 else r.choice([1, 2])
    if rows >= 40:   # keep the oracle's work small: fewer heads for the long calls
        ratio, n_head_kv = r.choice([(1, 2), (4, 1), (8, 1)])
    groups = r.randint(1, 2) if rows >= 40 else r.randint(1, 6)
    lens = []
    for _ in range(groups):
        kind = r.random()
        if kind < 0.2:
            L = rows                                        # nothing cached
        elif kind < 0.5:
            L = r.choice([1023, 1024, 1025, 2047, 2048, 2049, 4095, 4096, 4097]) + rows
        else:
            L = rows + r.randint(1, 3000 if rows < 40 else 2000)
        lens.append(max(L, rows))
    pages = math.ceil(max(lens) / page) + r.randint(0, 3)
    meta = {"head_dim": head_dim, "n_embd": 213 * ratio * n_head_kv} if head_dim == 256 else {}
    return wl.Config(f"rand{i}", groups, rows, ratio * n_head_kv, n_head_kv, head_dim, page, dtype, 7000 + i,
                     "fixed:" + ",".join(map(str, lens)), pages_per_seq=pages, meta=meta)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape_matches_oracle_everywhere(i):
    c, win = random_config(i), random_window(i)
    w = wl.make_workload(c, poison=True)
    dw = DevWorkload(w)
    out, err = dw.run(window=win)
    assert err == 0, (c, win, err)
    ref = oracle_rows(w, window=win or 0)
    assert_parity(as_f64(out), ref.out, dw.fp8, f"{c.name} window {win}: {c}")
