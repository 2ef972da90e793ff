"""GPU parity, row invariance and error-contract tests, through the C ABI.

Every expected value comes from the fp64 oracle (oracle/) on the same seeded
inputs; the CUDA path never produces a reference."""
import numpy as np
import pytest
import torch

from gpu_util import DevWorkload, as_f64, assert_parity, bits, oracle_rows
from paged_kv_attention_02_gb300 import binding as b
from paged_kv_attention_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

# Mid-size cases: several stages, several splits, ragged last pages, every
# call family, both head dims and both pool types, unused slots NaN-poisoned.
MID = {
    "dec128": wl.Config("dec128", 9, 1, 32, 8, 128, 16, wl.KV_BF16, 101,
                        "fixed:1,15,16,17,511,512,513,1500,3001", pages_per_seq=200),
    "dec256": wl.Config("dec256", 5, 1, 16, 2, 256, 32, wl.KV_BF16, 102, "fixed:1,33,700,1025,2500",
                        pages_per_seq=100, meta=dict(head_dim=256, n_embd=3408)),
    "dec_fp8_ratio1": wl.Config("dec_fp8_ratio1", 6, 1, 8, 8, 128, 16, wl.KV_FP8_E4M3, 103,
                                "fixed:3,64,700,1023,1024,1025", pages_per_seq=70),
    "dec_fp8_d256": wl.Config("dec_fp8_d256", 3, 1, 16, 2, 256, 32, wl.KV_FP8_E4M3, 104,
                              "fixed:40,900,1700", pages_per_seq=60),
    "ver_fp8": wl.Config("ver_fp8", 5, 8, 32, 8, 128, 16, wl.KV_FP8_E4M3, 105, "fixed:8,9,520,1000,2050",
                         pages_per_seq=130),
    # the e4m3 tcgen05 split kernel's 4096-key splits: lengths on both sides of 1, 2 and 3 splits
    "ver_fp8_splits": wl.Config("ver_fp8_splits", 6, 8, 32, 8, 128, 16, wl.KV_FP8_E4M3, 116,
                                "fixed:4095,4096,4097,8191,8193,12289", pages_per_seq=770),
    "dec_fp8_splits": wl.Config("dec_fp8_splits", 5, 1, 32, 8, 128, 32, wl.KV_FP8_E4M3, 117,
                                "fixed:4095,4096,4097,8192,8193", pages_per_seq=260),
    "ver_bf16": wl.Config("ver_bf16", 4, 8, 8, 2, 128, 16, wl.KV_BF16, 106, "fixed:8,100,513,1100",
                          pages_per_seq=70),
    "ver_wide_d256": wl.Config("ver_wide_d256", 3, 8, 16, 2, 256, 32, wl.KV_BF16, 107, "fixed:8,600,1500",
                               pages_per_seq=50),
    "ver_fp8_d256": wl.Config("ver_fp8_d256", 3, 8, 16, 2, 256, 32, wl.KV_FP8_E4M3, 112, "fixed:8,1100,2100",
                              pages_per_seq=70),
    "ratio16": wl.Config("ratio16", 3, 1, 16, 1, 128, 16, wl.KV_BF16, 108, "fixed:5,600,1200",
                         pages_per_seq=80),
    "chunk_split": wl.Config("chunk_split", 2, 40, 8, 2, 128, 16, wl.KV_BF16, 109, "fixed:40,1500",
                             pages_per_seq=100),
    "prefill": wl.Config("prefill", 2, 300, 8, 2, 128, 16, wl.KV_BF16, 110, "fixed:300,1000",
                         pages_per_seq=64),
    "prefill_fp8_d256": wl.Config("prefill_fp8_d256", 1, 260, 4, 1, 256, 32, wl.KV_FP8_E4M3, 111,
                                  "fixed:900", pages_per_seq=30),
    # head_dim 128 fp8 prefill chunks: the tcgen05 e4m3 kernel (ratios 4, 8, 1; both page sizes)
    "prefill_fp8": wl.Config("prefill_fp8", 2, 300, 8, 2, 128, 16, wl.KV_FP8_E4M3, 113, "fixed:300,1000",
                             pages_per_seq=64),
    "prefill_fp8_p32_r8": wl.Config("prefill_fp8_p32_r8", 1, 520, 16, 2, 128, 32, wl.KV_FP8_E4M3, 114,
                                    "fixed:1800", pages_per_seq=60),
    "prefill_fp8_r1": wl.Config("prefill_fp8_r1", 2, 272, 4, 4, 128, 16, wl.KV_FP8_E4M3, 115,
                                "fixed:272,2000", pages_per_seq=130),
    # head_dim-256 bf16 prefill chunks: the tcgen05 prefill kernel's 64-key-tile build (ratios 8, 1)
    "prefill_d256": wl.Config("prefill_d256", 2, 300, 16, 2, 256, 32, wl.KV_BF16, 118, "fixed:300,1500",
                              pages_per_seq=60, meta=dict(head_dim=256, n_embd=3408)),
    "prefill_d256_r1": wl.Config("prefill_d256_r1", 1, 272, 4, 4, 256, 16, wl.KV_BF16, 119, "fixed:900",
                                 pages_per_seq=64),
    # a GQA ratio (3) that does not tile the prefill kernels' 128-row blocks: the mma.sync wide tile
    "prefill_fp8_d256_r3": wl.Config("prefill_fp8_d256_r3", 1, 260, 6, 2, 256, 32, wl.KV_FP8_E4M3, 120,
                                     "fixed:900", pages_per_seq=30),
    "prefill_fp8_d256_2g": wl.Config("prefill_fp8_d256_2g", 2, 300, 16, 2, 256, 32, wl.KV_FP8_E4M3, 121,
                                     "fixed:300,1500", pages_per_seq=60),
    # uniform split calls with more than two items per SM: the e4m3 kernel and the head_dim-256
    # bf16 build take their items heaviest first (an order kernel sorts them before the launch)
    "ver_fp8_ordered": wl.Config("ver_fp8_ordered", 16, 8, 32, 8, 128, 16, wl.KV_FP8_E4M3, 122,
                                 "uniform:8,6000", pages_per_seq=600),
    "dec_d256_ordered": wl.Config("dec_d256_ordered", 48, 1, 16, 2, 256, 32, wl.KV_BF16, 123,
                                  "loguniform:1,12000", pages_per_seq=400, meta=dict(head_dim=256, n_embd=3408)),
    "dec_fp8_d256_ordered": wl.Config("dec_fp8_d256_ordered", 48, 1, 16, 2, 256, 32, wl.KV_FP8_E4M3, 124,
                                      "loguniform:1,12000", pages_per_seq=400),
}


@pytest.fixture(scope="module")
def mid():
    cache = {}

    def get(name):
        if name not in cache:
            w = wl.make_workload(MID[name], poison=True)
            cache[name] = (w, DevWorkload(w))
        return cache[name]
    return get


@pytest.mark.parametrize("name", list(MID))
def test_mid_size_matches_oracle_everywhere(mid, name):
    w, dw = mid(name)
    out, err = dw.run()
    assert err == 0
    ref = oracle_rows(w)
    assert ref.err_word == 0
    assert_parity(as_f64(out), ref.out, dw.fp8, name)


def test_tiny_decode_matches_oracle_everywhere():
    w = wl.make_workload("tiny_decode", poison=True)
    out, err = DevWorkload(w).run()
    assert err == 0
    assert_parity(as_f64(out), oracle_rows(w).out, False, "tiny_decode")


# ------------------------------------------------------------------ contexts past one combine chunk

# The combine kernel stages a row's partials 128 splits at a time: these contexts
# have more splits than that (2048-key splits on the bf16 tcgen05 split kernel,
# 4096 on the e4m3 one), so rows merge across chunk boundaries.
LONG = {
    "long_dec_bf16": wl.Config("long_dec_bf16", 2, 1, 8, 2, 128, 16, wl.KV_BF16, 121, "fixed:270000,1000",
                               pages_per_seq=16880),
    "long_ver_fp8": wl.Config("long_ver_fp8", 1, 8, 8, 2, 128, 32, wl.KV_FP8_E4M3, 122, "fixed:530000",
                              pages_per_seq=16570),
}


@pytest.mark.parametrize("name", list(LONG))
def test_contexts_past_one_combine_chunk_match_oracle(name):
    w = wl.make_workload(LONG[name], poison=True)
    dw = DevWorkload(w)
    out, err = dw.run()
    assert err == 0
    assert_parity(as_f64(out), oracle_rows(w).out, dw.fp8, name)
    del dw
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ full-size configurations

@pytest.fixture(scope="module")
def full():
    cache = {}

    def get(name):
        if name not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            w = wl.make_workload(name)
            cache[name] = (w, DevWorkload(w))
        return cache[name]
    return get


FULL = ["batched_decode", "hybrid_decode", "spec_verify", "prefill_chunk"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_rows_match_oracle(full, name):
    w, dw = full(name)
    out, err = dw.run()
    assert err == 0
    o = as_f64(out)
    assert np.all(np.isfinite(o))
    c = w.cfg
    rng = np.random.default_rng(7)
    n = 48
    rand = np.stack([rng.integers(0, w.groups, n), rng.integers(0, c.rows, n),
                     rng.integers(0, c.n_head, n)], axis=1)
    # one row of every sequence (so every context length is checked once), and
    # every head of the longest sequence's last row and of the shortest's first
    each = np.stack([np.arange(w.groups), rng.integers(0, c.rows, w.groups),
                     rng.integers(0, c.n_head, w.groups)], axis=1)
    heads = np.arange(c.n_head)
    longest = np.stack([np.full(c.n_head, int(np.argmax(w.seq_lens))), np.full(c.n_head, c.rows - 1), heads], axis=1)
    shortest = np.stack([np.full(c.n_head, int(np.argmin(w.seq_lens))), np.zeros(c.n_head, int), heads], axis=1)
    sel = np.concatenate([rand, each, longest, shortest]).astype(np.int64)
    ref = oracle_rows(w, sel)
    got = o[sel[:, 0], sel[:, 1], sel[:, 2]]
    assert_parity(got, ref.out, dw.fp8, name)


@pytest.mark.parametrize("name", ["batched_decode", "hybrid_decode", "spec_verify"])
def test_full_size_rows_are_bit_identical_across_batch_compositions(full, name):
    w, dw = full(name)
    out, _ = dw.run()
    base = bits(out)
    rng = np.random.default_rng(3)
    pick = rng.choice(w.groups, size=5, replace=False)
    # each sequence alone
    for g in pick[:3]:
        sub = w.select_groups([g])
        o, err = dw.run(q=dw.q[g:g + 1], table=dw.table[g:g + 1], lens=dw.lens[g:g + 1])
        assert err == 0
        assert np.array_equal(bits(o)[0], base[g]), f"group {g} alone"
        del sub
    # a shuffled subset padded with dummy sequences (seq_len = rows on page 0)
    order = np.concatenate([pick[::-1], [-1, -1, -1]])
    q = torch.cat([dw.q[g:g + 1] if g >= 0 else torch.zeros_like(dw.q[:1]) for g in order])
    table = torch.cat([dw.table[g:g + 1] if g >= 0 else torch.zeros_like(dw.table[:1]) for g in order])
    lens = torch.tensor([int(w.seq_lens[g]) if g >= 0 else w.cfg.rows for g in order], dtype=torch.int32,
                        device="cuda")
    o, err = dw.run(q=q, table=table, lens=lens)
    assert err == 0
    ob = bits(o)
    for i, g in enumerate(order):
        if g >= 0:
            assert np.array_equal(ob[i], base[g]), f"group {g} in a shuffled padded batch"


def test_full_size_prefill_chunk_is_bit_identical_alone_and_batched(full):
    # The 2048-row chunk over 8192 keys alone, and the same sequence as the
    # second group of a two-group call whose first group is another chunk of
    # 2048 rows (zero queries, the same pages, seq_len 2048): its rows must not
    # change with the other group.
    w, dw = full("prefill_chunk")
    alone, err = dw.run()
    assert err == 0
    R = w.cfg.rows
    q = torch.cat([torch.zeros_like(dw.q), dw.q])
    table = torch.cat([dw.table, dw.table])
    lens = torch.tensor([R, int(w.seq_lens[0])], dtype=torch.int32, device="cuda")
    both, err = dw.run(q=q, table=table, lens=lens)
    assert err == 0
    assert np.array_equal(bits(both)[1], bits(alone)[0])
    # and with the real sequence first, the padding group after it
    q = torch.cat([dw.q, torch.zeros_like(dw.q)])
    lens = torch.tensor([int(w.seq_lens[0]), R], dtype=torch.int32, device="cuda")
    both, err = dw.run(q=q, table=table, lens=lens)
    assert err == 0
    assert np.array_equal(bits(both)[0], bits(alone)[0])


@pytest.mark.parametrize("name", ["prefill", "prefill_fp8", "prefill_fp8_r1", "prefill_d256", "prefill_fp8_d256_2g"])
def test_prefill_rows_bit_identical_alone_and_batched(mid, name):
    w, dw = mid(name)
    out, _ = dw.run()
    o1, _ = dw.run(q=dw.q[1:2], table=dw.table[1:2], lens=dw.lens[1:2])
    assert np.array_equal(bits(o1)[0], bits(out)[1])


@pytest.mark.parametrize("name", ["ver_fp8_ordered", "dec_d256_ordered", "dec_fp8_d256_ordered"])
def test_heaviest_first_rows_equal_split_order_rows(mid, name):
    # the full call (more than two items per SM) takes its items heaviest first; two of its
    # sequences alone (a handful of items) take them in split order: same bits
    w, dw = mid(name)
    desc = b.describe(w.cfg.rows, w.cfg.n_head, w.cfg.n_head_kv, w.cfg.meta.get("head_dim", w.cfg.head_dim),
                      w.cfg.page_size, w.cfg.kv_dtype)
    assert "item_order" in desc
    out, err = dw.run()
    assert err == 0
    base = bits(out)
    for g in (int(np.argmax(w.seq_lens)), int(np.argmin(w.seq_lens))):
        o, err = dw.run(q=dw.q[g:g + 1], table=dw.table[g:g + 1], lens=dw.lens[g:g + 1])
        assert err == 0
        assert np.array_equal(bits(o)[0], base[g]), f"group {g} alone"


def test_repeated_calls_are_bit_identical(mid):
    w, dw = mid("dec128")
    a, _ = dw.run()
    for _ in range(3):
        c, _ = dw.run()
        assert np.array_equal(bits(a), bits(c))


@pytest.mark.parametrize("name", ["ver_fp8", "ver_bf16", "ver_wide_d256", "ver_fp8_d256"])
def test_verified_rows_equal_decode_rows_bit_for_bit(mid, name):
    # "Adding a model", step 4: every verified row must equal the decode
    # step's row bit for bit, or speculation is not lossless.  Row r of a
    # verify round over final length L is the decode step with length L-R+r+1.
    w, dw = mid(name)
    R = w.cfg.rows
    ver, err = dw.run()
    assert err == 0
    vb = bits(ver)
    for r in range(R):
        dec_cfg = wl.Config(name + "_dec", w.groups, 1, w.cfg.n_head, w.cfg.n_head_kv, w.cfg.head_dim,
                            w.cfg.page_size, w.cfg.kv_dtype, 0, "fixed:1", pages_per_seq=w.pages_per_seq)
        q = dw.q[:, r:r + 1].contiguous()
        lens = dw.lens - R + r + 1
        out = b.attn_paged(q, dw.k, dw.v, dw.table, lens, rows=1, n_head=dec_cfg.n_head,
                           n_head_kv=dec_cfg.n_head_kv, head_dim=dec_cfg.head_dim, page_size=dec_cfg.page_size,
                           scale=w.cfg.scale, kv_dtype=dec_cfg.kv_dtype, k_scales=dw.ks, v_scales=dw.vs)
        torch.cuda.synchronize()
        assert np.array_equal(bits(out)[:, 0], vb[:, r]), f"{name}: row {r} differs from its decode step"


# ------------------------------------------------------------------ errors never fault

def test_q_beyond_f16_range_flags_only_the_fp8_wide_tile(mid):
    """fp8 pools with head_dim 256 on the mma.sync wide tile (prefill chunks
    whose GQA ratio does not tile 128 rows) round q to f16: an element past its
    range raises RAD_ERRW_QRANGE (the other rows still match the oracle).  The
    tcgen05 e4m3 kernels split q exactly into two e4m3 terms with a per-row
    power-of-two scale and raise nothing, at either head_dim."""
    big = 100352.0   # a bf16 value past the f16 maximum (65504)
    for name, flagged in (("prefill_fp8_d256_r3", True), ("prefill_fp8_d256", False), ("dec_fp8_d256", False),
                          ("dec_fp8_ratio1", False)):
        w, dw = mid(name)
        q = w.q.copy()
        q[0, 0, 0, 5] = np.array([big], dtype=np.float32).view(np.uint32)[0] >> 16   # bf16 bits
        qd = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).view(torch.bfloat16).cuda()
        out, err = dw.run(q=qd)
        if flagged:
            assert err & b.RAD_ERRW_QRANGE
            ref = oracle_rows(w)
            o = as_f64(out)
            assert_parity(o[:, 1:], ref.out[:, 1:], True, name)   # rows of the other tokens
        else:
            assert err == 0
            assert np.all(np.isfinite(as_f64(out)))


def _bf16_bits(x):
    """float array -> bf16 bit patterns (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("name", ["ver_fp8", "ver_fp8_d256", "dec_fp8_ratio1", "dec_fp8_d256", "prefill_fp8"])
def test_fp8_query_row_scales_at_the_extremes(mid, name):
    """The e4m3 kernels split each query row q into two e4m3 terms of q 2^k,
    k from the row's largest magnitude (the split kernels gather it from four
    quarters of the row).  Rows of zeros, of bf16 subnormals, of huge values,
    and rows whose largest element sits alone in the last quarter must match
    the oracle like any other."""
    import copy
    w, dw = mid(name)
    c = w.cfg
    D = c.meta.get("head_dim", c.head_dim)
    q = w.q.copy()
    rng = np.random.default_rng(7)
    picks = [(0, t) for t in range(4)] if c.rows >= 4 else [(g, 0) for g in range(min(4, w.groups))]
    kinds = ["zero", "subnormal", "huge", "lone_max"]
    for (g, t), kind in zip(picks, kinds):
        for h in range(c.n_head):
            if kind == "zero":
                row = np.zeros(D)
            elif kind == "subnormal":
                row = rng.standard_normal(D) * 1e-39        # below bf16's smallest normal (1.2e-38)
            elif kind == "huge":
                row = rng.standard_normal(D) * 1e20
            else:
                row = rng.standard_normal(D) * 1e-3
                row[D - 3] = 3e3                              # the last quarter's element dominates
            q[g, t, h] = _bf16_bits(row)
    w2 = copy.copy(w)
    w2.q = q
    qd = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).view(torch.bfloat16).cuda()
    out, err = dw.run(q=qd)
    assert err == 0
    assert_parity(as_f64(out), oracle_rows(w2).out, True, name)


def test_bad_inputs_flag_errors_and_zero_only_their_group(mid):
    w, dw = mid("dec128")
    good, _ = dw.run()
    gb = bits(good)
    # a page id past the pool in group 8 (3001 keys: several splits)
    table = dw.table.clone()
    table[8, 100] = w.num_pages + 5
    o, err = dw.run(table=table)
    assert err == b.RAD_ERRW_PAGE
    ob = bits(o)
    assert np.all(ob[8] == 0) and np.array_equal(ob[:8], gb[:8])
    # negative page id in group 3 (17 keys: one split)
    table = dw.table.clone()
    table[3, 1] = -1
    o, err = dw.run(table=table)
    assert err == b.RAD_ERRW_PAGE
    ob = bits(o)
    assert np.all(ob[3] == 0) and np.array_equal(np.delete(ob, 3, 0), np.delete(gb, 3, 0))
    # seq_len 0 (< rows) and seq_len past the page table's capacity
    lens = dw.lens.clone()
    lens[0] = 0
    lens[5] = 200 * 16 + 1
    o, err = dw.run(lens=lens)
    assert err == b.RAD_ERRW_SEQLEN
    ob = bits(o)
    assert np.all(ob[0] == 0) and np.all(ob[5] == 0)
    keep = [1, 2, 3, 4, 6, 7, 8]
    assert np.array_equal(ob[keep], gb[keep])


def test_verify_bad_page_in_a_late_split_zeroes_every_row(mid):
    w, dw = mid("ver_fp8")
    good, _ = dw.run()
    table = dw.table.clone()
    table[4, 120] = 1 << 30
    o, err = dw.run(table=table)
    assert err == b.RAD_ERRW_PAGE
    ob, gb = bits(o), bits(good)
    assert np.all(ob[4] == 0) and np.array_equal(ob[:4], gb[:4])


@pytest.mark.parametrize("name", ["chunk_split", "prefill", "prefill_fp8_d256", "prefill_fp8", "prefill_d256",
                                  "prefill_fp8_d256_r3"])
def test_bad_last_page_zeroes_rows_of_every_query_tile(mid, name):
    # Calls with several query tiles per KV head: the early tiles never load
    # the last page, yet a bad id there zeroes every row of the group.
    w, dw = mid(name)
    good, _ = dw.run()
    g = w.groups - 1
    last = (int(w.seq_lens[g]) - 1) // w.cfg.page_size
    table = dw.table.clone()
    table[g, last] = -2
    o, err = dw.run(table=table)
    assert err == b.RAD_ERRW_PAGE
    ob, gb = bits(o), bits(good)
    assert np.all(ob[g] == 0) and np.array_equal(ob[:g], gb[:g])


@pytest.mark.parametrize("name", ["prefill", "dec128", "ver_fp8", "chunk_split", "prefill_fp8", "prefill_d256"])
@pytest.mark.parametrize("scale", [0.0, -0.07])
def test_zero_and_negative_scales_match_oracle(mid, name, scale):
    # scale 0: every visible key weighs the same; scale < 0 reverses the order
    # of the logits (the row max is taken after scaling).
    w, dw = mid(name)
    out, err = dw.run(scale=scale)
    assert err == 0
    ref = oracle_rows(w, scale=scale)
    assert_parity(as_f64(out), ref.out, dw.fp8, f"{name} scale {scale}")


def test_refused_shapes_write_nothing(mid):
    w, dw = mid("dec128")
    canary = torch.full((w.groups, 1, 32, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    for kw, code in ((dict(head_dim=96), b.RAD_E_DTYPE), (dict(page_size=24), b.RAD_E_DTYPE),
                     (dict(rows=0), b.RAD_E_SHAPE)):
        args = dict(rows=1, n_head=32, n_head_kv=8, head_dim=128, page_size=16, scale=0.08,
                    kv_dtype=b.RAD_KV_BF16)
        args.update(kw)
        with pytest.raises(b.RadAttnError) as e:
            b.attn_paged(dw.q, dw.k, dw.v, dw.table, dw.lens, out=canary, **args)
        assert e.value.status == code
    torch.cuda.synchronize()
    assert torch.all(canary == 7.0)


def test_head_dim_is_read_from_metadata_not_derived(mid):
    w, dw = mid("dec256")
    meta = w.cfg.meta
    derived = meta["n_embd"] // w.cfg.n_head      # 213 on the hybrid
    assert derived != meta["head_dim"]
    with pytest.raises(b.RadAttnError) as e:
        b.attn_paged(dw.q, dw.k, dw.v, dw.table, dw.lens, rows=1, n_head=16, n_head_kv=2,
                     head_dim=derived, page_size=32, scale=0.06)
    assert e.value.status == b.RAD_E_DTYPE


# ------------------------------------------------------------------ streams and graphs

def test_side_stream_and_cuda_graph_replay_are_bit_identical(mid):
    w, dw = mid("ver_fp8")
    eager, _ = dw.run()
    c = w.cfg
    out = torch.empty_like(eager)
    ws = torch.empty(b.workspace_bytes(w.groups, c.rows, c.n_head, c.n_head_kv, c.head_dim, c.page_size,
                                       w.pages_per_seq, c.kv_dtype), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dw.run(out=out, workspace=ws, stream=s)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), bits(eager))
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        b.attn_paged(dw.q, dw.k, dw.v, dw.table, dw.lens, rows=c.rows, n_head=c.n_head,
                     n_head_kv=c.n_head_kv, head_dim=c.head_dim, page_size=c.page_size, scale=c.scale,
                     kv_dtype=c.kv_dtype, k_scales=dw.ks, v_scales=dw.vs, out=out, workspace=ws)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), bits(eager))
