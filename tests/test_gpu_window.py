"""GPU tests of rad_attn_paged_window: attention over a sliding-window KV
group (RAD_KV_WINDOW, "Radiance architecture plugins", section "Declare:
buffers and KV groups"), where each row sees only its last W keys.

Expected values come from the fp64 oracle with the same window.  K/V slots
below each sequence's window start and the page ids of pages wholly below it
are poisoned (NaN codes, invalid ids): the kernels must never use them."""
import numpy as np
import pytest
import torch

from gpu_util import DevWorkload, as_f64, assert_parity, bits, oracle_rows
from paged_kv_attention_02_gb300 import binding as b
from paged_kv_attention_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

# (config, window): every call family, windows below, at and past a page, a
# stage and a split, and windows smaller than a verify round.
WIN = {
    "dec128_w1000": (wl.Config("dec128_w1000", 8, 1, 32, 8, 128, 16, wl.KV_BF16, 201,
                               "fixed:1,15,1000,1001,1024,1025,3000,5000", pages_per_seq=320), 1000),
    "dec128_w1": (wl.Config("dec128_w1", 4, 1, 8, 2, 128, 16, wl.KV_BF16, 202, "fixed:1,2,700,2049",
                            pages_per_seq=130), 1),
    "dec_fp8_d256_w700": (wl.Config("dec_fp8_d256_w700", 4, 1, 16, 2, 256, 32, wl.KV_FP8_E4M3, 203,
                                    "fixed:40,700,1900,4100", pages_per_seq=130,
                                    meta=dict(head_dim=256, n_embd=3408)), 700),
    "dec_d256_w48": (wl.Config("dec_d256_w48", 3, 1, 16, 2, 256, 32, wl.KV_BF16, 204, "fixed:47,48,2600",
                               pages_per_seq=90), 48),
    "ver_fp8_w513": (wl.Config("ver_fp8_w513", 5, 8, 32, 8, 128, 16, wl.KV_FP8_E4M3, 205,
                               "fixed:8,9,600,2100,4000", pages_per_seq=260), 513),
    # head_dim-128 fp8 decode (the tcgen05 split kernel, 16 query rows): windows across its
    # 4096-key splits, and one narrower than a 32-slot page
    "dec_fp8_w1000": (wl.Config("dec_fp8_w1000", 6, 1, 32, 8, 128, 16, wl.KV_FP8_E4M3, 214,
                                "fixed:1,15,1000,4095,4097,9000", pages_per_seq=570), 1000),
    "dec_fp8_p32_w20": (wl.Config("dec_fp8_p32_w20", 4, 1, 16, 4, 128, 32, wl.KV_FP8_E4M3, 215,
                                  "fixed:3,21,2100,4200", pages_per_seq=140), 20),
    "ver_bf16_w4": (wl.Config("ver_bf16_w4", 3, 8, 8, 2, 128, 16, wl.KV_BF16, 206, "fixed:8,30,1500",
                              pages_per_seq=100), 4),
    "ver_d256_w300": (wl.Config("ver_d256_w300", 3, 8, 16, 2, 256, 32, wl.KV_BF16, 207, "fixed:8,700,2500",
                                pages_per_seq=80), 300),
    "chunk_w300": (wl.Config("chunk_w300", 2, 40, 8, 2, 128, 16, wl.KV_BF16, 208, "fixed:40,2500",
                             pages_per_seq=160), 300),
    "prefill_tc_w257": (wl.Config("prefill_tc_w257", 3, 300, 8, 2, 128, 16, wl.KV_BF16, 209,
                                  "fixed:300,1000,2500", pages_per_seq=160), 257),
    "prefill_tc_w64": (wl.Config("prefill_tc_w64", 1, 520, 4, 1, 128, 32, wl.KV_BF16, 210, "fixed:1800",
                                 pages_per_seq=60), 64),
    "prefill_fp8_d256_w100": (wl.Config("prefill_fp8_d256_w100", 1, 260, 4, 1, 256, 32, wl.KV_FP8_E4M3,
                                        211, "fixed:900", pages_per_seq=30), 100),
    "prefill_d256_w100": (wl.Config("prefill_d256_w100", 2, 300, 16, 2, 256, 32, wl.KV_BF16, 216,
                                    "fixed:300,1800", pages_per_seq=60), 100),
    "prefill_fp8_w257": (wl.Config("prefill_fp8_w257", 3, 300, 8, 2, 128, 16, wl.KV_FP8_E4M3, 212,
                                   "fixed:300,1000,2500", pages_per_seq=160), 257),
    "prefill_fp8_w64": (wl.Config("prefill_fp8_w64", 1, 520, 4, 1, 128, 32, wl.KV_FP8_E4M3, 213, "fixed:1800",
                                  pages_per_seq=60), 64),
}


def poison_below_window(w: wl.Workload, window: int):
    """NaN codes in every slot below row 0's first visible key of each
    sequence; returns a page table whose ids wholly below it are invalid
    (alternately negative and past the pool)."""
    nan = wl.BF16_NAN if w.cfg.kv_dtype == wl.KV_BF16 else wl.E4M3_NAN
    P = w.cfg.page_size
    table = w.page_table.copy()
    for g in range(w.groups):
        n0 = int(w.seq_lens[g]) - w.cfg.rows + 1
        lo = n0 - window if n0 > window else 0
        for j in range(lo):
            pg = w.page_table[g, j // P]
            w.k_pool[pg, j % P] = nan
            w.v_pool[pg, j % P] = nan
        table[g, :lo // P] = -3 if g % 2 == 0 else w.num_pages + 11
    return table


@pytest.fixture(scope="module")
def win():
    cache = {}

    def get(name):
        if name not in cache:
            cfg, W = WIN[name]
            w = wl.make_workload(cfg, poison=True)
            w.page_table = poison_below_window(w, W)
            cache[name] = (w, DevWorkload(w), W)
        return cache[name]
    return get


@pytest.mark.parametrize("name", list(WIN))
def test_window_matches_oracle_everywhere(win, name):
    w, dw, W = win(name)
    out, err = dw.run(window=W)
    assert err == 0
    ref = oracle_rows(w, window=W)
    assert ref.err_word == 0
    assert_parity(as_f64(out), ref.out, dw.fp8, name)


@pytest.mark.parametrize("name", ["ver_fp8_w513", "prefill_tc_w257", "dec_d256_w48", "prefill_fp8_w257"])
def test_window_zero_and_window_past_the_context_equal_the_plain_op(name):
    w = wl.make_workload(WIN[name][0], poison=True)      # nothing poisoned below a window
    dw = DevWorkload(w)
    base, _ = dw.run()
    for W in (0, int(w.seq_lens.max()), 1 << 30):
        o, err = dw.run(window=W)
        assert err == 0
        assert np.array_equal(bits(o), bits(base)), f"window {W}"


@pytest.mark.parametrize("name", ["ver_fp8_w513", "ver_bf16_w4", "ver_d256_w300"])
def test_windowed_verified_rows_equal_windowed_decode_rows_bit_for_bit(win, name):
    w, dw, W = win(name)
    R = w.cfg.rows
    ver, err = dw.run(window=W)
    assert err == 0
    vb = bits(ver)
    c = w.cfg
    for r in range(R):
        out = b.attn_paged_window(dw.q[:, r:r + 1].contiguous(), dw.k, dw.v, dw.table, dw.lens - R + r + 1,
                                  rows=1, n_head=c.n_head, n_head_kv=c.n_head_kv, head_dim=c.head_dim,
                                  page_size=c.page_size, scale=c.scale, window=W, kv_dtype=c.kv_dtype,
                                  k_scales=dw.ks, v_scales=dw.vs)
        torch.cuda.synchronize()
        assert np.array_equal(bits(out)[:, 0], vb[:, r]), f"{name}: row {r} differs from its decode step"


@pytest.mark.parametrize("name", ["dec128_w1000", "ver_fp8_w513", "prefill_tc_w257", "prefill_fp8_w64"])
def test_windowed_rows_are_bit_identical_alone_and_batched(win, name):
    w, dw, W = win(name)
    out, _ = dw.run(window=W)
    for g in range(w.groups):
        o, err = dw.run(q=dw.q[g:g + 1], table=dw.table[g:g + 1], lens=dw.lens[g:g + 1], window=W)
        assert err == 0
        assert np.array_equal(bits(o)[0], bits(out)[g]), f"{name}: group {g}"


@pytest.mark.parametrize("name", ["dec128_w1000", "ver_fp8_w513", "chunk_w300", "prefill_tc_w257"])
def test_bad_page_inside_the_window_zeroes_its_group(win, name):
    w, dw, W = win(name)
    good, _ = dw.run(window=W)
    g = w.groups - 1
    P = w.cfg.page_size
    n0 = int(w.seq_lens[g]) - w.cfg.rows + 1
    first = (n0 - W if n0 > W else 0) // P            # the page holding row 0's first visible key
    table = dw.table.clone()
    table[g, first] = w.num_pages + 1
    o, err = dw.run(table=table, window=W)
    assert err == b.RAD_ERRW_PAGE
    ob, gb = bits(o), bits(good)
    assert np.all(ob[g] == 0) and np.array_equal(ob[:g], gb[:g])


def test_negative_window_is_refused(win):
    w, dw, W = win("dec128_w1")
    canary = torch.full((w.groups, 1, 8, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(b.RadAttnError) as e:
        dw.run(window=-1, out=canary)
    assert e.value.status == b.RAD_E_ARG
    torch.cuda.synchronize()
    assert torch.all(canary == 5.0)


def _ex_args(dw, window, out, ws, err, struct_size=None):
    import ctypes
    c = dw.w.cfg
    a = b.RadAttnPagedArgs()
    a.struct_size = ctypes.sizeof(b.RadAttnPagedArgs) if struct_size is None else struct_size
    a.q, a.k_pool, a.v_pool = dw.q.data_ptr(), dw.k.data_ptr(), dw.v.data_ptr()
    a.page_table, a.seq_lens = dw.table.data_ptr(), dw.lens.data_ptr()
    a.groups, a.rows, a.n_head, a.n_head_kv = dw.w.groups, c.rows, c.n_head, c.n_head_kv
    a.head_dim, a.page_size = c.head_dim, c.page_size
    a.pages_per_seq, a.num_pages = dw.table.shape[1], dw.k.shape[0]
    a.scale, a.kv_dtype = c.scale, c.kv_dtype
    a.k_scales = dw.ks.data_ptr() if dw.ks is not None else None
    a.v_scales = dw.vs.data_ptr() if dw.vs is not None else None
    a.out, a.workspace = out.data_ptr(), ws.data_ptr()
    a.workspace_bytes = ws.numel()
    a.err_word = err.data_ptr()
    a.window = window
    return a


@pytest.mark.parametrize("name", ["ver_fp8_w513", "dec128_w1000"])
def test_ex_entry_equals_the_window_and_plain_calls(win, name):
    import ctypes
    w, dw, W = win(name)
    c = w.cfg
    ref, _ = dw.run(window=W)
    need = b.workspace_bytes(w.groups, c.rows, c.n_head, c.n_head_kv, c.head_dim, c.page_size, w.pages_per_seq,
                             c.kv_dtype)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(ref, 3.0)
    assert b.attn_paged_ex(_ex_args(dw, W, out, ws, err)) == b.RAD_OK
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and np.array_equal(bits(out), bits(ref))
    # the base call's struct (ending before `window`): no window, whatever the field holds
    plain = DevWorkload(wl.make_workload(WIN[name][0], poison=True))
    pref, _ = plain.run()
    base = b.RadAttnPagedArgs.err_word.offset + ctypes.sizeof(ctypes.c_void_p)
    out2 = torch.full_like(ref, 3.0)
    assert b.attn_paged_ex(_ex_args(plain, 77, out2, ws, err, struct_size=base)) == b.RAD_OK
    torch.cuda.synchronize()
    assert np.array_equal(bits(out2), bits(pref))
