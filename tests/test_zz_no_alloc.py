"""rad_attn_paged_noalloc on the GPU, through the C ABI.

The entry point serves callers that cannot allocate device memory per call (a
runtime whose device memory is planned once at load time, or code handed only
the call's tensors); its scratch is a fixed array owned by the library and
shared by every call.  Both entry points run the same kernels on the same
inputs, so the no-alloc output must equal rad_attn_paged's bit for bit, and
both must match the oracle.

Each check first leaves the shared scratch dirty: a call of the same shape
whose K pool is all NaN (so every partial it writes is NaN), or a call of
another shape and pool type with longer contexts.  A combine that read a slot
the checked call did not write would then change the checked call's bits.
The checked call then runs twice in a row.  This file is collected last and
builds everything it needs, so it runs the same alone in a fresh process or
after the other tests.
"""
import numpy as np
import pytest
import torch

from gpu_util import DevWorkload, as_f64, assert_parity, bits, oracle_rows
from paged_kv_attention_02_gb300 import binding as b
from paged_kv_attention_02_gb300 import workloads as wl
from paged_kv_attention_02_gb300.build import build_library

pytestmark = pytest.mark.gpu

CASES = {
    # several splits per sequence, ragged last pages, bf16 and fp8, two call families
    "noalloc_decode": wl.Config("noalloc_decode", 9, 1, 32, 8, 128, 16, wl.KV_BF16, 201,
                                "fixed:1,15,16,17,511,512,513,1500,3001", pages_per_seq=200),
    "noalloc_verify_fp8": wl.Config("noalloc_verify_fp8", 5, 8, 32, 8, 128, 16, wl.KV_FP8_E4M3, 202,
                                    "fixed:8,9,520,1000,2050", pages_per_seq=130),
    "noalloc_decode_d256": wl.Config("noalloc_decode_d256", 4, 1, 16, 2, 256, 32, wl.KV_BF16, 203,
                                     "fixed:33,700,2500,5000", pages_per_seq=160,
                                     meta=dict(head_dim=256, n_embd=3408)),
    # the other shape of each pair: longer contexts, more splits
    "noalloc_long_fp8": wl.Config("noalloc_long_fp8", 6, 8, 32, 8, 128, 16, wl.KV_FP8_E4M3, 204,
                                  "fixed:9000,12000,3000,16000,7000,5000", pages_per_seq=1000),
    "noalloc_long_bf16": wl.Config("noalloc_long_bf16", 12, 1, 32, 8, 128, 16, wl.KV_BF16, 205,
                                   "uniform:6000,16000", pages_per_seq=1000),
}
# (checked case, the other-shape call run before it)
PAIRS = [("noalloc_decode", "noalloc_long_fp8"), ("noalloc_verify_fp8", "noalloc_long_bf16"),
         ("noalloc_decode_d256", "noalloc_long_fp8")]


@pytest.fixture(scope="module", autouse=True)
def library():
    build_library()
    b.load()


def need_of(w):
    c = w.cfg
    return b.workspace_bytes(w.groups, c.rows, c.n_head, c.n_head_kv, c.meta.get("head_dim", c.head_dim),
                             c.page_size, w.pages_per_seq, c.kv_dtype)


def noalloc(dw, k=None):
    """One rad_attn_paged_noalloc call on dw's inputs (k: another K pool);
    returns (out, error word)."""
    c = dw.w.cfg
    out = torch.full((dw.w.groups, c.rows, c.n_head, c.meta.get("head_dim", c.head_dim)), float("nan"),
                     dtype=torch.bfloat16, device="cuda")
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.attn_paged_noalloc(dw.q, dw.k if k is None else k, dw.v, dw.table, dw.lens, rows=c.rows, n_head=c.n_head,
                         n_head_kv=c.n_head_kv, head_dim=c.meta.get("head_dim", c.head_dim),
                         page_size=c.page_size, scale=c.scale, kv_dtype=c.kv_dtype, k_scales=dw.ks,
                         v_scales=dw.vs, out=out, err_word=e)
    torch.cuda.synchronize()
    return out, int(e.item())


def nan_pool(dw):
    """A K pool of the same shape and type whose every element is NaN."""
    if dw.fp8:
        return torch.full_like(dw.k, 0x7F)            # e4m3fn NaN code
    return torch.full_like(dw.k, float("nan"))


@pytest.mark.parametrize("pair", PAIRS, ids=[p[0] for p in PAIRS])
def test_noalloc_equals_workspace_entry_point_bit_for_bit_over_a_dirty_scratch(pair):
    name, other = pair
    w = wl.make_workload(CASES[name], poison=True)
    wo = wl.make_workload(CASES[other], poison=True)
    assert 0 < need_of(w) <= b.NOALLOC_SCRATCH_BYTES
    assert 0 < need_of(wo) <= b.NOALLOC_SCRATCH_BYTES
    dw, dwo = DevWorkload(w), DevWorkload(wo)
    ref, err = dw.run()                               # rad_attn_paged, caller-provided workspace
    assert err == 0
    oracle = oracle_rows(w)
    assert oracle.err_word == 0
    assert_parity(as_f64(ref), oracle.out, dw.fp8, f"{name} (workspace entry point)")

    # 1. the same shape with an all-NaN K pool: every partial slot it writes is NaN
    dirty, err = noalloc(dw, k=nan_pool(dw))
    assert err == 0
    assert torch.isnan(dirty.float()).any()
    for call in range(2):
        out, err = noalloc(dw)
        assert err == 0, f"{name} after a NaN call, call {call}: error word {err}"
        assert np.array_equal(bits(out), bits(ref)), f"{name} after a NaN call, call {call}"
    # 2. another shape and pool type, with more and longer splits
    o2, err = noalloc(dwo)
    assert err == 0
    r2, _ = dwo.run()
    assert np.array_equal(bits(o2), bits(r2)), other
    for call in range(2):
        out, err = noalloc(dw)
        assert err == 0, f"{name} after {other}, call {call}: error word {err}"
        assert np.array_equal(bits(out), bits(ref)), f"{name} after {other}, call {call}"
    assert_parity(as_f64(out), oracle.out, dw.fp8, f"{name} (no-alloc entry point)")


def test_noalloc_refuses_calls_beyond_its_scratch():
    cfg = wl.CONFIGS["batched_decode"]
    need = b.workspace_bytes(cfg.groups, cfg.rows, cfg.n_head, cfg.n_head_kv, cfg.head_dim, cfg.page_size,
                             cfg.pages_per_seq, cfg.kv_dtype)
    assert need > b.NOALLOC_SCRATCH_BYTES
    # pointers are never touched: the size check comes first
    q = torch.zeros(cfg.groups, 1, cfg.n_head, cfg.head_dim, dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros(4, cfg.page_size, cfg.n_head_kv, cfg.head_dim, dtype=torch.bfloat16, device="cuda")
    table = torch.zeros(cfg.groups, cfg.pages_per_seq, dtype=torch.int32, device="cuda")
    lens = torch.ones(cfg.groups, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 3.0)
    with pytest.raises(b.RadAttnError) as ex:
        b.attn_paged_noalloc(q, pool, pool, table, lens, rows=1, n_head=cfg.n_head, n_head_kv=cfg.n_head_kv,
                             head_dim=cfg.head_dim, page_size=cfg.page_size, scale=cfg.scale, out=out)
    assert ex.value.status == b.RAD_E_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
