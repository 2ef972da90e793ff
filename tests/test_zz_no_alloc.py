"""rad_attn_paged_noalloc on the GPU, through the C ABI.

The entry point serves callers that cannot allocate device memory per call (a
runtime whose device memory is planned once at load time, or code handed only
the call's tensors); its scratch is a fixed array owned by the library.  These
checks compare it with rad_attn_paged (caller-provided workspace) on the same
inputs, on two calls in a row so that the second sees the scratch the first
left behind.  This file is collected last and builds everything it needs, so
it runs the same alone in a fresh process or after the other tests.
"""
import numpy as np
import pytest
import torch

from gpu_util import DevWorkload, as_f64, assert_parity
from paged_kv_attention_02_gb300 import binding as b
from paged_kv_attention_02_gb300 import workloads as wl
from paged_kv_attention_02_gb300.build import build_library

pytestmark = pytest.mark.gpu

CASES = [
    # several splits per sequence, ragged last pages, bf16 and fp8, two call families
    wl.Config("noalloc_decode", 9, 1, 32, 8, 128, 16, wl.KV_BF16, 201,
              "fixed:1,15,16,17,511,512,513,1500,3001", pages_per_seq=200),
    wl.Config("noalloc_verify_fp8", 5, 8, 32, 8, 128, 16, wl.KV_FP8_E4M3, 202, "fixed:8,9,520,1000,2050",
              pages_per_seq=130),
]


@pytest.fixture(scope="module", autouse=True)
def library():
    build_library()
    b.load()


@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(cfg):
    w = wl.make_workload(cfg, poison=True)
    assert b.workspace_bytes(w.groups, cfg.rows, cfg.n_head, cfg.n_head_kv, cfg.head_dim, cfg.page_size,
                             w.pages_per_seq, cfg.kv_dtype) <= b.NOALLOC_SCRATCH_BYTES
    dw = DevWorkload(w)
    ref, err = dw.run()
    assert err == 0
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        e = torch.zeros(1, dtype=torch.int32, device="cuda")
        b.attn_paged_noalloc(dw.q, dw.k, dw.v, dw.table, dw.lens, rows=cfg.rows, n_head=cfg.n_head,
                             n_head_kv=cfg.n_head_kv, head_dim=cfg.head_dim, page_size=cfg.page_size,
                             scale=cfg.scale, kv_dtype=cfg.kv_dtype, k_scales=dw.ks, v_scales=dw.vs,
                             out=out, err_word=e)
        torch.cuda.synchronize()
        assert int(e.item()) == 0, f"call {call}: error word {int(e.item())}"
        assert_parity(as_f64(out), as_f64(ref), dw.fp8, f"{cfg.name} call {call}")


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
