"""The device error word's time-out bit, made to fire on purpose.

Every wait inside the kernels is bounded.  When one runs out the kernel sets
RAD_ERRW_TIMEOUT ("kern manifest v7", $defs.Fill `error`: the one-word error
flag the host reads after a call), unwinds its warp roles and returns, so the
context stays usable.  rad_attn_paged_fault_test lowers the wait limit and
makes the first CTA's K producer leave its first tile unissued: nothing ever
completes the waits on that tile, they run out, and the call must come back
with the bit set.  The same inputs then run normally on the same stream.
"""
import time

import numpy as np
import pytest
import torch

from gpu_util import DevWorkload, bits
from paged_kv_attention_02_gb300 import binding as b
from paged_kv_attention_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

LIMIT_NS = 50_000_000   # 50 ms per wait


def fault_call(dw, fault, limit_ns=LIMIT_NS, stream=None):
    c = dw.w.cfg
    out = torch.full_like(dw.q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.attn_paged_fault_test(dw.q, dw.k, dw.v, dw.table, dw.lens, rows=c.rows, n_head=c.n_head,
                            n_head_kv=c.n_head_kv, head_dim=c.head_dim, page_size=c.page_size, scale=c.scale,
                            wait_limit_ns=limit_ns, fault=fault, kv_dtype=c.kv_dtype, out=out, err_word=err,
                            stream=stream)
    torch.cuda.synchronize()
    return out, int(err.item())


def test_a_wait_that_runs_out_sets_the_timeout_bit_and_the_next_call_is_unaffected():
    w = wl.make_workload("tiny_decode", poison=True)
    c = w.cfg
    assert "attn_split_bf16_tc05" in b.describe(c.rows, c.n_head, c.n_head_kv, c.head_dim, c.page_size, c.kv_dtype)
    dw = DevWorkload(w)
    good, err = dw.run()
    assert err == 0

    # the hook with no fault and a lowered limit is the plain call
    out, err = fault_call(dw, b.RAD_FAULT_NONE)
    assert err == 0
    assert np.array_equal(bits(out), bits(good))

    # the injected fault: CTA 0 runs the first item (sequence 0, KV head 0)
    s = torch.cuda.Stream()
    t0 = time.monotonic()
    out, err = fault_call(dw, b.RAD_FAULT_SKIP_FIRST_K_TILE, stream=s)
    elapsed = time.monotonic() - t0
    assert err & b.RAD_ERRW_TIMEOUT, f"error word {err}"
    assert err == b.RAD_ERRW_TIMEOUT
    assert elapsed < 10.0
    ratio = c.n_head // c.n_head_kv
    ob, gb = bits(out), bits(good)
    # the other CTAs' items are untouched by the fault
    assert np.array_equal(ob[1:], gb[1:])
    assert np.array_equal(ob[0, :, ratio:], gb[0, :, ratio:])

    # the context is usable: the next calls, on the same stream and on the
    # default one, give the clean bits again
    out, err = fault_call(dw, b.RAD_FAULT_NONE, limit_ns=0, stream=s)
    assert err == 0
    assert np.array_equal(bits(out), bits(good))
    again, err = dw.run()
    assert err == 0
    assert np.array_equal(bits(again), bits(good))
