"""The C-ABI library without a GPU: it builds, loads, exports every function
include/rad_attn.h declares, and its host-side checks return the documented
status codes before touching any device."""
import ctypes
import os
import re

import numpy as np
import pytest

from paged_kv_attention_02_gb300 import binding as b
from paged_kv_attention_02_gb300 import workloads as wl
from paged_kv_attention_02_gb300.build import build_library

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "rad_attn.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    build_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rad_attn\w*)\s*\(", text)))


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert set(names) == set(b.EXPORTS)
    lib = ctypes.CDLL(b.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version():
    assert b.status_string(b.RAD_OK) == "RAD_OK"
    assert b.status_string(b.RAD_E_DTYPE) == "RAD_E_DTYPE"
    assert "sm_103a" in b.version()


def good_args(**over):
    a = dict(q_ptr=4096, k_ptr=8192, v_ptr=12288, table_ptr=16384, lens_ptr=20480, groups=4, rows=1,
             n_head=8, n_head_kv=2, head_dim=128, page_size=16, pages_per_seq=19, num_pages=64,
             scale=0.088, kv_dtype=b.RAD_KV_BF16, ks_ptr=0, vs_ptr=0, out_ptr=24576, ws_ptr=1 << 20,
             ws_bytes=1 << 30, err_ptr=0, stream_ptr=0)
    a.update(over)
    return a


@pytest.mark.parametrize("over,code", [
    (dict(rows=0), b.RAD_E_SHAPE),
    (dict(groups=0), b.RAD_E_SHAPE),
    (dict(n_head=6, n_head_kv=4), b.RAD_E_SHAPE),
    (dict(pages_per_seq=0), b.RAD_E_SHAPE),
    (dict(num_pages=0), b.RAD_E_SHAPE),
    (dict(num_pages=1 << 30, page_size=16), b.RAD_E_SHAPE),
    (dict(head_dim=96), b.RAD_E_DTYPE),
    (dict(head_dim=213), b.RAD_E_DTYPE),
    (dict(page_size=24), b.RAD_E_DTYPE),
    (dict(kv_dtype=7), b.RAD_E_DTYPE),
    (dict(q_ptr=0), b.RAD_E_ARG),
    (dict(out_ptr=0), b.RAD_E_ARG),
    (dict(k_ptr=8200), b.RAD_E_ARG),
    (dict(kv_dtype=b.RAD_KV_FP8_E4M3), b.RAD_E_ARG),
    (dict(scale=float("nan")), b.RAD_E_ARG),
    (dict(ws_ptr=0), b.RAD_E_WORKSPACE),
    (dict(ws_bytes=16), b.RAD_E_WORKSPACE),
])
def test_host_checks_refuse_before_any_device_access(over, code):
    assert b.call_raw(**good_args(**over)) == code


def test_zero_rows_precedes_every_other_check():
    a = good_args(rows=0, q_ptr=0, head_dim=96, ws_ptr=0)
    assert b.call_raw(**a) == b.RAD_E_SHAPE


def test_valid_call_without_a_gpu_fails_loudly():
    assert b.call_raw(**good_args()) in (b.RAD_E_CUDA, b.RAD_E_DEVICE)


def test_workspace_sizes():
    # decode splits: a flag, (max, sum) and an accumulator row per query row
    # for every possible split of every (sequence, KV head)
    split_len = int(re.search(r"split_len=(\d+)", b.describe(1, 32, 8, 128, 16)).group(1))
    max_splits = -(-512 * 16 // split_len)
    ws = b.workspace_bytes(256, 1, 32, 8, 128, 16, 512)
    assert ws >= 256 * 8 * max_splits * (4 * 130 * 4 + 4)
    assert b.workspace_bytes(1, 2048, 32, 8, 128, 16, 512) == 0      # bf16 prefill: no split
    assert b.workspace_bytes(1, 2048, 32, 8, 128, 16, 512, b.RAD_KV_FP8_E4M3) == 256   # fp8: the item counter
    assert b.workspace_bytes(1, 2048, 32, 8, 256, 16, 512) == 0      # head_dim-256 prefill (tile kernel): none
    assert b.workspace_bytes(0, 1, 32, 8, 128, 16, 512) == 0
    assert b.workspace_bytes(4, 1, 8, 2, 96, 16, 19) == 0


def bf16_tc(head_dim: int = 128) -> bool:
    """Whether the library was built with the bf16 tcgen05 split kernel for this head_dim (a compile-time switch)."""
    return "split_bf16_tc05" in b.describe(8, 32, 8, head_dim, 16)


def test_describe_names_the_kernel_choice():
    # bf16 pools with head_dim 128: decode and verify shapes share one family, the
    # bf16 tcgen05 split kernel when it is built in, else the tile kernel's decode
    # (<= 8 query rows per KV head) and verify tiles
    if bf16_tc():
        assert "family=split_bf16_tc05" in b.describe(1, 32, 8, 128, 16)
        assert "family=split_bf16_tc05" in b.describe(8, 32, 8, 128, 16)
    else:
        assert "family=decode" in b.describe(1, 32, 8, 128, 16)
        assert "family=verify" in b.describe(8, 32, 8, 128, 16)
    # bf16 pools with head_dim 256: the same, on the kernel's head_dim-256 build
    if bf16_tc(256):
        assert "family=split_bf16_tc05 head_dim=256" in b.describe(1, 16, 2, 256, 32)
        assert "keys_per_tile=64" in b.describe(1, 16, 2, 256, 32)
        assert "family=split_bf16_tc05 head_dim=256" in b.describe(8, 32, 8, 256, 16)
    else:
        assert "family=decode" in b.describe(1, 32, 8, 256, 16)
        assert "family=verify" in b.describe(8, 32, 8, 256, 16)
    # fp8 pools with head_dim 256: the e4m3 tcgen05 split kernel's head_dim-256 build
    assert "family=split_tc05 head_dim=256" in b.describe(8, 16, 2, 256, 32, b.RAD_KV_FP8_E4M3)
    assert "keys_per_tile=64" in b.describe(1, 16, 2, 256, 32, b.RAD_KV_FP8_E4M3)
    # fp8 pools with head_dim 128: decode and verify shapes share the tcgen05 split kernel
    assert "family=split_tc05" in b.describe(8, 32, 8, 128, 16, b.RAD_KV_FP8_E4M3)
    assert "family=split_tc05" in b.describe(1, 8, 8, 128, 16, b.RAD_KV_FP8_E4M3)
    assert "split_len=0" in b.describe(2048, 32, 8, 128, 16)
    with pytest.raises(b.RadAttnError):
        b.describe(1, 32, 8, 96, 16)


def test_describe_names_the_item_order_kernel_where_it_runs():
    # uniform calls on the e4m3 split kernel (both head dims) and on the head_dim-256 bf16
    # build sort their items heaviest first when they have more than two a CTA; the
    # head_dim-128 bf16 build and ragged calls keep split order
    assert "item_order" in b.describe(8, 32, 8, 128, 16, b.RAD_KV_FP8_E4M3)
    assert "item_order" in b.describe(1, 16, 2, 256, 32, b.RAD_KV_FP8_E4M3)
    if bf16_tc(256):
        assert "item_order" in b.describe(1, 16, 2, 256, 32)
    assert "item_order" not in b.describe(1, 32, 8, 128, 16)
    assert "item_order" not in b.ex_describe(b.shape_args(4, 8, 32, 8, 128, 16, 64, b.RAD_KV_FP8_E4M3, ragged=True))


def test_args_struct_matches_the_c_layout(tmp_path):
    """The binding's RadAttnPagedArgs mirror has the header's size and offsets."""
    fields = [f for f, _ in b.RadAttnPagedArgs._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "rad_attn.h"\nint main(void) {\n'
                   '  printf("%zu\\n", sizeof(RadAttnPagedArgs));\n' +
                   "".join(f'  printf("%zu\\n", offsetof(RadAttnPagedArgs, {f}));\n' for f in fields) +
                   "  return 0;\n}\n")
    exe = tmp_path / "layout"
    import subprocess
    subprocess.check_call(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)])
    got = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    assert got[0] == ctypes.sizeof(b.RadAttnPagedArgs)
    assert got[1:] == [getattr(b.RadAttnPagedArgs, f).offset for f in fields]


def _ex_status(struct_size, tail=b"", groups=0):
    """Status of rad_attn_paged_ex for an otherwise empty call (no device access)."""
    buf = ctypes.create_string_buffer(ctypes.sizeof(b.RadAttnPagedArgs) + len(tail))
    args = b.RadAttnPagedArgs.from_buffer(buf)
    args.struct_size = struct_size
    args.groups, args.rows = groups, 1
    ctypes.memmove(ctypes.addressof(buf) + ctypes.sizeof(b.RadAttnPagedArgs), tail, len(tail))
    return int(b.load().rad_attn_paged_ex(ctypes.byref(args), None))


def test_ex_struct_size_rules():
    full = ctypes.sizeof(b.RadAttnPagedArgs)
    base = b.RadAttnPagedArgs.err_word.offset + ctypes.sizeof(ctypes.c_void_p)
    assert int(b.load().rad_attn_paged_ex(None, None)) == b.RAD_E_ARG
    assert _ex_status(0) == b.RAD_E_ARG
    assert _ex_status(base - 1) == b.RAD_E_ARG
    # the base call (no window field) and the full struct reach the scalar checks: groups = 0
    assert _ex_status(base) == b.RAD_E_SHAPE
    assert _ex_status(full) == b.RAD_E_SHAPE
    # a newer caller: zero fields past the known ones are accepted, a non-zero one is refused
    assert _ex_status(full + 8, tail=bytes(8)) == b.RAD_E_SHAPE
    assert _ex_status(full + 8, tail=b"\0\0\0\1\0\0\0\0") == b.RAD_E_ARG


def _general_args(rows=8, cu=0, tree=0, window=0, head_dim=128, kv_dtype=b.RAD_KV_BF16):
    """A filled RadAttnPagedArgs with fake (aligned, never dereferenced) pointers."""
    a = b.RadAttnPagedArgs()
    a.struct_size = ctypes.sizeof(b.RadAttnPagedArgs)
    fake = 1 << 20
    a.q = a.k_pool = a.v_pool = a.out = fake
    a.page_table = a.seq_lens = a.k_scales = a.v_scales = fake
    a.groups, a.rows, a.n_head, a.n_head_kv, a.head_dim = 4, rows, 32, 8, head_dim
    a.page_size, a.pages_per_seq, a.num_pages, a.scale, a.kv_dtype = 16, 64, 256, 0.08, kv_dtype
    a.cu_seqlens, a.tree_mask, a.window = cu or None, tree or None, window
    return a


def test_ragged_and_tree_calls_the_host_refuses_before_any_device_access():
    fake = 1 << 20
    st = lambda a: int(b.load().rad_attn_paged_ex(ctypes.byref(a), None))
    assert st(_general_args(tree=fake, window=4)) == b.RAD_E_ARG        # tree rows take no window
    assert st(_general_args(rows=33, tree=fake)) == b.RAD_E_SHAPE       # a mask word covers 32 nodes
    assert st(_general_args(cu=fake + 2)) == b.RAD_E_ARG                # offsets not 4-byte aligned
    assert st(_general_args(tree=fake + 1)) == b.RAD_E_ARG              # mask words not 4-byte aligned
    assert st(_general_args(cu=fake, tree=fake, rows=0)) == b.RAD_E_SHAPE   # zero rows is not a call


def test_ex_workspace_follows_the_kernel_the_call_takes():
    fake = 1 << 20
    ws = lambda a: b.ex_workspace_bytes(a)
    for hd, dt in ((128, b.RAD_KV_BF16), (256, b.RAD_KV_FP8_E4M3), (128, b.RAD_KV_FP8_E4M3)):
        a = _general_args(head_dim=hd, kv_dtype=dt)
        assert ws(a) == b.workspace_bytes(4, 8, 32, 8, hd, 16, 64, dt) > 0
    # uniform, tree and ragged split calls run the tcgen05 split kernels at both
    # head dims and pool types; a ragged call adds its tile map (256 bytes here)
    for hd in (128, 256):
        for dt in (b.RAD_KV_BF16, b.RAD_KV_FP8_E4M3):
            uniform = b.workspace_bytes(4, 8, 32, 8, hd, 16, 64, dt)
            assert ws(_general_args(tree=fake, head_dim=hd, kv_dtype=dt)) == uniform
            assert ws(_general_args(cu=fake, head_dim=hd, kv_dtype=dt)) == uniform + 256
    # the caller's row total bounds the tiles: 4 sequences of up to 256 rows
    # (ratio 4, 32-row tiles: 32 tiles each) holding 40 rows in all need at
    # most ceil(160 / 32) + 4 = 9 tiles instead of 128
    big = _general_args(rows=256, cu=fake)
    small = _general_args(rows=256, cu=fake)
    small.total_rows = 40
    assert ws(small) < ws(big) // 10
    small.total_rows = -1
    assert ws(small) == 0
    assert int(b.load().rad_attn_paged_ex(ctypes.byref(small), None)) == b.RAD_E_ARG
    # chunks past the split limit need no partials: a uniform call over bf16
    # pools needs nothing, a ragged one (on the tile kernels) its tile maps
    # (4 x ceil(1200 / 64) tiles x 8 bytes for the wide tile, 4 x 8 bytes for
    # the decode tile, each rounded to 256)
    assert b.workspace_bytes(4, 300, 32, 8, 128, 16, 64) == 0
    assert ws(_general_args(rows=300, cu=fake)) == 768 + 256
    bad = _general_args()
    bad.struct_size = 8
    assert ws(bad) == 0


def test_ex_describe_names_the_kernels_of_ragged_and_tree_calls():
    shape = lambda **kw: b.shape_args(64, 8, 32, 8, 128, 16, 1024, b.RAD_KV_FP8_E4M3, **kw)
    assert "family=split_tc05" in b.ex_describe(shape())
    assert "family=split_tc05" in b.ex_describe(shape(tree=True))
    tree = b.ex_describe(b.shape_args(64, 8, 32, 8, 128, 16, 1024, tree=True))
    assert tree.startswith("attn_split_bf16_tc05 family=split_bf16_tc05" if bf16_tc() else "attn_tile family=verify")
    assert "attn_combine" in tree
    tree256 = b.ex_describe(b.shape_args(64, 8, 32, 8, 256, 16, 1024, tree=True))
    assert tree256.startswith("attn_split_bf16_tc05 family=split_bf16_tc05" if bf16_tc(256)
                              else "attn_tile family=verify") and "attn_combine" in tree256
    rag = b.ex_describe(shape(ragged=True))
    assert rag.startswith("ragged_tile_map + attn_split_tc05 family=split_tc05") and rag.count("attn_combine") == 1
    rag256 = b.ex_describe(b.shape_args(64, 8, 32, 8, 256, 16, 1024, b.RAD_KV_FP8_E4M3, ragged=True))
    assert rag256.startswith("ragged_tile_map + attn_split_tc05 family=split_tc05 head_dim=256")
    assert rag256.count("attn_combine") == 1
    chunk = b.ex_describe(b.shape_args(4, 300, 32, 8, 128, 16, 64, ragged=True))
    assert chunk.startswith("ragged_tile_map + attn_tile family=decode") and " + attn_tile family=wide" in chunk
    assert "attn_combine" not in chunk
    dec = b.ex_describe(b.shape_args(4, 2, 32, 8, 128, 16, 64, ragged=True))
    assert dec.startswith("ragged_tile_map + attn_split_bf16_tc05 family=split_bf16_tc05" if bf16_tc()
                          else "ragged_tile_map + attn_tile family=decode")
    dec256 = b.ex_describe(b.shape_args(4, 2, 32, 8, 256, 16, 64, ragged=True))
    if bf16_tc(256):
        assert dec256.startswith("ragged_tile_map + attn_split_bf16_tc05 family=split_bf16_tc05")
    else:
        assert dec256.startswith("ragged_tile_map + attn_tile family=decode") and dec256.count("attn_tile") == 1
    assert b.describe(300, 32, 8, 128, 16).startswith("attn_prefill_tc05")


def test_compact_pool_keeps_the_call():
    """A subset of sequences re-paged into a pool of only their pages gives the
    oracle's same bits."""
    import oracle
    w = wl.make_workload("tiny_decode")
    sub = w.select_groups([3, 1])
    small = wl.compact_pool(sub)
    assert small.num_pages == int(((sub.seq_lens + 15) // 16).sum())
    a = oracle.attn_paged(sub.q, sub.k_pool, sub.v_pool, sub.page_table, sub.seq_lens, **sub.call_args()).out
    c = oracle.attn_paged(small.q, small.k_pool, small.v_pool, small.page_table, small.seq_lens,
                          **small.call_args()).out
    assert np.array_equal(a, c)


def _fault_args(**over):
    """A RadAttnPagedArgs with fake, aligned device pointers (never touched:
    every case below is refused by the host checks)."""
    g = good_args(**over)
    a = b.shape_args(g["groups"], g["rows"], g["n_head"], g["n_head_kv"], g["head_dim"], g["page_size"],
                     g["pages_per_seq"], g["kv_dtype"])
    a.cu_seqlens = a.tree_mask = None
    a.q, a.k_pool, a.v_pool = g["q_ptr"], g["k_ptr"], g["v_ptr"]
    a.page_table, a.seq_lens, a.out = g["table_ptr"], g["lens_ptr"], g["out_ptr"]
    a.num_pages, a.scale = g["num_pages"], g["scale"]
    a.k_scales, a.v_scales = (4096, 4096) if g["kv_dtype"] == b.RAD_KV_FP8_E4M3 else (None, None)
    a.workspace, a.workspace_bytes = g["ws_ptr"], g["ws_bytes"]
    return a


@pytest.mark.parametrize("limit,fault,over", [
    (5, b.RAD_FAULT_NONE, {}),                                       # a limit below 1 ms
    (3_000_000_000, b.RAD_FAULT_NONE, {}),                           # above the 2 s default
    (0, 7, {}),                                                      # an unknown fault
    (0, b.RAD_FAULT_SKIP_FIRST_K_TILE, dict(kv_dtype=b.RAD_KV_FP8_E4M3)),   # e4m3 pools: not honoured
    (0, b.RAD_FAULT_SKIP_FIRST_K_TILE, dict(rows=300)),              # a prefill chunk: not honoured
])
def test_fault_test_hook_refuses_what_it_cannot_honour(limit, fault, over):
    lib = b.load()
    a = _fault_args(**over)
    assert lib.rad_attn_paged_fault_test(ctypes.byref(a), limit, fault, None) == b.RAD_E_ARG
