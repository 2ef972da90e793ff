"""Oracle for paged-KV attention -- TEST INFRASTRUCTURE ONLY.

A plain fp64 CPU definition of the `attn_paged` op (``ref_attn_paged.c``) and
this thin ctypes loader for it.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it.  It imports nothing
from the product package and the product never imports it.

Every function here works on host numpy arrays:

* ``q``           uint16 bf16 bit patterns, shape [groups, rows, n_head, head_dim]
* ``k_pool``/``v_pool``  uint16 (bf16) or uint8 (fp8 e4m3) codes,
                  shape [num_pages, page_size, n_head_kv, head_dim]
* ``page_table``  int32 [groups, pages_per_seq] physical page ids
* ``seq_lens``    int32 [groups], each sequence's length after the call
* ``k_scales``/``v_scales`` float32 [num_pages] (fp8 only)

and returns float64 results.  Parity status: every function is pinned by
``tests/test_oracle.py`` (brute force, closed forms, invariants, the fp8 and
bf16 format definitions) -- none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ref_attn_paged.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_attn_paged.so")

KV_BF16 = 0
KV_FP8_E4M3 = 1
ERRW_SEQLEN = 1
ERRW_PAGE = 2
ERRW_CUSEQ = 16
ERRW_MASK = 32

_lib = None


def build(force: bool = False) -> str:
    """Compiles the C oracle with gcc (-O2, OpenMP) into oracle/_build/."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32 = ctypes.c_int32
        i64 = ctypes.c_int64
        lib.oracle_attn_paged_rows.restype = ctypes.c_int
        lib.oracle_attn_paged_rows.argtypes = [
            P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, ctypes.c_double, i32, P, P,
            P, i64, P, P, i64, P, P, i32, i32, P, P]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def bf16_to_f64(bits: int) -> float:
    return float(_load().oracle_bf16_to_f64(int(bits)))


def e4m3_to_f64(code: int) -> float:
    return float(_load().oracle_e4m3_to_f64(int(code)))


class OracleError(RuntimeError):
    pass


@dataclass
class OracleResult:
    out: np.ndarray          # float64 [n_sel, head_dim] or [groups, rows, n_head, head_dim]
    err_word: int
    weights: np.ndarray | None = None   # float64 [n_sel, max_keys] (zero past n_keys)
    n_keys: np.ndarray | None = None    # int64 [n_sel]


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def attn_paged_rows(q, k_pool, v_pool, page_table, seq_lens, *, rows, n_head, n_head_kv, head_dim,
                    page_size, scale, kv_dtype=KV_BF16, k_scales=None, v_scales=None, sel=None,
                    want_weights=False, n_threads=0, window=0, cu_seqlens=None,
                    tree_mask=None) -> OracleResult:
    """Selected output rows of the op in fp64.

    ``sel`` is an int array of (g, r, h) triples; ``None`` selects every row and
    returns ``out`` shaped [groups, rows, n_head, head_dim].  ``window`` > 0
    limits each row to its last ``window`` keys (0: no window).

    ``cu_seqlens`` (int32 [groups + 1]) makes the rows ragged: group g has
    cu[g+1] - cu[g] rows at q rows cu[g] .., ``q`` is [q_rows, n_head, head_dim]
    and ``rows`` is the largest count.  The full selection then returns ``out``
    shaped like ``q`` (rows no group names stay zero), and a group with
    malformed entries is still touched, so that its error bit shows.
    ``tree_mask`` (uint32, one word per q row) makes each row see the cached
    keys plus the call's keys of its own bits (its path in a draft tree).
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    pool_dt = np.uint16 if kv_dtype == KV_BF16 else np.uint8
    k_pool = np.ascontiguousarray(k_pool, dtype=pool_dt)
    v_pool = np.ascontiguousarray(v_pool, dtype=pool_dt)
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    groups = int(seq_lens.shape[0])
    pages_per_seq = int(page_table.shape[1])
    num_pages = int(k_pool.shape[0])
    if k_scales is not None:
        k_scales = np.ascontiguousarray(k_scales, dtype=np.float32)
    if v_scales is not None:
        v_scales = np.ascontiguousarray(v_scales, dtype=np.float32)
    if cu_seqlens is not None:
        cu_seqlens = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        if cu_seqlens.shape != (groups + 1,):
            raise OracleError("cu_seqlens needs groups + 1 entries")
    if tree_mask is not None:
        tree_mask = np.ascontiguousarray(tree_mask, dtype=np.uint32)
    full = sel is None
    ragged_rows = None   # q row of every selected triple, ragged full selection only
    if full and cu_seqlens is None:
        gg, rr, hh = np.meshgrid(np.arange(groups), np.arange(rows), np.arange(n_head), indexing="ij")
        sel = np.stack([gg.ravel(), rr.ravel(), hh.ravel()], axis=1)
    elif full:
        trip, qrow = [], []
        for g in range(groups):
            a, b = int(cu_seqlens[g]), int(cu_seqlens[g + 1])
            if a < 0 or b < a or b - a > rows:
                trip.append((g, 0, 0))       # touched for its error bit, output dropped
                qrow.append(-1)
                continue
            for r in range(b - a):
                for h in range(n_head):
                    trip.append((g, r, h))
                    qrow.append(a + r)
        sel = np.array(trip, dtype=np.int32).reshape(-1, 3)
        ragged_rows = np.array(qrow, dtype=np.int64)
    sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int32).reshape(-1, 3))
    n_sel = sel.shape[0]
    out = np.zeros((n_sel, head_dim), dtype=np.float64)
    weights = None
    n_keys = np.zeros(n_sel, dtype=np.int64)
    wstride = 0
    if want_weights:
        wstride = int(max(int(seq_lens.max()), 1))
        weights = np.zeros((n_sel, wstride), dtype=np.float64)
    err = ctypes.c_uint32(0)
    rc = _load().oracle_attn_paged_rows(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(seq_lens), groups, rows, n_head,
        n_head_kv, head_dim, page_size, pages_per_seq, num_pages, float(np.float32(scale)), kv_dtype,
        _ptr(k_scales), _ptr(v_scales), _ptr(sel), n_sel, _ptr(out), _ptr(weights), wstride,
        _ptr(n_keys), ctypes.byref(err), int(n_threads), int(window), _ptr(cu_seqlens),
        _ptr(tree_mask))
    if rc != 0:
        raise OracleError(f"oracle refused the call: code {rc}")
    if full and ragged_rows is not None:
        flat = np.zeros((q.shape[0], n_head, head_dim), dtype=np.float64)
        keep = ragged_rows >= 0
        flat[ragged_rows[keep], sel[keep, 2]] = out[keep]
        out = flat
    elif full:
        out = out.reshape(groups, rows, n_head, head_dim)
    return OracleResult(out=out, err_word=int(err.value), weights=weights, n_keys=n_keys)


def attn_paged(q, k_pool, v_pool, page_table, seq_lens, **kw) -> OracleResult:
    """Every output row of the op, [groups, rows, n_head, head_dim] float64."""
    kw.pop("sel", None)
    return attn_paged_rows(q, k_pool, v_pool, page_table, seq_lens, sel=None, **kw)
