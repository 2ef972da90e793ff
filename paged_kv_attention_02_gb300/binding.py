"""Python binding of the C ABI in include/rad_attn.h (argument marshalling only).

Every step of the op runs in the CUDA library ``_lib/librad_attn.so``; this
module only turns torch tensors into pointers, sizes and a stream, and turns
status codes into exceptions.  If the library is missing it raises -- there is
no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

RAD_OK = 0
RAD_E_SHAPE = 1
RAD_E_DTYPE = 2
RAD_E_ARG = 3
RAD_E_WORKSPACE = 4
RAD_E_CUDA = 5
RAD_E_DEVICE = 6

RAD_KV_BF16 = 0
RAD_KV_FP8_E4M3 = 1

RAD_ERRW_SEQLEN = 1
RAD_ERRW_PAGE = 2
RAD_ERRW_QRANGE = 4
RAD_ERRW_TIMEOUT = 8
RAD_ERRW_CUSEQ = 16
RAD_ERRW_MASK = 32

EXPORTS = ("rad_attn_paged", "rad_attn_paged_workspace_bytes", "rad_attn_paged_describe",
           "rad_attn_status_string", "rad_attn_version", "rad_attn_paged_noalloc",
           "rad_attn_paged_window", "rad_attn_paged_ex", "rad_attn_paged_ex_workspace_bytes",
           "rad_attn_paged_ex_describe", "rad_attn_paged_fault_test")

# Test-only faults of rad_attn_paged_fault_test (include/rad_attn.h).
RAD_FAULT_NONE = 0
RAD_FAULT_SKIP_FIRST_K_TILE = 1


class RadAttnPagedArgs(ctypes.Structure):
    """Mirror of `RadAttnPagedArgs` in include/rad_attn.h (natural C alignment)."""
    _fields_ = [("struct_size", ctypes.c_size_t), ("q", ctypes.c_void_p), ("k_pool", ctypes.c_void_p),
                ("v_pool", ctypes.c_void_p), ("page_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("groups", ctypes.c_int32), ("rows", ctypes.c_int32), ("n_head", ctypes.c_int32),
                ("n_head_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("pages_per_seq", ctypes.c_int32), ("num_pages", ctypes.c_int32), ("scale", ctypes.c_float),
                ("kv_dtype", ctypes.c_int32), ("k_scales", ctypes.c_void_p), ("v_scales", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("err_word", ctypes.c_void_p), ("window", ctypes.c_int32), ("cu_seqlens", ctypes.c_void_p),
                ("tree_mask", ctypes.c_void_p), ("total_rows", ctypes.c_int32)]

# Size of the library-owned scratch of rad_attn_paged_noalloc (include/rad_attn.h).
NOALLOC_SCRATCH_BYTES = 16 << 20

_lib = None


class RadAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


def load(path: str | None = None) -> ctypes.CDLL:
    """Loads the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    i32, p, sz = ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
    lib.rad_attn_paged.restype = ctypes.c_int
    lib.rad_attn_paged.argtypes = [p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, i32,
                                   ctypes.c_float, i32, p, p, p, p, sz, p, p]
    lib.rad_attn_paged_workspace_bytes.restype = sz
    lib.rad_attn_paged_workspace_bytes.argtypes = [i32] * 8
    lib.rad_attn_paged_describe.restype = ctypes.c_int
    lib.rad_attn_paged_describe.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.c_char_p, sz]
    lib.rad_attn_status_string.restype = ctypes.c_char_p
    lib.rad_attn_status_string.argtypes = [ctypes.c_int]
    lib.rad_attn_version.restype = ctypes.c_char_p
    lib.rad_attn_version.argtypes = []
    lib.rad_attn_paged_window.restype = ctypes.c_int
    lib.rad_attn_paged_window.argtypes = [p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, i32,
                                          ctypes.c_float, i32, p, p, i32, p, p, sz, p, p]
    lib.rad_attn_paged_ex.restype = ctypes.c_int
    lib.rad_attn_paged_ex.argtypes = [p, p]
    lib.rad_attn_paged_ex_workspace_bytes.restype = sz
    lib.rad_attn_paged_ex_workspace_bytes.argtypes = [p]
    lib.rad_attn_paged_ex_describe.restype = ctypes.c_int
    lib.rad_attn_paged_ex_describe.argtypes = [p, ctypes.c_char_p, sz]
    lib.rad_attn_paged_fault_test.restype = ctypes.c_int
    lib.rad_attn_paged_fault_test.argtypes = [p, ctypes.c_uint64, i32, p]
    lib.rad_attn_paged_noalloc.restype = ctypes.c_int
    lib.rad_attn_paged_noalloc.argtypes = [p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, i32,
                                           ctypes.c_float, i32, p, p, p, p, p]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().rad_attn_status_string(int(status)).decode()


def version() -> str:
    return load().rad_attn_version().decode()


def workspace_bytes(groups, rows, n_head, n_head_kv, head_dim, page_size, pages_per_seq,
                    kv_dtype=RAD_KV_BF16) -> int:
    return int(load().rad_attn_paged_workspace_bytes(groups, rows, n_head, n_head_kv, head_dim,
                                                      page_size, pages_per_seq, kv_dtype))


def describe(rows, n_head, n_head_kv, head_dim, page_size, kv_dtype=RAD_KV_BF16) -> str:
    buf = ctypes.create_string_buffer(2048)
    rc = load().rad_attn_paged_describe(rows, n_head, n_head_kv, head_dim, page_size, kv_dtype, buf,
                                        len(buf))
    if rc != RAD_OK:
        raise RadAttnError(rc, "rad_attn_paged_describe")
    return buf.value.decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def attn_paged(q, k_pool, v_pool, page_table, seq_lens, *, rows, n_head, n_head_kv, head_dim,
               page_size, scale, kv_dtype=RAD_KV_BF16, k_scales=None, v_scales=None, out=None,
               workspace=None, err_word=None, stream=None):
    """Launches rad_attn_paged on `stream` (default: torch's current stream).

    q: bf16 [groups, rows, n_head, head_dim]; k_pool / v_pool: bf16 or uint8 (e4m3
    codes) [num_pages, page_size, n_head_kv, head_dim]; page_table: int32
    [groups, pages_per_seq]; seq_lens: int32 [groups]; k_scales / v_scales:
    float32 [num_pages] for fp8.  Returns `out` (bf16, allocated if None).
    A workspace is allocated with torch when none is given.
    """
    groups = int(seq_lens.shape[0])
    pages_per_seq = int(page_table.shape[1])
    num_pages = int(k_pool.shape[0])
    if out is None:
        out = torch.empty((groups, rows, n_head, head_dim), dtype=torch.bfloat16, device=q.device)
    need = workspace_bytes(groups, rows, n_head, n_head_kv, head_dim, page_size, pages_per_seq, kv_dtype)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().rad_attn_paged(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(seq_lens), groups, rows, n_head,
        n_head_kv, head_dim, page_size, pages_per_seq, num_pages, float(scale), kv_dtype,
        _ptr(k_scales), _ptr(v_scales), _ptr(out), _ptr(workspace), ws_bytes, _ptr(err_word),
        _stream_handle(stream))
    if rc != RAD_OK:
        raise RadAttnError(rc, "rad_attn_paged")
    return out


def attn_paged_window(q, k_pool, v_pool, page_table, seq_lens, *, rows, n_head, n_head_kv, head_dim,
                      page_size, scale, window, kv_dtype=RAD_KV_BF16, k_scales=None, v_scales=None,
                      out=None, workspace=None, err_word=None, stream=None):
    """Launches rad_attn_paged_window: attn_paged over a sliding-window KV group,
    each row seeing only its last `window` keys (0: no window).  Arguments and
    result as attn_paged."""
    groups = int(seq_lens.shape[0])
    pages_per_seq = int(page_table.shape[1])
    num_pages = int(k_pool.shape[0])
    if out is None:
        out = torch.empty((groups, rows, n_head, head_dim), dtype=torch.bfloat16, device=q.device)
    need = workspace_bytes(groups, rows, n_head, n_head_kv, head_dim, page_size, pages_per_seq, kv_dtype)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().rad_attn_paged_window(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(seq_lens), groups, rows, n_head,
        n_head_kv, head_dim, page_size, pages_per_seq, num_pages, float(scale), kv_dtype,
        _ptr(k_scales), _ptr(v_scales), int(window), _ptr(out), _ptr(workspace), ws_bytes,
        _ptr(err_word), _stream_handle(stream))
    if rc != RAD_OK:
        raise RadAttnError(rc, "rad_attn_paged_window")
    return out


def attn_paged_ex(args: RadAttnPagedArgs, stream=None) -> int:
    """rad_attn_paged_ex on a filled RadAttnPagedArgs; returns the status
    (callers that want an exception check it against RAD_OK)."""
    return int(load().rad_attn_paged_ex(ctypes.byref(args), _stream_handle(stream)))


def ex_workspace_bytes(args: RadAttnPagedArgs) -> int:
    return int(load().rad_attn_paged_ex_workspace_bytes(ctypes.byref(args)))


def shape_args(groups, rows, n_head, n_head_kv, head_dim, page_size, pages_per_seq, kv_dtype=RAD_KV_BF16,
               ragged=False, tree=False, total_rows=0) -> RadAttnPagedArgs:
    """A RadAttnPagedArgs carrying only a call's shape (and whether it has
    cu_seqlens / tree_mask), for the workspace and describe queries."""
    a = RadAttnPagedArgs()
    a.struct_size = ctypes.sizeof(RadAttnPagedArgs)
    a.groups, a.rows, a.n_head, a.n_head_kv, a.head_dim = groups, rows, n_head, n_head_kv, head_dim
    a.page_size, a.pages_per_seq, a.kv_dtype = page_size, pages_per_seq, kv_dtype
    a.cu_seqlens = 16 if ragged else None     # presence only: never dereferenced by the queries
    a.tree_mask = 16 if tree else None
    a.total_rows = total_rows
    return a


def ex_describe(args: RadAttnPagedArgs) -> str:
    buf = ctypes.create_string_buffer(2048)
    rc = load().rad_attn_paged_ex_describe(ctypes.byref(args), buf, len(buf))
    if rc != RAD_OK:
        raise RadAttnError(rc, "rad_attn_paged_ex_describe")
    return buf.value.decode()


def attn_paged_general(q, k_pool, v_pool, page_table, seq_lens, *, rows, n_head, n_head_kv, head_dim,
                       page_size, scale, kv_dtype=RAD_KV_BF16, k_scales=None, v_scales=None,
                       cu_seqlens=None, tree_mask=None, window=0, total_rows=None, out=None,
                       workspace=None, err_word=None, stream=None):
    """The op through rad_attn_paged_ex with every optional field.

    cu_seqlens: int32 [groups + 1] absolute row offsets (ragged rows; ``rows``
    is then the largest count and q is [q_rows, n_head, head_dim]); tree_mask:
    uint32 words (as int32) indexed like q's rows (draft-tree rows); window:
    sliding window.  Without cu_seqlens q is [groups, rows, n_head, head_dim].
    total_rows bounds the rows a ragged call names (default: q's rows, which
    hold every row the offsets may name).  Returns `out` (allocated like q
    when None; rows no group names are not written).
    """
    a, out, workspace = _general_args(q, k_pool, v_pool, page_table, seq_lens, rows, n_head, n_head_kv, head_dim,
                                      page_size, scale, kv_dtype, k_scales, v_scales, cu_seqlens, tree_mask,
                                      window, total_rows, out, workspace, err_word)
    rc = attn_paged_ex(a, stream)
    if rc != RAD_OK:
        raise RadAttnError(rc, "rad_attn_paged_ex")
    return out


def attn_paged_fault_test(q, k_pool, v_pool, page_table, seq_lens, *, rows, n_head, n_head_kv, head_dim,
                          page_size, scale, wait_limit_ns=0, fault=RAD_FAULT_NONE, kv_dtype=RAD_KV_BF16,
                          k_scales=None, v_scales=None, out=None, workspace=None, err_word=None, stream=None):
    """rad_attn_paged_fault_test: attn_paged_general's call with a test's
    wait limit (ns, 0 = the default) and injected fault.  Returns `out`."""
    a, out, workspace = _general_args(q, k_pool, v_pool, page_table, seq_lens, rows, n_head, n_head_kv, head_dim,
                                      page_size, scale, kv_dtype, k_scales, v_scales, None, None, 0, None, out,
                                      workspace, err_word)
    rc = int(load().rad_attn_paged_fault_test(ctypes.byref(a), int(wait_limit_ns), int(fault),
                                              _stream_handle(stream)))
    if rc != RAD_OK:
        raise RadAttnError(rc, "rad_attn_paged_fault_test")
    return out


def _general_args(q, k_pool, v_pool, page_table, seq_lens, rows, n_head, n_head_kv, head_dim, page_size, scale,
                  kv_dtype, k_scales, v_scales, cu_seqlens, tree_mask, window, total_rows, out, workspace,
                  err_word):
    """A filled RadAttnPagedArgs (with `out` and the workspace allocated by
    torch when not given); returns (args, out, workspace), the last two kept
    alive by the caller for the call."""
    groups = int(seq_lens.shape[0])
    if out is None:
        out = torch.empty(tuple(q.shape), dtype=torch.bfloat16, device=q.device)
    a = RadAttnPagedArgs()
    a.struct_size = ctypes.sizeof(RadAttnPagedArgs)
    a.q, a.k_pool, a.v_pool = q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr()
    a.page_table, a.seq_lens = page_table.data_ptr(), seq_lens.data_ptr()
    a.groups, a.rows, a.n_head, a.n_head_kv, a.head_dim = groups, rows, n_head, n_head_kv, head_dim
    a.page_size, a.pages_per_seq, a.num_pages = page_size, int(page_table.shape[1]), int(k_pool.shape[0])
    a.scale, a.kv_dtype = float(scale), kv_dtype
    a.k_scales = None if k_scales is None else k_scales.data_ptr()
    a.v_scales = None if v_scales is None else v_scales.data_ptr()
    a.cu_seqlens = None if cu_seqlens is None else cu_seqlens.data_ptr()
    a.tree_mask = None if tree_mask is None else tree_mask.data_ptr()
    a.window = int(window)
    if cu_seqlens is not None:
        a.total_rows = int(q.shape[0]) if total_rows is None else int(total_rows)
    a.out = out.data_ptr()
    need = ex_workspace_bytes(a)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    a.workspace = None if workspace is None else workspace.data_ptr()
    a.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    a.err_word = None if err_word is None else err_word.data_ptr()
    return a, out, workspace


def call_raw(q_ptr, k_ptr, v_ptr, table_ptr, lens_ptr, groups, rows, n_head, n_head_kv, head_dim,
             page_size, pages_per_seq, num_pages, scale, kv_dtype, ks_ptr, vs_ptr, out_ptr, ws_ptr,
             ws_bytes, err_ptr, stream_ptr) -> int:
    """The C call with raw integer pointers (for boundary tests); returns the status."""
    def vp(x):
        return ctypes.c_void_p(x) if x else None
    return int(load().rad_attn_paged(
        vp(q_ptr), vp(k_ptr), vp(v_ptr), vp(table_ptr), vp(lens_ptr), groups, rows, n_head, n_head_kv,
        head_dim, page_size, pages_per_seq, num_pages, float(scale), kv_dtype, vp(ks_ptr), vp(vs_ptr),
        vp(out_ptr), vp(ws_ptr), ws_bytes, vp(err_ptr), vp(stream_ptr)))


def attn_paged_noalloc(q, k_pool, v_pool, page_table, seq_lens, *, rows, n_head, n_head_kv, head_dim,
                       page_size, scale, kv_dtype=RAD_KV_BF16, k_scales=None, v_scales=None, out,
                       err_word=None, stream=None):
    """rad_attn_paged_noalloc: the op with the library's own fixed scratch.

    For callers that cannot allocate device memory per call (a runtime whose
    memory is planned once at load time, or code handed only the call's
    tensors).  `out` must be given; nothing is allocated here or in the
    library.  Raises RadAttnError with RAD_E_WORKSPACE when the call needs
    more than NOALLOC_SCRATCH_BYTES of scratch.
    """
    groups = int(seq_lens.shape[0])
    rc = load().rad_attn_paged_noalloc(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(seq_lens), groups, rows, n_head,
        n_head_kv, head_dim, page_size, int(page_table.shape[1]), int(k_pool.shape[0]), float(scale),
        kv_dtype, _ptr(k_scales), _ptr(v_scales), _ptr(out), _ptr(err_word), _stream_handle(stream))
    if rc != RAD_OK:
        raise RadAttnError(rc, "rad_attn_paged_noalloc")
    return out
