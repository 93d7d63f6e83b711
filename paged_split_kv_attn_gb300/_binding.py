"""ctypes binding of ``libpskv.so`` (the C ABI in ``include/pskv.h``).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and the current
stream; nothing here computes attention, and there is no CPU path: if the
library is missing the calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpskv.so")

PSKV_OK = 0
PSKV_ERR_INVALID_ARG = -1
PSKV_ERR_UNSUPPORTED = -2
PSKV_ERR_OVERFLOW = -3
PSKV_ERR_WORKSPACE_TOO_SMALL = -4
PSKV_ERR_PAST_PAGES = -5
PSKV_ERR_CUDA = -6

PSKV_DTYPE_F32 = 0
PSKV_DTYPE_BF16 = 1
PSKV_FORMAT_SPLIT = 0
PSKV_FORMAT_FOLDED = 1

PSKV_FAULT_BAD_PAGE = 1
PSKV_FAULT_PAST_PAGES = 2
PSKV_FAULT_BAD_LENGTH = 4
PSKV_FAULT_WAIT_TIMEOUT = 8
PSKV_FAULT_EMPTY_ROW = 16
PSKV_FAULT_BAD_STATE = 32
PSKV_FAULT_BAD_POSITION = 64
PSKV_FAULT_BAD_MASK = 128

PSKV_MAX_SPLITS = 1024
PSKV_AUTO_MAX_SPLITS = 256
PSKV_MERGE_GROUP = 16
PSKV_KEY_TILE = 16
PSKV_MAX_WINDOW_TOKENS = 64
PSKV_STATIC_SCRATCH_BYTES = 16 * 1024 * 1024

# Every function the header declares, in the header's order.
EXPORTS = ("paged_kv_layout_create", "paged_kv_layout_destroy", "kv_append_rows", "kv_prep_append",
           "decode_attn_splitkv", "decode_attn_windowed", "decode_attn_multirow",
           "decode_attn_tree", "prefill_attn_paged", "merge_partials",
           "decode_attn_workspace_bytes", "merge_partials_workspace_bytes",
           "prefill_attn_workspace_bytes", "decode_attn_multirow_workspace_bytes",
           "pskv_partial_scratch_bytes", "pskv_plan_splits", "decode_attn_splitkv_static",
           "pskv_check_flags", "pskv_strerror", "pskv_last_cuda_error", "pskv_kernel_launches",
           "pskv_version")


class PskvError(RuntimeError):
    def __init__(self, code: int, what: str):
        lib = _LIB
        msg = lib.pskv_strerror(code).decode() if lib is not None else str(code)
        if code == PSKV_ERR_CUDA and lib is not None:
            msg += " (" + lib.pskv_last_cuda_error().decode() + ")"
        super().__init__(f"{what}: {msg} [{code}]")
        self.code = code


class LayoutDesc(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int64), ("page_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim_k", ctypes.c_int32),
                ("head_dim_v", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("format", ctypes.c_int32), ("k_pool", ctypes.c_void_p),
                ("v_pool", ctypes.c_void_p), ("status", ctypes.c_void_p)]


class PrepDesc(ctypes.Structure):
    _fields_ = [("rot_dims", ctypes.c_int32), ("eps", ctypes.c_float), ("w_q", ctypes.c_void_p),
                ("w_k", ctypes.c_void_p), ("rope_cos", ctypes.c_void_p),
                ("rope_sin", ctypes.c_void_p), ("max_pos", ctypes.c_int32)]


class DecodeOpts(ctypes.Structure):
    _fields_ = [("merge_group", ctypes.c_int32), ("partial_begin", ctypes.c_void_p),
                ("partial_end", ctypes.c_void_p), ("append_k", ctypes.c_void_p),
                ("append_v", ctypes.c_void_p), ("append_pages", ctypes.c_void_p)]


_LIB = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (no fallback: raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m paged_split_kv_attn_gb300.build`")
    lib = ctypes.CDLL(path)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    F = ctypes.c_float
    lib.paged_kv_layout_create.argtypes = [ctypes.POINTER(LayoutDesc), ctypes.POINTER(P)]
    lib.paged_kv_layout_destroy.argtypes = [P]
    lib.paged_kv_layout_destroy.restype = None
    lib.kv_append_rows.argtypes = [P, P, P, P, P, I32, P, I32, P, I32, P, P, P, P]
    lib.kv_prep_append.argtypes = [P, ctypes.POINTER(PrepDesc), P, I64, I32, I32, I32, I32, I32,
                                   P, P, P, P, I32, P, I32, P, P, P, P, P]
    lib.decode_attn_splitkv.argtypes = [P, P, P, I32, P, P, I32, I32, F, I32, P, SZ, P, I32, P, P]
    lib.decode_attn_windowed.argtypes = [P, P, P, I32, P, P, P, P, I32, I32, F, I32, P, SZ, P,
                                         I32, P, P]
    lib.decode_attn_multirow.argtypes = [P, P, P, I32, P, P, I32, I32, I32, F, I32, P, SZ, P, I32,
                                         P, P]
    lib.decode_attn_tree.argtypes = [P, P, P, I32, P, P, P, I32, I32, I32, F, I32, P, SZ, P, I32,
                                     P, P]
    lib.prefill_attn_paged.argtypes = [P, P, P, P, P, I32, P, P, I32, I32, I32, F, I32, P, SZ, P,
                                       I32, P, P]
    lib.merge_partials.argtypes = [P, P, P, I32, I32, I32, P, I32, P, SZ, P, P, P]
    lib.decode_attn_workspace_bytes.argtypes = [I32, I32, I32, I32, ctypes.POINTER(SZ)]
    lib.merge_partials_workspace_bytes.argtypes = [I32, I32, I32, ctypes.POINTER(SZ)]
    lib.prefill_attn_workspace_bytes.argtypes = [P, P, P, I32, I32, I32, I32, I32,
                                                 ctypes.POINTER(SZ)]
    lib.decode_attn_multirow_workspace_bytes.argtypes = [P, P, I32, I32, I32, I32, I32, I32,
                                                         ctypes.POINTER(SZ)]
    lib.pskv_partial_scratch_bytes.argtypes = [I64, I64, I64, I64] + [ctypes.POINTER(SZ)] * 4
    lib.pskv_plan_splits.argtypes = [P, I32, I32, P, ctypes.POINTER(I32)]
    lib.decode_attn_splitkv_static.argtypes = [P, P, P, I32, P, P, I32, I32, F, I32, P, I32, P]
    lib.pskv_check_flags.argtypes = [P, I32, P, ctypes.POINTER(ctypes.c_uint32)]
    lib.pskv_strerror.argtypes = [ctypes.c_int]
    lib.pskv_strerror.restype = ctypes.c_char_p
    lib.pskv_last_cuda_error.argtypes = []
    lib.pskv_last_cuda_error.restype = ctypes.c_char_p
    lib.pskv_kernel_launches.argtypes = []
    lib.pskv_kernel_launches.restype = ctypes.c_uint64
    lib.pskv_version.argtypes = []
    _LIB = lib
    return lib


def _check(rc: int, what: str) -> None:
    if rc != PSKV_OK:
        raise PskvError(rc, what)


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return PSKV_DTYPE_BF16
    if t == torch.float32:
        return PSKV_DTYPE_F32
    raise TypeError(f"unsupported dtype {t}: bf16 or f32")


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _host_i32(x, name: str):
    """Host int32 array (list, numpy array or CPU tensor) -> ctypes array kept alive by the caller."""
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        if x.is_cuda:
            raise TypeError(f"{name} must be host memory")
        x = x.to(torch.int32).tolist()
    elif hasattr(x, "tolist"):
        x = x.tolist()
    return (ctypes.c_int32 * len(x))(*[int(v) for v in x])


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _event(ev):
    if ev is None:
        return None
    if isinstance(ev, torch.cuda.Event):
        if not ev.cuda_event:  # torch creates the event on its first record
            ev.record()
        return ev.cuda_event
    return int(ev)


def _opts(merge_group: int = 0, events=None, append=None, dtype=None):
    """Per-call options; ``append`` = (k_new, v_new, pages_of_row) writes each
    row's new K/V row (key seq_lens - 1) from inside the decode."""
    if not merge_group and events is None and append is None:
        return None
    begin, end = (None, None) if events is None else events
    ak = av = ap = None
    if append is not None:
        k_new, v_new, pages = append
        ak, av = _dev(k_new, "k_new", dtype), _dev(v_new, "v_new", dtype)
        ap = _dev(pages, "pages_of_row", torch.int32)
    return DecodeOpts(merge_group, _event(begin), _event(end), ak, av, ap)


# ---- layout ------------------------------------------------------------------

class Layout:
    """A layout handle together with the tensors it points at (kept alive)."""

    def __init__(self, handle, k_pool, v_pool, status, desc):
        self._handle = handle
        self.k_pool, self.v_pool, self.status, self.desc = k_pool, v_pool, status, desc

    @property
    def handle(self):
        return self._handle

    @property
    def num_kv_heads(self) -> int:
        return self.desc.num_kv_heads

    @property
    def head_dim(self) -> int:
        return self.desc.head_dim_k

    @property
    def page_size(self) -> int:
        return self.desc.page_size

    @property
    def dtype(self) -> torch.dtype:
        return self.k_pool.dtype

    def faults(self) -> int:
        """Read the device fault word (synchronises with the current stream)."""
        return 0 if self.status is None else int(self.status[0].item())

    def close(self) -> None:
        if self._handle is not None and _LIB is not None:
            _LIB.paged_kv_layout_destroy(self._handle)
        self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def paged_kv_layout_create(k_pool: torch.Tensor, v_pool: torch.Tensor,
                           status: torch.Tensor | None = None, fmt: int | None = None) -> Layout:
    """Wrap pools shaped [num_pages, num_kv_heads, page_size, head_dim]; a K pool
    narrower than the V pool is a folded pool unless ``fmt`` says otherwise."""
    lib = load_library()
    if k_pool.dim() != 4 or v_pool.dim() != 4 or k_pool.shape[:3] != v_pool.shape[:3]:
        raise ValueError("pools must be [num_pages, num_kv_heads, page_size, head_dim]")
    if fmt is None:
        fmt = PSKV_FORMAT_FOLDED if k_pool.shape[3] < v_pool.shape[3] else PSKV_FORMAT_SPLIT
    if k_pool.dtype != v_pool.dtype:
        raise TypeError("k_pool and v_pool must share a dtype")
    desc = LayoutDesc(k_pool.shape[0], k_pool.shape[2], k_pool.shape[1], k_pool.shape[3],
                      v_pool.shape[3], _dtype_code(k_pool.dtype), fmt,
                      _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"),
                      None if status is None else _dev(status, "status", torch.int32))
    handle = ctypes.c_void_p()
    _check(lib.paged_kv_layout_create(ctypes.byref(desc), ctypes.byref(handle)),
           "paged_kv_layout_create")
    return Layout(handle, k_pool, v_pool, status, desc)


# ---- calls -------------------------------------------------------------------

def kv_append_rows(layout: Layout, k_new, v_new, row_of, pos_of, page_tables, pages_of_row,
                   host=None, stream=None) -> None:
    """Copy rows k_new/v_new [n, num_kv_heads, head_dim] into their pages.
    ``host`` = (row_of, pos_of, pages_of_row) host copies for the up-front refusal."""
    lib = load_library()
    n = int(row_of.numel())
    hr = hp = hl = None
    if host is not None:
        hr, hp, hl = (_host_i32(x, name) for x, name in zip(host, ("row_of", "pos_of", "pages")))
    _check(lib.kv_append_rows(layout.handle, _dev(k_new, "k_new", layout.dtype),
                              _dev(v_new, "v_new", layout.dtype),
                              _dev(row_of, "row_of", torch.int32),
                              _dev(pos_of, "pos_of", torch.int32), n,
                              _dev(page_tables, "page_tables", torch.int32),
                              page_tables.shape[1], _dev(pages_of_row, "pages_of_row", torch.int32),
                              pages_of_row.numel(), hr, hp, hl, _stream(stream)),
           "kv_append_rows")


def kv_prep_append(layout: Layout, x, q_col: int, k_col: int, v_col: int, num_q_heads: int,
                   row_of, pos_of, page_tables, pages_of_row, rot_dims: int, eps: float,
                   w_q=None, w_k=None, rope_cos=None, rope_sin=None, first_pos=None, q_out=None,
                   host=None, stream=None) -> torch.Tensor:
    """K/V prep of n tokens with the page write fused in: ``x`` [n, stride] bf16
    projection rows; K and V rows go into the pages, the prepared queries into
    ``q_out`` [n, num_q_heads, head_dim] (returned).  ``host`` = (row_of, pos_of,
    pages_of_row) host copies for the up-front refusal."""
    lib = load_library()
    n = int(row_of.numel())
    d = layout.desc.head_dim_v
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be [n, stride] with unit column stride")
    if q_out is None:
        q_out = torch.empty((n, num_q_heads, d), dtype=torch.bfloat16, device=x.device)
    hr = hp = hl = None
    if host is not None:
        hr, hp, hl = (_host_i32(v, name) for v, name in zip(host, ("row_of", "pos_of", "pages")))
    opt = lambda t, name: None if t is None else _dev(t, name, torch.float32)
    desc = PrepDesc(rot_dims=rot_dims, eps=eps, w_q=opt(w_q, "w_q"), w_k=opt(w_k, "w_k"),
                    rope_cos=opt(rope_cos, "rope_cos"), rope_sin=opt(rope_sin, "rope_sin"),
                    max_pos=0 if rope_cos is None else rope_cos.shape[0])
    _check(lib.kv_prep_append(
        layout.handle, ctypes.byref(desc), _dev(x, "x", torch.bfloat16), x.stride(0), q_col, k_col,
        v_col, n, num_q_heads, _dev(row_of, "row_of", torch.int32),
        _dev(pos_of, "pos_of", torch.int32),
        None if first_pos is None else _dev(first_pos, "first_pos", torch.int32),
        _dev(page_tables, "page_tables", torch.int32), page_tables.shape[1],
        _dev(pages_of_row, "pages_of_row", torch.int32), pages_of_row.numel(), hr, hp, hl,
        _dev(q_out, "q_out", torch.bfloat16), _stream(stream)), "kv_prep_append")
    return q_out


def decode_attn_workspace_bytes(batch: int, num_q_heads: int, head_dim_v: int,
                                num_splits: int = 0) -> int:
    out = ctypes.c_size_t()
    _check(load_library().decode_attn_workspace_bytes(batch, num_q_heads, head_dim_v, num_splits,
                                                      ctypes.byref(out)),
           "decode_attn_workspace_bytes")
    return int(out.value)


def merge_partials_workspace_bytes(rows: int, num_splits: int, head_dim_v: int) -> int:
    out = ctypes.c_size_t()
    _check(load_library().merge_partials_workspace_bytes(rows, num_splits, head_dim_v,
                                                         ctypes.byref(out)),
           "merge_partials_workspace_bytes")
    return int(out.value)


def prefill_attn_workspace_bytes(layout: Layout, cu_q_host, seq_lens_host, table_stride: int,
                                 num_q_heads: int, window: int = 0, num_splits: int = 0) -> int:
    """Workspace bytes a prefill call needs under its plan (0: one partition, none needed)."""
    cu_h, lens_h = _host_i32(cu_q_host, "cu_q_host"), _host_i32(seq_lens_host, "seq_lens_host")
    out = ctypes.c_size_t()
    _check(load_library().prefill_attn_workspace_bytes(
        layout.handle, cu_h, lens_h, table_stride, len(lens_h), num_q_heads, int(window),
        num_splits, ctypes.byref(out)), "prefill_attn_workspace_bytes")
    return int(out.value)


def decode_attn_multirow_workspace_bytes(layout: Layout, seq_lens_host, table_stride: int,
                                         num_tokens: int, num_q_heads: int, tree: bool = False,
                                         num_splits: int = 0) -> int:
    """Workspace bytes a verify-window (or drafted-tree) call needs under its plan."""
    lens_h = _host_i32(seq_lens_host, "seq_lens_host")
    out = ctypes.c_size_t()
    _check(load_library().decode_attn_multirow_workspace_bytes(
        layout.handle, lens_h, table_stride, len(lens_h), num_tokens, num_q_heads, int(tree),
        num_splits, ctypes.byref(out)), "decode_attn_multirow_workspace_bytes")
    return int(out.value)


def _planned_workspace(nbytes: int, device):
    return None if nbytes == 0 else torch.empty(nbytes, dtype=torch.uint8, device=device)


def pskv_partial_scratch_bytes(batch: int, num_q_heads: int, head_dim_v: int, num_splits: int):
    vals = [ctypes.c_size_t() for _ in range(4)]
    _check(load_library().pskv_partial_scratch_bytes(batch, num_q_heads, head_dim_v, num_splits,
                                                      *[ctypes.byref(v) for v in vals]),
           "pskv_partial_scratch_bytes")
    return tuple(int(v.value) for v in vals)


def pskv_plan_splits(layout: Layout, num_q_heads: int, seq_lens_host) -> int:
    lens = _host_i32(seq_lens_host, "seq_lens_host")
    out = ctypes.c_int32()
    _check(load_library().pskv_plan_splits(layout.handle, len(lens), num_q_heads, lens,
                                           ctypes.byref(out)),
           "pskv_plan_splits")
    return int(out.value)


def workspace(batch: int, num_q_heads: int, head_dim_v: int, num_splits: int = 0,
              device=None) -> torch.Tensor:
    """A scratch tensor big enough for a decode call (allocated by PyTorch)."""
    n = decode_attn_workspace_bytes(batch, num_q_heads, head_dim_v, num_splits)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


_alloc_workspace = workspace


def _decode(windowed: bool, layout: Layout, q, page_tables, seq_lens, seq_lens_host, scale,
            num_splits, workspace_t, out, out_dtype, merge_group, events, stream,
            first_pos=None, window_lo=None, append=None):
    lib = load_library()
    if q.dim() != 3:
        raise ValueError("q must be [batch, num_q_heads, head_dim]")
    batch, hq = q.shape[0], q.shape[1]
    if out is None:
        out = torch.empty((batch, hq, layout.desc.head_dim_v), device=q.device,
                          dtype=out_dtype or torch.bfloat16)
    if workspace_t is None:
        workspace_t = workspace(batch, hq, layout.desc.head_dim_v, num_splits, q.device)
    lens_h = _host_i32(seq_lens_host, "seq_lens_host")
    if len(lens_h) != batch:
        raise ValueError("seq_lens_host must have one entry per row")
    opts = _opts(merge_group, events, append, layout.dtype)
    common = (_dev(q, "q", layout.dtype), _dev(page_tables, "page_tables", torch.int32),
              page_tables.shape[1], lens_h, _dev(seq_lens, "seq_lens", torch.int32))
    tail = (batch, hq, float(scale), num_splits, _dev(workspace_t, "workspace"),
            workspace_t.numel() * workspace_t.element_size(), _dev(out, "out"),
            _dtype_code(out.dtype), None if opts is None else ctypes.byref(opts), _stream(stream))
    if windowed:
        rc = lib.decode_attn_windowed(layout.handle, *common,
                                      _dev(first_pos, "first_pos", torch.int32),
                                      _dev(window_lo, "window_lo", torch.int32), *tail)
    else:
        rc = lib.decode_attn_splitkv(layout.handle, *common, *tail)
    _check(rc, "decode_attn_windowed" if windowed else "decode_attn_splitkv")
    return out


def decode_attn_splitkv(layout: Layout, q, page_tables, seq_lens, seq_lens_host, scale,
                        num_splits: int = 0, workspace=None, out=None, out_dtype=None,
                        merge_group: int = 0, events=None, stream=None,
                        append=None) -> torch.Tensor:
    """Split-KV decode; returns ``out`` [batch, num_q_heads, head_dim].
    ``append`` = (k_new, v_new, pages_of_row): each row's new K/V row, key
    seq_lens - 1, is written into its page by the decode itself."""
    return _decode(False, layout, q, page_tables, seq_lens, seq_lens_host, scale, num_splits,
                   workspace, out, out_dtype, merge_group, events, stream, append=append)


def decode_attn_windowed(layout: Layout, q, page_tables, seq_lens, seq_lens_host, first_pos,
                         window_lo, scale, num_splits: int = 0, workspace=None, out=None,
                         out_dtype=None, merge_group: int = 0, events=None,
                         stream=None, append=None) -> torch.Tensor:
    """Windowed split-KV decode; keys at positions below ``window_lo`` are masked."""
    return _decode(True, layout, q, page_tables, seq_lens, seq_lens_host, scale, num_splits,
                   workspace, out, out_dtype, merge_group, events, stream, first_pos, window_lo,
                   append)


def decode_attn_multirow(layout: Layout, q, page_tables, seq_lens, seq_lens_host, scale,
                         num_splits: int = 0, workspace=None, out=None, out_dtype=None,
                         merge_group: int = 0, events=None, stream=None) -> torch.Tensor:
    """Multi-row decode of a verify window: ``q`` is [batch, tokens, num_q_heads,
    head_dim]; token t of row b sits at key ``seq_lens[b] - tokens + t`` and
    attends keys up to itself.  Returns ``out`` [batch, tokens, num_q_heads, head_dim]."""
    lib = load_library()
    if q.dim() != 4:
        raise ValueError("q must be [batch, tokens, num_q_heads, head_dim]")
    batch, tokens, hq = q.shape[0], q.shape[1], q.shape[2]
    dv = layout.desc.head_dim_v
    if out is None:
        out = torch.empty((batch, tokens, hq, dv), device=q.device,
                          dtype=out_dtype or torch.bfloat16)
    lens_h = _host_i32(seq_lens_host, "seq_lens_host")
    if len(lens_h) != batch:
        raise ValueError("seq_lens_host must have one entry per row")
    if workspace is None:
        workspace = _planned_workspace(decode_attn_multirow_workspace_bytes(
            layout, lens_h, page_tables.shape[1], tokens, hq, False, num_splits), q.device)
    opts = _opts(merge_group, events)
    _check(lib.decode_attn_multirow(
        layout.handle, _dev(q, "q", layout.dtype), _dev(page_tables, "page_tables", torch.int32),
        page_tables.shape[1], lens_h, _dev(seq_lens, "seq_lens", torch.int32), batch, tokens, hq,
        float(scale), num_splits, None if workspace is None else _dev(workspace, "workspace"),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _dev(out, "out"), _dtype_code(out.dtype), None if opts is None else ctypes.byref(opts),
        _stream(stream)), "decode_attn_multirow")
    return out


def decode_attn_tree(layout: Layout, q, page_tables, seq_lens, seq_lens_host, tree_mask, scale,
                     num_splits: int = 0, workspace=None, out=None, out_dtype=None,
                     merge_group: int = 0, events=None, stream=None) -> torch.Tensor:
    """Tree attention over a drafted window: ``q`` is [batch, tokens, num_q_heads,
    head_dim]; the row's last ``tokens`` keys are the drafted tokens in an order
    where ancestors come first; ``tree_mask`` (device int64 or uint64 [batch,
    tokens]) holds each token's ancestor bits (itself included).  Token t
    attends every key before the window and the window tokens its mask marks.
    Returns ``out`` [batch, tokens, num_q_heads, head_dim]."""
    lib = load_library()
    if q.dim() != 4:
        raise ValueError("q must be [batch, tokens, num_q_heads, head_dim]")
    batch, tokens, hq = q.shape[0], q.shape[1], q.shape[2]
    if tuple(tree_mask.shape) != (batch, tokens):
        raise ValueError("tree_mask must be [batch, tokens]")
    if tree_mask.dtype not in (torch.int64, getattr(torch, "uint64", torch.int64)):
        raise TypeError("tree_mask must hold 64-bit integers (int64 or uint64 bit patterns)")
    dv = layout.desc.head_dim_v
    if out is None:
        out = torch.empty((batch, tokens, hq, dv), device=q.device,
                          dtype=out_dtype or torch.bfloat16)
    lens_h = _host_i32(seq_lens_host, "seq_lens_host")
    if len(lens_h) != batch:
        raise ValueError("seq_lens_host must have one entry per row")
    if workspace is None:
        workspace = _planned_workspace(decode_attn_multirow_workspace_bytes(
            layout, lens_h, page_tables.shape[1], tokens, hq, True, num_splits), q.device)
    opts = _opts(merge_group, events)
    _check(lib.decode_attn_tree(
        layout.handle, _dev(q, "q", layout.dtype), _dev(page_tables, "page_tables", torch.int32),
        page_tables.shape[1], lens_h, _dev(seq_lens, "seq_lens", torch.int32),
        _dev(tree_mask, "tree_mask"), batch, tokens, hq, float(scale), num_splits,
        None if workspace is None else _dev(workspace, "workspace"),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _dev(out, "out"), _dtype_code(out.dtype), None if opts is None else ctypes.byref(opts),
        _stream(stream)), "decode_attn_tree")
    return out


def prefill_attn_paged(layout: Layout, q, cu_q, cu_q_host, page_tables, seq_lens, seq_lens_host,
                       scale, window: int = 0, num_splits: int = 0, workspace=None, out=None,
                       out_dtype=None, merge_group: int = 0, events=None,
                       stream=None) -> torch.Tensor:
    """Paged prefill of variable-length chunks: ``q`` [total, num_q_heads,
    head_dim] packed by the row offsets ``cu_q`` (device) / ``cu_q_host``; row
    b's chunk is its last cu_q[b+1]-cu_q[b] keys, each token attending keys up
    to itself (within ``window`` keys when > 0).  Returns ``out`` [total,
    num_q_heads, head_dim]."""
    lib = load_library()
    if q.dim() != 3:
        raise ValueError("q must be [total, num_q_heads, head_dim]")
    total, hq = q.shape[0], q.shape[1]
    dv = layout.desc.head_dim_v
    if out is None:
        out = torch.empty((total, hq, dv), device=q.device, dtype=out_dtype or torch.bfloat16)
    cu_h = _host_i32(cu_q_host, "cu_q_host")
    lens_h = _host_i32(seq_lens_host, "seq_lens_host")
    batch = len(lens_h)
    if len(cu_h) != batch + 1:
        raise ValueError("cu_q_host must have batch + 1 entries")
    if workspace is None and num_splits != 1:
        workspace = _planned_workspace(prefill_attn_workspace_bytes(
            layout, cu_h, lens_h, page_tables.shape[1], hq, window, num_splits), q.device)
    opts = _opts(merge_group, events)
    _check(lib.prefill_attn_paged(
        layout.handle, _dev(q, "q", layout.dtype), cu_h, _dev(cu_q, "cu_q", torch.int32),
        _dev(page_tables, "page_tables", torch.int32), page_tables.shape[1], lens_h,
        _dev(seq_lens, "seq_lens", torch.int32), batch, hq, int(window), float(scale),
        num_splits, None if workspace is None else _dev(workspace, "workspace"),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _dev(out, "out"), _dtype_code(out.dtype), None if opts is None else ctypes.byref(opts),
        _stream(stream)), "prefill_attn_paged")
    return out


def decode_attn_splitkv_static(layout: Layout, q, page_tables, seq_lens, seq_lens_host, scale,
                               num_splits: int = 0, out=None, out_dtype=None,
                               stream=None) -> torch.Tensor:
    """Split-KV decode using the library's built-in scratch array instead of a
    workspace, for callers that cannot allocate device memory (see pskv.h)."""
    lib = load_library()
    if q.dim() != 3:
        raise ValueError("q must be [batch, num_q_heads, head_dim]")
    batch, hq = q.shape[0], q.shape[1]
    if out is None:
        out = torch.empty((batch, hq, layout.desc.head_dim_v), device=q.device,
                          dtype=out_dtype or torch.bfloat16)
    lens_h = _host_i32(seq_lens_host, "seq_lens_host")
    if len(lens_h) != batch:
        raise ValueError("seq_lens_host must have one entry per row")
    _check(lib.decode_attn_splitkv_static(
        layout.handle, _dev(q, "q", layout.dtype), _dev(page_tables, "page_tables", torch.int32),
        page_tables.shape[1], lens_h, _dev(seq_lens, "seq_lens", torch.int32), batch, hq,
        float(scale), num_splits, _dev(out, "out"), _dtype_code(out.dtype), _stream(stream)),
        "decode_attn_splitkv_static")
    return out


def merge_partials(m, l, o, out=None, out_dtype=None, workspace=None, status=None,
                   merge_group: int = 0, events=None, stream=None) -> torch.Tensor:
    """Merge partials m, l [rows, P] and o [rows, P, dv] into out [rows, dv]."""
    lib = load_library()
    rows, p, dv = o.shape
    if out is None:
        out = torch.empty((rows, dv), device=o.device, dtype=out_dtype or torch.float32)
    opts = _opts(merge_group, events)
    _check(lib.merge_partials(_dev(m, "m", torch.float32), _dev(l, "l", torch.float32),
                              _dev(o, "o", torch.float32), rows, p, dv, _dev(out, "out"),
                              _dtype_code(out.dtype),
                              None if workspace is None else _dev(workspace, "workspace"),
                              0 if workspace is None else workspace.numel() * workspace.element_size(),
                              None if status is None else _dev(status, "status", torch.int32),
                              None if opts is None else ctypes.byref(opts), _stream(stream)),
           "merge_partials")
    return out


def pskv_check_flags(layout: Layout, clear: bool = False, stream=None) -> int:
    """The layout's fault word (PSKV_FAULT_* bits) after the work enqueued so
    far; synchronizes the stream.  ``clear`` zeroes it for the next calls."""
    flags = ctypes.c_uint32()
    _check(load_library().pskv_check_flags(layout.handle, int(clear), _stream(stream),
                                           ctypes.byref(flags)), "pskv_check_flags")
    return int(flags.value)


def pskv_strerror(code: int) -> str:
    return load_library().pskv_strerror(code).decode()


def pskv_kernel_launches() -> int:
    return int(load_library().pskv_kernel_launches())


def pskv_version() -> int:
    return int(load_library().pskv_version())
