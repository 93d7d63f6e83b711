"""Plain fp64 CPU oracle for paged split-KV GQA decode attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may import this package.  It shares no code with the
CUDA library (``paged_split_kv_attn_gb300``) and never imports it.

The arithmetic lives in ``pskv_oracle.c``; this module only marshals numpy
arrays into it.  See that file for what is computed and which passage of the
source pages each step follows.

Arrays:
  * bf16 data is passed as ``uint16`` bit patterns, f32 data as ``float32``;
  * pools are ``[num_pages, num_kv_heads, page_size, head_dim]``; a K pool
    narrower than its V pool is a folded pool (see pskv_oracle.h);
  * ``q`` is ``[batch, num_q_heads, key width]`` (head_dim_k for a split pool,
    head_dim_v for a folded one), outputs are float64
    ``[batch, num_q_heads, head_dim_v]``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

ORC_OK = 0
ORC_ERR_INVALID = -1
ORC_ERR_PAST_PAGES = -2
ORC_ERR_OVERFLOW = -3
ORC_ERR_STATE = -4
ORC_ERR_BAD_PAGE = -5

_ERRORS = {
    ORC_ERR_INVALID: "invalid argument",
    ORC_ERR_PAST_PAGES: "position past the row's pages",
    ORC_ERR_OVERFLOW: "size overflow",
    ORC_ERR_STATE: "invalid softmax state",
    ORC_ERR_BAD_PAGE: "page id outside the pool",
}


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {_ERRORS.get(code, 'error')} ({code})")
        self.code = code


class _Pool(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dtype", ctypes.c_int),
                ("num_pages", ctypes.c_int64), ("page_size", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("head_dim_k", ctypes.c_int),
                ("head_dim_v", ctypes.c_int), ("format", ctypes.c_int)]


_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I, D, I64 = ctypes.c_int, ctypes.c_double, ctypes.c_int64
        lib.orc_attend_direct.argtypes = [P, P, P, I, I, I, I, D, P]
        lib.orc_online_partial.argtypes = [P, P, P, I, I, I, I, D, P, P, P]
        lib.orc_merge.argtypes = [D, D, P, D, D, P, I, P, P, P]
        lib.orc_finalize.argtypes = [D, D, P, I, P]
        lib.orc_attend_partitioned.argtypes = [P, P, P, I, I, P, I, I, D, P]
        lib.orc_attend_partitioned_f32.argtypes = [P, P, P, I, I, P, I, ctypes.c_float, P]
        lib.orc_gather.argtypes = [P, P, I, I, I, I, P, P]
        lib.orc_append_rows.argtypes = [P, P, P, P, P, P, P, I, P, I, P, I]
        lib.orc_decode_direct.argtypes = [P, P, P, I, P, P, P, I, I, D, P]
        lib.orc_decode_online.argtypes = [P, P, P, I, P, P, P, I, I, D, I, I, I, P]
        lib.orc_decode_multirow_direct.argtypes = [P, P, P, I, P, I, I, I, D, P]
        lib.orc_prefill_direct.argtypes = [P, P, P, P, I, P, I, I, I, D, P]
        lib.orc_decode_tree_direct.argtypes = [P, P, P, I, P, P, I, I, I, D, P]
        lib.orc_partial_scratch_bytes.argtypes = [I64, I64, I64, I64, P, P, P, P]
        lib.orc_num_threads.argtypes = []
        lib.orc_prep_head.argtypes = [P, I, D, P, I, P, P, P]
        lib.orc_prep_tokens.argtypes = [P, I, I64, I, I, I, I, I, I, I, I, D, P, P, P, P, I, P, I,
                                        P, P, P]
        _lib = lib
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != ORC_OK:
        raise OracleError(rc, what)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _data(a):
    """Contiguous view of pool / query data: uint16 (bf16 bits) or float32."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a, 1
    if a.dtype == np.float32:
        return a, 0
    raise TypeError(f"oracle data must be uint16 (bf16 bits) or float32, got {a.dtype}")


def num_threads() -> int:
    return int(_load().orc_num_threads())


# ---- dense, one query head -------------------------------------------------

def attend_direct(q, k, v, scale, begin=0, end=None):
    q, k, v = (_c(x, np.float64) for x in (q, k, v))
    end = k.shape[0] if end is None else end
    out = np.zeros(v.shape[1], np.float64)
    _check(_load().orc_attend_direct(_ptr(q), _ptr(k), _ptr(v), k.shape[1], v.shape[1],
                                     begin, end, scale, _ptr(out)), "attend_direct")
    return out


def online_partial(q, k, v, scale, begin, end):
    """Return (m, l, o) of the online state over keys [begin, end)."""
    q, k, v = (_c(x, np.float64) for x in (q, k, v))
    m, l = ctypes.c_double(), ctypes.c_double()
    o = np.zeros(v.shape[1], np.float64)
    _check(_load().orc_online_partial(_ptr(q), _ptr(k), _ptr(v), k.shape[1], v.shape[1], begin,
                                      end, scale, ctypes.byref(m), ctypes.byref(l), _ptr(o)),
           "online_partial")
    return m.value, l.value, o


def merge(a, b):
    """Merge two states (m, l, o) by the exact rescaling identity."""
    (ma, la, oa), (mb, lb, ob) = a, b
    oa, ob = _c(oa, np.float64), _c(ob, np.float64)
    m, l = ctypes.c_double(), ctypes.c_double()
    o = np.zeros_like(oa)
    _check(_load().orc_merge(ma, la, _ptr(oa), mb, lb, _ptr(ob), oa.shape[0], ctypes.byref(m),
                             ctypes.byref(l), _ptr(o)), "merge")
    return m.value, l.value, o


def finalize(state):
    m, l, o = state
    o = _c(o, np.float64)
    out = np.zeros_like(o)
    _check(_load().orc_finalize(m, l, _ptr(o), o.shape[0], _ptr(out)), "finalize")
    return out


def attend_partitioned(q, k, v, scale, bounds, group_size=16):
    q, k, v = (_c(x, np.float64) for x in (q, k, v))
    bounds = _c(bounds, np.int32)
    out = np.zeros(v.shape[1], np.float64)
    _check(_load().orc_attend_partitioned(_ptr(q), _ptr(k), _ptr(v), k.shape[1], v.shape[1],
                                          _ptr(bounds), len(bounds) - 1, group_size, scale,
                                          _ptr(out)), "attend_partitioned")
    return out


def attend_partitioned_f32(q, k, v, scale, bounds):
    q, k, v = (_c(x, np.float32) for x in (q, k, v))
    bounds = _c(bounds, np.int32)
    out = np.zeros(v.shape[1], np.float32)
    _check(_load().orc_attend_partitioned_f32(_ptr(q), _ptr(k), _ptr(v), k.shape[1], v.shape[1],
                                              _ptr(bounds), len(bounds) - 1, scale, _ptr(out)),
           "attend_partitioned_f32")
    return out


# ---- paged pool ------------------------------------------------------------

def _pool(k_pool, v_pool):
    k_pool, kt = _data(k_pool)
    v_pool, vt = _data(v_pool)
    if kt != vt or k_pool.ndim != 4 or v_pool.ndim != 4 or k_pool.shape[:3] != v_pool.shape[:3]:
        raise ValueError("k_pool / v_pool must be [num_pages, num_kv_heads, page_size, d] of one dtype")
    # a K region narrower than the V region is a folded pool
    fmt = 1 if k_pool.shape[3] < v_pool.shape[3] else 0
    p = _Pool(k_pool.ctypes.data, v_pool.ctypes.data, kt, k_pool.shape[0], k_pool.shape[2],
              k_pool.shape[1], k_pool.shape[3], v_pool.shape[3], fmt)
    return p, (k_pool, v_pool)


def gather(k_pool, v_pool, page_tables, b, g, length):
    """Keys (as a query meets them) and values of (row b, KV head g)."""
    pool, keep = _pool(k_pool, v_pool)
    tables = _c(page_tables, np.int32)
    k = np.zeros((length, pool.head_dim_v if pool.format else pool.head_dim_k), np.float64)
    v = np.zeros((length, pool.head_dim_v), np.float64)
    _check(_load().orc_gather(ctypes.byref(pool), _ptr(tables), tables.shape[1], b, g, length,
                              _ptr(k), _ptr(v)), "gather")
    return k, v


def append_rows(k_pool, v_pool, k_new, v_new, row_of, pos_of, page_tables, num_pages_of_row):
    """Append rows into the pools IN PLACE (they must be C-contiguous numpy arrays)."""
    for a in (k_pool, v_pool):
        if not a.flags.c_contiguous:
            raise ValueError("pools must be C-contiguous to be written in place")
    pool, _ = _pool(k_pool, v_pool)
    k_new, _ = _data(k_new)
    v_new, _ = _data(v_new)
    row_of, pos_of = _c(row_of, np.int32), _c(pos_of, np.int32)
    tables, lease = _c(page_tables, np.int32), _c(num_pages_of_row, np.int32)
    _check(_load().orc_append_rows(_ptr(k_pool), _ptr(v_pool), ctypes.byref(pool), _ptr(k_new),
                                   _ptr(v_new), _ptr(row_of), _ptr(pos_of), len(row_of),
                                   _ptr(tables), tables.shape[1], _ptr(lease), len(lease)),
           "append_rows")


def decode_direct(q, k_pool, v_pool, page_tables, seq_lens, scale, first_pos=None, window_lo=None):
    pool, keep = _pool(k_pool, v_pool)
    q, _ = _data(q)
    tables, lens = _c(page_tables, np.int32), _c(seq_lens, np.int32)
    fp, wl = _c(first_pos, np.int32), _c(window_lo, np.int32)
    out = np.zeros((q.shape[0], q.shape[1], pool.head_dim_v), np.float64)
    _check(_load().orc_decode_direct(ctypes.byref(pool), _ptr(q), _ptr(tables), tables.shape[1],
                                     _ptr(lens), _ptr(fp), _ptr(wl), q.shape[0], q.shape[1],
                                     scale, _ptr(out)), "decode_direct")
    return out


def decode_multirow_direct(q, k_pool, v_pool, page_tables, seq_lens, scale):
    """q [batch, tokens, num_q_heads, key width] -> out [batch, tokens, num_q_heads, dv]:
    token t of row b sits at key position len - tokens + t and attends causally."""
    pool, keep = _pool(k_pool, v_pool)
    q, _ = _data(q)
    tables, lens = _c(page_tables, np.int32), _c(seq_lens, np.int32)
    out = np.zeros((q.shape[0], q.shape[1], q.shape[2], pool.head_dim_v), np.float64)
    _check(_load().orc_decode_multirow_direct(ctypes.byref(pool), _ptr(q), _ptr(tables),
                                              tables.shape[1], _ptr(lens), q.shape[0], q.shape[1],
                                              q.shape[2], scale, _ptr(out)),
           "decode_multirow_direct")
    return out


def decode_tree_direct(q, k_pool, v_pool, page_tables, seq_lens, tree_mask, scale):
    """q [batch, tokens, num_q_heads, key width] -> out [batch, tokens, num_q_heads, dv]:
    the row's last `tokens` keys are a drafted tree in topological order;
    token t attends every key before the window and the window tokens whose
    bit is set in tree_mask[b, t] (uint64: its ancestors and itself)."""
    pool, keep = _pool(k_pool, v_pool)
    q, _ = _data(q)
    tables, lens = _c(page_tables, np.int32), _c(seq_lens, np.int32)
    mask = _c(tree_mask, np.uint64)
    if mask.shape != q.shape[:2]:
        raise ValueError("tree_mask must be [batch, tokens]")
    out = np.zeros((q.shape[0], q.shape[1], q.shape[2], pool.head_dim_v), np.float64)
    _check(_load().orc_decode_tree_direct(ctypes.byref(pool), _ptr(q), _ptr(tables),
                                          tables.shape[1], _ptr(lens), _ptr(mask), q.shape[0],
                                          q.shape[1], q.shape[2], scale, _ptr(out)),
           "decode_tree_direct")
    return out


def prefill_direct(q, cu_q, k_pool, v_pool, page_tables, seq_lens, scale, window=0):
    """q packed [total, num_q_heads, key width] -> out [total, num_q_heads, dv]:
    row b's last cu_q[b+1]-cu_q[b] keys are its new tokens, each attending
    causally (and within `window` keys when window > 0)."""
    pool, keep = _pool(k_pool, v_pool)
    q, _ = _data(q)
    cu = _c(cu_q, np.int32)
    tables, lens = _c(page_tables, np.int32), _c(seq_lens, np.int32)
    out = np.zeros((q.shape[0], q.shape[1], pool.head_dim_v), np.float64)
    _check(_load().orc_prefill_direct(ctypes.byref(pool), _ptr(q), _ptr(cu), _ptr(tables),
                                      tables.shape[1], _ptr(lens), int(window), lens.shape[0],
                                      q.shape[1], scale, _ptr(out)), "prefill_direct")
    return out


def decode_online(q, k_pool, v_pool, page_tables, seq_lens, scale, num_splits, chunk_tokens=None,
                  group_size=16, first_pos=None, window_lo=None):
    pool, keep = _pool(k_pool, v_pool)
    q, _ = _data(q)
    chunk_tokens = pool.page_size if chunk_tokens is None else chunk_tokens
    tables, lens = _c(page_tables, np.int32), _c(seq_lens, np.int32)
    fp, wl = _c(first_pos, np.int32), _c(window_lo, np.int32)
    out = np.zeros((q.shape[0], q.shape[1], pool.head_dim_v), np.float64)
    _check(_load().orc_decode_online(ctypes.byref(pool), _ptr(q), _ptr(tables), tables.shape[1],
                                     _ptr(lens), _ptr(fp), _ptr(wl), q.shape[0], q.shape[1],
                                     scale, chunk_tokens, num_splits, group_size, _ptr(out)),
           "decode_online")
    return out


def partial_scratch_bytes(batch, num_q_heads, head_dim_v, num_splits):
    """(maxima, denominators, numerators, total) bytes of the partial buffer."""
    vals = [ctypes.c_size_t() for _ in range(4)]
    _check(_load().orc_partial_scratch_bytes(batch, num_q_heads, head_dim_v, num_splits,
                                             *[ctypes.byref(x) for x in vals]),
           "partial_scratch_bytes")
    return tuple(int(x.value) for x in vals)


# ---- K/V prep ------------------------------------------------------------------

def prep_head(x, eps, w=None, cos=None, sin=None):
    """One head row: RMS-normalise, multiply by w, rotate the first 2*len(cos)
    columns as pairs (i, i + len(cos))."""
    x = _c(x, np.float64)
    w = _c(w, np.float64)
    cos, sin = _c(cos, np.float64), _c(sin, np.float64)
    rot = 0 if cos is None else 2 * cos.shape[0]
    out = np.zeros(x.shape[0], np.float64)
    _check(_load().orc_prep_head(_ptr(x), x.shape[0], eps, _ptr(w), rot, _ptr(cos), _ptr(sin),
                                 _ptr(out)), "prep_head")
    return out


def prep_tokens(x, q_col, k_col, v_col, num_q_heads, num_kv_heads, head_dim, eps, w_q, w_k,
                rope_cos, rope_sin, rope_pos, folded=False):
    """Prep n tokens from projection rows x [n, stride] (uint16 bf16 bits or
    float32).  rope_cos / rope_sin are float32 [max_pos, rot/2].  Returns fp64
    (q [n, Hq, D], k [n, Hkv, D], v [n, Hkv, D])."""
    x, xd = _data(x)
    n = x.shape[0]
    rope_cos, rope_sin = _c(rope_cos, np.float32), _c(rope_sin, np.float32)
    w_q, w_k = _c(w_q, np.float32), _c(w_k, np.float32)
    pos = _c(rope_pos, np.int32)
    rot = 2 * rope_cos.shape[1]
    q = np.zeros((n, num_q_heads, head_dim), np.float64)
    k = np.zeros((n, num_kv_heads, head_dim), np.float64)
    v = np.zeros((n, num_kv_heads, head_dim), np.float64)
    _check(_load().orc_prep_tokens(_ptr(x), xd, x.shape[1], q_col, k_col, v_col, n, num_q_heads,
                                   num_kv_heads, head_dim, rot, eps, _ptr(w_q), _ptr(w_k),
                                   _ptr(rope_cos), _ptr(rope_sin), rope_cos.shape[0], _ptr(pos),
                                   int(folded), _ptr(q), _ptr(k), _ptr(v)), "prep_tokens")
    return q, k, v
