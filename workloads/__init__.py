"""Seeded synthetic inputs for paged split-KV decode attention.

This module only MAKES inputs: random values, page permutations, lengths and
the placement of rows into pages.  It holds none of the attention arithmetic,
so both the CPU oracle's tests and the CUDA library's tests and bench can draw
from it without sharing any of the method.

Recipe (stated once, used everywhere):
  * values ~ N(0, 1) drawn as float32 from a PCG64 stream spawned from
    ``numpy.random.SeedSequence(seed)`` and, for bf16 data, rounded to
    nearest-even bf16 (carried as uint16 bits); the page order comes from a
    second spawned stream, so it never changes the values;
  * every row's pages are drawn without replacement from one shuffled pool
    of page ids, so page order in a table is a random permutation;
  * page ``num_pages - 1`` is a poison page filled with NaN; table entries past
    a row's pages point at it, and rows of the last page past the row's
    length are NaN too ("padding past the plan"): none of it may reach an output.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

BF16_NAN = np.uint16(0x7FC0)


def bf16_bits(x) -> np.ndarray:
    """Round float32 values to bf16 (nearest even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits) -> np.ndarray:
    """Exact float32 value of bf16 bit patterns."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal(rng, shape, dtype):
    x = rng.standard_normal(shape, dtype=np.float32)
    return bf16_bits(x) if dtype == "bf16" else x


def ragged_lengths(seed: int, n: int, hi: int) -> list[int]:
    """n lengths drawn log-uniform: L = max(1, floor(exp(U[0, ln hi))))."""
    rng = np.random.Generator(np.random.PCG64(seed))
    u = rng.uniform(0.0, math.log(hi), size=n)
    return [max(1, int(math.floor(math.exp(x)))) for x in u]


@dataclasses.dataclass
class PagedCase:
    """One synthetic decode problem over a paged pool."""
    dtype: str                  # "bf16" (uint16 bits) or "f32"
    q: np.ndarray               # [batch, num_q_heads, head_dim]
    k_pool: np.ndarray          # [num_pages, num_kv_heads, page_size, head_dim]
    v_pool: np.ndarray          # same shape as k_pool
    page_tables: np.ndarray     # int32 [batch, table_stride]
    seq_lens: np.ndarray        # int32 [batch]
    pages_of_row: np.ndarray    # int32 [batch]: pages each row holds
    poison_page: int
    scale: float
    first_pos: np.ndarray | None = None   # int32 [batch] (windowed cases)
    window_lo: np.ndarray | None = None   # int32 [batch] (windowed cases)
    dense_k: list | None = None           # per row [len, num_kv_heads, head_dim] (small cases)
    dense_v: list | None = None

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def num_q_heads(self) -> int:
        return self.q.shape[1]

    @property
    def num_kv_heads(self) -> int:
        return self.k_pool.shape[1]

    @property
    def head_dim(self) -> int:
        return self.v_pool.shape[3]

    @property
    def folded(self) -> bool:
        """True for a folded pool (the K region narrower than the V region)."""
        return self.k_pool.shape[3] < self.v_pool.shape[3]

    @property
    def page_size(self) -> int:
        return self.k_pool.shape[2]

    @property
    def num_pages(self) -> int:
        return self.k_pool.shape[0]

    def kv_bytes(self) -> int:
        """Bytes of K and V the attended keys occupy."""
        es = 2 if self.dtype == "bf16" else 4
        row_elems = self.k_pool.shape[3] + self.v_pool.shape[3]
        n = 0
        for b in range(self.batch):
            lo = 0
            if self.window_lo is not None:
                lo = min(max(int(self.window_lo[b]) - int(self.first_pos[b]), 0), int(self.seq_lens[b]))
            n += int(self.seq_lens[b]) - lo
        return n * self.num_kv_heads * row_elems * es


def make_paged_case(seed: int, seq_lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
                    page_size: int, dtype: str = "bf16", shuffle: bool = True,
                    extra_pages: int = 0, table_stride: int | None = None,
                    keep_dense: bool | None = None, scale: float | None = None,
                    k_dims: int | None = None) -> PagedCase:
    """Build a paged pool holding random K/V for every row, plus random queries.

    ``k_dims`` < head_dim makes a folded pool: the K region keeps k_dims
    columns per row, the V region head_dim (queries are head_dim wide)."""
    if dtype not in ("bf16", "f32"):
        raise ValueError(dtype)
    # values and page order come from independent streams, so a shuffled and an
    # identity table over the same seed hold the same values
    vals_seq, pages_seq = np.random.SeedSequence(seed).spawn(2)
    rng = np.random.Generator(np.random.PCG64(vals_seq))
    seq_lens = [int(x) for x in seq_lens]
    batch = len(seq_lens)
    pages_of_row = [max(1, -(-n // page_size)) for n in seq_lens]
    used = sum(pages_of_row)
    num_pages = used + extra_pages + 1
    poison = num_pages - 1
    stride = max(pages_of_row) if table_stride is None else table_stride
    if stride < max(pages_of_row):
        raise ValueError("table_stride too small for the longest row")
    if keep_dense is None:
        keep_dense = sum(seq_lens) * num_kv_heads * head_dim <= (1 << 22)

    ids = np.arange(num_pages - 1, dtype=np.int64)
    if shuffle:
        ids = np.random.Generator(np.random.PCG64(pages_seq)).permutation(ids)
    tables = np.full((batch, stride), poison, np.int32)
    cursor = 0
    for b, n in enumerate(pages_of_row):
        tables[b, :n] = ids[cursor:cursor + n]
        cursor += n

    dk = head_dim if k_dims is None else k_dims
    shape = (num_pages, num_kv_heads, page_size, head_dim)
    kshape = (num_pages, num_kv_heads, page_size, dk)
    if dtype == "bf16":
        k_pool = np.full(kshape, BF16_NAN, np.uint16)
        v_pool = np.full(shape, BF16_NAN, np.uint16)
    else:
        k_pool = np.full(kshape, np.nan, np.float32)
        v_pool = np.full(shape, np.nan, np.float32)

    dense_k, dense_v = ([], []) if keep_dense else (None, None)
    for b, n in enumerate(seq_lens):
        if keep_dense:
            dkk = _normal(rng, (n, num_kv_heads, dk), dtype)
            dvv = _normal(rng, (n, num_kv_heads, head_dim), dtype)
            dense_k.append(dkk)
            dense_v.append(dvv)
        for j in range(pages_of_row[b]):
            lo, hi = j * page_size, min(n, (j + 1) * page_size)
            if hi <= lo:
                continue
            page = tables[b, j]
            if keep_dense:
                kk = dkk[lo:hi].transpose(1, 0, 2)
                vv = dvv[lo:hi].transpose(1, 0, 2)
            else:
                kk = _normal(rng, (num_kv_heads, hi - lo, dk), dtype)
                vv = _normal(rng, (num_kv_heads, hi - lo, head_dim), dtype)
            k_pool[page, :, :hi - lo, :] = kk
            v_pool[page, :, :hi - lo, :] = vv

    q = _normal(rng, (batch, num_q_heads, head_dim), dtype)
    return PagedCase(dtype=dtype, q=q, k_pool=k_pool, v_pool=v_pool, page_tables=tables,
                     seq_lens=np.asarray(seq_lens, np.int32),
                     pages_of_row=np.asarray(pages_of_row, np.int32), poison_page=poison,
                     scale=(1.0 / math.sqrt(head_dim)) if scale is None else scale,
                     dense_k=dense_k, dense_v=dense_v)


def window_queries(case: PagedCase, tokens: int, seed: int = 0) -> np.ndarray:
    """Random queries for a verify window of ``tokens`` per row:
    [batch, tokens, num_q_heads, head_dim] in the case's dtype."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tokens])))
    return _normal(rng, (case.batch, tokens, case.num_q_heads, case.head_dim), case.dtype)


def with_window(case: PagedCase, window: int, first_pos=None) -> PagedCase:
    """Give every row a window lower bound so that the query (at position
    first_pos + len - 1) sees the last ``window`` positions, itself included."""
    fp = np.zeros(case.batch, np.int32) if first_pos is None else np.asarray(first_pos, np.int32)
    q_pos = fp.astype(np.int64) + case.seq_lens.astype(np.int64) - 1
    lo = np.maximum(0, q_pos - window + 1).astype(np.int32)
    return dataclasses.replace(case, first_pos=fp, window_lo=lo)


# ---- the named workloads ---------------------------------------------------

GLOBAL_SHAPE = dict(num_q_heads=32, num_kv_heads=4, head_dim=512, page_size=256)
WINDOW_SHAPE = dict(num_q_heads=32, num_kv_heads=16, head_dim=256, page_size=64)
WINDOW = 1024


def folded_case(context: int, seed: int = 0, batch: int = 1) -> PagedCase:
    """The global-layer shape in the folded format: per token and KV head the
    K region keeps the rotated quarter (128 columns), V all 512 (640 in all)."""
    return make_paged_case(seed, [context] * batch, dtype="bf16", k_dims=128, **GLOBAL_SHAPE)


def tiny_case(seed: int = 0) -> PagedCase:
    """Batch 1, 8 query heads on 1 KV head, head dim 512, 1,000 keys in 4 pages
    of 256 (last page partial), f32, scale 1/sqrt(512)."""
    return make_paged_case(seed, [1000], num_q_heads=8, num_kv_heads=1, head_dim=512,
                           page_size=256, dtype="f32")


def global_case(context: int, seed: int = 0, batch: int = 1) -> PagedCase:
    """Gemma-4-31B global-layer decode: 32 q heads, 4 KV heads, head dim 512,
    bf16, shuffled pages of 256."""
    return make_paged_case(seed, [context] * batch, dtype="bf16", **GLOBAL_SHAPE)


def window_case(residency: int, seed: int = 0, first_pos: int = 0) -> PagedCase:
    """Sliding-window decode: 32 q heads, 16 KV heads, head dim 256, window
    1,024, pages of 64, bf16."""
    c = make_paged_case(seed, [residency], dtype="bf16", **WINDOW_SHAPE)
    return with_window(c, WINDOW, [first_pos])


def ragged_case(seed: int = 0, n: int = 16, hi: int = 131072) -> PagedCase:
    """16 rows, lengths log-uniform in [1, 131,072], global-layer shape, one
    shared shuffled pool of pages of 256."""
    return make_paged_case(seed, ragged_lengths(seed, n, hi), dtype="bf16", **GLOBAL_SHAPE)


# ---- drafted token trees ---------------------------------------------------------

def random_tree_parents(seed: int, tokens: int, roots: float = 0.1) -> np.ndarray:
    """Parent index of each of `tokens` drafted tokens in topological order:
    token 0 is a root (-1: it hangs off the accepted prefix); token t > 0 is
    another root with probability `roots`, else the child of a uniformly
    drawn earlier token."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tokens, 5])))
    parents = np.full(tokens, -1, np.int64)
    for t in range(1, tokens):
        parents[t] = -1 if rng.random() < roots else int(rng.integers(0, t))
    return parents


def chain_parents(tokens: int) -> np.ndarray:
    """A chain: token t's parent is t - 1 (a plain causal verify window)."""
    return np.arange(-1, tokens - 1, dtype=np.int64)


def tree_masks(parents) -> np.ndarray:
    """uint64 ancestor masks: bit j of mask[t] is set iff window token j is t
    itself or one of its ancestors."""
    parents = np.asarray(parents, np.int64)
    masks = np.zeros(len(parents), np.uint64)
    for t, p in enumerate(parents):
        if not (-1 <= p < t):
            raise ValueError("parents must precede their children")
        masks[t] = np.uint64(1 << t) | (masks[p] if p >= 0 else np.uint64(0))
    return masks


# ---- K/V prep inputs -----------------------------------------------------------

@dataclasses.dataclass
class PrepInputs:
    """Projection rows of n new tokens and the prep's parameters."""
    x: np.ndarray            # bf16 bits [n, stride]: q band | K band | V band
    q_col: int
    k_col: int
    v_col: int               # == k_col when K and V share one projection
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    rot: int                 # leading columns rotated
    eps: float
    w_q: np.ndarray          # float32 [head_dim]
    w_k: np.ndarray          # float32 [head_dim]
    rope_cos: np.ndarray     # float32 [max_pos, rot / 2]
    rope_sin: np.ndarray


def rope_tables(max_pos: int, rot: int, theta: float = 10000.0):
    """cos / sin tables [max_pos, rot/2] (float32) of angles pos * theta^(-2i/rot)."""
    i = np.arange(rot // 2, dtype=np.float64)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * theta ** (-2.0 * i / rot)[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def make_prep_inputs(seed: int, n: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                     rot: int, max_pos: int, shared_kv: bool = False, eps: float = 1e-6,
                     theta: float = 10000.0) -> PrepInputs:
    """Random projection rows (each head row N(0,1) times a log-uniform scale in
    [0.1, 10]), norm multipliers 1 + 0.25 N(0,1), and rotation tables."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 77])))
    q_w = num_q_heads * head_dim
    kv_w = num_kv_heads * head_dim
    q_col, k_col = 0, q_w
    v_col = k_col if shared_kv else k_col + kv_w
    stride = v_col + kv_w
    heads = stride // head_dim
    x = rng.standard_normal((n, heads, head_dim), dtype=np.float32)
    x *= np.exp(rng.uniform(math.log(0.1), math.log(10.0), size=(n, heads, 1))).astype(np.float32)
    cos, sin = rope_tables(max_pos, rot, theta)
    return PrepInputs(x=bf16_bits(x.reshape(n, stride)), q_col=q_col, k_col=k_col, v_col=v_col,
                      num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                      rot=rot, eps=eps,
                      w_q=(1 + 0.25 * rng.standard_normal(head_dim)).astype(np.float32),
                      w_k=(1 + 0.25 * rng.standard_normal(head_dim)).astype(np.float32),
                      rope_cos=cos, rope_sin=sin)
