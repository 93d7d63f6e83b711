"""GPU parity of the key-major tensor-memory kernel (verify windows of 17 to
64 query columns per KV head) against the oracle; the 16-column cases check
the split-KV path the library keeps for them.

Token t of a T-token window sits at key len - T + t and attends keys up to
itself (TensorFold #1619: drafted verify windows read their keys through the
page table).  The kernel takes 128 keys per tile as the MMA's M and the
window's columns, zero-padded to 32 or 64, as its N; the library routes a
call there when its longest row has at least 8,192 keys, so every case below
holds such a row (LONG) beside its short ones.  Bars as for single-token
decode: max |out - fp64| <= 2e-3 in the fp32 output mode, the bf16 output the
round-to-nearest-even of the fp32 one."""
import numpy as np
import pytest
import torch

import oracle
import paged_split_kv_attn_gb300 as pskv
import workloads as W
from gpu_cases import TOL, DevCase, bf16_of, i32, max_err, to_dev

pytestmark = pytest.mark.gpu

LONG = 8300  # a row long enough for the key-major kernel (8,192 keys or more)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_split_kv_attn_gb300 import build
    build.build()
    pskv.load_library()


def run(dc, q, num_splits=0, out_dtype=torch.float32, lens=None, tables=None):
    c = dc.case
    return pskv.decode_attn_multirow(dc.layout, q, dc.tables if tables is None else tables,
                                     dc.lens if lens is None else lens, c.seq_lens, c.scale,
                                     num_splits=num_splits, out_dtype=out_dtype)


def check(case, tokens, splits=(0,), seed=0):
    dc = DevCase(case)
    qn = W.window_queries(case, tokens, seed)
    ref = oracle.decode_multirow_direct(qn, case.k_pool, case.v_pool, case.page_tables,
                                        case.seq_lens, case.scale)
    q = to_dev(qn, case.dtype)
    for p in splits:
        out32 = run(dc, q, p)
        out16 = run(dc, q, p, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert np.all(np.isfinite(out32.cpu().numpy())), f"non-finite output (splits={p})"
        err = max_err(out32, ref)
        assert err <= TOL, f"max |err| {err:.3e} > {TOL} (tokens={tokens}, splits={p})"
        assert torch.equal(out16, bf16_of(out32)), "bf16 output is not RNE of the fp32 output"
    assert dc.faults() == 0


def case_of(seed, lens, hq, hkv, d, ps, **kw):
    return W.make_paged_case(seed, lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                             page_size=ps, dtype="bf16", **kw)


@pytest.mark.parametrize("tokens", [2, 3, 4, 8])
def test_global_shape(tokens):
    """32 query heads on 4 KV heads, head dim 512, pages of 256: 16 to 64
    columns; rows of several tiles with ragged tails, one, several and more
    partitions than tiles (empty partitions)."""
    check(case_of(301 + tokens, [1000, 2900, 257, 130, LONG], 32, 4, 512, 256), tokens,
          splits=(0, 1, 3, 40, 90))


@pytest.mark.parametrize("group,tokens,ps", [(2, 8, 64), (2, 32, 64), (2, 13, 16), (1, 64, 64),
                                             (4, 16, 16), (8, 2, 64)])
def test_head_dim_256(group, tokens, ps):
    """Head dim 256 (two chunks per tile), pages of 64 (two pages per tile) and
    of 16 (16-row copies)."""
    hkv = 2
    check(case_of(310 + tokens + ps, [700, LONG, 1234], group * hkv, hkv, 256, ps), tokens,
          splits=(0, 1, 5))


@pytest.mark.parametrize("group,tokens", [(32, 2), (16, 4), (1, 16), (1, 64), (2, 32), (8, 5)])
def test_groups(group, tokens):
    """Query heads per KV head from 1 to 32 at head dim 512 (pages of 16 and
    of 256)."""
    hkv = 2
    check(case_of(320 + group + tokens, [900, 333, LONG], group * hkv, hkv, 512,
                  16 if group < 8 else 256), tokens, splits=(0, 4))


def test_rows_at_tile_edges():
    """len == T, and lengths one short of, at and one past a tile of 128 keys
    (the zeroed rows of a partial 16-key group, and whole groups skipped)."""
    check(case_of(330, [4, 127, 128, 129, 255, 256, 17, 8192], 16, 2, 512, 256), 4,
          splits=(0, 1, 2))


def test_page_outside_the_pool_is_skipped_and_flagged():
    """A table entry past the pool: its keys are skipped (no copy is issued)
    and PSKV_FAULT_BAD_PAGE is raised; the result is the oracle's over the row
    without that page (its keys all lie before the window, so every token
    sees the same keys either way)."""
    ps = 64
    case = case_of(331, [700, LONG], 32, 4, 512, ps)
    dc = DevCase(case)
    qn = W.window_queries(case, 4, 1)
    q = to_dev(qn, "bf16")
    tables = case.page_tables.copy()
    tables[0, 2] = case.page_tables.max() + 1000
    kept = case.page_tables.copy()
    kept[0] = np.concatenate([case.page_tables[0, :2], case.page_tables[0, 3:],
                              case.page_tables[0, :1]])
    lens_kept = case.seq_lens.copy()
    lens_kept[0] -= ps
    ref = oracle.decode_multirow_direct(qn, case.k_pool, case.v_pool, kept, lens_kept,
                                        case.scale)
    for p in (1, 3, 0):
        out = run(dc, q, p, tables=i32(tables))
        torch.cuda.synchronize()
        err = max_err(out, ref)
        assert err <= TOL, f"max |err| {err:.3e} (splits={p})"
    assert dc.faults() & pskv.PSKV_FAULT_BAD_PAGE


def test_device_length_below_the_window_is_flagged():
    """A device length shorter than the window (the host copy was fine) is
    clamped and flagged BAD_LENGTH, and nothing is read outside the row's pages."""
    case = case_of(332, [300, LONG], 32, 4, 512, 256)
    dc = DevCase(case)
    q = to_dev(W.window_queries(case, 4), "bf16")
    run(dc, q, 2, lens=i32([2, LONG]))
    torch.cuda.synchronize()
    assert dc.faults() & pskv.PSKV_FAULT_BAD_LENGTH


def test_run_to_run_deterministic():
    case = case_of(333, [LONG + 700, 3000], 32, 4, 512, 256)
    dc = DevCase(case)
    q = to_dev(W.window_queries(case, 4), "bf16")
    a, b = run(dc, q, 0), run(dc, q, 0)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("tokens", [2, 4, 8])
def test_bench_global_window_at_40002_keys(tokens):
    """The bench's verify windows at full size: one row of 40,002 keys, 32 q /
    4 KV heads, head dim 512, pages of 256 in a shuffled pool, the automatic
    plan; every output against the oracle."""
    case = W.make_paged_case(334, [40002], num_q_heads=32, num_kv_heads=4, head_dim=512,
                             page_size=256, dtype="bf16", keep_dense=False)
    check(case, tokens, splits=(0,), seed=tokens)
