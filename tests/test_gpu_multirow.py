"""GPU parity of multi-row decode (verify windows) against the oracle.

Token t of a T-token window sits at key len - T + t and attends keys up to
itself (TensorFold #1619: drafted verify windows read their keys through the
page table).  Bars as for single-token decode: max |out - fp64| <= 2e-3 in the
fp32 output mode, the bf16 output the round-to-nearest-even of the fp32 one."""
import numpy as np
import pytest
import torch

import oracle
import paged_split_kv_attn_gb300 as pskv
import workloads as W
from gpu_cases import TOL, DevCase, bf16_of, i32, max_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_split_kv_attn_gb300 import build
    build.build()
    pskv.load_library()


def run(dc, q, num_splits=0, out_dtype=torch.float32, lens=None, **kw):
    c = dc.case
    return pskv.decode_attn_multirow(dc.layout, q, dc.tables, dc.lens if lens is None else lens,
                                     c.seq_lens, c.scale, num_splits=num_splits,
                                     out_dtype=out_dtype, **kw)


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
        assert out32.shape == (case.batch, tokens, case.num_q_heads, case.head_dim)
        assert np.all(np.isfinite(out32.cpu().numpy())), "non-finite output"
        err = max_err(out32, ref)
        assert err <= TOL, f"max |err| {err:.3e} > {TOL} (tokens={tokens}, splits={p})"
        assert torch.equal(out16, bf16_of(out32)), "bf16 output is not RNE of the fp32 output"
    assert dc.faults() == 0


def small(seed, lens, hq, hkv, d, ps, **kw):
    return W.make_paged_case(seed, lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                             page_size=ps, dtype="bf16", **kw)


@pytest.mark.parametrize("tokens", [1, 2])
def test_global_shape_window(tokens):
    """32 query heads on 4 KV heads, head dim 512: two tokens fill two n-tiles."""
    check(small(71, [1000, 2900, 257], 32, 4, 512, 256), tokens, splits=(0, 1, 7, 40))


@pytest.mark.parametrize("group,tokens", [(8, 3), (8, 5), (4, 3), (2, 8), (1, 16), (1, 5),
                                          (2, 13)])
def test_column_blocks(group, tokens):
    """Columns past one n-tile: blocks of 16 per CTA, the last one padded."""
    hkv = 2
    check(small(72 + tokens, [700, 1234], group * hkv, hkv, 512, 256), tokens, splits=(0, 5))


def test_longest_window_at_head_dim_256():
    check(small(73, [300, 4000], 16, 2, 256, 64), pskv.PSKV_MAX_WINDOW_TOKENS, splits=(0, 3))


def test_rows_as_short_as_the_window():
    """len == T: token 0 sees key 0 alone, the last token every key; one row
    ends mid-tile, the other fills whole tiles."""
    check(small(74, [4, 17, 32, 4], 16, 2, 512, 256), 4, splits=(0, 1, 2))


def test_folded_pool_window():
    """The folded 640-column format: scores from K's stored quarter and V's rest."""
    check(W.make_paged_case(75, [1500, 600], num_q_heads=32, num_kv_heads=4, head_dim=512,
                            page_size=256, dtype="bf16", k_dims=128), 2, splits=(0, 9))


def test_one_token_equals_single_token_decode_bitwise():
    case = small(76, [3000, 777], 32, 4, 512, 256)
    dc = DevCase(case)
    for p in (1, 13, 0):
        a = run(dc, dc.q.unsqueeze(1), p)
        b = dc.decode(num_splits=p)
        torch.cuda.synchronize()
        assert torch.equal(a[:, 0], b)


def test_run_to_run_deterministic():
    case = small(77, [5000], 32, 4, 512, 256)
    dc = DevCase(case)
    q = to_dev(W.window_queries(case, 2), "bf16")
    a, b = run(dc, q, 0), run(dc, q, 0)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_device_length_below_the_window_is_flagged():
    """A device length shorter than the window (the host copy was fine) is
    clamped, flagged BAD_LENGTH, and nothing is read outside the row's pages."""
    case = small(78, [100], 16, 2, 512, 256)
    dc = DevCase(case)
    q = to_dev(W.window_queries(case, 4), "bf16")
    run(dc, q, 2, lens=i32([2]))
    torch.cuda.synchronize()
    assert dc.faults() & pskv.PSKV_FAULT_BAD_LENGTH


@pytest.mark.parametrize("hd,hq,hkv,tokens", [(256, 32, 2, 4), (512, 32, 2, 3)])
def test_wide_windows_of_large_groups(hd, hq, hkv, tokens):
    """16 query heads per KV head: windows of 64 / 48 columns run on the
    tensor-memory kernel (the split-KV kernels do not serve this group)."""
    check(small(79 + tokens, [900, 333], hq, hkv, hd, 64), tokens, splits=(0, 1, 4))
