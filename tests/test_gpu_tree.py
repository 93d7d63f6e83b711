"""GPU parity of tree attention over a drafted window against the oracle.

The window's tokens are the row's last keys in topological order; token t
attends every key before the window and the window tokens its ancestor mask
marks, itself included (TensorFold #1619, description "Reads" and review
thread: tree-attention rows read their keys through the page table).  Bars
as for single-token decode: max |out - fp64| <= 2e-3 in the fp32 output mode,
the bf16 output the round-to-nearest-even of the fp32 one."""
import numpy as np
import pytest
import torch

import oracle
import paged_split_kv_attn_gb300 as pskv
import workloads as W
from gpu_cases import TOL, DevCase, bf16_of, max_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_split_kv_attn_gb300 import build
    build.build()
    pskv.load_library()


def masks_of(case, tokens, seed, chain=False):
    """[batch, tokens] uint64 ancestor masks, one seeded tree per row."""
    if chain:
        return np.tile(W.tree_masks(W.chain_parents(tokens)), (case.batch, 1))
    return np.stack([W.tree_masks(W.random_tree_parents(seed * 131 + b, tokens))
                     for b in range(case.batch)])


def dev_masks(masks):
    return torch.from_numpy(np.ascontiguousarray(masks).view(np.int64)).cuda()


def run(dc, q, masks_dev, num_splits=0, out_dtype=torch.float32):
    c = dc.case
    return pskv.decode_attn_tree(dc.layout, q, dc.tables, dc.lens, c.seq_lens, masks_dev, c.scale,
                                 num_splits=num_splits, out_dtype=out_dtype)


def check(case, tokens, splits=(0,), seed=0, chain=False):
    dc = DevCase(case)
    qn = W.window_queries(case, tokens, seed)
    masks = masks_of(case, tokens, seed, chain)
    ref = oracle.decode_tree_direct(qn, case.k_pool, case.v_pool, case.page_tables,
                                    case.seq_lens, masks, case.scale)
    q, md = to_dev(qn, case.dtype), dev_masks(masks)
    for p in splits:
        out32 = run(dc, q, md, p)
        out16 = run(dc, q, md, p, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert np.all(np.isfinite(out32.cpu().numpy())), "non-finite output"
        err = max_err(out32, ref)
        assert err <= TOL, f"max |err| {err:.3e} > {TOL} (tokens={tokens}, splits={p})"
        assert torch.equal(out16, bf16_of(out32)), "bf16 output is not RNE of the fp32 output"
    assert dc.faults() == 0
    return dc, q, md


def small(seed, lens, hq, hkv, d, ps, **kw):
    return W.make_paged_case(seed, lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                             page_size=ps, dtype="bf16", **kw)


@pytest.mark.parametrize("tokens", [2, 3, 5, 8])
def test_global_shape_trees(tokens):
    """32 query heads on 4 KV heads, head dim 512: 16 to 64 columns per KV head
    in blocks of 16, several split counts (1: the direct path, no merge)."""
    check(small(101 + tokens, [1000, 2900, 257], 32, 4, 512, 256), tokens, splits=(0, 1, 7, 40),
          seed=tokens)


@pytest.mark.parametrize("group,tokens", [(1, 64), (2, 32), (4, 16), (8, 13)])
def test_large_trees(group, tokens):
    check(small(110 + tokens, [3000, tokens + 5], group * 2, 2, 512, 256), tokens, splits=(0, 3),
          seed=tokens)


def test_sliding_shape_tree():
    """32 query heads on 16 KV heads, head dim 256, pages of 64."""
    check(small(120, [1088, 600], 32, 16, 256, 64), 6, splits=(0, 5), seed=3)


def test_folded_pool_tree():
    check(W.make_paged_case(121, [1500, 600], num_q_heads=32, num_kv_heads=4, head_dim=512,
                            page_size=256, dtype="bf16", k_dims=128), 4, splits=(0, 9), seed=4)


def test_rows_that_hold_only_the_window():
    """len == T: a root sees its own key alone (its value, exactly, in f32)."""
    check(small(122, [8, 8, 21], 16, 2, 512, 256), 8, splits=(0, 1, 2), seed=5)


@pytest.mark.parametrize("tokens", [3, 4, 5, 8])
def test_key_major_kernel_trees(tokens):
    """17 to 64 columns per KV head on rows of 8,192 keys or more run on the
    key-major tensor-memory kernel (24 / 32 / 40 / 64 columns here)."""
    check(small(130 + tokens, [9000, 12345], 32, 4, 512, 256), tokens, splits=(0, 1, 5),
          seed=tokens)


def test_key_major_kernel_trees_at_head_dim_256():
    """16 query heads per KV head (a group the split-KV consumer does not serve):
    4 tokens are 64 columns on the key-major kernel."""
    check(small(136, [9000, 8192], 32, 2, 256, 64), 4, splits=(0, 3), seed=11)


def test_long_row():
    """40,002 keys of the global shape with an 8-token tree, automatic plan."""
    check(W.global_case(40002, seed=123), 8, splits=(0,), seed=6)


def test_chain_equals_the_causal_window_on_the_key_major_kernel():
    case = small(137, [20000], 32, 4, 512, 256)
    for tokens in (4, 8):
        dc, q, md = check(case, tokens, splits=(0,), chain=True)
        for p in (0, 3):
            a = run(dc, q, md, p)
            b = pskv.decode_attn_multirow(dc.layout, q, dc.tables, dc.lens, case.seq_lens,
                                          case.scale, num_splits=p, out_dtype=torch.float32)
            torch.cuda.synchronize()
            assert torch.equal(a, b)


def test_chain_equals_the_causal_window_bitwise():
    """A chain mask gives decode_attn_multirow's causal window, bit for bit, on
    the kernels both run on (16 columns per KV head; 24 on rows below 8,192 keys)."""
    for tokens, lens in ((2, [40002]), (3, [5000, 777])):
        case = small(124 + tokens, lens, 32, 4, 512, 256)
        dc, q, md = check(case, tokens, splits=(0,), chain=True)
        for p in (0, 1, 11):
            a = run(dc, q, md, p)
            b = pskv.decode_attn_multirow(dc.layout, q, dc.tables, dc.lens, case.seq_lens,
                                          case.scale, num_splits=p, out_dtype=torch.float32)
            torch.cuda.synchronize()
            assert torch.equal(a, b)


def test_run_to_run_deterministic():
    case = small(126, [9000], 32, 4, 512, 256)
    dc, q, md = check(case, 5, seed=7)
    a, b = run(dc, q, md), run(dc, q, md)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("length", [700, 9000])
def test_masks_with_later_bits_are_flagged_and_cut(length):
    """A mask bit above the token's own is flagged BAD_MASK and ignored: the
    result is the oracle's for the mask without it (split-KV kernels at 700
    keys, the key-major kernel at 9,000)."""
    tokens = 4
    case = small(127, [length], 16, 2, 512, 256)
    dc = DevCase(case)
    qn = W.window_queries(case, tokens, 8)
    masks = masks_of(case, tokens, 8)
    bad = masks.copy()
    bad[0, 1] |= np.uint64(1 << 3)
    ref = oracle.decode_tree_direct(qn, case.k_pool, case.v_pool, case.page_tables,
                                    case.seq_lens, masks, case.scale)
    out = run(dc, to_dev(qn, "bf16"), dev_masks(bad))
    torch.cuda.synchronize()
    assert dc.faults() & pskv.PSKV_FAULT_BAD_MASK
    assert max_err(out, ref) <= TOL


def test_refusals():
    case = small(128, [700], 16, 2, 512, 256)
    dc = DevCase(case)
    q = to_dev(W.window_queries(case, 4, 9), "bf16")
    with pytest.raises(ValueError):  # a mask of the wrong shape
        run(dc, q, dev_masks(np.zeros((1, 3), np.uint64)))
    f32 = W.make_paged_case(129, [300], num_q_heads=8, num_kv_heads=1, head_dim=512,
                            page_size=256, dtype="f32")
    dcf = DevCase(f32)
    qf = to_dev(W.window_queries(f32, 2, 1), "f32")
    with pytest.raises(pskv.PskvError) as e:  # f32 pools run on the CUDA-core consumer
        run(dcf, qf, dev_masks(masks_of(f32, 2, 1)))
    assert e.value.code == pskv.PSKV_ERR_UNSUPPORTED


@pytest.mark.parametrize("tokens,length", [(8, 9092), (16, 9100), (5, 12419)])
def test_key_major_window_across_two_tiles(tokens, length):
    """The drafted window straddles a 128-key tile boundary (its first key at
    row 124 or 126 of a tile): each softmax thread meets its window key in one
    tile or the next, and chains still equal the causal window bit for bit."""
    assert (length - tokens) % 128 > 128 - tokens
    hq, hkv = (16, 2) if tokens == 8 else (8, 2) if tokens == 16 else (32, 4)
    case = small(140 + tokens, [length, 9000], hq, hkv, 512, 256)
    check(case, tokens, splits=(0, 3), seed=tokens)
    dc, q, md = check(case, tokens, splits=(0,), chain=True)
    a = run(dc, q, md, 0)
    b = pskv.decode_attn_multirow(dc.layout, q, dc.tables, dc.lens, case.seq_lens, case.scale,
                                  out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_widest_tree_on_the_key_major_kernel():
    """64 drafted tokens of one query head per KV head: 64 columns per KV head."""
    check(small(145, [8300, 9000], 4, 4, 256, 64), 64, splits=(0, 2), seed=9)
