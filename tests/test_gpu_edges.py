"""GPU edge cases: the largest split count, merge group sizes, wide ragged
batches, one-key rows (closed form), and device lengths past the table."""
import numpy as np
import pytest
import torch

import oracle
import paged_split_kv_attn_gb300 as pskv
import workloads as W
from gpu_cases import TOL, DevCase, i32, max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_split_kv_attn_gb300 import build
    build.build()
    pskv.load_library()


def ref_direct(c):
    return oracle.decode_direct(c.q, c.k_pool, c.v_pool, c.page_tables, c.seq_lens, c.scale,
                                c.first_pos, c.window_lo)


def test_the_largest_split_count():
    """PSKV_MAX_SPLITS partitions over 40,002 keys (2,501 tiles): most hold two
    or three tiles, the merge folds 64 groups of 16."""
    c = W.global_case(40002, seed=121)
    dc = DevCase(c)
    out = dc.decode(num_splits=pskv.PSKV_MAX_SPLITS)
    torch.cuda.synchronize()
    assert max_err(out, ref_direct(c)) <= TOL
    assert dc.faults() == 0


@pytest.mark.parametrize("group,splits", [(1, 48), (5, 48), (16, 48), (3, 7)])
def test_merge_group_sizes(group, splits):
    c = W.global_case(10602, seed=122)
    dc = DevCase(c)
    out = dc.decode(num_splits=splits, merge_group=group)
    torch.cuda.synchronize()
    assert max_err(out, ref_direct(c)) <= TOL
    assert dc.faults() == 0


def test_wide_ragged_batch():
    """64 rows of 1 to 3,000 keys in one call (grid z = 64), automatic plan."""
    rng = np.random.default_rng(123)
    lens = [1, 2, 15, 16, 17] + [int(x) for x in rng.integers(1, 3000, 59)]
    c = W.make_paged_case(123, lens, num_q_heads=32, num_kv_heads=4, head_dim=512,
                          page_size=256)
    dc = DevCase(c)
    out = dc.decode()
    torch.cuda.synchronize()
    assert max_err(out, ref_direct(c)) <= TOL
    assert dc.faults() == 0


@pytest.mark.parametrize("splits", [1, 4])
def test_one_key_rows_return_their_value_exactly(splits):
    """With one key the softmax weight is exactly 1: the output is the value
    row itself, bit for bit, in both output types."""
    c = W.make_paged_case(124, [1, 1, 700], num_q_heads=32, num_kv_heads=4, head_dim=512,
                          page_size=256)
    dc = DevCase(c)
    out32 = dc.decode(num_splits=splits, out_dtype=torch.float32)
    out16 = dc.decode(num_splits=splits, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    for b in (0, 1):
        page = int(c.page_tables[b, 0])
        v = torch.from_numpy(W.bf16_to_f32(c.v_pool[page, :, 0, :]))  # [Hkv, D]
        exp = v.repeat_interleave(8, dim=0)  # query head h reads KV head h // 8
        assert torch.equal(out32[b].cpu(), exp)
        assert torch.equal(out16[b].cpu().float(), exp)


def test_device_length_past_the_table_is_flagged():
    """A device length beyond table_stride * page_size is clamped to the table
    (entries there point at an in-bounds page) and flagged PSKV_FAULT_BAD_LENGTH."""
    c = W.make_paged_case(125, [300], num_q_heads=8, num_kv_heads=1, head_dim=512,
                          page_size=256)
    dc = DevCase(c)
    pskv.decode_attn_splitkv(dc.layout, dc.q, dc.tables, i32([1 << 30]), c.seq_lens, c.scale,
                             num_splits=3)
    torch.cuda.synchronize()
    assert dc.faults() & pskv.PSKV_FAULT_BAD_LENGTH
    # the library's reader sees the same word, and clears it on request
    assert pskv.pskv_check_flags(dc.layout, clear=True) & pskv.PSKV_FAULT_BAD_LENGTH
    assert pskv.pskv_check_flags(dc.layout) == 0


def test_device_lengths_rule_over_the_host_copy():
    """The kernels read the device lengths; the host copy only plans.  A
    device length that differs
    from the host copy -- as in a captured graph replayed after the device
    lengths moved -- still decodes exactly its own keys."""
    import dataclasses
    c = W.global_case(12000, seed=126)
    dc = DevCase(c)
    for dev_len in (9000, 11999, 12000):
        out = pskv.decode_attn_splitkv(dc.layout, dc.q, dc.tables, i32([dev_len]), c.seq_lens,
                                       c.scale, num_splits=0, out_dtype=torch.float32)
        torch.cuda.synchronize()
        ref = ref_direct(dataclasses.replace(c, seq_lens=np.array([dev_len], np.int32)))
        assert max_err(out, ref) <= TOL, dev_len
    assert dc.faults() == 0


@pytest.mark.parametrize("host_len,dev_len,splits", [
    (9000, 8500, 0),    # the plan from the host length, the keys from the device one
    (9000, 8990, 16),   # the same table slots in use, shifted partition bounds
    (9000, 9000, 64),   # agreeing copies (the page ids fetched from the host length kept)
    (700, 9000, 0),     # a device length past the host's: planned for 700 keys
])
def test_device_lengths_rule_over_the_host_copy(host_len, dev_len, splits):
    """The kernels take a row's keys from the device lengths; the host copy only
    plans the call (split count, and the page ids fetched before the device
    length arrives, kept only when the device length puts the partition on the
    same table slots).  A graph replayed after the lengths advanced relies on it."""
    import dataclasses
    c = W.make_paged_case(131, [9000, 2000], **W.GLOBAL_SHAPE)
    dc = DevCase(c)
    lens_dev = i32([dev_len, 2000])
    lens_host = np.array([host_len, 2000], np.int32)
    out = pskv.decode_attn_splitkv(dc.layout, dc.q, dc.tables, lens_dev, lens_host, c.scale,
                                   num_splits=splits, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = ref_direct(dataclasses.replace(c, seq_lens=np.array([dev_len, 2000], np.int32)))
    assert max_err(out, ref) <= TOL
    assert dc.faults() == 0


def test_workspace_queries_give_the_automatic_plans_bytes():
    """The size queries plan exactly as the calls: a long prefill chunk and a
    verify window on the key-major kernel (one CTA per SM per KV head: 38
    partitions on 152 SMs), answered on the device's own SM count."""
    c = W.global_case(40002, seed=132)
    dc = DevCase(c)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    cu = np.array([0, 512], np.int32)
    assert pskv.prefill_attn_workspace_bytes(dc.layout, cu, c.seq_lens, c.page_tables.shape[1],
                                             32) == 0  # the blocks fill the SM pairs: one partition
    want = pskv.decode_attn_workspace_bytes(4, 32, 512, n_sm // 4)
    assert pskv.decode_attn_multirow_workspace_bytes(dc.layout, c.seq_lens,
                                                     c.page_tables.shape[1], 4, 32) == want
    # and the call runs in exactly that workspace
    q = torch.randn(1, 4, 32, 512, device="cuda").to(torch.bfloat16)
    ws = torch.empty(want, dtype=torch.uint8, device="cuda")
    pskv.decode_attn_multirow(dc.layout, q, dc.tables, dc.lens, c.seq_lens, c.scale, workspace=ws)
    with pytest.raises(pskv.PskvError) as e:
        pskv.decode_attn_multirow(dc.layout, q, dc.tables, dc.lens, c.seq_lens, c.scale,
                                  workspace=ws[:want - 256])
    assert e.value.code == pskv.PSKV_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert dc.faults() == 0
