"""GPU parity of paged prefill on the tensor-memory (tcgen05) kernel against
the oracle: head dim 256 on one CTA, head dim 512 on a CTA pair.

The kernel serves blocks of 128 query columns (tokens x the KV group's
heads), 64-key tiles brought in by tensor copies in 16- or 64-row boxes
(pages of 16 or 32 keys, pages of 64 or more), one CTA (pair) per block and
partition.  Cases cover several blocks with a ragged last one, every group
size, windows that cut tiles anywhere, empty partitions, pages outside the
pool and the NaN-filled rows the generator leaves past each row's keys.
Bars as for decode: max |out - fp64| <= 2e-3 in the fp32 output mode, the
bf16 output the round-to-nearest-even of the fp32 one."""
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


def _cu(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def _q(case, counts, seed=0):
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 11])))
    q = rng.standard_normal((int(sum(counts)), case.num_q_heads, case.head_dim), dtype=np.float32)
    return W.bf16_bits(q)


def _case(seed, lens, hq, hkv, ps, **kw):
    return W.make_paged_case(seed, lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=256,
                             page_size=ps, dtype="bf16", **kw)


def run(dc, q, cu, window=0, splits=0, out_dtype=torch.float32, tables=None):
    c = dc.case
    return pskv.prefill_attn_paged(dc.layout, q, i32(cu), cu,
                                   dc.tables if tables is None else tables, dc.lens, c.seq_lens,
                                   c.scale, window=window, num_splits=splits, out_dtype=out_dtype)


def check(case, counts, window=0, splits=(0,), seed=0):
    dc = DevCase(case)
    qn = _q(case, counts, seed)
    cu = _cu(counts)
    ref = oracle.prefill_direct(qn, cu, case.k_pool, case.v_pool, case.page_tables,
                                case.seq_lens, case.scale, window)
    q = to_dev(qn, "bf16")
    for p in splits:
        out32 = run(dc, q, cu, window, p)
        out16 = run(dc, q, cu, window, p, torch.bfloat16)
        torch.cuda.synchronize()
        assert np.all(np.isfinite(out32.cpu().numpy())), f"non-finite output (splits={p})"
        err = max_err(out32, ref)
        assert err <= TOL, f"max |err| {err:.3e} > {TOL} (splits={p})"
        assert torch.equal(out16, bf16_of(out32)), "bf16 output is not RNE of the fp32 output"
    assert dc.faults() == 0


def test_causal_prompt_several_blocks():
    """32 q / 16 KV heads (G = 2), pages of 64: a whole prompt of 300 tokens
    (600 columns: four full blocks and one of 88) and a chunk of 40 at 517
    keys; one partition, three, and the automatic plan."""
    check(_case(201, [300, 517], 32, 16, 64), [300, 40], splits=(0, 1, 3))


def test_window_cuts_tiles():
    """A window of 100 keys (not a multiple of the 64-key tile) on the same
    shapes: every block starts and ends mid-tile."""
    check(_case(202, [300, 517], 32, 16, 64), [300, 40], window=100, splits=(0, 1, 2))


def test_group_of_eight_large_pages():
    """8 q / 1 KV head (G = 8), pages of 256: a chunk of 100 tokens at 700
    keys (800 columns: six full blocks and one of 32)."""
    check(_case(203, [700], 8, 1, 256), [100], splits=(0, 1, 2))


def test_group_of_one_small_pages():
    """4 q / 4 KV heads (G = 1), pages of 16 (16-row copies): a chunk of 130
    tokens at 250 keys (two blocks, the second of 2 columns)."""
    check(_case(204, [250, 31], 4, 4, 16), [130, 31], splits=(0, 1, 4))


def test_group_of_four_pages_of_32_with_empty_and_single_chunks():
    """8 q / 2 KV heads (G = 4), pages of 32: chunks of 1, 0 and 77 tokens."""
    check(_case(205, [5, 64, 200], 8, 2, 32), [1, 0, 77], window=50, splits=(0, 1, 3))


def test_more_partitions_than_tiles():
    """Sixteen partitions over rows of at most five tiles: most CTAs see no
    key and write empty states the merge must skip."""
    check(_case(206, [300, 90], 32, 16, 64), [20, 90], splits=(16,))


def test_long_context_chunk_with_window_and_short_rows():
    """A chunk of 256 tokens at 4,000 keys with a window of 1,024 beside two
    short whole prompts (the sliding family's prefill)."""
    check(_case(207, [4000, 130, 65], 32, 16, 64), [256, 130, 65], window=1024, splits=(0, 1))


def test_one_token_chunk_matches_windowed_decode():
    """A one-token chunk with a window is the windowed decode with
    window_lo = own - W + 1 (the prefill of head dim 256 runs on its own
    kernel, so the two agree to the fp32 bar, not bit for bit)."""
    case = _case(208, [1088, 700], 32, 16, 64)
    dc = DevCase(case)
    wnd = 1024
    q = to_dev(case.q, "bf16")
    own = case.seq_lens - 1
    fp, wl = i32([0, 0]), i32(np.maximum(0, own - wnd + 1))
    ref = oracle.decode_direct(case.q, case.k_pool, case.v_pool, case.page_tables,
                               case.seq_lens, case.scale, np.zeros(2, np.int32),
                               np.maximum(0, own - wnd + 1).astype(np.int32))
    for p in (1, 6):
        a = run(dc, q, _cu([1, 1]), window=wnd, splits=p)
        b = pskv.decode_attn_windowed(dc.layout, q, dc.tables, dc.lens, case.seq_lens, fp, wl,
                                      case.scale, num_splits=p, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert max_err(a, ref) <= TOL and max_err(b, ref) <= TOL
        assert float((a - b).abs().max()) <= TOL
    assert dc.faults() == 0


def test_page_outside_the_pool_is_skipped_and_flagged():
    """A table entry past the pool: its keys are skipped (no copy is issued),
    PSKV_FAULT_BAD_PAGE is raised, and the outputs stay finite."""
    case = _case(209, [400], 32, 16, 64)
    dc = DevCase(case)
    tables = case.page_tables.copy()
    tables[0, 2] = case.page_tables.max() + 1000
    q = to_dev(_q(case, [200]), "bf16")
    for p in (1, 3):
        out = run(dc, q, _cu([200]), splits=p, tables=i32(tables))
        torch.cuda.synchronize()
        assert np.all(np.isfinite(out.cpu().numpy()))
    assert dc.faults() & pskv.PSKV_FAULT_BAD_PAGE


def test_bench_sliding_prompt_sampled_tokens():
    """The bench's sliding prompt at full size (4,096 tokens, 32 q / 16 KV
    heads, pages of 64, a window of 1,024 keys) in the automatic plan, checked
    on sampled tokens: each equals the oracle's windowed decode of its row cut
    at its own key."""
    n = 4096
    case = _case(210, [n], 32, 16, 64, keep_dense=False)
    dc = DevCase(case)
    qn = _q(case, [n], seed=3)
    q = to_dev(qn, "bf16")
    out = run(dc, q, _cu([n]), window=1024, splits=0)
    torch.cuda.synchronize()
    assert dc.faults() == 0
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    for t in (0, 1, 63, 64, 127, 1000, 1023, 1024, 2047, 3000, 4094, 4095):
        lens = np.array([t + 1], np.int32)
        ref = oracle.decode_direct(qn[t:t + 1], case.k_pool, case.v_pool, case.page_tables, lens,
                                   case.scale, np.zeros(1, np.int32),
                                   np.array([max(0, t - 1023)], np.int32))
        err = float(np.abs(got[t:t + 1].astype(np.float64) - ref).max())
        assert err <= TOL, f"token {t}: max |err| {err:.3e}"


def test_bench_global_prompt_sampled_tokens():
    """The bench's global prompt at full size (4,096 tokens, 32 q / 4 KV heads,
    head dim 512 on a CTA pair, pages of 256, causal) in the automatic plan,
    checked on sampled tokens against the oracle's decode of the row cut at
    each token's own key."""
    n = 4096
    case = W.make_paged_case(211, [n], num_q_heads=32, num_kv_heads=4, head_dim=512,
                             page_size=256, dtype="bf16", keep_dense=False)
    dc = DevCase(case)
    qn = _q(case, [n], seed=4)
    q = to_dev(qn, "bf16")
    out = run(dc, q, _cu([n]), splits=0)
    torch.cuda.synchronize()
    assert dc.faults() == 0
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    for t in (0, 1, 15, 16, 63, 64, 255, 1000, 2047, 4094, 4095):
        ref = oracle.decode_direct(qn[t:t + 1], case.k_pool, case.v_pool, case.page_tables,
                                   np.array([t + 1], np.int32), case.scale)
        err = float(np.abs(got[t:t + 1].astype(np.float64) - ref).max())
        assert err <= TOL, f"token {t}: max |err| {err:.3e}"


def test_pair_group_of_one_small_pages_and_splits():
    """Head dim 512 with one query head per KV head (G = 1) and pages of 16
    (16-row copies): a chunk of 150 tokens at 400 keys, one and four
    partitions (partials merged)."""
    case = W.make_paged_case(212, [400, 37], num_q_heads=2, num_kv_heads=2, head_dim=512,
                             page_size=16, dtype="bf16")
    check(case, [150, 37], window=90, splits=(0, 1, 4))


@pytest.mark.parametrize("hd,hq,hkv,ps", [(256, 4, 2, 64), (512, 8, 1, 256)])
def test_bad_device_offsets_and_lengths_are_flagged(hd, hq, hkv, ps):
    """Device offsets past the packed rows, and a device length shorter than
    the row's chunk, are refused per row on the device (PSKV_FAULT_BAD_LENGTH),
    with nothing outside q / out addressed and the other row still right."""
    case = W.make_paged_case(213, [300, 300], num_q_heads=hq, num_kv_heads=hkv, head_dim=hd,
                             page_size=ps, dtype="bf16")
    dc = DevCase(case)
    counts = [40, 40]
    qn = _q(case, counts)
    q = to_dev(qn, "bf16")
    cu = _cu(counts)
    ref = oracle.prefill_direct(qn, cu, case.k_pool, case.v_pool, case.page_tables,
                                case.seq_lens, case.scale, 0)
    # row 1's offsets point past the 80 packed rows
    out = pskv.prefill_attn_paged(dc.layout, q, i32([0, 40, 1 << 20]), cu, dc.tables, dc.lens,
                                  case.seq_lens, case.scale, num_splits=1,
                                  out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert dc.faults() & pskv.PSKV_FAULT_BAD_LENGTH
    assert max_err(out[:40], ref[:40]) <= TOL
    # row 0's device length shorter than its chunk: that row reads no key
    dc.status.zero_()
    bad_lens = i32([10, 300])
    out = pskv.prefill_attn_paged(dc.layout, q, i32(cu), cu, dc.tables, bad_lens,
                                  case.seq_lens, case.scale, num_splits=1,
                                  out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert dc.faults() & pskv.PSKV_FAULT_BAD_LENGTH
    assert max_err(out[40:], ref[40:]) <= TOL
    assert np.all(np.isfinite(out.cpu().numpy()))


@pytest.mark.parametrize("hd,hq,hkv,lens,counts,window", [
    (256, 32, 2, [300, 37], [100, 37], 0),    # G = 16: 8 tokens per block
    (256, 32, 1, [130], [40], 50),            # G = 32: 4 tokens per block
    (512, 32, 2, [200, 70], [50, 9], 0),      # G = 16 on the CTA pair
])
def test_large_groups(hd, hq, hkv, lens, counts, window):
    """Groups the decode kernels do not serve (16 or 32 query heads per KV
    head) prefill on the tensor-memory kernel: 128 / G tokens per block."""
    case = W.make_paged_case(214 + hq // hkv, lens, num_q_heads=hq, num_kv_heads=hkv,
                             head_dim=hd, page_size=64, dtype="bf16")
    check(case, counts, window=window, splits=(0, 1, 3))


def test_random_shapes_against_the_oracle():
    """Forty seeded random prefills (head dim 256 / 512, 1-16 query heads per
    KV head, pages of 16-256, 1-3 rows with chunks of any length including
    empty ones, windows, one to five partitions) against the oracle."""
    rng = np.random.default_rng(2024)
    for it in range(40):
        hd = int(rng.choice([256, 512]))
        g = int(rng.choice([1, 2, 4, 8, 16]))
        hkv = int(rng.choice([1, 2]))
        ps = int(rng.choice([16, 32, 64, 128, 256]))
        lens = [int(rng.integers(1, 700)) for _ in range(int(rng.integers(1, 4)))]
        counts = [int(rng.integers(0, n + 1)) for n in lens]
        if sum(counts) == 0:
            counts[0] = lens[0]
        window = int(rng.choice([0, 0, int(rng.integers(1, 300))]))
        splits = int(rng.choice([0, 1, 2, 5]))
        case = W.make_paged_case(int(rng.integers(1 << 30)), lens, num_q_heads=g * hkv,
                                 num_kv_heads=hkv, head_dim=hd, page_size=ps, dtype="bf16")
        dc = DevCase(case)
        qn = _q(case, counts, seed=it)
        cu = _cu(counts)
        ref = oracle.prefill_direct(qn, cu, case.k_pool, case.v_pool, case.page_tables,
                                    case.seq_lens, case.scale, window)
        out = run(dc, to_dev(qn, "bf16"), cu, window, splits)
        torch.cuda.synchronize()
        err = max_err(out, ref)
        assert err <= TOL and dc.faults() == 0, (it, hd, g, hkv, ps, lens, counts, window,
                                                  splits, err)
