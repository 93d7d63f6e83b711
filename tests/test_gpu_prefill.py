"""GPU parity of the paged varlen prefill (prefill_attn_paged) against the oracle.

Row b's new tokens are its last T_b keys; token t at key own = L_b - T_b + t
attends keys [max(0, own - W + 1), own] (W = 0: all).  Bars as for decode:
max |out - fp64| <= 2e-3 in the fp32 output mode, the bf16 output the
round-to-nearest-even of the fp32 one."""
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
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 5])))
    q = rng.standard_normal((int(sum(counts)), case.num_q_heads, case.head_dim), dtype=np.float32)
    return W.bf16_bits(q)


def run(dc, q, cu, window=0, splits=0, out_dtype=torch.float32, cu_dev=None):
    c = dc.case
    return pskv.prefill_attn_paged(dc.layout, q, i32(cu) if cu_dev is None else cu_dev, cu,
                                   dc.tables, dc.lens, c.seq_lens, c.scale, window=window,
                                   num_splits=splits, out_dtype=out_dtype)


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
        assert np.all(np.isfinite(out32.cpu().numpy())), "non-finite output"
        err = max_err(out32, ref)
        assert err <= TOL, f"max |err| {err:.3e} > {TOL} (splits={p})"
        assert torch.equal(out16, bf16_of(out32)), "bf16 output is not RNE of the fp32 output"
    assert dc.faults() == 0


def _case(seed, lens, hq, hkv, d, ps, **kw):
    return W.make_paged_case(seed, lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                             page_size=ps, dtype="bf16", **kw)


def test_global_varlen_chunks():
    """32 q / 4 KV heads, head dim 512: chunks of 16, 300 and 1 token, one
    partition (each CTA writes its output) and three (partials + merge)."""
    check(_case(101, [300, 1000, 77], 32, 4, 512, 256), [16, 300, 1], splits=(0, 1, 3))


def test_whole_prompts_and_empty_chunks():
    check(_case(102, [700, 50, 129], 32, 4, 512, 256), [700, 0, 129], splits=(0, 2))


def test_sliding_window_prompt():
    """32 q / 16 KV heads, head dim 256, pages of 64, a window of 256 keys:
    a whole prompt of 600 tokens and a chunk of 100 at 1,500 keys."""
    check(_case(103, [600, 1500], 32, 16, 256, 64), [600, 100], window=256, splits=(0, 4))


def test_folded_pool_prefill():
    check(_case(104, [400, 260], 32, 4, 512, 256, k_dims=128), [64, 260], splits=(0,))


@pytest.mark.parametrize("group", [1, 2, 4])
def test_small_groups(group):
    check(_case(105 + group, [333, 90], 2 * group, 2, 512, 256), [45, 90], splits=(0, 2))


def test_one_token_chunks_match_windowed_decode():
    """A chunk of one token with a window is the windowed decode with
    window_lo = own - W + 1.  Prefill runs on the tensor-memory kernel, the
    windowed decode on the split-KV kernels: the two agree to the fp32 bar
    (different summation orders), each against the oracle."""
    case = _case(109, [1088, 700], 32, 4, 512, 256)
    dc = DevCase(case)
    wnd = 1024
    q = to_dev(case.q, "bf16")
    own = case.seq_lens - 1
    wl_host = np.maximum(0, own - wnd + 1).astype(np.int32)
    fp, wl = i32([0, 0]), i32(wl_host)
    ref = oracle.decode_direct(case.q, case.k_pool, case.v_pool, case.page_tables,
                               case.seq_lens, case.scale, np.zeros(2, np.int32), wl_host)
    for p in (1, 6):
        a = run(dc, q, _cu([1, 1]), window=wnd, splits=p)
        b = pskv.decode_attn_windowed(dc.layout, q, dc.tables, dc.lens, case.seq_lens, fp, wl,
                                      case.scale, num_splits=p, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert max_err(a, ref) <= TOL and max_err(b, ref) <= TOL
        assert float((a - b).abs().max()) <= TOL
    assert dc.faults() == 0


def test_device_offsets_outside_the_rows_are_flagged():
    """Device offsets that point past the packed rows are refused per row on
    the device (PSKV_FAULT_BAD_LENGTH): nothing outside q/out is addressed."""
    case = _case(110, [100, 100], 8, 1, 512, 256)
    dc = DevCase(case)
    q = to_dev(_q(case, [5, 5]), "bf16")
    run(dc, q, _cu([5, 5]), splits=1, cu_dev=i32([0, 5, 1 << 20]))
    torch.cuda.synchronize()
    assert dc.faults() & pskv.PSKV_FAULT_BAD_LENGTH
