"""The scratch-free decode entry point, through the C ABI.

decode_attn_splitkv_static serves callers that cannot allocate device memory
(no cudaMalloc allowed where they run, or a host framework that owns all
device memory): it uses a scratch array built into the library instead of a
caller workspace.  At the same split count it must give the workspace entry
point's output bit for bit (same kernels, same partition, same merge order),
and both must stay within the fp64 tolerance of the oracle.

This file runs last so that, if it fails, a run stopping at the first failure
has already run every other test; it must pass both alone in a fresh process
and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_split_kv_attn_gb300 as pskv
import workloads as W
from gpu_cases import TOL, DevCase

pytestmark = pytest.mark.gpu

SCRATCH = pskv.PSKV_STATIC_SCRATCH_BYTES


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_split_kv_attn_gb300 import build
    build.build()
    pskv.load_library()


def _static(dc, num_splits, out_dtype=torch.float32):
    c = dc.case
    return pskv.decode_attn_splitkv_static(dc.layout, dc.q, dc.tables, dc.lens, c.seq_lens,
                                           c.scale, num_splits=num_splits, out_dtype=out_dtype)


def _reference(case):
    return oracle.decode_direct(case.q, case.k_pool, case.v_pool, case.page_tables,
                                case.seq_lens, case.scale)


def _check_against(dc, ref64, got, expect):
    """got equals the workspace entry point's output bit for bit and is within
    the tolerance of the fp64 oracle; no fault bit is set."""
    torch.cuda.synchronize()
    assert torch.equal(got, expect)
    err = float(np.abs(got.double().cpu().numpy() - ref64).max())
    assert np.isfinite(err) and err <= TOL, err
    assert dc.faults() == 0


def _workspace_split_count(batch, num_q_heads, head_dim_v, num_splits):
    return pskv.decode_attn_workspace_bytes(batch, num_q_heads, head_dim_v, num_splits)


def test_static_scratch_equals_the_workspace_entry_point_twice_in_a_row():
    cases = [W.global_case(9000, seed=41), W.make_paged_case(42, [3000, 17, 700], **W.GLOBAL_SHAPE)]
    for case in cases:
        dc = DevCase(case)
        ref64 = _reference(case)
        plan = pskv.pskv_plan_splits(dc.layout, case.num_q_heads, case.seq_lens)
        assert _workspace_split_count(case.batch, 32, 512, plan) <= SCRATCH
        for _ in range(2):  # the second call finds the first call's leftovers in the array
            expect = dc.decode(num_splits=plan, out_dtype=torch.float32)
            got = _static(dc, 0)
            _check_against(dc, ref64, got, expect)
            # and at an explicit split count other than the plan's
            expect = dc.decode(num_splits=7, out_dtype=torch.float32)
            got = _static(dc, 7)
            _check_against(dc, ref64, got, expect)
        # the bf16 output is the round-to-nearest-even of the f32 one
        got16 = _static(dc, 0, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert torch.equal(got16, _static(dc, 0).to(torch.bfloat16))


def test_static_scratch_at_the_largest_explicit_split_count_that_fits():
    # one row of 32 query heads at head dim 512: 255 partitions need exactly the
    # array's 16 MiB (two 256-byte aligned 32,640-byte state sections plus
    # 16,711,680 bytes of numerators); 256 need one numerator block more
    assert _workspace_split_count(1, 32, 512, 255) == SCRATCH
    assert _workspace_split_count(1, 32, 512, 256) > SCRATCH
    case = W.global_case(9000, seed=44)
    dc = DevCase(case)
    ref64 = _reference(case)
    for _ in range(2):
        expect = dc.decode(num_splits=255, out_dtype=torch.float32)
        got = _static(dc, 255)
        _check_against(dc, ref64, got, expect)
    with pytest.raises(pskv.PskvError) as e:
        _static(dc, 256)
    assert e.value.code == pskv.PSKV_ERR_WORKSPACE_TOO_SMALL


def test_static_scratch_lowers_an_automatic_plan_too_big_for_it():
    # eight rows, one long: the automatic plan asks for more partials than the
    # array holds (8 rows x 32 heads x P x 2 KiB of numerators), so the static
    # entry point lowers it to the largest split count that fits (31 here)
    case = W.make_paged_case(45, [20000] + [100] * 7, **W.GLOBAL_SHAPE)
    dc = DevCase(case)
    plan = pskv.pskv_plan_splits(dc.layout, 32, case.seq_lens)
    assert _workspace_split_count(8, 32, 512, plan) > SCRATCH
    assert _workspace_split_count(8, 32, 512, 31) <= SCRATCH < _workspace_split_count(8, 32, 512, 32)
    ref64 = _reference(case)
    for _ in range(2):
        expect = dc.decode(num_splits=31, out_dtype=torch.float32)
        got = _static(dc, 0)
        _check_against(dc, ref64, got, expect)


def test_static_scratch_plan_with_sixteen_query_heads_per_kv_head():
    # 32 query heads on 2 KV heads at head dim 256 (the CUDA-core consumer):
    # the static entry point's automatic plan (pskv_plan_splits) is the one
    # decode_attn_splitkv picks with num_splits = 0, so all three agree bit for bit
    case = W.make_paged_case(46, [5000], num_q_heads=32, num_kv_heads=2, head_dim=256,
                             page_size=64)
    dc = DevCase(case)
    ref64 = _reference(case)
    plan = pskv.pskv_plan_splits(dc.layout, 32, case.seq_lens)
    assert plan > 1
    for _ in range(2):
        expect = dc.decode(num_splits=plan, out_dtype=torch.float32)
        auto = dc.decode(num_splits=0, out_dtype=torch.float32)
        got = _static(dc, 0)
        _check_against(dc, ref64, got, expect)
        assert torch.equal(auto, expect)


def test_static_scratch_refuses_a_plan_too_big_for_it():
    case = W.make_paged_case(43, [64] * 8, **W.GLOBAL_SHAPE)
    dc = DevCase(case)
    need = pskv.decode_attn_workspace_bytes(8, 32, 512, 1024)
    assert need > SCRATCH
    with pytest.raises(pskv.PskvError) as e:
        _static(dc, 1024)
    assert e.value.code == pskv.PSKV_ERR_WORKSPACE_TOO_SMALL
