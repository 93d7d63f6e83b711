"""The scratch-free decode entry point, through the C ABI.

decode_attn_splitkv_static serves callers that cannot allocate device memory
(no cudaMalloc allowed where they run, or a host framework that owns all
device memory): it uses a scratch array built into the library instead of a
caller workspace.  This file runs last so that, if it fails, a run stopping
at the first failure has already run every other test; it must pass both
alone in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import paged_split_kv_attn_gb300 as pskv
import workloads as W
from gpu_cases import TOL, DevCase

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_split_kv_attn_gb300 import build
    build.build()
    pskv.load_library()


def test_static_scratch_matches_the_workspace_entry_point_twice_in_a_row():
    cases = [W.global_case(9000, seed=41), W.make_paged_case(42, [3000, 17, 700], **W.GLOBAL_SHAPE)]
    for case in cases:  # two calls in a row; the second finds the first's leftovers
        dc = DevCase(case)
        ref = dc.decode(num_splits=0, out_dtype=torch.float32)
        got = pskv.decode_attn_splitkv_static(dc.layout, dc.q, dc.tables, dc.lens, case.seq_lens,
                                              case.scale, num_splits=0, out_dtype=torch.float32)
        torch.cuda.synchronize()
        err = float((got - ref).abs().max())
        assert np.isfinite(err) and err <= TOL, err
        assert dc.faults() == 0


def test_static_scratch_refuses_a_plan_too_big_for_it():
    case = W.make_paged_case(43, [64] * 8, **W.GLOBAL_SHAPE)
    dc = DevCase(case)
    need = pskv.decode_attn_workspace_bytes(8, 32, 512, 1024)
    assert need > pskv.PSKV_STATIC_SCRATCH_BYTES
    with pytest.raises(pskv.PskvError) as e:
        pskv.decode_attn_splitkv_static(dc.layout, dc.q, dc.tables, dc.lens, case.seq_lens,
                                        case.scale, num_splits=1024)
    assert e.value.code == pskv.PSKV_ERR_WORKSPACE_TOO_SMALL
