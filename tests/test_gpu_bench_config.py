"""The benchmark's own step, at full size and in the launch configuration it
times (automatic plans, the new K/V row written by the decode itself, bf16
output), against the oracle: the global-layer calls at 10,602, 40,002, 81,653
and 163,336 keys and the sliding-window call at residency 1,088."""
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


# half a bf16 ulp of outputs in [-4, 4) on top of the fp32-mode bar
BF16_TOL = TOL + 2.0 ** -7


@pytest.mark.parametrize("name,make", [
    ("global_10602", lambda: W.global_case(10602, seed=10602)),
    ("global_40002", lambda: W.global_case(40002, seed=40002)),
    ("global_81653", lambda: W.global_case(81653, seed=81653)),
    ("global_163336", lambda: W.global_case(163336, seed=163336)),
    ("window_1088", lambda: W.window_case(1088, seed=7)),
])
def test_bench_step_call(name, make):
    c = make()
    dc = DevCase(c)
    # the step's new row of each table row: its last key, taken from the pool
    pos = int(c.seq_lens[0]) - 1
    page = int(c.page_tables[0, pos // c.page_size])
    k_new = dc.k_pool[page, :, pos % c.page_size].unsqueeze(0).contiguous()
    v_new = dc.v_pool[page, :, pos % c.page_size].unsqueeze(0).contiguous()
    pages = i32(c.pages_of_row)
    out = dc.decode(num_splits=0, out_dtype=torch.bfloat16, append=(k_new, v_new, pages))
    torch.cuda.synchronize()
    assert dc.faults() == 0
    ref = oracle.decode_direct(c.q, c.k_pool, c.v_pool, c.page_tables, c.seq_lens, c.scale,
                               c.first_pos, c.window_lo)
    assert np.all(np.isfinite(out.float().cpu().numpy()))
    assert max_err(out, ref) <= BF16_TOL
