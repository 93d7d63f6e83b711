"""The append fused into the decode (pskv_decode_opts.append_*) against the
separate kv_append_rows + decode: the same pool bytes after the call and the
same output bits (at a fixed split count), on every partial-kernel family."""
import numpy as np
import pytest
import torch

import paged_split_kv_attn_gb300 as pskv
import workloads as W
from gpu_cases import DevCase, i32, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_split_kv_attn_gb300 import build
    build.build()
    pskv.load_library()


def new_rows(case, seed):
    rng = np.random.default_rng(seed)
    shp_k = (case.batch, case.num_kv_heads, case.k_pool.shape[3])
    shp_v = (case.batch, case.num_kv_heads, case.v_pool.shape[3])
    k = rng.standard_normal(shp_k).astype(np.float32)
    v = rng.standard_normal(shp_v).astype(np.float32)
    if case.dtype == "bf16":
        return to_dev(W.bf16_bits(k), "bf16"), to_dev(W.bf16_bits(v), "bf16")
    return to_dev(k, "f32"), to_dev(v, "f32")


def both(case, splits, pages=None, seed=0):
    """(separate, fused): outputs and pool bytes of the two ways."""
    res = []
    for fused in (False, True):
        dc = DevCase(case)
        k_new, v_new = new_rows(case, seed)
        por = i32(case.pages_of_row if pages is None else pages)
        if not fused:
            pos = [int(n) - 1 for n in case.seq_lens]
            pskv.kv_append_rows(dc.layout, k_new, v_new, i32(range(case.batch)), i32(pos),
                                dc.tables, por)
        out = dc.decode(num_splits=splits, out_dtype=torch.float32,
                        append=(k_new, v_new, por) if fused else None)
        torch.cuda.synchronize()
        res.append((out, dc.k_pool.clone(), dc.v_pool.clone(), dc.faults()))
    return res


@pytest.mark.parametrize("name,case,splits", [
    ("global", lambda: W.make_paged_case(111, [300, 1000, 257], num_q_heads=32, num_kv_heads=4,
                                         head_dim=512, page_size=256), 7),
    ("global-auto", lambda: W.make_paged_case(112, [4000], num_q_heads=32, num_kv_heads=4,
                                              head_dim=512, page_size=256), 0),
    ("folded", lambda: W.make_paged_case(113, [900, 33], num_q_heads=32, num_kv_heads=4,
                                         head_dim=512, page_size=256, k_dims=128), 5),
    ("window", lambda: W.with_window(W.make_paged_case(114, [1088, 70], num_q_heads=32,
                                                       num_kv_heads=16, head_dim=256,
                                                       page_size=64), 1024), 0),
    ("f32", lambda: W.make_paged_case(115, [500, 129], num_q_heads=8, num_kv_heads=2,
                                      head_dim=512, page_size=256, dtype="f32"), 3),
    ("bf16-g16", lambda: W.make_paged_case(116, [700], num_q_heads=32, num_kv_heads=2,
                                           head_dim=256, page_size=64), 4),
])
def test_fused_equals_separate(name, case, splits):
    c = case()
    (o1, k1, v1, f1), (o2, k2, v2, f2) = both(c, splits)
    assert f1 == 0 and f2 == 0
    assert torch.equal(k1.view(torch.uint8), k2.view(torch.uint8)), "K pools differ"
    assert torch.equal(v1.view(torch.uint8), v2.view(torch.uint8)), "V pools differ"
    assert torch.equal(o1, o2), "outputs differ"


def test_past_pages_flagged_and_nothing_written():
    c = W.make_paged_case(117, [256, 40], num_q_heads=8, num_kv_heads=1, head_dim=512,
                          page_size=256)
    dc = DevCase(c)
    before = dc.k_pool.clone()
    k_new, v_new = new_rows(c, 1)
    dc.decode(num_splits=2, append=(k_new, v_new, i32([0, 1])))  # row 0 leases no page
    torch.cuda.synchronize()
    assert dc.faults() & pskv.PSKV_FAULT_PAST_PAGES
    page0 = int(c.page_tables[0, 0])
    assert torch.equal(dc.k_pool[page0].view(torch.uint8), before[page0].view(torch.uint8))


def test_row_written_when_the_window_excludes_every_key():
    """A window bound past the query: the output row is zeros (EMPTY_ROW) and
    the new row is still written, as the separate append would."""
    c = W.make_paged_case(118, [100], num_q_heads=32, num_kv_heads=16, head_dim=256,
                          page_size=64)
    c = W.with_window(c, 1024)
    c.window_lo[:] = 500  # beyond every key
    (o1, k1, v1, f1), (o2, k2, v2, f2) = both(c, 3)
    assert torch.equal(k1.view(torch.uint8), k2.view(torch.uint8))
    assert torch.equal(v1.view(torch.uint8), v2.view(torch.uint8))
    assert f1 & pskv.PSKV_FAULT_EMPTY_ROW and f2 & pskv.PSKV_FAULT_EMPTY_ROW
