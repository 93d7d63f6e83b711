"""GPU parity of the K/V prep with the fused page write (kv_prep_append).

The kernel computes in f32 and rounds to nearest-even bf16; the oracle gives
the exact (fp64) prepared rows.  Bar per element: |got - exact| <= half a bf16
ulp of the exact value (the rounding) + 1e-5 x the row's largest magnitude
(the f32 arithmetic before it).  Bytes the call does not own stay bit-equal."""
import numpy as np
import pytest
import torch

import oracle
import paged_split_kv_attn_gb300 as pskv
import workloads as W
from gpu_cases import TOL, DevCase, i32, max_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_split_kv_attn_gb300 import build
    build.build()
    pskv.load_library()


def half_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 8), 2.0 ** -134)


def assert_rows_close(got_bits: np.ndarray, exact: np.ndarray, what: str):
    got = W.bf16_to_f32(got_bits).astype(np.float64)
    slack = 1e-5 * np.abs(exact).max(axis=-1, keepdims=True)
    bad = np.abs(got - exact) > half_ulp(exact) + slack
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off, worst " \
        f"{float(np.abs(got - exact).max()):.3e}"


def bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def run_prep(dc, p, row_of, pos_of, first_pos=None, host=True):
    c = dc.case
    x = to_dev(p.x, "bf16")
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    return pskv.kv_prep_append(
        dc.layout, x, p.q_col, p.k_col, p.v_col, p.num_q_heads, i32(row_of), i32(pos_of),
        dc.tables, i32(c.pages_of_row), p.rot, p.eps, w_q=f(p.w_q), w_k=f(p.w_k),
        rope_cos=f(p.rope_cos), rope_sin=f(p.rope_sin),
        first_pos=None if first_pos is None else i32(first_pos),
        host=(row_of, pos_of, c.pages_of_row) if host else None)


def expected(p, row_of, pos_of, first_pos=None, folded=False):
    rope_pos = np.asarray(pos_of) + (0 if first_pos is None else np.asarray(first_pos)[row_of])
    return oracle.prep_tokens(p.x, p.q_col, p.k_col, p.v_col, p.num_q_heads, p.num_kv_heads,
                              p.head_dim, p.eps, p.w_q, p.w_k, p.rope_cos, p.rope_sin, rope_pos,
                              folded=folded)


def check_case(case, p, row_of, pos_of, first_pos=None):
    dc = DevCase(case)
    k_before, v_before = bits(dc.k_pool), bits(dc.v_pool)
    q = run_prep(dc, p, row_of, pos_of, first_pos)
    torch.cuda.synchronize()
    assert dc.faults() == 0
    eq, ek, ev = expected(p, row_of, pos_of, first_pos, folded=case.folded)
    assert_rows_close(bits(q), eq, "q_out")
    k_after, v_after = bits(dc.k_pool), bits(dc.v_pool)
    ps, kw = case.page_size, case.k_pool.shape[3]
    owned = np.zeros(k_after.shape[:3], bool)
    for t, (b, pos) in enumerate(zip(row_of, pos_of)):
        page = case.page_tables[b, pos // ps]
        owned[page, :, pos % ps] = True
        assert_rows_close(k_after[page, :, pos % ps], ek[t][:, :kw], f"K row {t}")
        assert_rows_close(v_after[page, :, pos % ps], ev[t], f"V row {t}")
    assert np.array_equal(k_after[~owned], k_before[~owned]), "K bytes outside the new rows changed"
    assert np.array_equal(v_after[~owned], v_before[~owned]), "V bytes outside the new rows changed"
    return dc, q


def test_global_split_rows():
    """32 q heads / 4 KV heads, head dim 512, the first quarter rotated, K and V
    from separate bands; the step's new token at the end of each row."""
    case = W.make_paged_case(81, [300, 1000, 257], num_q_heads=32, num_kv_heads=4, head_dim=512,
                             page_size=256)
    p = W.make_prep_inputs(81, 3, 32, 4, 512, 128, 2048)
    check_case(case, p, [0, 1, 2], [299, 999, 256])


def test_global_folded_rows():
    case = W.make_paged_case(82, [300, 1000], num_q_heads=32, num_kv_heads=4, head_dim=512,
                             page_size=256, k_dims=128)
    p = W.make_prep_inputs(82, 4, 32, 4, 512, 128, 2048, shared_kv=True)
    check_case(case, p, [0, 1, 1, 0], [299, 999, 998, 17])


def test_sliding_rows_with_first_pos():
    """Head dim 256 fully rotated, pages of 64; the rotation position is
    first_pos + key index."""
    case = W.make_paged_case(83, [1088, 70], num_q_heads=32, num_kv_heads=16, head_dim=256,
                             page_size=64)
    p = W.make_prep_inputs(83, 2, 32, 16, 256, 256, 9000)
    check_case(case, p, [0, 1], [1087, 69], first_pos=[5000, 17])


@pytest.mark.parametrize("folded", [False, True])
def test_prepped_rows_decode_to_the_definition(folded):
    """Every key of two rows comes from the prep (into a split or a folded
    pool); decoding each row's last token matches the fp64 definition over the
    oracle's prepared rows rounded to bf16 as stored (for the folded pool: the
    stored K quarter, V's other columns and the folded query).  The two formats
    agree exactly only before rounding, so each is held to its own rows."""
    lens = [37, 300]
    n = sum(lens)
    case = W.make_paged_case(84, lens, num_q_heads=32, num_kv_heads=4, head_dim=512,
                             page_size=256, k_dims=128 if folded else None)
    p = W.make_prep_inputs(84, n, 32, 4, 512, 128, 512, shared_kv=True)
    row_of = [b for b, L in enumerate(lens) for _ in range(L)]
    pos_of = [i for L in lens for i in range(L)]
    dc = DevCase(case)
    q = run_prep(dc, p, row_of, pos_of)
    last = [sum(lens[:b + 1]) - 1 for b in range(len(lens))]
    out = pskv.decode_attn_splitkv(dc.layout, q[last].contiguous(), dc.tables, dc.lens,
                                   case.seq_lens, case.scale, num_splits=3,
                                   out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert dc.faults() == 0
    eq, ek, ev = expected(p, row_of, pos_of, folded=folded)
    stored = lambda a: W.bf16_to_f32(W.bf16_bits(a.astype(np.float32))).astype(np.float64)
    eq, ek, ev = stored(eq), stored(ek), stored(ev)
    if folded:  # the key a folded query meets: stored quarter, then V's columns
        ek = np.concatenate([ek[..., :128], ev[..., 128:]], axis=-1)
    ref = np.zeros((2, 32, 512))
    for b in range(2):
        rows = [t for t in range(n) if row_of[t] == b]
        for h in range(32):
            s = case.scale * (ek[rows, h // 8] @ eq[last[b], h])
            w = np.exp(s - s.max())
            ref[b, h] = (w / w.sum()) @ ev[rows, h // 8]
    err = max_err(out, ref)
    assert err <= TOL, f"{err:.3e}"


def test_bad_position_is_flagged_and_skipped():
    case = W.make_paged_case(85, [100], num_q_heads=8, num_kv_heads=1, head_dim=512,
                             page_size=256)
    p = W.make_prep_inputs(85, 1, 8, 1, 512, 128, 64)  # table of 64 positions, key 99
    dc = DevCase(case)
    k_before = bits(dc.k_pool)
    run_prep(dc, p, [0], [99])
    torch.cuda.synchronize()
    assert dc.faults() & pskv.PSKV_FAULT_BAD_POSITION
    assert np.array_equal(bits(dc.k_pool), k_before)


def test_past_pages_refused_on_the_host():
    case = W.make_paged_case(86, [100], num_q_heads=8, num_kv_heads=1, head_dim=512,
                             page_size=256)
    p = W.make_prep_inputs(86, 1, 8, 1, 512, 128, 1024)
    dc = DevCase(case)
    with pytest.raises(pskv.PskvError) as e:
        run_prep(dc, p, [0], [256])  # the row leases one page
    assert e.value.code == pskv.PSKV_ERR_PAST_PAGES
