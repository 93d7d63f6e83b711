"""GPU parity: the CUDA library (called through its C ABI) against the CPU oracle.

Bars: appends and gathers bit-exact; decode within max|out - fp64| <= 2e-3 in
the fp32 output mode, the bf16 output equal to the round-to-nearest-even of
the fp32 one; run-to-run bit-identical at a fixed split count."""
import math

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


def ref_direct(case):
    return oracle.decode_direct(case.q, case.k_pool, case.v_pool, case.page_tables, case.seq_lens,
                                case.scale, case.first_pos, case.window_lo)


def check_decode(dc, ref, num_splits=0, tol=TOL, **kw):
    out32 = dc.decode(num_splits=num_splits, out_dtype=torch.float32, **kw)
    out16 = dc.decode(num_splits=num_splits, out_dtype=torch.bfloat16, **kw)
    torch.cuda.synchronize()
    err = max_err(out32, ref)
    assert np.all(np.isfinite(out32.cpu().numpy())), "non-finite output"
    assert err <= tol, f"max |err| {err:.3e} > {tol} (splits={num_splits})"
    assert torch.equal(out16, bf16_of(out32)), "bf16 output is not RNE of the fp32 output"
    assert dc.faults() == 0
    return err


# ---- append ----------------------------------------------------------------------

@pytest.mark.parametrize("dtype,d,ps", [("bf16", 512, 256), ("f32", 512, 256), ("bf16", 256, 64)])
def test_append_rebuilds_the_pool_bit_exactly(dtype, d, ps):
    case = W.make_paged_case(21, [1, 300, 1000], num_q_heads=8, num_kv_heads=2, head_dim=d,
                             page_size=ps, dtype=dtype, keep_dense=True)
    # expected pool: the oracle's append into an empty pool
    exp_k, exp_v = np.zeros_like(case.k_pool), np.zeros_like(case.v_pool)
    rows = [(b, i) for b in range(case.batch) for i in range(int(case.seq_lens[b]))]
    rng = np.random.default_rng(1)
    rng.shuffle(rows)
    kn = np.stack([case.dense_k[b][i] for b, i in rows])
    vn = np.stack([case.dense_v[b][i] for b, i in rows])
    row_of, pos_of = [r[0] for r in rows], [r[1] for r in rows]
    oracle.append_rows(exp_k, exp_v, kn, vn, row_of, pos_of, case.page_tables, case.pages_of_row)

    k_pool = torch.zeros_like(to_dev(case.k_pool, dtype))
    v_pool = torch.zeros_like(k_pool)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    layout = pskv.paged_kv_layout_create(k_pool, v_pool, status)
    pskv.kv_append_rows(layout, to_dev(kn, dtype), to_dev(vn, dtype), i32(row_of), i32(pos_of),
                        i32(case.page_tables), i32(case.pages_of_row),
                        host=(row_of, pos_of, case.pages_of_row))
    torch.cuda.synchronize()
    view = np.int16 if dtype == "bf16" else np.float32
    got_k = k_pool.cpu().view(torch.int16 if dtype == "bf16" else torch.float32).numpy()
    got_v = v_pool.cpu().view(torch.int16 if dtype == "bf16" else torch.float32).numpy()
    assert got_k.tobytes() == exp_k.view(view).tobytes()
    assert got_v.tobytes() == exp_v.view(view).tobytes()
    assert int(status[0].item()) == 0


def test_append_past_pages_is_refused():
    case = W.make_paged_case(22, [20, 40], num_q_heads=8, num_kv_heads=1, head_dim=512,
                             page_size=256)
    dc = DevCase(case)
    before_k, before_v = dc.k_pool.clone(), dc.v_pool.clone()
    kn = torch.full((2, 1, 512), 1000.0, dtype=torch.bfloat16, device="cuda")  # never drawn
    row_of, pos_of = [0, 1], [5, 256]   # row 1 holds one page: position 256 is past it
    with pytest.raises(pskv.PskvError) as e:   # host copies given: refused before launch
        pskv.kv_append_rows(dc.layout, kn, kn, i32(row_of), i32(pos_of), dc.tables,
                            i32(case.pages_of_row), host=(row_of, pos_of, case.pages_of_row))
    assert e.value.code == pskv.PSKV_ERR_PAST_PAGES
    # device-only arrays: the kernel skips the bad row and flags it, the good row lands
    pskv.kv_append_rows(dc.layout, kn, kn, i32(row_of), i32(pos_of), dc.tables,
                        i32(case.pages_of_row))
    assert dc.faults() & pskv.PSKV_FAULT_PAST_PAGES
    page0 = int(case.page_tables[0, 0])
    bits = lambda t: t.view(torch.int16)  # compare bit patterns: the pools hold NaN padding
    changed = (bits(dc.k_pool) != bits(before_k)).nonzero()
    assert changed.shape[0] == 512 and torch.all(changed[:, 0] == page0)
    assert torch.all(changed[:, 2] == 5)
    assert torch.equal(bits(dc.v_pool) != bits(before_v), bits(dc.k_pool) != bits(before_k))


# ---- the tiny decode (f32, CUDA-core kernel) ---------------------------------------

@pytest.mark.parametrize("splits", [1, 2, 3, 4, 7, 16])
def test_tiny_f32_decode(splits):
    case = W.tiny_case(0)
    dc = DevCase(case)
    ref = ref_direct(case)
    err = check_decode(dc, ref, num_splits=splits)
    assert err < 1e-5  # f32 all the way: far inside the gate


def test_empty_partitions_on_the_gpu():
    """More partitions than key tiles: trailing partitions are empty."""
    case = W.make_paged_case(23, [40, 7], num_q_heads=32, num_kv_heads=4, head_dim=512,
                             page_size=256)
    dc = DevCase(case)
    ref = ref_direct(case)
    for splits in (3, 7, 16, 40):
        check_decode(dc, ref, num_splits=splits)


# ---- the global-layer shape (bf16, tensor-core kernel) ---------------------------

@pytest.mark.parametrize("context", [10602, 40002])
def test_global_decode(context):
    case = W.global_case(context, seed=1)
    dc = DevCase(case)
    ref = ref_direct(case)
    auto = pskv.pskv_plan_splits(dc.layout, 32, case.seq_lens)
    assert 1 <= auto <= pskv.PSKV_AUTO_MAX_SPLITS
    for splits in (0, 1, 8, 64, 256):
        check_decode(dc, ref, num_splits=splits)


@pytest.mark.parametrize("context", [81653, 163336])
def test_global_decode_long_split_sweep(context):
    case = W.global_case(context, seed=2)
    dc = DevCase(case)
    ref = ref_direct(case)
    for splits in (0, 8, 16, 32, 64, 128, 256):
        check_decode(dc, ref, num_splits=splits)


def test_global_decode_is_deterministic_and_page_order_free():
    lens = [5000]
    a = W.make_paged_case(24, lens, shuffle=True, **W.GLOBAL_SHAPE)
    b = W.make_paged_case(24, lens, shuffle=False, **W.GLOBAL_SHAPE)
    da, db = DevCase(a), DevCase(b)
    for splits in (0, 5, 33):
        o1 = da.decode(num_splits=splits)
        o2 = da.decode(num_splits=splits)
        o3 = db.decode(num_splits=splits)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2), "not run-to-run deterministic"
        assert torch.equal(o1, o3), "shuffled and identity tables differ"


# ---- the sliding-window variant -----------------------------------------------------

@pytest.mark.parametrize("residency", [1088, 1040, 1024, 528, 1])
def test_windowed_decode(residency):
    case = W.window_case(residency, seed=3)
    dc = DevCase(case)
    ref = ref_direct(case)
    for splits in (0, 1, 3, 9):
        check_decode(dc, ref, num_splits=splits)
    if residency == 1:  # one key: the output is that key's value, bit for bit
        out = dc.decode(out_dtype=torch.bfloat16)
        v0 = dc.v_pool[int(case.page_tables[0, 0]), :, 0, :]  # [Hkv, D]
        assert torch.equal(out[0], v0.repeat_interleave(2, dim=0))


def test_windowed_offset_rows_and_tensor_core_group():
    """Several rows with offsets, on both kernels (G = 2 CUDA cores, G = 8 tensor cores)."""
    for hq, hkv in ((32, 16), (32, 4)):
        base = W.make_paged_case(25, [1088, 700, 64, 1], num_q_heads=hq, num_kv_heads=hkv,
                                 head_dim=256, page_size=64)
        case = W.with_window(base, 1024, first_pos=[0, 5000, 17, 3])
        case.window_lo[1] = 5000 + 600  # a bound past the window rule: keys < 600 masked
        dc = DevCase(case)
        ref = ref_direct(case)
        for splits in (0, 2, 5):
            check_decode(dc, ref, num_splits=splits)


# ---- ragged batch with hostile padding ------------------------------------------------

def test_ragged_batch_with_nan_padding():
    case = W.ragged_case(seed=0)
    dc = DevCase(case)
    ref = ref_direct(case)
    for splits in (0, 16, 64):
        n_used = pskv.decode_attn_workspace_bytes(case.batch, 32, 512, splits)
        big_ws = torch.full((n_used + 4096,), 0x5A, dtype=torch.uint8, device="cuda")
        out = torch.full((case.batch + 1, 32, 512), float("nan"), device="cuda")
        view = out[:case.batch]
        dc.decode(num_splits=splits, out_dtype=torch.float32, out=view, workspace=big_ws[:n_used])
        torch.cuda.synchronize()
        assert torch.all(torch.isnan(out[case.batch])), "padding past the output was written"
        assert torch.all(big_ws[n_used:] == 0x5A), "padding past the workspace was written"
        err = max_err(view, ref)
        assert err <= TOL, err
    assert dc.faults() == 0


# ---- other shapes on the CUDA-core kernel ---------------------------------------------

@pytest.mark.parametrize("dtype,d,hq,hkv", [
    ("bf16", 512, 4, 4), ("bf16", 512, 8, 4), ("bf16", 512, 16, 4), ("bf16", 256, 64, 4),
    ("bf16", 256, 32, 4), ("f32", 256, 32, 2), ("f32", 512, 4, 2), ("f32", 256, 8, 8),
])
def test_other_group_sizes(dtype, d, hq, hkv):
    case = W.make_paged_case(26, [1, 77, 513, 2049], num_q_heads=hq, num_kv_heads=hkv,
                             head_dim=d, page_size=64, dtype=dtype)
    dc = DevCase(case)
    ref = ref_direct(case)
    for splits in (0, 1, 6):
        check_decode(dc, ref, num_splits=splits)


# ---- merge ---------------------------------------------------------------------------

def _oracle_partials(rng, rows, parts, dv, empty_every=0):
    m = np.zeros((rows, parts)); l = np.zeros((rows, parts)); o = np.zeros((rows, parts, dv))
    q = rng.standard_normal(16)
    for r in range(rows):
        k = rng.standard_normal((parts * 5, 16)); v = rng.standard_normal((parts * 5, dv))
        for p in range(parts):
            if empty_every and (p + r) % empty_every == 0:
                m[r, p], l[r, p] = -math.inf, 0.0
                continue
            m[r, p], l[r, p], o[r, p] = oracle.online_partial(q, k, v, 0.25, 5 * p, 5 * p + 5)
    return m, l, o


def _oracle_merge(m, l, o, group=16):
    out = []
    for r in range(m.shape[0]):
        tot = (-math.inf, 0.0, np.zeros(o.shape[2]))
        for g0 in range(0, m.shape[1], group):
            grp = (-math.inf, 0.0, np.zeros(o.shape[2]))
            for p in range(g0, min(g0 + group, m.shape[1])):
                st = (m[r, p], l[r, p], o[r, p] if m[r, p] != -math.inf else np.zeros(o.shape[2]))
                grp = oracle.merge(grp, st)
            tot = oracle.merge(tot, grp)
        out.append(oracle.finalize(tot))
    return np.stack(out)


@pytest.mark.parametrize("parts,empty_every", [(1, 0), (7, 3), (16, 0), (17, 4), (100, 7),
                                               (1024, 0)])
def test_merge_partials_matches_the_oracle(parts, empty_every):
    rng = np.random.default_rng(parts)
    m, l, o = _oracle_partials(rng, 3, parts, 64, empty_every)
    ref = _oracle_merge(m, l, o)
    t = lambda a: torch.tensor(a, dtype=torch.float32, device="cuda")
    o_t = t(o)
    if empty_every:  # o of an empty state is never read: poison it
        o_t[torch.tensor(m, device="cuda") == -math.inf] = float("nan")
    out = pskv.merge_partials(t(m), t(l), o_t)
    torch.cuda.synchronize()
    err = float(np.abs(out.cpu().numpy() - ref).max())
    assert err < 1e-5, err


def test_merge_with_empty_state_changes_nothing():
    rng = np.random.default_rng(5)
    m, l, o = _oracle_partials(rng, 2, 1, 32)
    t = lambda a: torch.tensor(a, dtype=torch.float32, device="cuda")
    single = pskv.merge_partials(t(m), t(l), t(o))
    m2 = np.concatenate([m, np.full((2, 3), -math.inf)], 1)
    l2 = np.concatenate([l, np.zeros((2, 3))], 1)
    o2 = np.concatenate([o, np.full((2, 3, 32), np.nan)], 1)
    padded = pskv.merge_partials(t(m2), t(l2), t(o2))
    torch.cuda.synchronize()
    assert torch.equal(single, padded)


def test_decode_partials_then_merge_equals_decode():
    case = W.global_case(3000, seed=6)
    dc = DevCase(case)
    splits = 24
    n = pskv.decode_attn_workspace_bytes(1, 32, 512, splits)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    out = dc.decode(num_splits=splits, workspace=ws)
    rows = 32
    align = lambda x: -(-x // 256) * 256
    m = ws[:rows * splits * 4].view(torch.float32).view(rows, splits)
    l_off = align(rows * splits * 4)
    l = ws[l_off:l_off + rows * splits * 4].view(torch.float32).view(rows, splits)
    o_off = align(l_off + rows * splits * 4)
    o = ws[o_off:o_off + rows * splits * 512 * 4].view(torch.float32).view(rows, splits, 512)
    merged = pskv.merge_partials(m.clone(), l.clone(), o.clone())
    torch.cuda.synchronize()
    assert torch.equal(merged.view(1, 32, 512), out)


# ---- device-side faults are flagged, never trapped -------------------------------------

def test_bad_page_id_is_flagged_not_read():
    case = W.make_paged_case(27, [600], **W.GLOBAL_SHAPE)
    dc = DevCase(case)
    tables = dc.tables.clone()
    tables[0, 1] = case.num_pages + 5  # outside the pool: the kernel must not dereference it
    out = pskv.decode_attn_splitkv(dc.layout, dc.q, tables, dc.lens, case.seq_lens, case.scale,
                                   num_splits=4, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert dc.faults() & pskv.PSKV_FAULT_BAD_PAGE
    assert torch.all(torch.isfinite(out))


# ---- the folded format (K keeps the rotated quarter, V in full) ------------------------

def _split_twin_dev(case):
    """The split pool a folded pool stands for: K = [stored K, V's remaining columns]."""
    import dataclasses
    dk = case.k_pool.shape[3]
    k_full = np.ascontiguousarray(np.concatenate([case.k_pool, case.v_pool[..., dk:]], axis=3))
    return dataclasses.replace(case, k_pool=k_full)


@pytest.mark.parametrize("context", [10602, 40002])
def test_folded_decode(context):
    case = W.folded_case(context, seed=51)
    dc = DevCase(case)
    ref = ref_direct(case)
    for splits in (0, 8, 64):
        check_decode(dc, ref, num_splits=splits)


def test_folded_equals_its_split_twin_bit_for_bit():
    case = W.make_paged_case(52, [5000, 333, 1], k_dims=128, **W.GLOBAL_SHAPE)
    twin = _split_twin_dev(case)
    a, b = DevCase(case), DevCase(twin)
    # the same partition on both sides (the automatic plans may differ: folded
    # CTAs are smaller, so more of them fit on an SM)
    for splits in (7, 76):
        oa = a.decode(num_splits=splits)
        ob = b.decode(num_splits=splits)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob)


@pytest.mark.parametrize("d,hq,hkv", [(256, 32, 16), (256, 32, 4), (512, 16, 4)])
def test_folded_other_shapes_and_window(d, hq, hkv):
    base = W.make_paged_case(53, [700, 64, 1, 300], num_q_heads=hq, num_kv_heads=hkv,
                             head_dim=d, page_size=64, k_dims=d // 4)
    for case in (base, W.with_window(base, 256, first_pos=[0, 10, 3, 1000])):
        dc = DevCase(case)
        ref = ref_direct(case)
        for splits in (0, 3):
            check_decode(dc, ref, num_splits=splits)


def test_folded_append_is_bit_exact():
    case = W.make_paged_case(54, [40, 300], num_q_heads=8, num_kv_heads=2, head_dim=512,
                             page_size=256, k_dims=128, keep_dense=True)
    exp_k, exp_v = np.zeros_like(case.k_pool), np.zeros_like(case.v_pool)
    rows = [(b, i) for b in range(case.batch) for i in range(int(case.seq_lens[b]))]
    kn = np.stack([case.dense_k[b][i] for b, i in rows])
    vn = np.stack([case.dense_v[b][i] for b, i in rows])
    row_of, pos_of = [r[0] for r in rows], [r[1] for r in rows]
    oracle.append_rows(exp_k, exp_v, kn, vn, row_of, pos_of, case.page_tables, case.pages_of_row)
    k_pool = torch.zeros_like(to_dev(case.k_pool, "bf16"))
    v_pool = torch.zeros_like(to_dev(case.v_pool, "bf16"))
    layout = pskv.paged_kv_layout_create(k_pool, v_pool)
    assert layout.desc.format == pskv.PSKV_FORMAT_FOLDED
    pskv.kv_append_rows(layout, to_dev(kn, "bf16"), to_dev(vn, "bf16"), i32(row_of), i32(pos_of),
                        i32(case.page_tables), i32(case.pages_of_row))
    torch.cuda.synchronize()
    assert k_pool.cpu().view(torch.int16).numpy().tobytes() == exp_k.view(np.int16).tobytes()
    assert v_pool.cpu().view(torch.int16).numpy().tobytes() == exp_v.view(np.int16).tobytes()
