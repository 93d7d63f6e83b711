"""Pins for the CPU oracle: each test checks it against something other than
itself -- a brute-force dense computation on the unpaged tensors, a closed
form, an invariant of the merge identity, or a value or error bound the
source pages print (fixtures under tests/golden/, each with its citation)."""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def dense_f64(case, b):
    """Dense K, V of row b as float64 [len, Hkv, D] from the arrays the pool was built from."""
    conv = (lambda a: W.bf16_to_f32(a)) if case.dtype == "bf16" else (lambda a: a)
    return (conv(case.dense_k[b]).astype(np.float64), conv(case.dense_v[b]).astype(np.float64))


def q_f64(case):
    return (W.bf16_to_f32(case.q) if case.dtype == "bf16" else case.q).astype(np.float64)


def brute_force(case):
    """softmax(scale * q K^T) V on the dense tensors, with scipy's softmax; query
    head h reads KV head h // (Hq / Hkv).  For a folded pool the key is the
    stored K columns followed by V's remaining columns."""
    q = q_f64(case)
    G = case.num_q_heads // case.num_kv_heads
    out = np.zeros((case.batch, case.num_q_heads, case.head_dim))
    for b in range(case.batch):
        K, V = dense_f64(case, b)
        if case.folded:
            K = np.concatenate([K, V[:, :, K.shape[2]:]], axis=2)
        lo = 0
        if case.window_lo is not None:
            lo = max(0, int(case.window_lo[b]) - int(case.first_pos[b]))
        for h in range(case.num_q_heads):
            k, v = K[lo:, h // G, :], V[lo:, h // G, :]
            out[b, h] = softmax(case.scale * (k @ q[b, h])) @ v
    return out


def run_direct(case):
    return oracle.decode_direct(case.q, case.k_pool, case.v_pool, case.page_tables, case.seq_lens,
                                case.scale, case.first_pos, case.window_lo)


# ---- gather and the direct path against brute force -----------------------

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gather_is_bit_exact(dtype, seed):
    case = W.make_paged_case(seed, [1, 37, 130], num_q_heads=4, num_kv_heads=2, head_dim=24,
                             page_size=16, dtype=dtype)
    for b in range(case.batch):
        K, V = dense_f64(case, b)
        for g in range(case.num_kv_heads):
            k, v = oracle.gather(case.k_pool, case.v_pool, case.page_tables, b, g,
                                 int(case.seq_lens[b]))
            assert np.array_equal(k, K[:, g, :]) and np.array_equal(v, V[:, g, :])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", [(4, 2, 17, 8), (8, 1, 32, 16), (6, 3, 20, 4)])
def test_direct_matches_brute_force(dtype, shape):
    hq, hkv, d, ps = shape
    case = W.make_paged_case(11, [1, 13, 50, 129], num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                             page_size=ps, dtype=dtype)
    np.testing.assert_allclose(run_direct(case), brute_force(case), rtol=0, atol=1e-12)


def test_direct_matches_brute_force_windowed():
    case = W.make_paged_case(5, [1, 40, 90, 64], num_q_heads=4, num_kv_heads=2, head_dim=16,
                             page_size=8)
    case = W.with_window(case, window=24, first_pos=[0, 3, 100, 7])
    np.testing.assert_allclose(run_direct(case), brute_force(case), rtol=0, atol=1e-12)


def test_head_mapping_is_grouped():
    """Query head h reads KV head h // G: make KV head g's values all equal to g."""
    case = W.make_paged_case(3, [20], num_q_heads=6, num_kv_heads=3, head_dim=8, page_size=8,
                             dtype="f32")
    for g in range(3):
        case.v_pool[:, g, :, :] = float(g)
    out = run_direct(case)
    for h in range(6):
        np.testing.assert_allclose(out[0, h], float(h // 2), rtol=0, atol=1e-14)


# ---- closed forms ----------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_single_key_returns_its_value_exactly(dtype):
    case = W.make_paged_case(7, [1, 1], num_q_heads=4, num_kv_heads=2, head_dim=32, page_size=16,
                             dtype=dtype)
    out = run_direct(case)
    onl = oracle.decode_online(case.q, case.k_pool, case.v_pool, case.page_tables, case.seq_lens,
                               case.scale, num_splits=3, chunk_tokens=16)
    for b in range(2):
        _, V = dense_f64(case, b)
        for h in range(4):
            assert np.array_equal(out[b, h], V[0, h // 2])
            assert np.array_equal(onl[b, h], V[0, h // 2])


def test_zero_query_gives_mean_of_values():
    case = W.make_paged_case(8, [77], num_q_heads=2, num_kv_heads=1, head_dim=16, page_size=16,
                             dtype="f32")
    case.q[:] = 0.0
    _, V = dense_f64(case, 0)
    out = run_direct(case)
    np.testing.assert_allclose(out[0, 0], V[:, 0, :].mean(axis=0), rtol=0, atol=1e-14)


def test_dominant_key_selects_its_value():
    case = W.make_paged_case(9, [50], num_q_heads=1, num_kv_heads=1, head_dim=16, page_size=16,
                             dtype="f32")
    q = case.q[0, 0].astype(np.float64)
    j = 23
    page, row = case.page_tables[0, j // 16], j % 16
    case.k_pool[page, 0, row, :] = (q * 200.0).astype(np.float32)  # score ~ 200 |q|^2 / 4
    _, V = dense_f64(case, 0)
    out = run_direct(case)
    assert np.array_equal(out[0, 0], V[j, 0])


# ---- the merge identity ----------------------------------------------------

def fixture_13x17(seed=0):
    fx = golden("gem_partition_fixture.json")
    rng = np.random.default_rng(seed)
    n, d = fx["tokens"], fx["dims"]
    return (rng.standard_normal(d), rng.standard_normal((n, d)), rng.standard_normal((n, d)),
            fx["ways"])


def ceil_bounds(n, parts):
    per = -(-n // parts)
    return [min(n, p * per) for p in range(parts + 1)]


@pytest.mark.parametrize("group", [1, 2, 3, 16])
def test_partitions_agree_with_direct(group):
    q, k, v, ways = fixture_13x17()
    scale = 1.0 / math.sqrt(17)
    ref = oracle.attend_direct(q, k, v, scale)
    rng = np.random.default_rng(1)
    for parts in ways:
        cuts = [ceil_bounds(13, parts)]
        for _ in range(5):  # random cuts, repeats allowed (empty partitions)
            inner = np.sort(rng.integers(0, 14, size=parts - 1))
            cuts.append([0, *inner.tolist(), 13])
        for bounds in cuts:
            out = oracle.attend_partitioned(q, k, v, scale, bounds, group_size=group)
            np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    # the 16-way split of 13 keys necessarily holds empty partitions
    b16 = ceil_bounds(13, 16)
    assert any(b16[p] == b16[p + 1] for p in range(16))


def test_merge_with_empty_is_identity_bitwise():
    q, k, v, _ = fixture_13x17(2)
    x = oracle.online_partial(q, k, v, 0.3, 2, 11)
    empty = (-math.inf, 0.0, np.zeros(17))
    for a, b in ((x, empty), (empty, x)):
        m, l, o = oracle.merge(a, b)
        assert m == x[0] and l == x[1] and np.array_equal(o, x[2])
    assert oracle.online_partial(q, k, v, 0.3, 5, 5)[:2] == (-math.inf, 0.0)


def test_merge_associative_and_commutative():
    q, k, v, _ = fixture_13x17(3)
    a, b, c = (oracle.online_partial(q, k, v, 0.7, lo, hi) for lo, hi in ((0, 4), (4, 9), (9, 13)))
    left = oracle.merge(oracle.merge(a, b), c)
    right = oracle.merge(a, oracle.merge(b, c))
    swapped = oracle.merge(c, oracle.merge(b, a))
    for s in (right, swapped):
        assert abs(s[0] - left[0]) < 1e-12 and abs(s[1] - left[1]) < 1e-12 * left[1]
        np.testing.assert_allclose(s[2], left[2], rtol=1e-12, atol=1e-12)
    whole = oracle.online_partial(q, k, v, 0.7, 0, 13)
    np.testing.assert_allclose(oracle.finalize(left), oracle.finalize(whole), rtol=0, atol=1e-13)


@pytest.mark.parametrize("bad", [
    (-math.inf, 1.0, 0.0),      # empty max carrying mass
    (-math.inf, 0.0, 1.0),      # empty max carrying a numerator
    (math.nan, 1.0, 0.0),
    (math.inf, 1.0, 0.0),
    (0.5, 0.0, 0.0),            # finite max, zero sum
    (0.5, -1.0, 0.0),
    (0.5, math.inf, 0.0),
    (0.5, 1.0, math.nan),
    (0.5, 1.0, math.inf),
])
def test_invalid_states_fail_closed(bad):
    m, l, o0 = bad
    good = (0.1, 2.0, np.ones(4))
    badst = (m, l, np.full(4, o0))
    for a, b in ((good, badst), (badst, good)):
        with pytest.raises(oracle.OracleError) as e:
            oracle.merge(a, b)
        assert e.value.code == oracle.ORC_ERR_STATE
    with pytest.raises(oracle.OracleError):
        oracle.finalize(badst)


def test_finalize_empty_fails():
    with pytest.raises(oracle.OracleError):
        oracle.finalize((-math.inf, 0.0, np.zeros(3)))


# ---- the gem design's accuracy audit ----------------------------------------

def _audit(length, seed=0):
    g = golden("gem_online_merge_audit.json")
    rng = np.random.default_rng(seed)
    d = g["head_dim_v"]
    q = rng.standard_normal((8, d), dtype=np.float32)
    k = rng.standard_normal((length, d), dtype=np.float32)
    v = rng.standard_normal((length, d), dtype=np.float32)
    scale = 1.0 / math.sqrt(d)
    bounds = ceil_bounds(length, g["num_splits"])
    ref = np.stack([oracle.attend_direct(q[h], k, v, scale) for h in range(8)])
    f32 = np.stack([oracle.attend_partitioned_f32(q[h], k, v, scale, bounds) for h in range(8)])
    f32b = np.stack([oracle.attend_partitioned_f32(q[h], k, v, scale, bounds) for h in range(8)])
    assert np.array_equal(f32, f32b) and np.all(np.isfinite(f32))  # repeat-deterministic, finite
    diff = f32.astype(np.float64) - ref
    corr = np.corrcoef(f32.ravel().astype(np.float64), ref.ravel())[0, 1]
    nmse = float((diff ** 2).sum() / (ref ** 2).sum())
    assert corr >= g["min_correlation"]
    assert nmse <= g["max_nmse"]
    assert np.abs(diff).max() < g["max_abs_error_below"]


@pytest.mark.parametrize("length", [8191, 8192, 8193])
def test_single_precision_audit_bounds(length):
    _audit(length)


@pytest.mark.slow
@pytest.mark.parametrize("length", [65536, 131072])
def test_single_precision_audit_bounds_long(length):
    _audit(length)


# ---- masks and hostile padding -----------------------------------------------

def test_window_equals_sliced_direct():
    base = W.make_paged_case(4, [1088, 1040, 1024, 528, 1], num_q_heads=4, num_kv_heads=2,
                             head_dim=32, page_size=64)
    case = W.with_window(base, 1024)
    assert case.window_lo.tolist() == [64, 16, 0, 0, 0]
    np.testing.assert_allclose(run_direct(case), brute_force(case), rtol=0, atol=1e-12)


def test_nan_padding_never_reaches_the_output():
    case = W.make_paged_case(6, [5, 33, 64], num_q_heads=4, num_kv_heads=2, head_dim=16,
                             page_size=16, extra_pages=2)
    out = run_direct(case)
    assert np.all(np.isfinite(out))
    clean = W.make_paged_case(6, [5, 33, 64], num_q_heads=4, num_kv_heads=2, head_dim=16,
                              page_size=16, extra_pages=2)
    # replace every NaN (padding rows, poison page) by zeros: same output, bit for bit
    clean.k_pool[np.isnan(W.bf16_to_f32(clean.k_pool))] = 0
    clean.v_pool[np.isnan(W.bf16_to_f32(clean.v_pool))] = 0
    assert np.array_equal(run_direct(clean), out)


def test_shuffled_table_equals_identity_table():
    lens = [300, 17, 129]
    a = W.make_paged_case(12, lens, num_q_heads=8, num_kv_heads=2, head_dim=16, page_size=32,
                          shuffle=True)
    b = W.make_paged_case(12, lens, num_q_heads=8, num_kv_heads=2, head_dim=16, page_size=32,
                          shuffle=False)
    assert not np.array_equal(a.page_tables, b.page_tables)
    assert np.array_equal(run_direct(a), run_direct(b))


# ---- append --------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_append_rebuilds_the_pool_bit_exactly(dtype):
    case = W.make_paged_case(13, [3, 40, 17], num_q_heads=4, num_kv_heads=2, head_dim=8,
                             page_size=16, dtype=dtype)
    k_pool = np.zeros_like(case.k_pool)
    v_pool = np.zeros_like(case.v_pool)
    rows = [(b, i) for b in range(case.batch) for i in range(int(case.seq_lens[b]))]
    rng = np.random.default_rng(0)
    rng.shuffle(rows)
    kn = np.stack([case.dense_k[b][i] for b, i in rows])
    vn = np.stack([case.dense_v[b][i] for b, i in rows])
    oracle.append_rows(k_pool, v_pool, kn, vn, [r[0] for r in rows], [r[1] for r in rows],
                       case.page_tables, case.pages_of_row)
    for b in range(case.batch):
        for i in range(int(case.seq_lens[b])):
            page, row = case.page_tables[b, i // 16], i % 16
            assert np.array_equal(k_pool[page, :, row], case.k_pool[page, :, row])
            assert np.array_equal(v_pool[page, :, row], case.v_pool[page, :, row])
            assert k_pool[page, :, row].tobytes() == case.dense_k[b][i].tobytes()


def test_append_past_pages_is_refused_and_writes_nothing():
    case = W.make_paged_case(14, [20], num_q_heads=2, num_kv_heads=1, head_dim=8, page_size=16)
    k_pool, v_pool = case.k_pool.copy(), case.v_pool.copy()
    kn = np.ones((2, 1, 8), np.uint16)
    with pytest.raises(oracle.OracleError) as e:
        # the first row is fine, the second lands past the row's 2 pages
        oracle.append_rows(k_pool, v_pool, kn, kn, [0, 0], [5, 32], case.page_tables,
                           case.pages_of_row)
    assert e.value.code == oracle.ORC_ERR_PAST_PAGES
    assert np.array_equal(k_pool, case.k_pool) and np.array_equal(v_pool, case.v_pool)


# ---- the tiny decode: paged online path against the direct path -----------------

def test_tiny_decode_partitions():
    case = W.tiny_case(0)
    assert case.pages_of_row.tolist() == [4] and case.seq_lens.tolist() == [1000]
    ref = run_direct(case)
    np.testing.assert_allclose(ref, brute_force(case), rtol=0, atol=1e-12)
    for parts in golden("gem_partition_fixture.json")["ways"]:
        for chunk in (256, 16):
            out = oracle.decode_online(case.q, case.k_pool, case.v_pool, case.page_tables,
                                       case.seq_lens, case.scale, num_splits=parts,
                                       chunk_tokens=chunk, group_size=3)
            np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_online_windowed_matches_direct():
    case = W.with_window(W.make_paged_case(15, [300, 97], num_q_heads=4, num_kv_heads=1,
                                           head_dim=16, page_size=16), 40, first_pos=[5, 0])
    ref = run_direct(case)
    for parts in (1, 3, 7):
        out = oracle.decode_online(case.q, case.k_pool, case.v_pool, case.page_tables,
                                   case.seq_lens, case.scale, num_splits=parts, chunk_tokens=16,
                                   first_pos=case.first_pos, window_lo=case.window_lo)
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


# ---- the scratch byte contract ---------------------------------------------------

def test_scratch_contract_matches_the_page():
    g = golden("gem_scratch_contract.json")
    s = g["shape"]
    for c in g["cases"]:
        got = oracle.partial_scratch_bytes(s["batch"], s["num_q_heads"], s["head_dim_v"],
                                           c["num_splits"])
        assert got == (c["maxima"], c["denominators"], c["numerators"], c["total"])
    for p, mib in g["numerator_mib_by_splits"].items():
        got = oracle.partial_scratch_bytes(s["batch"], s["num_q_heads"], s["head_dim_v"], int(p))
        assert got[2] == mib * (1 << 20)


def test_scratch_contract_overflow_fails_closed():
    with pytest.raises(oracle.OracleError) as e:
        oracle.partial_scratch_bytes(1 << 30, 1 << 20, 512, 1 << 10)
    assert e.value.code == oracle.ORC_ERR_OVERFLOW
    with pytest.raises(oracle.OracleError):
        oracle.partial_scratch_bytes(0, 32, 512, 32)


def test_refuses_empty_rows():
    case = W.make_paged_case(1, [4], num_q_heads=2, num_kv_heads=1, head_dim=8, page_size=8)
    with pytest.raises(oracle.OracleError):
        oracle.decode_direct(case.q, case.k_pool, case.v_pool, case.page_tables, [0], case.scale)


# ---- the folded format ----------------------------------------------------------

def split_twin(case):
    """The split pool a folded pool stands for: K = [stored K, V's remaining columns]."""
    import dataclasses
    dk = case.k_pool.shape[3]
    k_full = np.concatenate([case.k_pool, case.v_pool[..., dk:]], axis=3)
    return dataclasses.replace(case, k_pool=np.ascontiguousarray(k_full))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_folded_equals_its_split_twin_exactly(dtype):
    case = W.make_paged_case(31, [1, 70, 257], num_q_heads=8, num_kv_heads=2, head_dim=32,
                             page_size=16, dtype=dtype, k_dims=8)
    assert case.folded
    twin = split_twin(case)
    assert np.array_equal(run_direct(case), run_direct(twin))
    for parts in (1, 5):
        a = oracle.decode_online(case.q, case.k_pool, case.v_pool, case.page_tables,
                                 case.seq_lens, case.scale, num_splits=parts, chunk_tokens=16)
        b = oracle.decode_online(twin.q, twin.k_pool, twin.v_pool, twin.page_tables,
                                 twin.seq_lens, twin.scale, num_splits=parts, chunk_tokens=16)
        assert np.array_equal(a, b)


def test_folded_matches_brute_force():
    case = W.make_paged_case(32, [3, 90, 140], num_q_heads=4, num_kv_heads=2, head_dim=24,
                             page_size=8, k_dims=6)
    np.testing.assert_allclose(run_direct(case), brute_force(case), rtol=0, atol=1e-12)
    k, v = oracle.gather(case.k_pool, case.v_pool, case.page_tables, 1, 1, 90)
    K, V = dense_f64(case, 1)
    assert np.array_equal(k[:, :6], K[:, 1]) and np.array_equal(k[:, 6:], V[:, 1, 6:])


def test_folded_stored_columns_reach_the_score():
    """Changing a stored K column changes the output; changing V's first columns
    (which a folded key does not use) changes only the value side."""
    case = W.make_paged_case(33, [20], num_q_heads=2, num_kv_heads=1, head_dim=16, page_size=16,
                             dtype="f32", k_dims=4)
    base = run_direct(case)
    page = case.page_tables[0, 0]
    k_saved = case.k_pool.copy()
    case.k_pool[page, 0, 3, 0] += 5.0  # one key's stored column (a shift of all keys would cancel)
    assert not np.allclose(run_direct(case), base)
    case.k_pool[:] = k_saved
    case.v_pool[page, 0, 3, 1] += 5.0  # V column 1 < k_dims: only the value side moves
    out = run_direct(case)
    moved = np.abs(out - base).max(axis=(0, 1))
    assert moved[1] > 0 and np.all(moved[np.arange(16) != 1] == 0)


# ---- multi-row decode (verify windows) ----------------------------------------------

@pytest.mark.parametrize("tokens", [1, 2, 3, 8])
def test_multirow_token_equals_single_decode_of_the_truncated_row(tokens):
    """Token t of a T-token window is the single-token decode of the row cut at
    its own position (the same keys, the same order: bit for bit)."""
    import dataclasses
    case = W.make_paged_case(61, [40, 9, 300], num_q_heads=4, num_kv_heads=2, head_dim=16,
                             page_size=16, dtype="f32")
    rng = np.random.default_rng(tokens)
    q = rng.standard_normal((case.batch, tokens, 4, 16)).astype(np.float32)
    out = oracle.decode_multirow_direct(q, case.k_pool, case.v_pool, case.page_tables,
                                        case.seq_lens, case.scale)
    for t in range(tokens):
        lens = case.seq_lens - tokens + t + 1
        single = dataclasses.replace(case, q=np.ascontiguousarray(q[:, t]), seq_lens=lens)
        assert np.array_equal(out[:, t], run_direct(single))


def test_multirow_matches_causal_brute_force():
    case = W.make_paged_case(62, [33, 70], num_q_heads=4, num_kv_heads=1, head_dim=8, page_size=8,
                             dtype="bf16")
    T = 4
    rng = np.random.default_rng(0)
    q = W.bf16_bits(rng.standard_normal((case.batch, T, 4, 8)).astype(np.float32))
    out = oracle.decode_multirow_direct(q, case.k_pool, case.v_pool, case.page_tables,
                                        case.seq_lens, case.scale)
    qf = W.bf16_to_f32(q).astype(np.float64)
    for b in range(case.batch):
        K, V = dense_f64(case, b)
        L = int(case.seq_lens[b])
        for t in range(T):
            for h in range(4):
                s_ = case.scale * (K[:, 0, :] @ qf[b, t, h])
                s_[L - T + t + 1:] = -np.inf  # causal: keys after the token's own position
                ref = softmax(s_) @ V[:, 0, :]
                np.testing.assert_allclose(out[b, t, h], ref, rtol=0, atol=1e-12)


def test_multirow_refuses_rows_shorter_than_the_window():
    case = W.make_paged_case(63, [2], num_q_heads=2, num_kv_heads=1, head_dim=8, page_size=8)
    q = np.zeros((1, 3, 2, 8), np.uint16)
    with pytest.raises(oracle.OracleError):
        oracle.decode_multirow_direct(q, case.k_pool, case.v_pool, case.page_tables,
                                      case.seq_lens, case.scale)
