"""Pins of the oracle's paged varlen prefill (CPU only).

Row b's new tokens are its last T_b keys; token t sits at key index
own = L_b - T_b + t and attends keys [max(0, own - W + 1), own] (W = 0: no
window).  Checked against decode of truncated rows (the same keys in the
same order: bit for bit), an explicit causal/window mask on the dense
tensors, and refusals."""
import dataclasses

import numpy as np
import pytest
from scipy.special import softmax

import oracle
import workloads as W


def _case(seed, lens, hq=4, hkv=2, d=16, ps=8, dtype="bf16", k_dims=None):
    return W.make_paged_case(seed, lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                             page_size=ps, dtype=dtype, keep_dense=True, k_dims=k_dims)


def _queries(case, counts, seed=0):
    rng = np.random.default_rng(seed)
    total = int(sum(counts))
    q = rng.standard_normal((total, case.num_q_heads, case.head_dim)).astype(np.float32)
    return W.bf16_bits(q) if case.dtype == "bf16" else q


def _cu(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


@pytest.mark.parametrize("window", [0, 5, 40])
def test_each_token_is_the_decode_of_its_truncated_row(window):
    case = _case(91, [37, 9, 60])
    counts = [5, 9, 1]
    q = _queries(case, counts)
    cu = _cu(counts)
    out = oracle.prefill_direct(q, cu, case.k_pool, case.v_pool, case.page_tables, case.seq_lens,
                                case.scale, window)
    for b, T in enumerate(counts):
        for t in range(T):
            own = int(case.seq_lens[b]) - T + t
            lo = max(0, own - window + 1) if window else 0
            one = dataclasses.replace(case, q=q[cu[b] + t][None], page_tables=case.page_tables[b:b + 1],
                                      seq_lens=np.array([own + 1], np.int32))
            ref = oracle.decode_direct(one.q, one.k_pool, one.v_pool, one.page_tables,
                                       one.seq_lens, one.scale, np.array([0], np.int32),
                                       np.array([lo], np.int32))
            assert np.array_equal(out[cu[b] + t], ref[0])


def test_matches_an_explicit_causal_window_mask():
    case = _case(92, [23, 40], hq=4, hkv=1, d=8, dtype="f32")
    counts, window = [23, 7], 6  # the first row is a whole prompt
    q = _queries(case, counts, 1)
    cu = _cu(counts)
    out = oracle.prefill_direct(q, cu, case.k_pool, case.v_pool, case.page_tables, case.seq_lens,
                                case.scale, window)
    for b, T in enumerate(counts):
        K = case.dense_k[b][:, 0, :].astype(np.float64)
        V = case.dense_v[b][:, 0, :].astype(np.float64)
        L = int(case.seq_lens[b])
        for t in range(T):
            own = L - T + t
            for h in range(4):
                s = case.scale * (K @ q[cu[b] + t, h].astype(np.float64))
                idx = np.arange(L)
                s[(idx > own) | (idx < own - window + 1)] = -np.inf
                np.testing.assert_allclose(out[cu[b] + t, h], softmax(s) @ V, rtol=0,
                                           atol=1e-12)


def test_a_window_longer_than_the_row_changes_nothing():
    case = _case(93, [30, 12])
    counts = [4, 12]
    q = _queries(case, counts, 2)
    cu = _cu(counts)
    a = oracle.prefill_direct(q, cu, case.k_pool, case.v_pool, case.page_tables, case.seq_lens,
                              case.scale, 0)
    b = oracle.prefill_direct(q, cu, case.k_pool, case.v_pool, case.page_tables, case.seq_lens,
                              case.scale, 31)
    assert np.array_equal(a, b)


def test_empty_chunks_and_folded_pools():
    """A row with no new tokens contributes no output row; a folded pool gives
    the same result as the split pool it stands for."""
    case = _case(94, [20, 33, 8], d=32, k_dims=None)
    counts = [3, 0, 8]
    q = _queries(case, counts, 3)
    cu = _cu(counts)
    split = oracle.prefill_direct(q, cu, case.k_pool, case.v_pool, case.page_tables,
                                  case.seq_lens, case.scale, 0)
    assert split.shape == (11, case.num_q_heads, 32)
    # the folded pool of the same keys: K keeps its first quarter, the rest of
    # each key is V's columns
    kf = case.k_pool[..., :8].copy()
    vf = case.v_pool.copy()
    vf[..., 8:] = case.k_pool[..., 8:]  # now V[8:] holds what K held there
    folded = oracle.prefill_direct(q, cu, kf, vf, case.page_tables, case.seq_lens, case.scale, 0)
    ref = oracle.prefill_direct(q, cu, case.k_pool, vf, case.page_tables, case.seq_lens,
                                case.scale, 0)
    np.testing.assert_allclose(folded, ref, rtol=0, atol=1e-12)


def test_refusals():
    case = _case(95, [5])
    q = _queries(case, [6])
    with pytest.raises(oracle.OracleError):  # more new tokens than keys
        oracle.prefill_direct(q, [0, 6], case.k_pool, case.v_pool, case.page_tables,
                              case.seq_lens, case.scale)
    with pytest.raises(oracle.OracleError):  # offsets must start at 0
        oracle.prefill_direct(q[:4], [1, 5], case.k_pool, case.v_pool, case.page_tables,
                              case.seq_lens, case.scale)
    with pytest.raises(oracle.OracleError):
        oracle.prefill_direct(q[:2], [0, 2], case.k_pool, case.v_pool, case.page_tables,
                              case.seq_lens, case.scale, -1)
