"""Pins of the oracle's K/V prep (CPU only).

The prep (pegainfer #1055 and #1057, Description) normalises each head row by
its root mean square, multiplies by the head's norm multiplier, turns the
first R columns as pairs (i, i + R/2), and for the folded format moves K's
multiplier into the query.  Nothing here retypes the oracle's formula: each
check is a closed form, an invariant or an identity the definition implies."""
import math

import numpy as np
import pytest

import oracle
import workloads as W


def test_constant_row_normalises_to_its_sign_times_the_multiplier():
    w = np.linspace(0.5, 2.0, 16)
    for c in (3.0, -0.25, 1e-3):
        out = oracle.prep_head(np.full(16, c), 0.0, w=w)
        np.testing.assert_allclose(out, math.copysign(1.0, c) * w, rtol=0, atol=1e-15)


def test_one_hot_row_gives_sqrt_d():
    x = np.zeros(64)
    x[17] = -5.0
    out = oracle.prep_head(x, 0.0)
    exp = np.zeros(64)
    exp[17] = -8.0  # sqrt(64)
    np.testing.assert_allclose(out, exp, rtol=0, atol=1e-14)


def test_mean_square_after_normalising_is_ms_over_ms_plus_eps():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(512) * 0.01
    ms = float(np.mean(x * x))
    for eps in (0.0, 1e-6, 1e-4):
        out = oracle.prep_head(x, eps)
        assert abs(float(np.mean(out * out)) - ms / (ms + eps)) < 1e-13


def test_zero_angle_is_no_rotation():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(32)
    plain = oracle.prep_head(x, 1e-6)
    turned = oracle.prep_head(x, 1e-6, cos=np.ones(8), sin=np.zeros(8))
    assert np.array_equal(plain, turned)


def test_quarter_turn_maps_pairs_exactly():
    """cos = 0, sin = 1 sends (a, b) to (-b, a) for each pair (i, i + R/2)."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal(32)
    plain = oracle.prep_head(x, 1e-6)
    turned = oracle.prep_head(x, 1e-6, cos=np.zeros(8), sin=np.ones(8))
    assert np.array_equal(turned[0:8], -plain[8:16])
    assert np.array_equal(turned[8:16], plain[0:8])
    assert np.array_equal(turned[16:], plain[16:])  # columns past R untouched


def test_rotation_keeps_each_pair_norm():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(64)
    ang = rng.uniform(-3, 3, 16)
    plain = oracle.prep_head(x, 0.0)
    turned = oracle.prep_head(x, 0.0, cos=np.cos(ang), sin=np.sin(ang))
    np.testing.assert_allclose(turned[:16] ** 2 + turned[16:32] ** 2,
                               plain[:16] ** 2 + plain[16:32] ** 2, rtol=1e-13)


def test_scores_depend_only_on_the_position_difference():
    """Rotating q and k by their positions' angles makes q.k a function of the
    offset alone: the same rows at (m, n) and (m + s, n + s) score alike."""
    p = W.make_prep_inputs(4, 1, 1, 1, 64, 64, 200)
    dot = []
    for m, n in ((40, 7), (140, 107), (33, 0)):
        q, k, _ = oracle.prep_tokens(np.concatenate([p.x, p.x]), p.q_col, p.k_col, p.v_col, 1, 1,
                                     64, p.eps, p.w_q, p.w_k, p.rope_cos, p.rope_sin, [m, n])
        dot.append(float(q[0, 0] @ k[1, 0]))
    assert abs(dot[0] - dot[1]) < 1e-4 * abs(dot[0])  # float32 tables: angles to ~1e-7
    assert abs(dot[0] - dot[2]) < 1e-4 * abs(dot[0])


def test_folded_query_scores_equal_split_scores():
    """With K and V from one projection row, q_split . k_full equals
    q_fold[:R] . k[:R] + q_fold[R:] . v[R:] (pegainfer #1055, Description:
    K's norm weight folded into the query)."""
    p = W.make_prep_inputs(5, 6, 8, 2, 128, 32, 64, shared_kv=True)
    pos = np.arange(6) * 9
    args = (p.x, p.q_col, p.k_col, p.v_col, 8, 2, 128, p.eps, p.w_q, p.w_k, p.rope_cos,
            p.rope_sin, pos)
    qs, k, v = oracle.prep_tokens(*args)
    qf, k2, v2 = oracle.prep_tokens(*args, folded=True)
    assert np.array_equal(k, k2) and np.array_equal(v, v2)
    R = 32
    for t in range(6):
        for h in range(8):
            g = h // 4
            for u in range(6):
                split = qs[t, h] @ k[u, g]
                fold = qf[t, h, :R] @ k[u, g, :R] + qf[t, h, R:] @ v[u, g, R:]
                assert abs(split - fold) <= 1e-12 * (1 + abs(split))


def test_value_rows_are_normalised_only():
    p = W.make_prep_inputs(6, 2, 2, 1, 32, 8, 16)
    _, k, v = oracle.prep_tokens(p.x, p.q_col, p.k_col, p.v_col, 2, 1, 32, p.eps, p.w_q, p.w_k,
                                 p.rope_cos, p.rope_sin, [3, 9])
    xv = W.bf16_to_f32(p.x[:, p.v_col:p.v_col + 32]).astype(np.float64)
    for t in range(2):
        # normalised: mean square ms/(ms+eps); direction that of the input row
        ms = float(np.mean(xv[t] ** 2))
        assert abs(float(np.mean(v[t, 0] ** 2)) - ms / (ms + p.eps)) < 1e-12
        cos = float(v[t, 0] @ xv[t]) / (np.linalg.norm(v[t, 0]) * np.linalg.norm(xv[t]))
        assert abs(cos - 1.0) < 1e-14


def test_position_outside_the_table_is_refused():
    p = W.make_prep_inputs(7, 1, 1, 1, 16, 4, 8)
    with pytest.raises(oracle.OracleError):
        oracle.prep_tokens(p.x, p.q_col, p.k_col, p.v_col, 1, 1, 16, p.eps, p.w_q, p.w_k,
                           p.rope_cos, p.rope_sin, [8])


def test_folded_needs_one_projection_row():
    p = W.make_prep_inputs(8, 1, 1, 1, 16, 4, 8, shared_kv=False)
    with pytest.raises(oracle.OracleError):
        oracle.prep_tokens(p.x, p.q_col, p.k_col, p.v_col, 1, 1, 16, p.eps, p.w_q, p.w_k,
                           p.rope_cos, p.rope_sin, [1], folded=True)
