"""Pins of the oracle's tree attention over a drafted window (TensorFold
#1619, description "Reads" and review thread: tree-attention rows read their
keys from a page table).  The window's T tokens are the row's last T keys in
topological order; token t attends every key before the window, its
ancestors in the window and itself."""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
import workloads as W


def dense_f64(case, b):
    conv = (lambda a: W.bf16_to_f32(a)) if case.dtype == "bf16" else (lambda a: a)
    return (conv(case.dense_k[b]).astype(np.float64), conv(case.dense_v[b]).astype(np.float64))


def queries(case, T, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((case.batch, T, case.num_q_heads, case.head_dim)).astype(np.float32)
    return W.bf16_bits(q) if case.dtype == "bf16" else q


def q64(case, q):
    return (W.bf16_to_f32(q) if case.dtype == "bf16" else q).astype(np.float64)


def tree(case, q, masks):
    return oracle.decode_tree_direct(q, case.k_pool, case.v_pool, case.page_tables,
                                     case.seq_lens, masks, case.scale)


def ancestors(parents, t):
    """t and its ancestors, by walking the parent links (not through the masks)."""
    seen = []
    while t >= 0:
        seen.append(t)
        t = int(parents[t])
    return seen


def test_masks_hold_the_ancestor_sets():
    for seed in range(5):
        parents = W.random_tree_parents(seed, 40)
        masks = W.tree_masks(parents)
        for t in range(40):
            bits = {j for j in range(64) if (int(masks[t]) >> j) & 1}
            assert bits == set(ancestors(parents, t))


@pytest.mark.parametrize("T", [1, 2, 5, 16])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_chain_equals_the_causal_verify_window_bitwise(T, dtype):
    case = W.make_paged_case(70 + T, [40, T, 300], num_q_heads=4, num_kv_heads=2, head_dim=16,
                             page_size=16, dtype=dtype)
    q = queries(case, T, T)
    masks = np.tile(W.tree_masks(W.chain_parents(T)), (case.batch, 1))
    got = tree(case, q, masks)
    ref = oracle.decode_multirow_direct(q, case.k_pool, case.v_pool, case.page_tables,
                                        case.seq_lens, case.scale)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("seed,T", [(0, 6), (1, 13), (2, 32), (3, 64)])
def test_random_trees_match_brute_force(seed, T):
    lens = [T, T + 7, T + 130]
    case = W.make_paged_case(80 + seed, lens, num_q_heads=6, num_kv_heads=2, head_dim=8,
                             page_size=8, dtype="bf16")
    q = queries(case, T, seed)
    parents = [W.random_tree_parents(100 * seed + b, T) for b in range(case.batch)]
    masks = np.stack([W.tree_masks(p) for p in parents])
    got = tree(case, q, masks)
    qf = q64(case, q)
    G = case.num_q_heads // case.num_kv_heads
    for b in range(case.batch):
        K, V = dense_f64(case, b)
        w0 = int(case.seq_lens[b]) - T
        for t in range(T):
            keys = list(range(w0)) + sorted(w0 + j for j in ancestors(parents[b], t))
            for h in range(case.num_q_heads):
                s_ = case.scale * (K[keys, h // G, :] @ qf[b, t, h])
                ref = softmax(s_) @ V[keys, h // G, :]
                np.testing.assert_allclose(got[b, t, h], ref, rtol=0, atol=1e-12)


def test_a_token_that_sees_only_itself_and_the_prefix():
    """Mask = its own bit: the dense direct attention over the prefix keys and
    the token's own key, put side by side in one contiguous buffer."""
    T = 5
    case = W.make_paged_case(90, [70], num_q_heads=2, num_kv_heads=1, head_dim=16,
                             page_size=16, dtype="f32")
    q = queries(case, T, 3)
    masks = np.array([[np.uint64(1 << t) for t in range(T)]], np.uint64)
    got = tree(case, q, masks)
    K, V = dense_f64(case, 0)
    w0 = 70 - T
    for t in range(T):
        keys = list(range(w0)) + [w0 + t]
        k = np.ascontiguousarray(K[keys, 0, :].astype(np.float32))
        v = np.ascontiguousarray(V[keys, 0, :].astype(np.float32))
        for h in range(2):
            ref = oracle.attend_direct(q[0, t, h], k, v, case.scale)
            assert np.array_equal(got[0, t, h], ref)


def test_a_root_with_no_prefix_returns_its_value_exactly():
    """A row that holds only the window: a root sees one key, its own, and
    gets that key's value exactly; a child of that root sees two keys."""
    T = 3
    case = W.make_paged_case(91, [T], num_q_heads=2, num_kv_heads=1, head_dim=16, page_size=16,
                             dtype="bf16")
    q = queries(case, T, 4)
    masks = W.tree_masks([-1, 0, -1])[None, :]
    got = tree(case, q, masks)
    _, V = dense_f64(case, 0)
    for h in range(2):
        assert np.array_equal(got[0, 0, h], V[0, 0])
        assert np.array_equal(got[0, 2, h], V[2, 0])
        assert not np.array_equal(got[0, 1, h], V[1, 0])


def test_folded_tree_equals_its_split_twin():
    import dataclasses
    T = 7
    case = W.make_paged_case(92, [30, 100], num_q_heads=4, num_kv_heads=2, head_dim=32,
                             page_size=16, dtype="bf16", k_dims=8)
    k_full = np.concatenate([case.k_pool, case.v_pool[..., 8:]], axis=3)
    twin = dataclasses.replace(case, k_pool=np.ascontiguousarray(k_full))
    q = queries(case, T, 5)
    masks = np.stack([W.tree_masks(W.random_tree_parents(b, T)) for b in range(2)])
    assert np.array_equal(tree(case, q, masks), tree(twin, q, masks))


@pytest.mark.parametrize("bad", ["no_self", "later_bit", "short_row", "too_many"])
def test_invalid_trees_fail_closed(bad):
    T = 65 if bad == "too_many" else 4
    lens = [3] if bad == "short_row" else [80]
    case = W.make_paged_case(93, lens, num_q_heads=2, num_kv_heads=1, head_dim=8, page_size=8)
    q = np.zeros((1, T, 2, 8), np.uint16)
    masks = W.tree_masks(W.chain_parents(T)) if T <= 64 else np.ones(T, np.uint64)
    masks = masks[None, :].copy()
    if bad == "no_self":
        masks[0, 2] &= ~np.uint64(1 << 2)
    elif bad == "later_bit":
        masks[0, 1] |= np.uint64(1 << 3)
    with pytest.raises(oracle.OracleError):
        tree(case, q, masks)
