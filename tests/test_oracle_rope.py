"""Pins for the RoPE and path-weight oracles (CPU, no GPU).

The pages print no RoPE values, so the pins come from the mathematics of the
rotation (RoFormer, Su et al. 2023) and from the pages' own claims: eq. 9
positions make tree RoPE equal per-path RoPE (§3.2 "Position Embedding"), and
the weighted tree loss equals the weighted sum of per-path losses (§3.1, the
general lambda_t after eq. 5).
"""
import math

import numpy as np
import pytest

import treegen
from oracle import rope as R
from oracle import trie as T

def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)

@pytest.mark.parametrize("rotate_half", [False, True])
def test_two_dims_turn_by_pos_radians(rotate_half):
    # D = 2: theta_0 = base^0 = 1, so position p turns (1, 0) to (cos p, sin p)
    x = np.array([[[1.0, 0.0]], [[1.0, 0.0]], [[0.0, 2.0]]])
    y = R.rope(x, [1, 3, 2], base=500.0, rotate_half=rotate_half)
    assert np.allclose(y[0, 0], [math.cos(1), math.sin(1)], atol=1e-15)
    assert np.allclose(y[1, 0], [math.cos(3), math.sin(3)], atol=1e-15)
    assert np.allclose(y[2, 0], [-2 * math.sin(2), 2 * math.cos(2)], atol=1e-15)

def test_second_pair_uses_base_to_the_minus_half():
    # D = 4, base 10000: pair 1 has theta = 10000^(-1/2) = 0.01
    x = np.zeros((1, 1, 4))
    x[0, 0, 2] = 1.0
    y = R.rope(x, [7], base=10000.0)
    assert np.allclose(y[0, 0], [0, 0, math.cos(0.07), math.sin(0.07)], atol=1e-15)
    x = np.zeros((1, 1, 4))
    x[0, 0, 1] = 1.0  # split halves: pair 1 is dims (1, 3)
    y = R.rope(x, [7], base=10000.0, rotate_half=True)
    assert np.allclose(y[0, 0], [0, math.cos(0.07), 0, math.sin(0.07)], atol=1e-15)

@pytest.mark.parametrize("rotate_half", [False, True])
def test_position_zero_is_identity_and_norms_are_kept(rotate_half):
    x = _rand((5, 3, 16), 0)
    assert np.array_equal(R.rope(x, [0] * 5, rotate_half=rotate_half), x)
    y = R.rope(x, [0, 1, 17, 1000, 123456], rotate_half=rotate_half)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)

@pytest.mark.parametrize("rotate_half", [False, True])
def test_scores_depend_on_relative_position_only(rotate_half):
    # <R(p) q, R(p') k> = <R(p - p') q, k>: the property RoPE exists for
    q = _rand((1, 1, 64), 1)
    k = _rand((1, 1, 64), 2)
    for p, pp in [(5, 2), (100, 37), (4000, 3999), (3, 9)]:
        lhs = float(np.sum(R.rope(q, [p], rotate_half=rotate_half) * R.rope(k, [pp], rotate_half=rotate_half)))
        rhs = float(np.sum(R.rope(q, [p - pp], rotate_half=rotate_half) * k))
        assert abs(lhs - rhs) < 1e-9 * max(1.0, abs(rhs))

@pytest.mark.parametrize("rotate_half", [False, True])
def test_inverse_undoes_the_rotation(rotate_half):
    x = _rand((6, 2, 32), 3)
    pos = [0, 1, 2, 50, 900, 70000]
    y = R.rope(R.rope(x, pos, rotate_half=rotate_half), pos, rotate_half=rotate_half, inverse=True)
    assert np.allclose(y, x, atol=1e-12)

def test_the_two_pairings_differ_by_a_fixed_permutation():
    D = 8
    perm = np.array([0, 4, 1, 5, 2, 6, 3, 7])  # split-halves pair i -> interleaved slots 2i, 2i+1
    x = _rand((4, 2, D), 4)
    pos = [3, 11, 0, 250]
    a = R.rope(x, pos, rotate_half=True)
    b = R.rope(x[..., perm], pos, rotate_half=False)
    assert np.allclose(a[..., perm], b, atol=1e-14)

@pytest.mark.parametrize("rotate_half", [False, True])
def test_tree_rope_equals_rope_on_each_path(rotate_half):
    # §3.2 "Position Embedding": with eq. 9 positions every token of the tree is
    # rotated exactly as in each standalone root-to-leaf sequence (positions 0..L-1)
    for wi, seed in [(1, 0), (1, 1)]:
        w = treegen.workload(wi, seed)
        N = int(np.sum(w.lengths))
        x = _rand((N, 2, 16), seed + 10)
        tree = R.rope(x, T.position_ids(w.parents, w.lengths), rotate_half=rotate_half)
        for _, ids in T.base_serialization(w.parents, w.lengths):
            path = R.rope(x[ids], np.arange(len(ids)), rotate_half=rotate_half)
            assert np.allclose(tree[ids], path, atol=1e-12)

def test_path_weights_reduce_to_g_over_K_and_to_g():
    for wi, seed in [(1, 0), (3, 0), (4, 0)]:
        w = treegen.workload(wi, seed)
        K = T.paths_per_trie(w.parents)
        roots, trie_id = T.tries(w.parents)
        order, _ = T.dfs_serialize(w.parents, w.lengths)
        leaf_set = set(T.leaves(w.parents))
        dfs_leaves = [s for s in order if s in leaf_set]
        inv_k = np.array([1.0 / K[trie_id[s]] for s in dfs_leaves])
        got = T.path_weight_tokens(w.parents, w.lengths, inv_k)
        ref = T.token_weights(w.parents, w.lengths)
        # both round an fp64 value to fp32; the sums of 1/K may differ from g/K
        # in the last fp64 bits, so allow one fp32 ulp
        assert np.all(np.abs(got.astype(np.float64) - ref) <= np.spacing(np.abs(ref)))
        ones = T.path_weight_tokens(w.parents, w.lengths, np.ones(len(dfs_leaves)))
        g = T.paths_through(w.parents)
        tok = T.token_segments(w.parents, w.lengths)
        assert np.array_equal(ones, np.array([g[s] for s in tok], dtype=np.float32))

def test_weighted_tree_loss_equals_weighted_sum_of_path_losses():
    # §3.1 after eq. 5: sum_t lambda_t l_t = sum_k w_k sum_{t in p_k} l_t
    rng = np.random.default_rng(7)
    for wi, seed in [(1, 2), (3, 1)]:
        w = treegen.workload(wi, seed)
        N = int(np.sum(w.lengths))
        loss = rng.standard_normal(N)
        paths = T.base_serialization(w.parents, w.lengths)
        order, _ = T.dfs_serialize(w.parents, w.lengths)
        rank = {s: i for i, s in enumerate(order)}
        paths.sort(key=lambda p: rank[p[0]])  # number the paths by their leaves in DFS order
        pw = rng.uniform(0.1, 2.0, len(paths))
        lam = T.path_weight_tokens(w.parents, w.lengths, pw).astype(np.float64)
        tree_loss = float(np.dot(lam, loss))
        path_loss = float(sum(pw[k] * loss[ids].sum() for k, (_, ids) in enumerate(paths)))
        # lambda_t is rounded to fp32: relative error at most 2^-24 per term
        assert abs(tree_loss - path_loss) <= 2.0 ** -23 * float(np.dot(np.abs(lam), np.abs(loss))) + 1e-9
