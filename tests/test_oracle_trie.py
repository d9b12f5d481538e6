"""Pins of the oracle's trie layer against the pages' definitions.

Tree Training (arXiv 2511.00413): §3.1 eq. 1-4, eq. 7-8; §3.2 eq. 9 and
"Loss Weights"; §4.1 eq. 12 with the Figure 5 numbers.
"""
import json
import os

import numpy as np
import pytest

import treegen
from oracle import mask as M
from oracle import tiles as TL
from oracle import trie as T

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_por_printed_example():
    g = _gold("por_partition_example.json")
    assert abs(100 * T.por(g["n_tree"], g["n_base"]) - g["por_percent_printed"]) <= g["printed_precision"]


def test_hand_worked_trie():
    g = _gold("small_trie_hand.json")
    p, L = g["parents"], g["lengths"]
    order, seg_start = T.dfs_serialize(p, L)
    assert order == g["dfs_order"]
    assert seg_start == g["seg_start"]
    assert sorted(map(tuple, T.paths(p))) == sorted(map(tuple, g["paths"]))
    assert T.paths_through(p) == g["g"]
    assert T.paths_per_trie(p) == [g["K"]]
    assert T.token_segments(p, L) == g["token_seg"]
    assert T.position_ids(p, L) == g["pos_id"]
    assert T.token_weights(p, L).tolist() == g["weights"]
    dense = M.dense_mask_appendix(p, L)
    for i, vis in enumerate(g["visible"]):
        assert np.flatnonzero(dense[i]).tolist() == vis
    assert TL.key_end(p, L).tolist() == g["key_end"]
    assert int(dense.sum()) == g["visible_pairs"]
    assert M.TrieView(p, L).visible_count() == g["visible_pairs"]
    assert sum(len(ids) for _, ids in T.base_serialization(p, L)) == g["base_tokens"]
    assert T.trie_por(p, L) == pytest.approx(g["por"], abs=1e-15)


def _forests(n, seed=0, max_segments=14):
    rng = np.random.default_rng(seed)
    for t in range(n):
        S = int(rng.integers(1, max_segments + 1))
        yield treegen.random_forest(rng, S, max_len=int(rng.integers(1, 9)),
                                    n_roots=int(rng.integers(1, 4)))


def test_dfs_visits_every_token_once_and_subtrees_are_contiguous():
    for p, L in _forests(200, seed=1):
        order, seg_start = T.dfs_serialize(p, L)
        assert sorted(order) == list(range(len(p)))
        tok = T.token_segments(p, L)
        assert len(tok) == int(np.sum(L))
        # each segment's tokens appear once, contiguously, at seg_start
        for s in range(len(p)):
            idx = [i for i, x in enumerate(tok) if x == s]
            assert idx == list(range(seg_start[s], seg_start[s] + int(L[s])))
        # pre-order: a parent precedes its children; a subtree is one token range
        for s in range(len(p)):
            if p[s] >= 0:
                assert seg_start[p[s]] < seg_start[s]
            desc = [d for d in range(len(p)) if s in T.ancestors(list(p), d)] + [s]
            toks = sorted(i for d in desc for i in range(seg_start[d], seg_start[d] + int(L[d])))
            assert toks == list(range(toks[0], toks[0] + len(toks)))
        # children in ascending id are visited in ascending id
        children, roots = T.children_of(list(p))
        assert [s for s in order if p[s] == -1] == roots
        for s in range(len(p)):
            assert [seg_start[c] for c in children[s]] == sorted(seg_start[c] for c in children[s])


def test_position_ids_equal_per_path_offsets():
    """eq. 9: every token gets the index it has in each per-path sequence (eq. 7)."""
    for p, L in _forests(150, seed=2):
        pos = T.position_ids(p, L)
        for _, ids in T.base_serialization(p, L):
            assert [pos[t] for t in ids] == list(range(len(ids)))


def test_siblings_share_position_ranges():
    p, L = [-1, 0, 0, 0], [5, 3, 4, 2]
    pos = T.position_ids(p, L)
    _, seg_start = T.dfs_serialize(p, L)
    for s in (1, 2, 3):
        assert pos[seg_start[s]] == 5


def test_g_counts_paths_and_loss_identity():
    """eq. 2-3: sum over paths of path tokens' losses == sum_t g_t l_t == K * L_tree."""
    rng = np.random.default_rng(3)
    for p, L in _forests(150, seed=3):
        if len(T.children_of(list(p))[1]) != 1:
            continue  # one trie: a single K
        N = int(np.sum(L))
        ell = rng.standard_normal(N)
        K = T.paths_per_trie(p)[0]
        sep_avg = sum(ell[ids].sum() for _, ids in T.base_serialization(p, L)) / K
        w = T.token_weights(p, L).astype(np.float64)
        assert float(np.dot(w, ell)) == pytest.approx(sep_avg, rel=1e-6, abs=1e-6)
        g = T.paths_through(list(p))
        tok = T.token_segments(p, L)
        assert sum(g[tok[t]] * ell[t] for t in range(N)) == pytest.approx(K * sep_avg, rel=1e-12, abs=1e-9)


def test_weight_sum_is_mean_path_length():
    for p, L in _forests(100, seed=4):
        _, trie_id = T.tries(list(p))
        K = T.paths_per_trie(list(p))
        w = T.token_weights(p, L).astype(np.float64)
        tok = T.token_segments(p, L)
        for r in range(len(K)):
            lens = [len(ids) for leaf, ids in T.base_serialization(p, L) if trie_id[leaf] == r]
            assert sum(w[t] for t in range(len(tok)) if trie_id[tok[t]] == r) == pytest.approx(
                sum(lens) / K[r], rel=1e-6)


def test_chain_weights_are_one_and_gk_exact():
    p, L = treegen.chain(37)
    assert T.token_weights(p, L).tolist() == [1.0] * 37
    # g/K formed in fp64 and rounded once equals the exact rational rounded to fp32
    from fractions import Fraction
    for g, K in [(1, 3), (2, 7), (5, 11), (1, 1000003), (999, 1000)]:
        exact = Fraction(g, K)
        f32 = np.float32(g / K)
        below = np.nextafter(f32, np.float32(-1))
        above = np.nextafter(f32, np.float32(2))
        assert abs(Fraction(float(f32)) - exact) <= abs(Fraction(float(below)) - exact)
        assert abs(Fraction(float(f32)) - exact) <= abs(Fraction(float(above)) - exact)


def test_invalid_inputs():
    with pytest.raises(T.TrieError) as e:
        T.validate([1, 0], [1, 1])
    assert e.value.kind == "cycle"
    with pytest.raises(T.TrieError) as e:
        T.validate([-1, 5], [1, 1])
    assert e.value.kind == "invalid"
    with pytest.raises(T.TrieError) as e:
        T.validate([0], [1])
    assert e.value.kind == "invalid"
    with pytest.raises(T.TrieError) as e:
        T.validate([-1, 0], [1, 0])
    assert e.value.kind == "empty"


def test_workload_generators_shapes():
    w1 = treegen.workload(1)
    assert w1.parents.tolist() == [-1, 0, 0, 1, 1, 2, 2]
    assert all(8 <= x <= 32 for x in w1.lengths)
    w2 = treegen.workload(2)
    assert w2.num_tokens == 4096
    w3 = treegen.workload(3)
    assert w3.lengths[0] == 2048 and len(w3.lengths) == 17
    assert all(512 <= x <= 2048 for x in w3.lengths[1:])
    w4 = treegen.workload(4)
    assert w4.num_tokens == 65536
    assert max(len(T.ancestors(list(w4.parents), s)) for s in range(len(w4.parents))) <= 5
    w5 = treegen.workload(5)
    assert w5.num_tokens == 131072
    roots = [s for s in range(len(w5.parents)) if w5.parents[s] == -1]
    assert len(roots) == 32
    p = list(w5.parents)
    sizes = {}
    for s in range(len(p)):
        r = T.root_of(p, s)
        sizes[r] = sizes.get(r, 0) + int(w5.lengths[s])
    assert all(2048 <= x <= 8192 for x in sizes.values())
