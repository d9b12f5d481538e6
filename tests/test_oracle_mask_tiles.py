"""Pins of the oracle's mask and tile map.

Tree Training (arXiv 2511.00413) §3.2 "Attention Mask" (j <= i and a common
root-to-leaf path) against App. A.1 (ancestor chunks in full, own chunk
causal), and the tile counts against brute force over the dense mask.
"""
import numpy as np

import treegen
from oracle import mask as M
from oracle import tiles as TL
from oracle import trie as T


def _forests(n, seed, max_segments=12, max_len=9):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        S = int(rng.integers(1, max_segments + 1))
        yield treegen.random_forest(rng, S, max_len=int(rng.integers(1, max_len + 1)),
                                    n_roots=int(rng.integers(1, 4)))


def test_two_mask_statements_agree():
    for p, L in _forests(200, seed=10):
        a = M.dense_mask_appendix(p, L)
        b = M.dense_mask_paths(p, L)
        assert np.array_equal(a, b)


def test_row_intervals_and_key_end_match_dense():
    for p, L in _forests(120, seed=11):
        dense = M.dense_mask_appendix(p, L)
        N = dense.shape[0]
        ke = TL.key_end(p, L)
        view = M.TrieView(p, L)
        for i in range(N):
            row = np.zeros(N, dtype=bool)
            for (c, d) in M.row_intervals(p, L, i):
                row[c:d] = True
            assert np.array_equal(row, dense[i])
            assert np.array_equal(np.flatnonzero(dense[i]), view.visible_keys(i))
        for j in range(N):
            seen = np.flatnonzero(dense[:, j])
            assert ke[j] == seen.max() + 1
            # key_end is the column form: rows j..key_end-1 see j, no others
            assert seen.tolist() == list(range(j, ke[j]))
        assert view.visible_count() == int(dense.sum())


def test_tile_map_matches_brute_force():
    for bm in (1, 3, 4, 8):
        for p, L in _forests(40, seed=20 + bm, max_segments=10, max_len=12):
            dense = M.dense_mask_appendix(p, L)
            N = dense.shape[0]
            f = TL.plan_fields(p, L, bm, bm)
            Tq = (N + bm - 1) // bm
            kinds = {}
            for qt in range(Tq):
                for kt in range(Tq):
                    blk = dense[qt * bm:(qt + 1) * bm, kt * bm:(kt + 1) * bm]
                    c = int(blk.sum())
                    if c:
                        kinds[(qt, kt)] = TL.FULL if c == bm * bm else TL.PARTIAL
            got = {}
            for qt in range(Tq):
                for e in range(f["qt_ptr"][qt], f["qt_ptr"][qt + 1]):
                    got[(qt, int(f["qt_kt"][e]))] = int(f["qt_kind"][e])
            assert got == kinds
            for qt in range(Tq):
                kts = f["qt_kt"][f["qt_ptr"][qt]:f["qt_ptr"][qt + 1]]
                assert list(kts) == sorted(kts)


def test_backward_ranges_are_contiguous():
    """Every q-tile between kt_qlo and kt_qhi sees the k-tile (the column union is one range)."""
    for bm in (2, 4, 8):
        for p, L in _forests(60, seed=30 + bm, max_segments=12, max_len=12):
            f = TL.plan_fields(p, L, bm, bm)
            Tq = len(f["qt_ptr"]) - 1
            nonempty = set()
            for qt in range(Tq):
                for e in range(f["qt_ptr"][qt], f["qt_ptr"][qt + 1]):
                    nonempty.add((qt, int(f["qt_kt"][e])))
            for kt in range(Tq):
                qs = sorted(qt for (qt, k) in nonempty if k == kt)
                assert qs == list(range(f["kt_qlo"][kt], f["kt_qhi"][kt]))


def test_orders_and_pair_lists():
    for p, L in _forests(60, seed=40, max_segments=12, max_len=20):
        f = TL.plan_fields(p, L, 4, 4)
        Tq = len(f["qt_ptr"]) - 1
        npairs = (Tq + 1) // 2
        assert f["fwd_order"].tolist() == list(range(Tq))[::-1]
        assert f["bwd_order"].tolist() == list(range(Tq))
        assert f["qp_order"].tolist() == list(range(npairs))[::-1]
        assert len(f["qp_ptr"]) == npairs + 1
        for pr in range(npairs):
            lst = f["qp_kt"][f["qp_ptr"][pr]:f["qp_ptr"][pr + 1]].tolist()
            kinds = f["qp_kind"][f["qp_ptr"][pr]:f["qp_ptr"][pr + 1]].tolist()
            for slot in (0, 1):
                qt = 2 * pr + slot
                mine = [kt for kt, kd in zip(lst, kinds) if (kd >> (2 * slot)) & 3]
                if qt < Tq:
                    exp = f["qt_kt"][f["qt_ptr"][qt]:f["qt_ptr"][qt + 1]].tolist()
                    assert mine == exp
                else:
                    assert mine == []
            assert lst == sorted(set(lst))


def test_chain_tiles_are_causal_blocks():
    p, L = treegen.chain(1000)
    f = TL.plan_fields(p, L, 128, 128)
    Tq = 8
    for qt in range(Tq):
        kts = f["qt_kt"][f["qt_ptr"][qt]:f["qt_ptr"][qt + 1]].tolist()
        kinds = f["qt_kind"][f["qt_ptr"][qt]:f["qt_ptr"][qt + 1]].tolist()
        assert kts == list(range(qt + 1))
        if qt < Tq - 1:
            assert kinds == [TL.FULL] * qt + [TL.PARTIAL]
        else:  # rows past N make the last q-tile partial everywhere
            assert kinds == [TL.PARTIAL] * (qt + 1)
    assert f["visible_pairs"] == 1000 * 1001 // 2
    assert f["kt_qhi"].tolist() == [8] * 8
