"""The partition planner (C-ABI, host) against brute force and the pages'
definitions (§3.3 "Partitioning"; App. B.2, B.4 eq. 17). CPU only."""
import json
import os

import numpy as np
import pytest

import treegen
import tree_packed_attention_gb300 as tpa
from oracle import partition as PO
from oracle import trie as T


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _random_forest(rng, S_max, len_max):
    S = int(rng.integers(1, S_max + 1))
    parents = [-1] + [int(rng.integers(-1, s)) for s in range(1, S)]
    lengths = [int(x) for x in rng.integers(1, len_max + 1, S)]
    return parents, lengths


def _check_against_oracle(parents, lengths, cap, exact_count):
    plan = tpa.tree_plan_build(parents, lengths)
    r = tpa.tree_partition(plan, cap)
    part = [int(x) for x in r["part_of_segment"]]
    assert PO.is_valid_partition(parents, lengths, cap, part)
    assert r["num_parts"] == len(set(part))
    if exact_count:
        assert r["num_parts"] == PO.min_partitions_bruteforce(parents, lengths, cap)
    rec = PO.partition_records(parents, lengths, part)
    pos = T.position_ids(parents, lengths)
    _, seg_start = T.dfs_serialize(parents, lengths)
    for i in range(r["num_parts"]):
        o = rec[i]
        assert r["root"][i] == o["root"] and r["parent"][i] == o["parent"], i
        assert r["tokens"][i] == o["tokens"] <= cap
        assert r["pos_offset"][i] == o["pos_offset"]  # eq. 17 as a recursion
        assert r["pos_offset"][i] == pos[seg_start[o["root"]]]  # eq. 9 of the root's first token
        assert r["past_len"][i] == o["past_len"]
        if o["parent"] >= 0:
            assert o["parent"] < i  # parents first
    assert r["peak_path_tokens"] == PO.peak_path_tokens(parents, lengths, part)
    return r


def test_fewest_partitions_equal_brute_force_on_small_forests():
    rng = np.random.default_rng(0)
    for _ in range(150):
        parents, lengths = _random_forest(rng, 12, 40)
        cap = int(rng.integers(max(lengths), max(lengths) * 4 + 1))
        _check_against_oracle(parents, lengths, cap, exact_count=True)


def test_worked_example_three_pieces():
    # root 10 tokens, two children of 5, each with two 3-token leaves; cap 15:
    # 32 tokens need at least 3 pieces, e.g. {root}, {1, 3, 4}, {2, 5, 6}
    parents, lengths = [-1, 0, 0, 1, 1, 2, 2], [10, 5, 5, 3, 3, 3, 3]
    r = _check_against_oracle(parents, lengths, 15, exact_count=True)
    assert r["num_parts"] == 3
    assert sorted(r["tokens"].tolist()) == [10, 11, 11]


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_workloads_are_partitioned_validly(index):
    w = treegen.workload(index)
    for cap in sorted({max(w.lengths), 4096, 16384, 1 << 20}):
        if cap < max(w.lengths):
            continue
        r = _check_against_oracle(w.parents, w.lengths, cap, exact_count=False)
        N = int(np.sum(w.lengths))
        assert r["num_parts"] >= max(-(-N // cap), len(T.tries(w.parents)[0]))


def test_a_cap_at_the_forest_size_keeps_one_partition_per_trie():
    w = treegen.workload(5)
    r = tpa.tree_partition(tpa.tree_plan_build(w.parents, w.lengths), 1 << 30)
    assert r["num_parts"] == len(T.tries(w.parents)[0]) == 32
    assert (r["parent"] == -1).all() and (r["past_len"] == 0).all() and (r["pos_offset"] == 0).all()


def test_caps_below_a_segment_are_rejected():
    plan = tpa.tree_plan_build([-1, 0], [10, 30])
    with pytest.raises(tpa.TreeAttnError) as e:
        tpa.tree_partition(plan, 29)
    assert e.value.status == 5 and "segment 1" in str(e.value)
    with pytest.raises(tpa.TreeAttnError) as e:
        tpa.tree_partition(plan, 0)
    assert e.value.status == 1
    r = tpa.tree_partition(tpa.tree_plan_build(np.zeros(0, np.int32), np.zeros(0, np.int32)), 5)
    assert r["num_parts"] == 0 and r["peak_path_tokens"] == 0


def test_hand_worked_gateway_example():
    """App. B.2-B.4 worked by hand on a three-level chain of partitions whose
    gateways hold a non-ancestor sibling (the App. B.3 case)."""
    with open(os.path.join(GOLDEN, "partition_gateway_example.json")) as f:
        g = json.load(f)
    parents, lengths, cap = g["parents"], g["lengths"], g["cap"]
    assert PO.min_partitions_bruteforce(parents, lengths, cap) == g["num_parts"]
    part = g["part_of_segment"]
    assert PO.is_valid_partition(parents, lengths, cap, part)
    rec = PO.partition_records(parents, lengths, part)
    for i in range(g["num_parts"]):
        for key in ("root", "parent", "tokens", "past_len", "pos_offset"):
            assert rec[i][key] == g[key][i], (key, i)
    assert PO.peak_path_tokens(parents, lengths, part) == g["peak_path_tokens"]
    r = tpa.tree_partition(tpa.tree_plan_build(parents, lengths), cap)
    assert r["part_of_segment"].tolist() == part
    for key in ("root", "parent", "tokens", "past_len", "pos_offset"):
        assert r[key].tolist() == g[key], key
    assert r["peak_path_tokens"] == g["peak_path_tokens"]


def _gateway_len_by_tokens(parents, lengths, part):
    """App. B.2 counted token by token in the global DFS sequence: the gateway
    of piece C holds, for every piece A above C on its chain, A's tokens that
    come before the end of A's cut node (the deepest segment of A on the way
    down to C's root). A piece is a connected subtree, so the global DFS order
    restricted to A is A's own DFS order."""
    order, seg_start = T.dfs_serialize(parents, lengths)
    seg = T.token_segments(parents, lengths)
    out = {}
    for c in set(part):
        top = next(s for s in order if part[s] == c)
        chain = T.ancestors(parents, top)  # root first
        total = 0
        for a in {part[s] for s in chain}:
            cut = [s for s in chain if part[s] == a][-1]
            end = seg_start[cut] + lengths[cut]
            total += sum(1 for t in range(end) if part[seg[t]] == a)
        out[c] = total
    return out


def _peak_by_tokens(parents, lengths, part):
    """Peak partition tokens along a path, from each path's token list (eq. 7
    layout): the pieces its tokens fall in, summed by piece size."""
    seg = T.token_segments(parents, lengths)
    size = {}
    for t in range(len(seg)):
        size[part[seg[t]]] = size.get(part[seg[t]], 0) + 1
    best = 0
    for _, ids in T.base_serialization(parents, lengths):
        best = max(best, sum(size[p] for p in {part[seg[t]] for t in ids}))
    return best


def test_gateway_lengths_and_peak_by_token_counting():
    rng = np.random.default_rng(7)
    cases = [treegen.workload(1, s) for s in range(3)]
    forests = [_random_forest(rng, 14, 30) for _ in range(80)]
    for parents, lengths in [(w.parents, w.lengths) for w in cases] + forests:
        parents = [int(x) for x in parents]
        lengths = [int(x) for x in lengths]
        for cap in (max(lengths), max(lengths) * 2, sum(lengths)):
            r = tpa.tree_partition(tpa.tree_plan_build(parents, lengths), cap)
            part = [int(x) for x in r["part_of_segment"]]
            rec = PO.partition_records(parents, lengths, part)
            by_tokens = _gateway_len_by_tokens(parents, lengths, part)
            for i in range(r["num_parts"]):
                assert rec[i]["past_len"] == by_tokens[i] == r["past_len"][i]
            peak = _peak_by_tokens(parents, lengths, part)
            assert PO.peak_path_tokens(parents, lengths, part) == peak == r["peak_path_tokens"]


def test_bench_gateway_pieces_follow_the_definition():
    """bench.py builds the pieces it times (--op gateway) from the library's plan
    fields; they must be the pieces of App. B.2-B.3 as the test helper builds
    them from the definition, and their visible pairs, own plus gateway, must
    add up to the whole trie's."""
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    from partition_util import pieces
    rng = np.random.default_rng(31)
    for _ in range(12):
        S = int(rng.integers(2, 14))
        parents = [-1] + [int(rng.integers(0, s)) for s in range(1, S)]
        lengths = [int(x) for x in rng.integers(1, 90, S)]
        whole = tpa.tree_plan_build(parents, lengths)
        r = tpa.tree_partition(whole, max(max(lengths), sum(lengths) // 3))
        part = [int(x) for x in r["part_of_segment"]]
        got = bench.gateway_pieces(parents, lengths, part, whole)
        ref = pieces(parents, lengths, part)
        assert len(got) == len(ref) == r["num_parts"]
        pairs = 0
        for X, Y in zip(got, ref):
            for key in ("parents", "lengths", "tokens", "gw", "vis"):
                assert list(X[key]) == list(Y[key]), key
            plan = tpa.tree_plan_build_partition(X["parents"], X["lengths"], X["vis"])
            pairs += plan.info["visible_pairs"] + len(X["tokens"]) * plan.info["past_visible"]
        assert pairs == whole.info["visible_pairs"]
