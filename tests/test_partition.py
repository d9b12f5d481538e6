"""The partition planner (C-ABI, host) against brute force and the pages'
definitions (§3.3 "Partitioning"; App. B.2, B.4 eq. 17). CPU only."""
import numpy as np
import pytest

import treegen
import tree_packed_attention_gb300 as tpa
from oracle import partition as PO
from oracle import trie as T


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
