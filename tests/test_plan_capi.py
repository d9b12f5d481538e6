"""The C++ plan builder (through the C-ABI) against the oracle, bit for bit, on CPU.

Also: the library loads and exports every symbol the public header declares,
error statuses for invalid tries, and the g/K weights.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import treegen
import tree_packed_attention_gb300 as tpa
from oracle import tiles as TL
from oracle import trie as T

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_library_exports_every_declared_symbol():
    with open(os.path.join(ROOT, "include", "treeattn.h")) as f:
        header = f.read()
    declared = set(re.findall(r"^\S[^\n(]*?\b(tree_\w+)\(", header, flags=re.M))
    assert declared == set(tpa.EXPORTS)
    lib = ctypes.CDLL(tpa.LIB_PATH)
    for name in declared:
        assert getattr(lib, name) is not None


def _assert_plan_equal(p, L):
    plan = tpa.tree_plan_build(p, L)
    ref = TL.plan_fields(p, L, 128, 128)
    got = plan.fields()
    for name in tpa.FIELDS:
        assert got[name].dtype == np.int32
        assert np.array_equal(got[name], ref[name]), name
    info = plan.info
    assert info["num_tokens"] == ref["num_tokens"]
    assert info["num_segments"] == ref["num_segments"]
    assert info["num_tries"] == ref["num_tries"]
    assert info["visible_pairs"] == ref["visible_pairs"]
    assert info["nnz_tiles"] == len(ref["qt_kt"])
    assert info["num_pairs"] == len(ref["qp_ptr"]) - 1
    w = tpa.tree_weights(plan)
    assert np.array_equal(w.view(np.uint32), T.token_weights(p, L).view(np.uint32))
    return plan


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_workload_plans_bit_exact(index):
    w = treegen.workload(index)
    _assert_plan_equal(w.parents, w.lengths)


def test_random_forests_bit_exact():
    rng = np.random.default_rng(100)
    for _ in range(60):
        S = int(rng.integers(1, 40))
        p, L = treegen.random_forest(rng, S, max_len=int(rng.integers(1, 300)),
                                     n_roots=int(rng.integers(1, 5)))
        _assert_plan_equal(p, L)


def test_degenerate_tries_bit_exact():
    cases = [
        ([-1], [1]),                                     # a single token
        ([-1], [128]),                                   # exactly one tile
        ([-1], [129]),                                   # one tile plus one row
        ([-1] + list(range(0, 299)), [1] * 300),         # deep chain of 1-token segments
        ([-1] + list(range(0, 99)), [127] * 100),        # deep chain of 127-token segments
        ([-1] + [0] * 1000, [3] + [1] * 1000),           # 1000-way fan-out
        ([3, 3, 3, -1], [5, 7, 9, 11]),                  # root listed after its children
        ([-1, -1, -1], [129, 127, 1]),                   # forest of chains around tile edges
    ]
    for p, L in cases:
        _assert_plan_equal(np.array(p), np.array(L))


def test_empty_plan():
    plan = tpa.tree_plan_build(np.zeros(0, np.int32), np.zeros(0, np.int32))
    assert plan.info["num_tokens"] == 0
    assert plan.field("cu_seqlens").tolist() == [0]
    assert tpa.tree_weights(plan).size == 0


@pytest.mark.parametrize("parents,lengths,status", [
    ([1, 0], [1, 1], "TREE_ERR_CYCLE"),
    ([-1, 2, 1], [1, 1, 1], "TREE_ERR_CYCLE"),
    ([-1, 5], [1, 1], "TREE_ERR_INVALID_ARG"),
    ([-2], [1], "TREE_ERR_INVALID_ARG"),
    ([0], [1], "TREE_ERR_INVALID_ARG"),
    ([-1, 0], [1, 0], "TREE_ERR_EMPTY_SEGMENT"),
    ([-1], [-3], "TREE_ERR_EMPTY_SEGMENT"),
    ([-1, 0, 0], [2**30, 2**30, 2**30], "TREE_ERR_OVERFLOW"),
])
def test_invalid_tries_are_rejected(parents, lengths, status):
    with pytest.raises(tpa.TreeAttnError) as e:
        tpa.tree_plan_build(parents, lengths)
    assert e.value.status_name == status
    if status != "TREE_ERR_OVERFLOW":
        kind = {"TREE_ERR_CYCLE": "cycle", "TREE_ERR_INVALID_ARG": "invalid",
                "TREE_ERR_EMPTY_SEGMENT": "empty"}[status]
        with pytest.raises(T.TrieError) as e2:
            T.validate(parents, lengths)
        assert e2.value.kind == kind


def test_field_size_mismatch_and_null_args():
    plan = tpa.tree_plan_build([-1, 0], [3, 4])
    buf = np.zeros(5, np.int32)
    st = tpa.lib.tree_plan_get(plan.handle, 0, buf.ctypes.data, 4)
    assert st == 1
    assert b"bytes" in tpa.lib.tree_last_error()
    h = ctypes.c_void_p()
    assert tpa.lib.tree_plan_build(None, None, 3, ctypes.byref(h)) == 1


def test_device_calls_without_device_copy_are_rejected():
    """Host-side validation runs before any launch (no GPU needed)."""
    # The plan has no device copy, so none of these calls could reach a launch
    # even if a check were skipped. Pointers are NULL wherever the case does
    # not test the pointers themselves.
    plan = tpa.tree_plan_build([-1], [8])
    nul = (None,) * 5  # q, k, v, o, lse
    # D = 96 is rejected before the device is touched
    st = tpa.lib.tree_attn_fwd(plan.handle, *nul, 1, 1, 96, 1, 0.0, None)
    assert st == 5
    st = tpa.lib.tree_attn_fwd(plan.handle, *nul, 3, 2, 128, 1, 0.0, None)
    assert st == 1
    st = tpa.lib.tree_attn_fwd(plan.handle, *nul, 1, 1, 128, 1, 0.0, None)
    assert st == 1 and b"NULL" in tpa.lib.tree_last_error()
    st = tpa.lib.tree_attn_fwd(plan.handle, 17, 16, 16, 16, 16, 1, 1, 128, 1, 0.0, None)
    assert st == 1  # misaligned pointer
    # each backward phase checks the pointers it uses
    args = (16, 16, 16, 16)  # dout, q, k, v
    st = tpa.lib.tree_attn_bwd_dq(plan.handle, *args, None, 16, 16, 2, 1, 128, 1, 1, 0.0, 16, 1 << 20, None)
    assert st == 1 and b"NULL" in tpa.lib.tree_last_error()  # o
    st = tpa.lib.tree_attn_bwd_dkdv(plan.handle, *args, 16, 16, None, 2, 1, 128, 1, 1, 0.0, 16, 1 << 20, None)
    assert st == 1 and b"NULL" in tpa.lib.tree_last_error()  # dv
    nul4 = (None,) * 4
    st = tpa.lib.tree_attn_bwd_dkdv(plan.handle, *nul4, None, None, None, 2, 1, 96, 1, 1, 0.0, None, 1 << 20, None)
    assert st == 5  # D = 96 unsupported for bf16
    st = tpa.lib.tree_attn_bwd_dq(plan.handle, *args, 16, 16, 16, 2, 1, 128, 1, 1, 0.0, 16, 4, None)
    assert st == 1 and b"workspace too small" in tpa.lib.tree_last_error()
    # bf16 workspace: lse*log2(e) and Delta, fp32 [hq, 128 * q-tiles] each
    assert tpa.lib.tree_attn_bwd_workspace_bytes(plan.handle, 2, 128, 1) == 2 * 2 * 128 * 4
    # fp32 workspace: Delta [hq, N], rounded up to 256 bytes
    assert tpa.lib.tree_attn_bwd_workspace_bytes(plan.handle, 2, 64, 0) == 256


def _dfs_leaf_count(parents, lengths):
    order, _ = T.dfs_serialize(parents, lengths)
    leaf_set = set(T.leaves(parents))
    return sum(1 for s in order if s in leaf_set)


@pytest.mark.parametrize("index,seed", [(1, 0), (3, 0), (4, 0), (5, 0), (1, 2)])
def test_path_weights_match_the_oracle(index, seed):
    w = treegen.workload(index, seed)
    plan = tpa.tree_plan_build(w.parents, w.lengths)
    nk = _dfs_leaf_count(w.parents, w.lengths)
    pw = np.random.default_rng(seed + 100).uniform(-1.0, 3.0, nk)
    got = tpa.tree_weights_paths(plan, pw)
    ref = T.path_weight_tokens(w.parents, w.lengths, pw)
    # same fp64 additions in the same order, one rounding to fp32
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_path_weights_of_random_forests_match_the_oracle():
    rng = np.random.default_rng(11)
    for _ in range(20):
        S = int(rng.integers(1, 40))
        parents = [-1] + [int(rng.integers(-1, s)) for s in range(1, S)]
        lengths = [int(x) for x in rng.integers(1, 300, S)]
        plan = tpa.tree_plan_build(parents, lengths)
        pw = rng.standard_normal(_dfs_leaf_count(parents, lengths))
        got = tpa.tree_weights_paths(plan, pw)
        assert np.array_equal(got.view(np.uint32), T.path_weight_tokens(parents, lengths, pw).view(np.uint32))


def test_path_weights_and_rope_validate_their_arguments():
    plan = tpa.tree_plan_build([-1, 0, 0], [4, 3, 5])  # two paths
    with pytest.raises(tpa.TreeAttnError) as e:
        tpa.tree_weights_paths(plan, [1.0, 2.0, 3.0])
    assert e.value.status == 1 and "2 paths" in str(e.value)
    with pytest.raises(tpa.TreeAttnError):
        tpa.tree_weights_paths(plan, [1.0, float("nan")])
    # tree_rope: checks that need no device (the last argument is the stream)
    lib = tpa.lib
    assert lib.tree_rope(None, None, 2, 64, 1, 10000.0, 0, 0, None) == 1
    assert lib.tree_rope(plan.handle, None, 2, 63, 1, 10000.0, 0, 0, None) == 5  # odd head_dim
    assert lib.tree_rope(plan.handle, None, 2, 130, 1, 10000.0, 0, 0, None) == 5  # above 128
    assert lib.tree_rope(plan.handle, None, 0, 64, 1, 10000.0, 0, 0, None) == 1  # heads
    assert lib.tree_rope(plan.handle, None, 2, 64, 7, 10000.0, 0, 0, None) == 1  # dtype
    assert lib.tree_rope(plan.handle, None, 2, 64, 1, 0.0, 0, 0, None) == 1  # base
    assert lib.tree_rope(plan.handle, None, 2, 64, 1, float("inf"), 0, 0, None) == 1
    assert lib.tree_rope(plan.handle, None, 2, 64, 1, 10000.0, 2, 0, None) == 1  # rotate_half
    assert lib.tree_rope(plan.handle, None, 2, 64, 1, 10000.0, 0, 3, None) == 1  # inverse
    # tree_rope_qk: a missing or overlapping second tensor is refused before any
    # device use (host buffers stand in for the tensors; the plan is not uploaded,
    # so a call that got past these checks would stop at TREE_ERR_NOT_ON_DEVICE)
    buf = np.zeros(plan.info["num_tokens"] * 4 * 64 + 64, dtype=np.float32)
    a0 = buf.ctypes.data
    assert lib.tree_rope_qk(plan.handle, a0, 2, None, 2, 64, 0, 10000.0, 0, 0, None) == 1
    assert lib.tree_rope_qk(plan.handle, a0, 2, a0 + 64, 2, 64, 0, 10000.0, 0, 0, None) == 1
    assert b"overlap" in lib.tree_last_error()
    assert lib.tree_rope_qk(plan.handle, a0, 2, a0, 0, 64, 0, 10000.0, 0, 0, None) == 1  # heads
    assert lib.tree_rope(plan.handle, None, 2, 64, 1, 10000.0, 0, 0, None) == 1  # NULL x
    assert lib.tree_rope(plan.handle, 20, 2, 64, 1, 10000.0, 0, 0, None) == 1  # misaligned


def test_conv_validates_its_arguments():
    plan = tpa.tree_plan_build([-1, 0], [5, 7])
    lib = tpa.lib
    assert lib.tree_conv_prepare(None, 4, None) == 1
    assert lib.tree_conv_prepare(plan.handle, 0, None) == 5  # kernel size out of range
    assert lib.tree_conv_prepare(plan.handle, 9, None) == 5
    # checks that need no device: channels, dtype, activation
    args = (None, None, None, None)  # x, weight, bias, y: rejected before they are read
    assert lib.tree_conv_fwd(None, *args, 8, 1, 1, None) == 1
    assert lib.tree_conv_fwd(plan.handle, *args, 12, 1, 1, None) == 5  # not a multiple of 8
    assert lib.tree_conv_fwd(plan.handle, *args, 8, 5, 1, None) == 1  # dtype
    assert lib.tree_conv_fwd(plan.handle, *args, 8, 1, 2, None) == 1  # activation
    assert lib.tree_conv_bwd_workspace_bytes(plan.handle, 8) == 0  # nothing prepared yet


def test_weighted_ce_host_checks():
    """Rejected before any device use: bad vocab, dtype, grad_scale, NULL pointers."""
    plan = tpa.tree_plan_build([-1, 0], [3, 2])
    L = tpa.lib.tree_weighted_ce
    assert L(plan.handle, None, None, None, None, 7, 1, 1.0, None, None, None) == 1
    assert b"multiple of 8" in tpa.lib.tree_last_error()
    assert L(plan.handle, None, None, None, None, 8, 9, 1.0, None, None, None) == 1
    assert L(plan.handle, None, None, None, None, 8, 1, float("inf"), None, None, None) == 1
    assert L(plan.handle, None, None, None, None, 8, 1, 1.0, None, None, None) == 1
    assert b"NULL" in tpa.lib.tree_last_error()
    assert L(None, None, None, None, None, 8, 1, 1.0, None, None, None) == 1


def test_gdn_levels_count_branch_points_on_paths():
    """The GDN forward launches once per level: 1 + the most segments with
    several children met on one root-to-leaf path (a chain of only children is
    one unit)."""
    rng = np.random.default_rng(5)
    cases = [([-1], [3]), ([-1, 0, 1, 2], [2, 2, 2, 2]), ([-1, 0, 0], [4, 1, 1]),
             ([-1, -1, 0, 0, 1], [1, 2, 3, 4, 5]), ([], [])]
    for _ in range(40):
        S = int(rng.integers(1, 30))
        parents = [-1] + [int(rng.integers(-1, s)) if rng.random() < 0.1 else int(rng.integers(0, s))
                          for s in range(1, S)]
        cases.append((parents, [int(x) for x in rng.integers(1, 9, S)]))
    for i in (1, 2, 3, 4, 5):
        w = treegen.workload(i)
        cases.append((w.parents.tolist(), w.lengths.tolist()))
    for parents, lengths in cases:
        S = len(parents)
        nchild = [0] * S
        for p in parents:
            if p >= 0:
                nchild[p] += 1
        best = 0
        for s in range(S):
            if nchild[s] == 0:  # a leaf: count the branch points above it
                n, a = 0, parents[s]
                while a >= 0:
                    n += nchild[a] >= 2
                    a = parents[a]
                best = max(best, n + 1)
        plan = tpa.tree_plan_build(parents, lengths)
        assert plan.info["gdn_levels"] == best, (parents, lengths)


def test_diagnostic_wait_checks_its_limit_before_any_launch():
    # outside [1e3, 1e10] ns: refused on the host, nothing launched
    for bad in (0, 999, -5, 10 ** 10 + 1):
        assert tpa.lib.tree_diag_wait_timeout(bad, None) == 1
        assert b"limit_ns" in tpa.lib.tree_last_error()
