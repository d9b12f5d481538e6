"""Pins for the gateway attention oracle (App. B.2-B.5), CPU only.

The pin is the claim of App. B ("zero-overhead partition boundaries"): run
piece by piece, each child piece attending to its gateway under the
ancestor-aware bias, a partitioned trie gives the same outputs for every
token as the whole trie in one pass, and the gradients of each token's key
and value -- its own piece's plus those that arrive through every gateway
holding it -- add up to the whole trie's (B.6 chain rule). The whole-trie
side is the tree-attention oracle, itself pinned by per-path brute force.
"""
import numpy as np
import pytest
import torch

import treegen
import tree_packed_attention_gb300 as tpa
from oracle import attention as A
from oracle import gateway as GW
from oracle import mask as M
from oracle import partition as PT
from oracle import tiles as TL
from partition_util import cut_forest, pieces, to_np


def _draw(N, hq, hkv, D, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(N, hq, D, generator=g, dtype=torch.float64)
    k = torch.randn(N, hkv, D, generator=g, dtype=torch.float64)
    v = torch.randn(N, hkv, D, generator=g, dtype=torch.float64)
    do = torch.randn(N, hq, D, generator=g, dtype=torch.float64)
    return q, k, v, do


def _cases():
    rng = np.random.default_rng(3)
    out = []
    w = treegen.workload(1, 0)
    out.append((w.parents.tolist(), w.lengths.tolist(), [0, 0, 0, 1, 1, 2, 2]))  # no cut
    out.append(([-1, 0, 1, 1, 3, 4, 4, 6], [4, 3, 2, 5, 6, 3, 4, 11], [0, 0, 0, 0, 4, 4, 4, 7]))
    for _ in range(10):
        S = int(rng.integers(3, 14))
        parents = [-1] + [int(rng.integers(0, s)) for s in range(1, S)]
        lengths = [int(x) for x in rng.integers(1, 12, S)]
        out.append((parents, lengths, cut_forest(rng, parents, lengths)))
    return out


@pytest.mark.parametrize("case", range(12))
def test_partitioned_run_equals_the_whole_trie(case):
    parents, lengths, part = _cases()[case]
    N = sum(lengths)
    hq, hkv, D = 4, 2, 16
    q, k, v, do = _draw(N, hq, hkv, D, case)
    o_full, lse_full = A.forward(q, k, v, parents, lengths)
    dq_full, dk_full, dv_full = A.backward(q, k, v, do, parents, lengths)
    dk_sum = torch.zeros_like(k)
    dv_sum = torch.zeros_like(v)
    for X in pieces(parents, lengths, part):
        tok, gw = to_np(X["tokens"]), to_np(X["gw"])
        args = (q[tok], k[tok], v[tok], k[gw], v[gw])
        o, lse = GW.forward_dense(*args, X["parents"], X["lengths"], X["vis"])
        assert torch.allclose(o, o_full[tok], atol=1e-12)
        assert torch.allclose(lse, lse_full[:, tok], atol=1e-12)
        dq, dk, dv, dpk, dpv = GW.backward_dense(*args, do[tok], X["parents"], X["lengths"], X["vis"])
        assert torch.allclose(dq, dq_full[tok], atol=1e-11)
        dk_sum[tok] += dk
        dv_sum[tok] += dv
        dk_sum.index_add_(0, torch.as_tensor(gw, dtype=torch.long), dpk)
        dv_sum.index_add_(0, torch.as_tensor(gw, dtype=torch.long), dpv)
    assert torch.allclose(dk_sum, dk_full, atol=1e-11)
    assert torch.allclose(dv_sum, dv_full, atol=1e-11)


def test_row_and_key_forms_match_the_dense_form():
    parents, lengths, part = _cases()[1]
    N = sum(lengths)
    q, k, v, do = _draw(N, 4, 2, 16, 9)
    X = pieces(parents, lengths, part)[1]
    tok, gw = to_np(X["tokens"]), to_np(X["gw"])
    args = (q[tok], k[tok], v[tok], k[gw], v[gw])
    o, lse = GW.forward_dense(*args, X["parents"], X["lengths"], X["vis"])
    dq, dk, dv, _, _ = GW.backward_dense(*args, do[tok], X["parents"], X["lengths"], X["vis"])
    rows = list(range(len(tok)))
    o2, lse2 = GW.forward_rows(*args, X["parents"], X["lengths"], X["vis"], rows)
    assert torch.allclose(o2, o, atol=1e-12) and torch.allclose(lse2, lse, atol=1e-12)
    dq2 = GW.backward_rows(*args, do[tok], X["parents"], X["lengths"], X["vis"], rows)
    assert torch.allclose(dq2, dq, atol=1e-11)
    dk2, dv2 = GW.backward_own_keys(*args, do[tok], X["parents"], X["lengths"], X["vis"], rows)
    assert torch.allclose(dk2, dk, atol=1e-11) and torch.allclose(dv2, dv, atol=1e-11)


def test_hidden_gateway_keys_change_nothing_and_no_gateway_is_tree_attention():
    parents, lengths = [-1, 0, 0], [5, 3, 4]
    N = 12
    q, k, v, do = _draw(N, 2, 1, 8, 1)
    pk, pv = torch.randn(7, 1, 8, dtype=torch.float64), torch.randn(7, 1, 8, dtype=torch.float64)
    vis = [1, 0, 1, 1, 0, 0, 1]
    o1, l1 = GW.forward_dense(q, k, v, pk, pv, parents, lengths, vis)
    pk2, pv2 = pk.clone(), pv.clone()
    for j, x in enumerate(vis):
        if not x:
            pk2[j] += 5.0
            pv2[j] -= 3.0
    o2, l2 = GW.forward_dense(q, k, v, pk2, pv2, parents, lengths, vis)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    e = torch.zeros(0, 1, 8, dtype=torch.float64)
    o3, l3 = GW.forward_dense(q, k, v, e, e, parents, lengths, [])
    o4, l4 = A.forward(q, k, v, parents, lengths)
    assert torch.allclose(o3, o4, atol=1e-12) and torch.allclose(l3, l4, atol=1e-12)
    m = GW.combined_mask(parents, lengths, vis)
    assert m.shape == (N, 7 + N)
    assert (m[:, :7] == np.asarray(vis, bool)).all()
    assert (m[:, 7:] == M.dense_mask_appendix(parents, lengths)).all()


def test_partition_plans_match_the_oracle_bit_for_bit():
    """Gathered tiles with gateway tiles, GW_KEND and GW_KT of partition plans."""
    rng = np.random.default_rng(12)
    cases = _cases()
    w4 = treegen.workload(4)
    cases.append((w4.parents.tolist(), w4.lengths.tolist(), None))
    for parents, lengths, part in cases:
        if part is None:
            r = tpa.tree_partition(tpa.tree_plan_build(parents, lengths), 16384)
            part = [int(x) for x in r["part_of_segment"]]
        for X in pieces(parents, lengths, part)[:4]:
            plan = tpa.tree_plan_build_partition(X["parents"], X["lengths"], X["vis"])
            ref = TL.plan_fields(X["parents"], X["lengths"], past_visible=X["vis"])
            got = plan.fields()
            for name in tpa.FIELDS:
                assert np.array_equal(got[name], ref[name]), name
            assert plan.info["past_len"] == len(X["vis"])
            assert plan.info["past_visible"] == int(np.sum(X["vis"]))
    # random visibility patterns, including none visible and long runs
    for n in range(8):
        S = int(rng.integers(1, 8))
        parents = [-1] + [int(rng.integers(0, s)) for s in range(1, S)]
        lengths = [int(x) for x in rng.integers(1, 200, S)]
        vis = (rng.random(int(rng.integers(0, 700))) < [0.0, 0.3, 0.9, 1.0][n % 4]).tolist()
        plan = tpa.tree_plan_build_partition(parents, lengths, vis)
        ref = TL.plan_fields(parents, lengths, past_visible=vis)
        got = plan.fields()
        for name in tpa.FIELDS:
            assert np.array_equal(got[name], ref[name]), name


def test_partition_positions_continue_the_path_above():
    """App. B.4 eq. 17: a partition plan built with the planner's pos_offset
    gives every token the position id it has in the whole trie (eq. 9), so
    RoPE on the pieces equals RoPE on the whole trie; the oracle's plan fields
    agree."""
    cases = [(p, L, None) for p, L, _ in _cases()]
    w4 = treegen.workload(4)
    cases.append((w4.parents.tolist(), w4.lengths.tolist(), 16384))
    cases.append(([-1, 0, 1, 1, 0, 4], [40, 30, 20, 50, 10, 60], 64))
    for parents, lengths, cap in cases:
        whole = tpa.tree_plan_build(parents, lengths)
        cap = cap or max(max(lengths), sum(lengths) // 3)
        r = tpa.tree_partition(whole, cap)
        pos = whole.field("pos_id")
        got_pieces = pieces(parents, lengths, [int(x) for x in r["part_of_segment"]])
        assert len(got_pieces) == r["num_parts"]
        for i, X in enumerate(got_pieces):
            off = int(r["pos_offset"][i])
            _check_piece(X, off, pos)
            if r["parent"][i] < 0:
                assert off == 0
    # hand-made and random cuts, offsets from the eq. 17 recursion
    for parents, lengths, part in _cases():
        pos = tpa.tree_plan_build(parents, lengths).field("pos_id")
        rec = PT.partition_records(parents, lengths, part)
        for X in pieces(parents, lengths, part):
            _check_piece(X, rec[part[X["segs"][0]]]["pos_offset"], pos)


def _check_piece(X, off, pos):
    plan = tpa.tree_plan_build_partition(X["parents"], X["lengths"], X["vis"], off)
    assert np.array_equal(plan.field("pos_id"), pos[X["tokens"]])
    if len(X["tokens"]) < 5000:
        ref = TL.plan_fields(X["parents"], X["lengths"], past_visible=X["vis"], pos_offset=off)
        assert np.array_equal(plan.field("pos_id"), ref["pos_id"])


def test_partition_plan_arguments_are_checked():
    import ctypes
    h = ctypes.c_void_p()
    p = np.array([-1], np.int32)
    L = np.array([4], np.int32)
    assert tpa.lib.tree_plan_build_partition(p.ctypes.data, L.ctypes.data, 1, None, -1, 0,
                                             ctypes.byref(h)) == 1
    assert tpa.lib.tree_plan_build_partition(p.ctypes.data, L.ctypes.data, 1, None, 3, 0,
                                             ctypes.byref(h)) == 1
    assert tpa.lib.tree_plan_build_partition(p.ctypes.data, L.ctypes.data, 1, None, 0, -1,
                                             ctypes.byref(h)) == 1
    assert tpa.lib.tree_plan_build_partition(p.ctypes.data, L.ctypes.data, 1, None, 0,
                                             2 ** 31 - 4, ctypes.byref(h)) == 4  # overflow
    plan = tpa.tree_plan_build_partition([-1], [4], [1, 1])
    # a plan with a gateway is refused by the plain calls (before any device use)
    st = tpa.lib.tree_attn_fwd(plan.handle, None, None, None, None, None, 1, 1, 128, 1, 0.0, None)
    assert st == 1 and b"gateway" in tpa.lib.tree_last_error()
    # gateway attention is bf16 only
    st = tpa.lib.tree_attn_fwd_gateway(plan.handle, None, None, None, None, None, None, None, 1, 1,
                                       64, 0, 0.0, None)
    assert st == 5
