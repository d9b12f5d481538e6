"""GPU parity of partition-gateway attention (App. B.2-B.5) through the C-ABI.

Each piece of a partitioned trie runs with its gateway (keys and values of
earlier pieces, visible or hidden per App. B.3) and is compared with the fp64
gateway oracle; at full size, sampled rows and keys are compared with the
oracle and, at every row and key, the pieces together are compared with one
whole-trie run of the library (outputs equal; each token's key and value
gradients -- its own piece's plus those accumulated in fp32 through every
gateway that holds it -- add up to the whole trie's). Tolerances as the other
bf16 parity tests: max-abs 2e-2, mean-abs 2e-3, plus bf16 storage rounding for
bf16-stored outputs.
"""
import numpy as np
import pytest
import torch

import treegen
import tree_packed_attention_gb300 as tpa
from oracle import gateway as GW
from partition_util import cut_forest, pieces, to_np

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN = 2e-2, 2e-3


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _check(name, got, ref, store_bf16=False):
    d = (got.double().cpu() - ref).abs()
    bound = BF16_MAX + (2.0 ** -8 * ref.abs() if store_bf16 else 0.0)
    worst = float((d - bound).max()) if d.numel() else 0.0
    assert worst <= 0, f"{name}: error exceeds bound by {worst:.3g} (max {float(d.max()):.3g})"
    if d.numel():
        mean_bound = BF16_MEAN + (2.0 ** -9 * float(ref.abs().mean()) if store_bf16 else 0.0)
        assert float(d.mean()) <= mean_bound, f"{name}: mean abs err {float(d.mean()):.3g}"


def _run_piece(X, q, k, v, do, acc_k=None, acc_v=None):
    """GPU forward + backward of one piece with its gateway (fp32 gradients)."""
    tok, gw = to_np(X["tokens"]), to_np(X["gw"])
    plan = tpa.tree_plan_build_partition(X["parents"], X["lengths"], X["vis"])
    qd, kd, vd, dod = (x[tok].contiguous().cuda() for x in (q, k, v, do))
    pkd, pvd = (x[gw].contiguous().cuda() for x in (k, v))
    o, lse = tpa.tree_attn_fwd_gateway(plan, qd, kd, vd, pkd, pvd)
    dq, dk, dv, ak, av = tpa.tree_attn_bwd_gateway(plan, dod, qd, kd, vd, pkd, pvd, o, lse, acc_k, acc_v,
                                                   grad_dtype=torch.float32)
    tpa.tree_status_sync()
    return (o, lse, dq, dk, dv, ak, av), (qd, kd, vd, pkd, pvd, dod, plan)


def _small_cases():
    rng = np.random.default_rng(21)
    out = [([-1, 0, 1, 1, 3, 4, 4, 6], [140, 60, 90, 129, 200, 70, 130, 150],
            [0, 0, 0, 0, 4, 4, 4, 7])]
    for _ in range(3):
        S = int(rng.integers(4, 12))
        parents = [-1] + [int(rng.integers(0, s)) for s in range(1, S)]
        lengths = [int(x) for x in rng.integers(20, 260, S)]
        out.append((parents, lengths, cut_forest(rng, parents, lengths)))
    return out


@pytest.mark.parametrize("case", range(4))
def test_gateway_pieces_match_the_oracle(case):
    _need_gpu()
    parents, lengths, part = _small_cases()[case]
    N = sum(lengths)
    hq, hkv, D = 4, 2, 128
    q, k, v, do = treegen.draw_tensors(N, hq, hkv, D, "bf16", seed=case)
    for X in pieces(parents, lengths, part):
        P = len(X["gw"])
        g = torch.Generator().manual_seed(P)
        init_k = torch.randn(P, hkv, D, generator=g)
        init_v = torch.randn(P, hkv, D, generator=g)
        (o, lse, dq, dk, dv, ak, av), _ = _run_piece(X, q, k, v, do, init_k.cuda(), init_v.cuda())
        tok, gw = to_np(X["tokens"]), to_np(X["gw"])
        args = (q[tok], k[tok], v[tok], k[gw], v[gw])
        ro, rlse = GW.forward_dense(*args, X["parents"], X["lengths"], X["vis"])
        rdq, rdk, rdv, rpk, rpv = GW.backward_dense(*args, do[tok], X["parents"], X["lengths"], X["vis"])
        _check("o", o, ro, store_bf16=True)
        _check("lse", lse, rlse)
        for name, got, ref in (("dq", dq, rdq), ("dk", dk, rdk), ("dv", dv, rdv)):
            _check(name, got, ref)
        # the gateway gradients were added to the accumulators
        _check("past dk", ak.cpu() - init_k, rpk)
        _check("past dv", av.cpu() - init_v, rpv)


def test_gateway_without_past_keys_is_tree_attention_and_repeats():
    _need_gpu()
    parents, lengths = treegen.grpo_tree(2, prompt=200, n_leaves=3, lo=60, hi=150)
    N = int(np.sum(lengths))
    q, k, v, do = (x.cuda() for x in treegen.draw_tensors(N, 4, 2, 128, "bf16", 5))
    plain = tpa.tree_plan_build(parents, lengths)
    part = tpa.tree_plan_build_partition(parents, lengths, [])
    o1, l1 = tpa.tree_attn_fwd(plain, q, k, v)
    e = torch.zeros(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    o2, l2 = tpa.tree_attn_fwd_gateway(part, q, k, v, e, e)
    g1 = tpa.tree_attn_bwd(plain, do, q, k, v, o1, l1)
    g2 = tpa.tree_attn_bwd_gateway(part, do, q, k, v, e, e, o2, l2)
    tpa.tree_status_sync()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for a, b in zip(g1, g2[:3]):
        assert torch.equal(a, b)
    # with a gateway: two runs give the same bits, NaN-prefilled outputs all written
    parents, lengths, part_of = _small_cases()[0]
    Nf = sum(lengths)
    q, k, v, do = treegen.draw_tensors(Nf, 4, 2, 128, "bf16", 7)
    X = pieces(parents, lengths, part_of)[2]
    runs = []
    for _ in range(2):
        res, _ = _run_piece(X, q, k, v, do)
        for t in res:
            assert torch.isfinite(t).all()
        runs.append(res)
    for a, b in zip(*runs):
        assert torch.equal(a, b)


def test_agentic_trie_partitioned_at_16384_tokens():
    """Workload 4 (64k tokens, depth 6, 16 heads) cut into partitions of at
    most 16,384 tokens by the planner: every piece with its gateway against
    one whole-trie run, and sampled rows and keys of the pieces against the
    oracle."""
    _need_gpu()
    w = treegen.workload(4)
    N, hq, hkv, D = w.num_tokens, w.hq, w.hkv, w.head_dim
    q, k, v, do = treegen.draw_tensors(N, hq, hkv, D, w.dtype, 0)
    r = tpa.tree_partition(tpa.tree_plan_build(w.parents, w.lengths), 16384)
    part = [int(x) for x in r["part_of_segment"]]
    Xs = pieces(w.parents, w.lengths, part)
    assert len(Xs) == r["num_parts"] > 1
    full = tpa.tree_plan_build(w.parents, w.lengths)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o_full, lse_full = tpa.tree_attn_fwd(full, qd, kd, vd)
    dq_full, dk_full, dv_full = tpa.tree_attn_bwd(full, dod, qd, kd, vd, o_full, lse_full,
                                                  grad_dtype=torch.float32)
    dk_sum = torch.zeros(N, hkv, D, device="cuda")
    dv_sum = torch.zeros(N, hkv, D, device="cuda")
    rng = np.random.default_rng(4)
    checked = 0
    for X in Xs:
        (o, lse, dq, dk, dv, ak, av), _ = _run_piece(X, q, k, v, do)
        tok = torch.as_tensor(to_np(X["tokens"]), device="cuda")
        gw = torch.as_tensor(to_np(X["gw"]), dtype=torch.long, device="cuda")
        # the pieces against the whole-trie run (both on the GPU), every row
        _check("o vs whole", o, o_full[tok].double().cpu(), store_bf16=True)
        _check("lse vs whole", lse, lse_full[:, tok].double().cpu())
        _check("dq vs whole", dq, dq_full[tok].double().cpu())
        dk_sum[tok] += dk
        dv_sum[tok] += dv
        if len(X["gw"]):
            dk_sum.index_add_(0, gw, ak)
            dv_sum.index_add_(0, gw, av)
        # sampled rows and keys of the larger child pieces against the oracle
        if len(X["gw"]) and checked < 2 and len(X["tokens"]) > 2000:
            checked += 1
            n = len(X["tokens"])
            rows = sorted(set([0, n - 1] + rng.integers(0, n, 8).tolist()))
            tk, gk = to_np(X["tokens"]), to_np(X["gw"])
            args = (q[tk], k[tk], v[tk], k[gk], v[gk])
            ro, rlse = GW.forward_rows(*args, X["parents"], X["lengths"], X["vis"], rows)
            _check("o rows", o[rows], ro, store_bf16=True)
            _check("lse rows", lse[:, rows], rlse)
            rdq = GW.backward_rows(*args, do[tk], X["parents"], X["lengths"], X["vis"], rows)
            _check("dq rows", dq[rows], rdq)
            keys = sorted(set([n - 1, n - 2] + rng.integers(max(0, n - 60), n, 2).tolist()))
            rdk, rdv = GW.backward_own_keys(*args, do[tk], X["parents"], X["lengths"], X["vis"], keys)
            _check("dk keys", dk[keys], rdk)
            _check("dv keys", dv[keys], rdv)
    assert checked >= 1
    _check("dk summed over pieces vs whole", dk_sum, dk_full.double().cpu())
    _check("dv summed over pieces vs whole", dv_sum, dv_full.double().cpu())


def test_rope_on_pieces_equals_rope_on_the_whole_trie():
    """App. B.4 eq. 17: with the planner's pos_offset, RoPE applied to each
    piece of workload 4 (cut at 16,384 tokens) gives bit for bit what RoPE on
    the whole trie gives for the same tokens (same position ids, same kernel)."""
    _need_gpu()
    w = treegen.workload(4)
    N = w.num_tokens
    full = tpa.tree_plan_build(w.parents, w.lengths)
    r = tpa.tree_partition(full, 16384)
    Xs = pieces(w.parents, w.lengths, [int(x) for x in r["part_of_segment"]])
    x = treegen.draw_tensors(N, w.hq, w.hkv, w.head_dim, w.dtype, 3)[0].cuda()
    whole = tpa.tree_rope(full, x.clone())
    for i, X in enumerate(Xs):
        plan = tpa.tree_plan_build_partition(X["parents"], X["lengths"], X["vis"],
                                             int(r["pos_offset"][i]))
        tok = torch.as_tensor(to_np(X["tokens"]), device="cuda")
        got = tpa.tree_rope(plan, x[tok].contiguous())
        assert torch.equal(got, whole[tok]), i
        if i and r["pos_offset"][i] > 0:  # without the offset the rotation differs
            plain = tpa.tree_plan_build_partition(X["parents"], X["lengths"], X["vis"])
            assert not torch.equal(tpa.tree_rope(plain, x[tok].contiguous()), whole[tok])
    tpa.tree_status_sync()
