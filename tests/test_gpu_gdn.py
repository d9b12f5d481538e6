"""GPU parity of the GDN tree state routing (eq. 10, App. A.2) through the
C-ABI, against the fp64 oracle (token recurrence with tree routing).

Tolerance: fp32 arithmetic on the same (dtype-rounded) inputs; the state is
contractive for unit-norm keys and beta in (0, 1), so errors stay at fp32
rounding level: outputs and segment end states max-abs 2e-4 + 1e-4 |ref|;
bf16-stored outputs add the storage rounding 2^-8 |ref|.
"""
import numpy as np
import pytest
import torch

import treegen
import tree_packed_attention_gb300 as tpa
from oracle import gdn as GD

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _close(name, got, ref, bf16_store=False):
    d = (got.double().cpu() - ref).abs()
    bound = 2e-4 + 1e-4 * ref.abs() + (2.0 ** -8 * ref.abs() if bf16_store else 0.0)
    worst = float((d - bound).max())
    assert worst <= 0, f"{name}: max err {float(d.max()):.3g}"


def _run(parents, lengths, hk, hv, dtype, seed, with_state=True):
    N = int(np.sum(lengths))
    q, k, v, g, beta, s0 = treegen.draw_gdn(N, hk, hv, 128, dtype, seed, with_state)
    plan = tpa.tree_plan_build(parents, lengths)
    o, states = tpa.tree_gdn_fwd(plan, q.cuda(), k.cuda(), v.cuda(), g.cuda(), beta.cuda(),
                                 None if s0 is None else s0.cuda())
    tpa.tree_status_sync()
    return (q, k, v, g, beta, s0), o, states


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("seed", range(3))
def test_gdn_matches_the_oracle_on_tries_and_forests(dtype, seed):
    _need_gpu()
    rng = np.random.default_rng(seed)
    cases = [treegen.tiny_trie(seed), treegen.grpo_tree(seed, prompt=70, n_leaves=4, lo=10, hi=50),
             treegen.random_forest(rng, 12, 30, n_roots=3)]
    for n, (parents, lengths) in enumerate(cases):
        (q, k, v, g, beta, s0), o, states = _run(parents, lengths, 2, 4, dtype, seed * 7 + n,
                                                 with_state=n != 1)
        ro, rs = GD.tree_forward(q, k, v, g, beta, parents, lengths, s0)
        _close("o", o, ro, bf16_store=dtype == "bf16")
        _close("segment states", states, rs)


def test_gdn_repeats_and_equals_per_path_runs():
    """Bit-for-bit repeats; and every leaf's path, run on its own as a chain,
    gives the same outputs on its tokens (the pages' claim, on the GPU)."""
    _need_gpu()
    parents, lengths = treegen.grpo_tree(4, prompt=90, n_leaves=3, lo=20, hi=70)
    (q, k, v, g, beta, s0), o1, st1 = _run(parents, lengths, 1, 2, "fp32", 11)
    plan = tpa.tree_plan_build(parents, lengths)
    o2, st2 = tpa.tree_gdn_fwd(plan, q.cuda(), k.cuda(), v.cuda(), g.cuda(), beta.cuda(), s0.cuda())
    tpa.tree_status_sync()
    assert torch.equal(o1, o2) and torch.equal(st1, st2)
    from oracle import trie as T
    for leaf, ids in T.base_serialization(parents, lengths):
        idx = torch.as_tensor(ids)
        chain = tpa.tree_plan_build([-1], [len(ids)])
        oc, _ = tpa.tree_gdn_fwd(chain, q[idx].cuda(), k[idx].cuda(), v[idx].cuda(), g[idx].cuda(),
                                 beta[idx].cuda(), s0.cuda())
        tpa.tree_status_sync()
        assert torch.allclose(oc.cpu(), o1[idx.cuda()].cpu(), atol=1e-5, rtol=1e-5)


def test_gdn_on_the_grpo_workload_trie():
    """Workload 3's trie (22,637 tokens: a 2048-token prompt and 16 leaves),
    2 query/key heads and 4 value heads, bf16: every output and every segment
    end state against the oracle."""
    _need_gpu()
    w = treegen.workload(3)
    (q, k, v, g, beta, s0), o, states = _run(w.parents, w.lengths, 2, 4, "bf16", 3)
    ro, rs = GD.tree_forward(q, k, v, g, beta, w.parents, w.lengths, s0)
    _close("o", o, ro, bf16_store=True)
    _close("segment states", states, rs)


def test_gdn_reset_gates_and_many_branch_levels():
    """Gates that wipe the state (g = -30: one step's decay below 2^-40, so the
    kernel renormalises; g = -200: the decay underflows fp32 to 0, the state
    is reset to k delta^T), on a single token, a heap-shaped tree and a spine
    whose every segment branches (20 levels of branch points, one launch
    each), against the oracle in fp64."""
    _need_gpu()
    rng = np.random.default_rng(5)
    spine = [-1] + [2 * ((s - 1) // 2) for s in range(1, 41)]  # segment 2m: a leaf 2m+1 and 2m+2
    cases = [([-1], [1]),
             ([-1] + [(s - 1) // 2 for s in range(1, 31)], [int(x) for x in rng.integers(1, 4, 31)]),
             (spine, [int(x) for x in rng.integers(1, 6, len(spine))])]
    for n, (parents, lengths) in enumerate(cases):
        N = int(np.sum(lengths))
        q, k, v, g, beta, s0 = treegen.draw_gdn(N, 1, 2, 128, "fp32", 40 + n)
        pick = torch.as_tensor(rng.random((N, 2)))
        g = torch.where(pick < 0.15, torch.full_like(g, -30.0), g)
        g = torch.where(pick > 0.9, torch.full_like(g, -200.0), g)
        plan = tpa.tree_plan_build(parents, lengths)
        if n == 2:
            assert plan.info["gdn_levels"] >= 20
        o, states = tpa.tree_gdn_fwd(plan, q.cuda(), k.cuda(), v.cuda(), g.cuda(), beta.cuda(), s0.cuda())
        tpa.tree_status_sync()
        ro, rs = GD.tree_forward(q, k, v, g, beta, parents, lengths, s0)
        assert torch.isfinite(o).all() and torch.isfinite(states).all()
        _close("o", o, ro)
        _close("segment states", states, rs)
