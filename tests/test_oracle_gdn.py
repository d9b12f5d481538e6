"""Pins for the GDN tree state routing oracle (eq. 10, App. A.2), CPU only.

- The pages' chunk algorithm (within-chunk WY correction by a triangular
  solve, then the cross-chunk term) equals the token recurrence: two different
  computations of the gated delta rule.
- Closed forms: beta = 0 leaves only decay (o_t = exp(sum g) q_t^T S0); with no
  decay, beta = 1 and orthonormal keys the state is an exact key-value memory
  (writing v under key e_i replaces row i; querying e_i returns it).
- The pages' claim: with tree routing every token's output equals that of a
  standalone run of its root-to-leaf path laid out on its own; sequential
  routing (the chunk before in DFS order) breaks it on a branching trie.
"""
import numpy as np
import pytest
import torch

from oracle import gdn as GD
from oracle import trie as T


def _draw(N, hk, hv, Dk, Dv, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.nn.functional.normalize(torch.randn(N, hk, Dk, generator=g, dtype=torch.float64), dim=-1)
    k = torch.nn.functional.normalize(torch.randn(N, hk, Dk, generator=g, dtype=torch.float64), dim=-1)
    v = torch.randn(N, hv, Dv, generator=g, dtype=torch.float64)
    gg = -0.5 * torch.rand(N, hv, generator=g, dtype=torch.float64)
    beta = torch.rand(N, hv, generator=g, dtype=torch.float64)
    S0 = torch.randn(hv, Dk, Dv, generator=g, dtype=torch.float64) * 0.3
    return q, k, v, gg, beta, S0


@pytest.mark.parametrize("L", [1, 2, 7, 33])
def test_chunk_form_equals_the_recurrence(L):
    q, k, v, g, beta, S0 = _draw(L, 1, 1, 16, 8, L)
    o1, s1 = GD.recurrence(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S0[0])
    o2, s2 = GD.chunk_form(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S0[0])
    assert torch.allclose(o1, o2, atol=1e-12) and torch.allclose(s1, s2, atol=1e-12)


def test_closed_forms():
    L, Dk, Dv = 9, 8, 5
    q, k, v, g, _, S0 = _draw(L, 1, 1, Dk, Dv, 3)
    o, S = GD.recurrence(q[:, 0], k[:, 0], v[:, 0], g[:, 0], torch.zeros(L, dtype=torch.float64), S0[0])
    decay = torch.exp(torch.cumsum(g[:, 0], 0))
    assert torch.allclose(o, decay[:, None] * (q[:, 0] @ S0[0]), atol=1e-12)
    assert torch.allclose(S, decay[-1] * S0[0], atol=1e-12)
    # key-value memory: keys e_0, e_3, e_0 (overwrite), no decay, beta 1
    keys = torch.zeros(3, Dk, dtype=torch.float64)
    keys[0, 0] = keys[1, 3] = keys[2, 0] = 1.0
    vals = torch.randn(3, Dv, dtype=torch.float64)
    z = torch.zeros(3, dtype=torch.float64)
    _, S = GD.recurrence(keys, keys, vals, z, torch.ones(3, dtype=torch.float64),
                         torch.zeros(Dk, Dv, dtype=torch.float64))
    assert torch.allclose(S[0], vals[2]) and torch.allclose(S[3], vals[1])
    assert torch.count_nonzero(S[[1, 2, 4, 5, 6, 7]]) == 0


def _forest(seed):
    rng = np.random.default_rng(seed)
    S = int(rng.integers(2, 10))
    parents = [-1] + [int(rng.integers(-1, s)) if rng.random() < 0.15 else int(rng.integers(0, s))
                      for s in range(1, S)]
    lengths = [int(x) for x in rng.integers(1, 7, S)]
    return parents, lengths


@pytest.mark.parametrize("seed", range(8))
def test_tree_routing_equals_standalone_paths(seed):
    parents, lengths = _forest(seed)
    N = sum(lengths)
    hk, hv, Dk, Dv = 2, 4, 8, 6
    q, k, v, g, beta, S0 = _draw(N, hk, hv, Dk, Dv, seed)
    o, S_end = GD.tree_forward(q, k, v, g, beta, parents, lengths, S0)
    o2, S_end2 = GD.tree_forward(q, k, v, g, beta, parents, lengths, S0, step="chunk")
    assert torch.allclose(o, o2, atol=1e-11) and torch.allclose(S_end, S_end2, atol=1e-11)
    _, seg_start = T.dfs_serialize(parents, lengths)
    for leaf, ids in T.base_serialization(parents, lengths):
        idx = torch.as_tensor(ids)
        for h in range(hv):
            op, sp = GD.recurrence(q[idx, h // 2], k[idx, h // 2], v[idx, h], g[idx, h], beta[idx, h], S0[h])
            assert torch.allclose(op, o[idx, h], atol=1e-12)
            assert torch.allclose(sp, S_end[leaf, h], atol=1e-12)


def test_sequential_routing_differs_on_a_branching_trie():
    parents, lengths = [-1, 0, 0], [3, 2, 2]
    N = 7
    q, k, v, g, beta, S0 = _draw(N, 1, 1, 4, 3, 0)
    o_tree, _ = GD.tree_forward(q, k, v, g, beta, parents, lengths, S0)
    o_seq, _ = GD.recurrence(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S0[0])
    assert torch.allclose(o_tree[:5, 0], o_seq[:5])  # root and first child: same context
    assert not torch.allclose(o_tree[5:, 0], o_seq[5:])  # the second child must not see the first
