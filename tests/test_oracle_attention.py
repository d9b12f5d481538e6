"""Pins of the oracle's fp64 attention against independent routes.

Tree Training (arXiv 2511.00413) §3.1 eq. 6 (forward equivalence with every
per-path run), eq. 5 (gradient equivalence of the g_t/K-weighted tree loss
with the sep-avg loss of eq. 1), and the chain special case (ordinary causal
attention). Library routes: torch SDPA, torch.autograd, gradcheck.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import treegen
from oracle import attention as A
from oracle import mask as M
from oracle import trie as T


def _sdpa_path(q, k, v, ids, scale):
    """Plain causal attention over one path (token ids in path order), fp64, via SDPA."""
    hq, hkv = q.shape[1], k.shape[1]
    G = hq // hkv
    qq = q[ids].permute(1, 0, 2)                      # [hq, L, D]
    kk = k[ids].permute(1, 0, 2).repeat_interleave(G, 0)
    vv = v[ids].permute(1, 0, 2).repeat_interleave(G, 0)
    o = F.scaled_dot_product_attention(qq[None], kk[None], vv[None], is_causal=True, scale=scale)[0]
    s = scale * qq @ kk.transpose(1, 2)
    L = len(ids)
    s = s.masked_fill(torch.triu(torch.ones(L, L, dtype=torch.bool), 1), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)                  # [hq, L]
    return o.permute(1, 0, 2), lse


def _inputs(p, L, hq, hkv, D, seed):
    N = int(np.sum(L))
    q, k, v, do = treegen.draw_tensors(N, hq, hkv, D, "fp32", seed)
    return [x.double() for x in (q, k, v, do)]


def test_forward_equals_every_path_run_alone():
    """eq. 6: tree (o, lse) of every token equals its value on each path through it."""
    cases = [treegen.tiny_trie(0) + (1, 1, 16)]
    rng = np.random.default_rng(5)
    for _ in range(20):
        p, L = treegen.random_forest(rng, int(rng.integers(1, 9)), max_len=7, n_roots=int(rng.integers(1, 3)))
        cases.append((p, L, 4, 2, 8))
    for n, (p, L, hq, hkv, D) in enumerate(cases):
        q, k, v, _ = _inputs(p, L, hq, hkv, D, seed=n)
        scale = 0.37 if n % 2 else None
        o, lse = A.forward(q, k, v, p, L, scale)
        sc = A.default_scale(D) if scale is None else scale
        for _, ids in T.base_serialization(p, L):
            po, plse = _sdpa_path(q, k, v, ids, sc)
            assert torch.allclose(o[ids], po, atol=1e-12, rtol=0)
            assert torch.allclose(lse[:, ids], plse, atol=1e-12, rtol=0)


def test_chain_equals_causal_sdpa():
    p, L = treegen.chain(200)
    q, k, v, _ = _inputs(p, L, 4, 4, 16, seed=1)
    o, lse = A.forward(q, k, v, p, L)
    ref = F.scaled_dot_product_attention(q.permute(1, 0, 2)[None], k.permute(1, 0, 2)[None],
                                         v.permute(1, 0, 2)[None], is_causal=True)[0].permute(1, 0, 2)
    assert torch.allclose(o, ref, atol=1e-12, rtol=0)


def test_closed_forms():
    p, L = treegen.tiny_trie(3)
    N = int(L.sum())
    view = M.TrieView(p, L)
    q, k, v, _ = _inputs(p, L, 2, 1, 8, seed=2)
    # all value rows equal to c -> every output row is c
    c = torch.linspace(-1, 1, 8, dtype=torch.float64)
    o, _ = A.forward(q, k, c.expand(N, 1, 8).clone(), p, L)
    assert torch.allclose(o, c.expand(N, 2, 8), atol=1e-13)
    # q = 0 -> uniform weights: o_i = mean of visible v_j, lse_i = ln |vis(i)|
    o, lse = A.forward(torch.zeros_like(q), k, v, p, L)
    for i in range(N):
        vis = view.visible_keys(i)
        assert torch.allclose(o[i, 0], v[vis, 0].mean(0), atol=1e-13)
        assert lse[0, i].item() == pytest.approx(np.log(len(vis)), abs=1e-13)
    # the first token of a root sees only itself: o_0 = v_0, lse_0 = scale * q_0.k_0
    o, lse = A.forward(q, k, v, p, L)
    assert torch.allclose(o[0, 0], v[0, 0], atol=1e-14)
    assert lse[0, 0].item() == pytest.approx((q[0, 0] @ k[0, 0]).item() / np.sqrt(8), abs=1e-13)


def test_segment_form_equals_dense_form():
    rng = np.random.default_rng(6)
    for n in range(12):
        p, L = treegen.random_forest(rng, int(rng.integers(1, 10)), max_len=9, n_roots=int(rng.integers(1, 3)))
        q, k, v, do = _inputs(p, L, 4, 2, 8, seed=10 + n)
        mask = M.dense_mask_appendix(p, L)
        o1, l1 = A.forward(q, k, v, p, L)
        o2, l2 = A.forward_dense(q, k, v, mask)
        assert torch.allclose(o1, o2, atol=1e-13) and torch.allclose(l1, l2, atol=1e-13)
        g1 = A.backward(q, k, v, do, p, L)
        g2 = A.backward_dense(q, k, v, o2, l2, do, mask)
        for a, b in zip(g1, g2):
            assert torch.allclose(a, b, atol=1e-12)


def test_backward_equals_autograd_and_gradcheck():
    p, L = treegen.tiny_trie(0)
    mask = M.dense_mask_appendix(p, L)
    q, k, v, do = _inputs(p, L, 2, 1, 8, seed=7)
    qa, ka, va = (x.clone().requires_grad_(True) for x in (q, k, v))
    # autograd through a plain differentiable masked softmax
    m = torch.as_tensor(mask)

    def f(qx, kx, vx):
        outs = []
        for h in range(2):
            s = (qx[:, h] @ kx[:, 0].T) / np.sqrt(8)
            s = s.masked_fill(~m, float("-inf"))
            outs.append(torch.softmax(s, dim=1) @ vx[:, 0])
        return torch.stack(outs, 1)

    out = f(qa, ka, va)
    out.backward(do)
    o, lse = A.forward(q, k, v, p, L)
    dq, dk, dv = A.backward(q, k, v, do, p, L)
    assert torch.allclose(dq, qa.grad, atol=1e-12)
    assert torch.allclose(dk, ka.grad, atol=1e-12)
    assert torch.allclose(dv, va.grad, atol=1e-12)
    # finite differences on a smaller slice
    p2, L2 = [-1, 0, 0], [3, 2, 2]
    mask2 = torch.as_tensor(M.dense_mask_appendix(p2, L2))
    q2, k2, v2, _ = _inputs(p2, L2, 1, 1, 4, seed=8)

    def f2(qx, kx, vx):
        s = (qx[:, 0] @ kx[:, 0].T) / 2.0
        s = s.masked_fill(~mask2, float("-inf"))
        return torch.softmax(s, dim=1) @ vx[:, 0]

    assert torch.autograd.gradcheck(f2, tuple(x.clone().requires_grad_(True) for x in (q2, k2, v2)))
    do2 = torch.randn(7, 1, 4, dtype=torch.float64, generator=torch.Generator().manual_seed(1))
    qa, ka, va = (x.clone().requires_grad_(True) for x in (q2, k2, v2))
    f2(qa, ka, va).backward(do2[:, 0])
    g = A.backward(q2, k2, v2, do2, p2, L2)
    assert torch.allclose(g[0], qa.grad, atol=1e-12)
    assert torch.allclose(g[1], ka.grad, atol=1e-12)
    assert torch.allclose(g[2], va.grad, atol=1e-12)


def test_tree_gradient_equals_sep_avg_gradient():
    """eq. 5: with l_t = <c_t, o_t>, averaging per-path gradients over the K paths
    equals the tree backward with dO_t = (g_t/K) c_t."""
    rng = np.random.default_rng(9)
    cases = [treegen.tiny_trie(1)]
    for _ in range(6):
        cases.append(treegen.random_forest(rng, int(rng.integers(2, 9)), max_len=6, n_roots=1))
    for n, (p, L) in enumerate(cases):
        q, k, v, c = _inputs(p, L, 2, 1, 8, seed=20 + n)
        K = T.paths_per_trie(p)[0]
        w = torch.as_tensor(T.token_weights(p, L).astype(np.float64))
        gq = torch.zeros_like(q)
        gk = torch.zeros_like(k)
        gv = torch.zeros_like(v)
        for _, ids in T.base_serialization(p, L):
            qa, ka, va = (x[ids].clone().requires_grad_(True) for x in (q, k, v))
            G = 2
            qq = qa.permute(1, 0, 2)
            kk = ka.permute(1, 0, 2).repeat_interleave(G, 0)
            vv = va.permute(1, 0, 2).repeat_interleave(G, 0)
            o = F.scaled_dot_product_attention(qq[None], kk[None], vv[None], is_causal=True)[0].permute(1, 0, 2)
            (o * c[ids]).sum().div(K).backward()
            gq[ids] += qa.grad
            gk[ids] += ka.grad
            gv[ids] += va.grad
        # w is fp32-rounded g/K; these small K are exact in fp32 except for 1/3-like ratios
        do = c * w[:, None, None]
        dq, dk, dv = A.backward(q, k, v, do, p, L)
        assert torch.allclose(dq, gq, atol=1e-6, rtol=1e-6)
        assert torch.allclose(dk, gk, atol=1e-6, rtol=1e-6)
        assert torch.allclose(dv, gv, atol=1e-6, rtol=1e-6)


def test_sampled_rows_and_keys_match_full_backward():
    p, L = treegen.grpo_tree(0, prompt=40, n_leaves=5, lo=10, hi=30)
    q, k, v, do = _inputs(p, L, 4, 2, 8, seed=30)
    dq, dk, dv = A.backward(q, k, v, do, p, L)
    rows = [0, 17, 39, 40, 55, int(L.sum()) - 1]
    assert torch.allclose(A.backward_rows(q, k, v, do, p, L, rows), dq[rows], atol=1e-12)
    keys = [0, 39, 41, int(L.sum()) - 1]
    sk, sv = A.backward_keys(q, k, v, do, p, L, keys)
    assert torch.allclose(sk, dk[keys], atol=1e-12)
    assert torch.allclose(sv, dv[keys], atol=1e-12)
    o, lse = A.forward(q, k, v, p, L)
    o2, l2 = A.forward(q, k, v, p, L, rows=rows)
    assert torch.allclose(o2, o[rows]) and torch.allclose(l2, lse[:, rows])
