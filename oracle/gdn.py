"""Gated DeltaNet over a DFS-serialized trie with tree state routing (fp64,
torch CPU): test infrastructure only.

Tree Training (arXiv 2511.00413) §3.2 "SSM Layers (GDN)" eq. 10 and App. A.2.
Each tree node's token segment is one chunk, the unit of state transfer, and
a chunk starts from the final state of its parent chunk, not from the chunk
before it in DFS order (h_c^(0) = h_pi(c)^(end); a root starts from the
initial state, zero unless given).

The gated delta rule (Yang et al. 2025c), per head, state S of shape
[Dk, Dv], token t with query q_t, key k_t, value v_t, log decay g_t <= 0 and
write strength beta_t, as the pages' chunk form computes it (a chunk of one
token reduces to this):

    S_t = exp(g_t) S_{t-1} + k_t (beta_t (v_t - exp(g_t) S_{t-1}^T k_t))^T
    o_t = S_t^T q_t

Reading: the listing takes the query and key as given; the GDN layer's own
L2 normalisation of q and k and its 1/sqrt(Dk) query scale belong to the
caller (the inputs here are drawn already normalised). Heads: hv value heads
share hk = hv / G query/key heads (value head h reads q/k head h // G).

Functions:
  * ``recurrence`` -- the token recurrence on one sequence (the definition);
  * ``chunk_form`` -- the pages' chunked algorithm on one chunk (within-chunk
    WY correction by a unit lower-triangular solve, then the cross-chunk
    state term), a second computation of the same thing;
  * ``tree_forward`` -- eq. 10's routing over the trie with either step.
"""
from __future__ import annotations

import numpy as np
import torch

from . import trie as T


def _f64(x):
    return torch.as_tensor(x).detach().to(torch.float64)


def recurrence(q, k, v, g, beta, S0):
    """One sequence, one head. q, k [L, Dk], v [L, Dv], g, beta [L], S0 [Dk, Dv].
    Returns (o [L, Dv], S_end [Dk, Dv])."""
    q, k, v, g, beta, S = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta), _f64(S0).clone()
    o = torch.zeros(q.shape[0], v.shape[1], dtype=torch.float64)
    for t in range(q.shape[0]):
        a = torch.exp(g[t])
        delta = beta[t] * (v[t] - a * (S.T @ k[t]))
        S = a * S + torch.outer(k[t], delta)
        o[t] = S.T @ q[t]
    return o, S


def chunk_form(q, k, v, g, beta, S0):
    """The pages' chunk algorithm on one chunk of L tokens, one head.

    With G_i = sum_{s<=i} g_s (cumulative log decay inside the chunk):
      A[i, j]  = beta_i (k_i . k_j) exp(G_i - G_j) for j < i, else 0
      T        = (I + A)^-1                                   (unit lower triangular)
      U        = T (beta v)                 W = T (beta k exp(G))
      V'       = U - W S0                                     (the corrected values)
      o_i      = exp(G_i) q_i^T S0 + sum_{j<=i} (q_i . k_j) exp(G_i - G_j) V'_j
      S_end    = exp(G_L) S0 + sum_j exp(G_L - G_j) k_j V'_j^T
    """
    q, k, v, g, beta, S0 = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta), _f64(S0)
    L = q.shape[0]
    G = torch.cumsum(g, dim=0)
    D = G[:, None] - G[None, :]
    lower = torch.tril(torch.ones(L, L, dtype=torch.bool), diagonal=-1)
    A = torch.where(lower, beta[:, None] * (k @ k.T) * torch.exp(torch.where(lower, D, 0.0)), 0.0)
    Tm = torch.linalg.solve_triangular(torch.eye(L, dtype=torch.float64) + A,
                                       torch.eye(L, dtype=torch.float64), upper=False, unitriangular=True)
    U = Tm @ (beta[:, None] * v)
    W = Tm @ (beta[:, None] * k * torch.exp(G)[:, None])
    Vn = U - W @ S0
    incl = torch.tril(torch.ones(L, L, dtype=torch.bool))
    P = torch.where(incl, (q @ k.T) * torch.exp(torch.where(incl, D, 0.0)), 0.0)
    o = torch.exp(G)[:, None] * (q @ S0) + P @ Vn
    S_end = torch.exp(G[-1]) * S0 + (k * torch.exp(G[-1] - G)[:, None]).T @ Vn
    return o, S_end


def tree_forward(q, k, v, g, beta, parents, lengths, S0=None, step="recurrence"):
    """eq. 10 over the trie. q, k [N, hk, Dk], v [N, hv, Dv], g, beta [N, hv],
    S0 [hv, Dk, Dv] or None (zeros). Returns (o [N, hv, Dv], S_end [S, hv, Dk, Dv]),
    S_end[s] the state after segment s (by segment id)."""
    parents, lengths = T.validate(parents, lengths)
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    N, hk, Dk = q.shape
    hv, Dv = v.shape[1], v.shape[2]
    G = hv // hk
    S0 = torch.zeros(hv, Dk, Dv, dtype=torch.float64) if S0 is None else _f64(S0)
    order, seg_start = T.dfs_serialize(parents, lengths)
    fn = recurrence if step == "recurrence" else chunk_form
    o = torch.zeros(N, hv, Dv, dtype=torch.float64)
    S_end = torch.zeros(len(parents), hv, Dk, Dv, dtype=torch.float64)
    for s in order:  # parents come before children in DFS order
        a, b = seg_start[s], seg_start[s] + lengths[s]
        for h in range(hv):
            init = S0[h] if parents[s] < 0 else S_end[parents[s], h]
            o[a:b, h], S_end[s, h] = fn(q[a:b, h // G], k[a:b, h // G], v[a:b, h], g[a:b, h],
                                        beta[a:b, h], init)
    return o, S_end
