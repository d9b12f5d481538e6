"""Attention of one partition with its gateway (fp64, torch CPU): test infrastructure only.

Tree Training (arXiv 2511.00413) App. B.2-B.4. A child partition C of a
partitioned trie runs its own DFS token sequence (N tokens) with, in front of
it, a gateway of past_len cached keys: the parent partition's own gateway
followed by the parent's DFS tokens up to the end of the cut node. Eq. 14
gives the mask over the concatenated keys [gateway (past_len), own (N)]:

    M[i, j] = attn_bias[j]                 for j <  past_len
    M[i, j] = tree mask[i, j - past_len]   for j >= past_len

and eq. 16 makes attn_bias 0 on the parent's own gateway and on the cut
node's ancestor chain inside the parent (eq. 15), -inf elsewhere; here that
is the boolean ``past_visible`` [past_len]. B.5 accumulates the gateway keys'
gradients of several children in fp32; in fp64 here that is a plain sum.

Everything below is plain masked-softmax attention over that concatenated key
set, computed by the dense functions of ``oracle.attention`` (small N) or row
by row / key by key (larger N), in fp64.
"""
from __future__ import annotations

import numpy as np
import torch

from . import attention as A
from . import mask as M
from .mask import TrieView


def combined_mask(parents, lengths, past_visible) -> np.ndarray:
    """Eq. 14 written out: [N, past_len + N] bool, the gateway columns first."""
    vis = np.asarray(past_visible, dtype=bool)
    tree = M.dense_mask_appendix(parents, lengths)
    N = tree.shape[0]
    return np.concatenate([np.broadcast_to(vis, (N, vis.size)), tree], axis=1)


def _cat(past, own):
    return torch.cat([past.detach().to(torch.float64), own.detach().to(torch.float64)], dim=0)


def forward_dense(q, k, v, past_k, past_v, parents, lengths, past_visible, scale=None):
    """(o [N, Hq, D], lse [Hq, N]) over the gateway and own keys (small N)."""
    m = combined_mask(parents, lengths, past_visible)
    return A.forward_dense(q, _cat(past_k, k), _cat(past_v, v), m, scale)


def backward_dense(q, k, v, past_k, past_v, do, parents, lengths, past_visible, scale=None):
    """(dq, dk, dv, d past_k, d past_v): the analytic backward over the
    concatenated keys, split back into the partition's own keys and the
    gateway's (small N)."""
    m = combined_mask(parents, lengths, past_visible)
    K, V = _cat(past_k, k), _cat(past_v, v)
    o, lse = A.forward_dense(q, K, V, m, scale)
    dq, dK, dV = A.backward_dense(q, K, V, o, lse, do, m, scale)
    P = past_k.shape[0]
    return dq, dK[P:], dV[P:], dK[:P], dV[:P]


def _row_keys(view, past_vis_idx, past_len, i):
    """Row i's visible keys in the concatenated key space."""
    return np.concatenate([past_vis_idx, past_len + view.visible_keys(i)])


def forward_rows(q, k, v, past_k, past_v, parents, lengths, past_visible, rows, scale=None):
    """(o [len(rows), Hq, D], lse [Hq, len(rows)]) for the rows asked for."""
    view = TrieView(parents, lengths)
    past_vis_idx = np.flatnonzero(np.asarray(past_visible, dtype=bool))
    P = past_k.shape[0]
    hq, hkv, D = q.shape[1], k.shape[1], q.shape[2]
    G = hq // hkv
    scale = A.default_scale(D) if scale is None else scale
    o = torch.zeros(len(rows), hq, D, dtype=torch.float64)
    lse = torch.zeros(hq, len(rows), dtype=torch.float64)
    for n, i in enumerate(rows):
        keys = torch.as_tensor(_row_keys(view, past_vis_idx, P, int(i)))
        kp = keys[keys < P]
        ko = keys[keys >= P] - P
        for h in range(hq):
            kv = h // G
            kk = torch.cat([past_k[kp, kv].to(torch.float64), k[ko, kv].to(torch.float64)])
            vv = torch.cat([past_v[kp, kv].to(torch.float64), v[ko, kv].to(torch.float64)])
            s = scale * (kk @ q[int(i), h].to(torch.float64))
            l = torch.logsumexp(s, dim=0)
            o[n, h] = torch.exp(s - l) @ vv
            lse[h, n] = l
    return o, lse


def backward_rows(q, k, v, past_k, past_v, do, parents, lengths, past_visible, rows, scale=None):
    """dq for the rows asked for: [len(rows), Hq, D]."""
    view = TrieView(parents, lengths)
    past_vis_idx = np.flatnonzero(np.asarray(past_visible, dtype=bool))
    P = past_k.shape[0]
    hq, hkv, D = q.shape[1], k.shape[1], q.shape[2]
    G = hq // hkv
    scale = A.default_scale(D) if scale is None else scale
    o, lse = forward_rows(q, k, v, past_k, past_v, parents, lengths, past_visible, rows, scale)
    dq = torch.zeros(len(rows), hq, D, dtype=torch.float64)
    for n, i in enumerate(rows):
        keys = torch.as_tensor(_row_keys(view, past_vis_idx, P, int(i)))
        kp = keys[keys < P]
        ko = keys[keys >= P] - P
        for h in range(hq):
            kv = h // G
            kk = torch.cat([past_k[kp, kv].to(torch.float64), k[ko, kv].to(torch.float64)])
            vv = torch.cat([past_v[kp, kv].to(torch.float64), v[ko, kv].to(torch.float64)])
            qi, doi = q[int(i), h].to(torch.float64), do[int(i), h].to(torch.float64)
            p = torch.exp(scale * (kk @ qi) - lse[h, n])
            delta = (doi * o[n, h]).sum()
            ds = p * (vv @ doi - delta)
            dq[n, h] = scale * (ds @ kk)
    return dq


def backward_own_keys(q, k, v, past_k, past_v, do, parents, lengths, past_visible, keys, scale=None):
    """dk, dv of the partition's own keys asked for: [len(keys), Hkv, D] each.
    Key j is seen by the rows of oracle.attention.rows_seeing (the gateway
    does not change which rows see an own key, only their softmax)."""
    view = TrieView(parents, lengths)
    hq, hkv, D = q.shape[1], k.shape[1], q.shape[2]
    G = hq // hkv
    scale = A.default_scale(D) if scale is None else scale
    seen = [A.rows_seeing(view, int(j)) for j in keys]
    union = np.unique(np.concatenate(seen)) if len(keys) else np.zeros(0, np.int64)
    o_all, lse_all = forward_rows(q, k, v, past_k, past_v, parents, lengths, past_visible, union, scale)
    dk = torch.zeros(len(keys), hkv, D, dtype=torch.float64)
    dv = torch.zeros(len(keys), hkv, D, dtype=torch.float64)
    for n, j in enumerate(keys):
        rows = seen[n]
        at = torch.as_tensor(np.searchsorted(union, rows))
        rr = torch.as_tensor(rows)
        for h in range(hq):
            kv = h // G
            qr = q[rr, h].to(torch.float64)
            dor = do[rr, h].to(torch.float64)
            p = torch.exp(scale * (qr @ k[int(j), kv].to(torch.float64)) - lse_all[h, at])
            delta = (dor * o_all[at, h]).sum(dim=1)
            ds = p * (dor @ v[int(j), kv].to(torch.float64) - delta)
            dk[n, kv] += scale * (ds @ qr)
            dv[n, kv] += p @ dor
    return dk, dv
