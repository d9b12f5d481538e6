"""fp64 tree attention: forward (o, lse) and analytic backward (dq, dk, dv).

What is computed is plain masked softmax attention over the DFS sequence with
the tree mask of "Tree Training" (arXiv 2511.00413) §3.2 "Attention Mask" /
App. A.1; by §3.1 eq. 6 this equals running every root-to-leaf path alone,
which the tests check by brute force per path.

Conventions (the pages leave them open):
  * q [N, Hq, D], k and v [N, Hkv, D], dO [N, Hq, D], token-major;
  * grouped heads: q head h reads kv head h // (Hq / Hkv);
  * softmax scale defaults to 1/sqrt(D);
  * lse [Hq, N] is the natural log of the softmax denominator (with the scale
    applied to the logits);
  * the diagonal is visible, so every row has at least one key.

Backward (standard softmax calculus, written out):
  P = exp(scale*S - lse), Delta_i = sum_d dO_id O_id, dP = dO V^T,
  dS = P * (dP - Delta), dQ = scale * dS K, dK = scale * dS^T Q (summed over
  the q heads of a group), dV = P^T dO (summed likewise).

All arithmetic is torch fp64 on the CPU; inputs are the dtype-rounded tensors
upcast to fp64.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from .mask import TrieView


def _f64(x):
    return x.detach().to(torch.float64)


class _Upcast:
    """Index first, then upcast the slice to fp64 (no fp64 copy of a whole large tensor)."""

    def __init__(self, x):
        self.x = x.detach()
        self.shape = x.shape

    def __getitem__(self, idx):
        return self.x[idx].to(torch.float64)


def _lazy(x):
    if isinstance(x, _Upcast):
        return x
    return x.detach() if x.dtype == torch.float64 else _Upcast(x)


def _group(hq, hkv):
    if hq % hkv:
        raise ValueError("hq must be a multiple of hkv")
    return hq // hkv


def default_scale(head_dim):
    return 1.0 / math.sqrt(head_dim)


# ---------------------------------------------------------------- dense form

def forward_dense(q, k, v, mask, scale=None):
    """Forward with an explicit [N, N] bool mask (small N)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    N, hq, D = q.shape
    G = _group(hq, k.shape[1])
    scale = default_scale(D) if scale is None else scale
    m = torch.as_tensor(np.asarray(mask), dtype=torch.bool)
    o = torch.zeros_like(q)
    lse = torch.zeros(hq, N, dtype=torch.float64)
    for h in range(hq):
        kv = h // G
        s = scale * (q[:, h] @ k[:, kv].T)
        s = s.masked_fill(~m, float("-inf"))
        lse[h] = torch.logsumexp(s, dim=1)
        p = torch.exp(s - lse[h][:, None])
        o[:, h] = p @ v[:, kv]
    return o, lse


def backward_dense(q, k, v, o, lse, do, mask, scale=None):
    """Analytic backward with an explicit [N, N] bool mask (small N)."""
    q, k, v, o, lse, do = map(_f64, (q, k, v, o, lse, do))
    N, hq, D = q.shape
    hkv = k.shape[1]
    G = _group(hq, hkv)
    scale = default_scale(D) if scale is None else scale
    m = torch.as_tensor(np.asarray(mask), dtype=torch.bool)
    dq = torch.zeros_like(q)
    dk = torch.zeros_like(k)
    dv = torch.zeros_like(v)
    for h in range(hq):
        kv = h // G
        s = scale * (q[:, h] @ k[:, kv].T)
        p = torch.exp(s - lse[h][:, None]).masked_fill(~m, 0.0)
        delta = (do[:, h] * o[:, h]).sum(dim=1)
        dp = do[:, h] @ v[:, kv].T
        ds = p * (dp - delta[:, None])
        dq[:, h] = scale * (ds @ k[:, kv])
        dk[:, kv] += scale * (ds.T @ q[:, h])
        dv[:, kv] += p.T @ do[:, h]
    return dq, dk, dv


# ------------------------------------------------------ segment-gathered form

def _segment_rows(view, rows):
    """Group the requested rows by segment: {segment: sorted row array}."""
    rows = np.asarray(rows, dtype=np.int64)
    segs = view.token_seg[rows]
    out = {}
    for s in np.unique(segs):
        out[int(s)] = np.sort(rows[segs == s])
    return out


def _keys_and_mask(view, s, rows):
    """Visible key indices for rows of segment s and their [rows, keys] mask."""
    a = view.seg_start[s]
    anc = view.ancestor_keys(s)
    own = np.arange(a, int(rows.max()) + 1)
    keys = np.concatenate([anc, own])
    mask = np.ones((len(rows), len(keys)), dtype=bool)
    mask[:, len(anc):] = own[None, :] <= rows[:, None]  # causal inside the own segment
    return keys, torch.as_tensor(mask)


def forward(q, k, v, parents, lengths, scale=None, rows=None, view=None):
    """Forward over the rows asked for (all rows by default).

    Returns (o [len(rows), Hq, D], lse [Hq, len(rows)]) in the order of ``rows``.
    """
    q, k, v = _lazy(q), _lazy(k), _lazy(v)
    view = view or TrieView(parents, lengths)
    N, hq, D = q.shape
    G = _group(hq, k.shape[1])
    scale = default_scale(D) if scale is None else scale
    rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    where = {int(r): n for n, r in enumerate(rows)}
    o = torch.zeros(len(rows), hq, D, dtype=torch.float64)
    lse = torch.zeros(hq, len(rows), dtype=torch.float64)
    for s, srows in _segment_rows(view, rows).items():
        keys, m = _keys_and_mask(view, s, srows)
        kk = torch.as_tensor(keys)
        rr = torch.as_tensor(srows)
        idx = torch.as_tensor([where[int(r)] for r in srows])
        for h in range(hq):
            kv = h // G
            sc = scale * (q[rr, h] @ k[kk, kv].T)
            sc = sc.masked_fill(~m, float("-inf"))
            l = torch.logsumexp(sc, dim=1)
            p = torch.exp(sc - l[:, None])
            o[idx, h] = p @ v[kk, kv]
            lse[h, idx] = l
    return o, lse


def backward(q, k, v, do, parents, lengths, scale=None, view=None):
    """Full analytic backward (recomputes the forward); returns dq, dk, dv."""
    q, k, v, do = map(_f64, (q, k, v, do))
    view = view or TrieView(parents, lengths)
    N, hq, D = q.shape
    hkv = k.shape[1]
    G = _group(hq, hkv)
    scale = default_scale(D) if scale is None else scale
    o, lse = forward(q, k, v, parents, lengths, scale, view=view)
    dq = torch.zeros_like(q)
    dk = torch.zeros_like(k)
    dv = torch.zeros_like(v)
    for s, srows in _segment_rows(view, np.arange(N)).items():
        keys, m = _keys_and_mask(view, s, srows)
        kk = torch.as_tensor(keys)
        rr = torch.as_tensor(srows)
        for h in range(hq):
            kv = h // G
            sc = scale * (q[rr, h] @ k[kk, kv].T)
            p = torch.exp(sc - lse[h, rr][:, None]).masked_fill(~m, 0.0)
            delta = (do[rr, h] * o[rr, h]).sum(dim=1)
            dp = do[rr, h] @ v[kk, kv].T
            ds = p * (dp - delta[:, None])
            dq[rr, h] = scale * (ds @ k[kk, kv])
            dk[kk, kv] += scale * (ds.T @ q[rr, h])
            dv[kk, kv] += p.T @ do[rr, h]
    return dq, dk, dv


def backward_rows(q, k, v, do, parents, lengths, rows, scale=None, view=None):
    """dq for the rows asked for only: [len(rows), Hq, D]."""
    q, k, v, do = map(_lazy, (q, k, v, do))
    view = view or TrieView(parents, lengths)
    N, hq, D = q.shape
    G = _group(hq, k.shape[1])
    scale = default_scale(D) if scale is None else scale
    rows = np.asarray(rows, dtype=np.int64)
    o, lse = forward(q, k, v, parents, lengths, scale, rows=rows, view=view)
    where = {int(r): n for n, r in enumerate(rows)}
    dq = torch.zeros(len(rows), hq, D, dtype=torch.float64)
    for s, srows in _segment_rows(view, rows).items():
        keys, m = _keys_and_mask(view, s, srows)
        kk = torch.as_tensor(keys)
        rr = torch.as_tensor(srows)
        idx = torch.as_tensor([where[int(r)] for r in srows])
        for h in range(hq):
            kv = h // G
            sc = scale * (q[rr, h] @ k[kk, kv].T)
            p = torch.exp(sc - lse[h, idx][:, None]).masked_fill(~m, 0.0)
            delta = (do[rr, h] * o[idx, h]).sum(dim=1)
            dp = do[rr, h] @ v[kk, kv].T
            ds = p * (dp - delta[:, None])
            dq[idx, h] = scale * (ds @ k[kk, kv])
    return dq


def rows_seeing(view, j):
    """All rows that attend to key j: its own segment from j on, and every
    token of every segment that has seg(j) among its ancestors."""
    s = int(view.token_seg[j])
    segs = [d for d in range(view.S) if s in view.anc[d]]
    parts = [np.arange(j, view.seg_range(s)[1])] + [np.arange(*view.seg_range(d)) for d in segs]
    return np.sort(np.concatenate(parts))


def backward_keys(q, k, v, do, parents, lengths, keys, scale=None, view=None):
    """dk, dv for the keys asked for only: [len(keys), Hkv, D] each."""
    q, k, v, do = map(_lazy, (q, k, v, do))
    view = view or TrieView(parents, lengths)
    N, hq, D = q.shape
    hkv = k.shape[1]
    G = _group(hq, hkv)
    scale = default_scale(D) if scale is None else scale
    keys = np.asarray(keys, dtype=np.int64)
    dk = torch.zeros(len(keys), hkv, D, dtype=torch.float64)
    dv = torch.zeros(len(keys), hkv, D, dtype=torch.float64)
    seen = [rows_seeing(view, int(j)) for j in keys]
    # o and lse of every row that sees one of the keys, computed once
    union = np.unique(np.concatenate(seen)) if len(keys) else np.zeros(0, np.int64)
    o_all, lse_all = forward(q, k, v, parents, lengths, scale, rows=union, view=view)
    for n, j in enumerate(keys):
        rows = seen[n]
        at = torch.as_tensor(np.searchsorted(union, rows))
        o, lse = o_all[at], lse_all[:, at]
        rr = torch.as_tensor(rows)
        for h in range(hq):
            kv = h // G
            sc = scale * (q[rr, h] @ k[int(j), kv])
            p = torch.exp(sc - lse[h])
            delta = (do[rr, h] * o[:, h]).sum(dim=1)
            dp = do[rr, h] @ v[int(j), kv]
            ds = p * (dp - delta)
            dk[n, kv] += scale * (ds @ q[rr, h])
            dv[n, kv] += p @ do[rr, h]
    return dk, dv
