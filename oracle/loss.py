"""Weighted next-token cross-entropy over a DFS-serialized trie (fp64, torch CPU):
test infrastructure only.

Tree Training (arXiv 2511.00413) §3.1 eq. 3-5 and §3.2 "Loss Weights": the
tree loss is one weighted sum over unique tokens, sum_t lambda_t * l_t, with
l_t the per-token objective of a path through t (for SFT, -log p(y_t | x)).

Reading (the pages do not say which logits row predicts which token): on
every root-to-leaf path, the token after position a is predicted from the
logits of a. In the DFS layout that is the previous token of the same
segment, or, for a segment's first token, the last token of its parent
segment; a root's first token is predicted by nothing. Several tokens (the
first tokens of all children of a segment) are predicted from one row, each
with its own weight. The weight of a prediction is the weight lambda_t of the
predicted token t (g_t / K for the sep-avg objective), so that every path
counts each of its predictions once.

    L        = sum over predictions (r -> t) of lambda_t * (logsumexp(z_r) - z_r[x_t])
    dL/dz_r  = grad_scale * sum over (r -> t) of lambda_t * (softmax(z_r) - onehot(x_t))
"""
from __future__ import annotations

import numpy as np
import torch

from . import trie as T


def path_successors(parents, lengths):
    """For each DFS row a, the DFS indices of the tokens that follow a on some
    root-to-leaf path (ascending), from the paths themselves."""
    N = int(np.sum(lengths))
    succ = [set() for _ in range(N)]
    for _, ids in T.base_serialization(parents, lengths):
        for a, b in zip(ids[:-1], ids[1:]):
            succ[a].add(b)
    return [sorted(s) for s in succ]


def weighted_ce(logits, tokens, lam, parents, lengths, grad_scale=1.0, rows=None):
    """(loss, row_loss, dlogits) in fp64.

    logits [N, V] (any float dtype, upcast), tokens [N] token ids of the DFS
    sequence (a negative id: the token is not predicted), lam [N] weight of
    the prediction of each token. row_loss[r] is the weighted loss of the
    predictions made from row r. With ``rows``, only those rows are computed
    and row_loss / dlogits hold them in that order (loss is then their sum).
    """
    z = torch.as_tensor(logits)
    x = np.asarray(tokens, dtype=np.int64)
    w = np.asarray(lam, dtype=np.float64)
    N, V = z.shape
    succ_all = path_successors(parents, lengths)
    rows = list(range(N)) if rows is None else [int(r) for r in rows]
    row_loss = torch.zeros(len(rows), dtype=torch.float64)
    dz = torch.zeros(len(rows), V, dtype=torch.float64)
    for n, r in enumerate(rows):
        succ = [t for t in succ_all[r] if x[t] >= 0]
        if not succ:
            continue
        zr = z[r].to(torch.float64)
        lse = torch.logsumexp(zr, dim=0)
        p = torch.exp(zr - lse)
        for t in succ:
            row_loss[n] += w[t] * (lse - zr[x[t]])
            dz[n] += grad_scale * w[t] * p
            dz[n, x[t]] -= grad_scale * w[t]
    return float(row_loss.sum()), row_loss, dz
