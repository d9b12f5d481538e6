"""Tree-correct causal depthwise convolution (fp64, torch CPU): test infrastructure only.

Tree Training (arXiv 2511.00413) App. A.3 "Tree-Correct Causal Convolution"
(eq. 11): a causal conv of width K must, for every token, mix the K-1 tokens
that precede it on its own root-to-leaf path, not the K-1 tokens that precede
it in the DFS sequence (those may belong to a sibling branch). Stated per
token, which is the definition this module writes out:

    y[t] = act(b + sum_{k=0}^{K-1} w[:, K-1-k] * x[pred_k(t)])

with pred_0(t) = t, pred_k(t) the k-th token before t on t's root-to-leaf path
(the path's token sequence: its ancestors' segments root first, then t's own
segment up to t), and x[pred_k(t)] = 0 when the path has fewer than k tokens
before t. The pages reach the same result segment by segment (each segment
convolved with its parent's last K-1 effective tokens prepended); the pin in
the tests is the pages' claim itself, that the result equals a plain causal
conv1d run on every root-to-leaf path alone.

``causal_conv`` is the plain causal conv1d of one sequence:
y[i] = act(b + sum_k w[:, k] x[i-(K-1)+k]), zeros before the start.
Everything is torch fp64, so autograd gives the backward.
"""
import torch

from . import trie as T


def causal_conv(x, w, b=None, act="silu"):
    """x [L, C], w [C, K], b [C] or None (torch fp64) -> [L, C]."""
    L, C = x.shape
    K = w.shape[1]
    xp = torch.cat([torch.zeros(K - 1, C, dtype=x.dtype), x], dim=0)
    y = torch.zeros(L, C, dtype=x.dtype) if b is None else b.expand(L, C).clone()
    for k in range(K):
        y = y + w[:, k] * xp[k:k + L]
    return torch.nn.functional.silu(y) if act == "silu" else y


def path_predecessors(parents, lengths, K):
    """pred[t, k] for k = 0..K-1 (int64 [N, K]): the k-th token before t on its
    root-to-leaf path (t itself for k = 0), or -1 past the root. Walks back
    along the path: inside t's segment first, then from the last token of the
    parent segment, and so on up to the root."""
    parents, lengths = T.validate(parents, lengths)
    _, seg_start = T.dfs_serialize(parents, lengths)
    seg = T.token_segments(parents, lengths)
    N = len(seg)
    pred = torch.full((N, K), -1, dtype=torch.int64)
    for t in range(N):
        u = t
        for k in range(K):
            if u < 0:
                break
            pred[t, k] = u
            s = seg[u]
            if u > seg_start[s]:  # the previous token of the same segment
                u -= 1
            else:  # the path continues at the parent's last token
                p = parents[s]
                u = seg_start[p] + lengths[p] - 1 if p >= 0 else -1
    return pred


def tree_conv(parents, lengths, x, w, b=None, act="silu"):
    """x [N, C] in the DFS token layout -> [N, C], per the definition above."""
    N, C = x.shape
    K = w.shape[1]
    pred = path_predecessors(parents, lengths, K)
    xz = torch.cat([x, torch.zeros(1, C, dtype=x.dtype)], dim=0)  # row N: the zero past the root
    idx = torch.where(pred >= 0, pred, torch.full_like(pred, N))
    y = torch.zeros(N, C, dtype=x.dtype) if b is None else b.expand(N, C).clone()
    for k in range(K):
        y = y + w[:, K - 1 - k] * xz[idx[:, k]]
    return torch.nn.functional.silu(y) if act == "silu" else y
