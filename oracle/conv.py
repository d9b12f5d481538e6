"""Tree-correct causal depthwise convolution (fp64, torch CPU): test infrastructure only.

Tree Training (arXiv 2511.00413) App. A.3 "Tree-Correct Causal Convolution"
(eq. 11): in DFS order the K-1 tokens before a child segment belong to a
sibling branch, so each segment is convolved with its parent's last K-1
effective tokens prepended as left context (and those outputs dropped); a
segment's own last K-1 effective tokens -- its context plus its tokens,
zero-padded at a root -- become the context of its children.

``tree_conv`` takes those steps segment by segment in DFS order, in torch
fp64 so that autograd gives the backward. ``causal_conv`` is the plain causal
conv1d of one sequence: y[i] = act(b + sum_k w[:, k] x[i-(K-1)+k]), zeros
before the start.
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


def tree_conv(parents, lengths, x, w, b=None, act="silu"):
    """x [N, C] in the DFS token layout -> [N, C], per App. A.3."""
    parents, lengths = T.validate(parents, lengths)
    order, seg_start = T.dfs_serialize(parents, lengths)
    K = w.shape[1]
    C = x.shape[1]
    out = [None] * len(parents)
    state = {}
    for s in order:  # parents come before their children
        chunk = x[seg_start[s]:seg_start[s] + lengths[s]]
        if parents[s] >= 0:
            ext = torch.cat([state[parents[s]], chunk], dim=0)
            out[s] = causal_conv(ext, w, b, act)[K - 1:]
        else:
            ext = torch.cat([torch.zeros(K - 1, C, dtype=x.dtype), chunk], dim=0)
            out[s] = causal_conv(chunk, w, b, act)
        state[s] = ext[ext.shape[0] - (K - 1):]  # last K-1 effective tokens (empty when K = 1)
    return torch.cat([out[s] for s in order], dim=0)
