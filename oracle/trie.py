"""Trie, DFS serialization, ancestors, g_n, K, position ids, weights, POR.

Follows "Tree Training" (arXiv 2511.00413):
  * §3.1: a trajectory tree; node n holds segment T_n; K root-to-leaf paths;
    g_n = number of paths through n.
  * §3.1 eq. 8: X_DFS(i) = Concat[token(i), X_DFS(child(0,i)), X_DFS(child(1,i)), ...].
  * §3.1 eq. 7: the baseline serialization repeating the prefix per path.
  * §3.2 eq. 9: pos(t) = sum of |T_n'| over the ancestors n' != n, plus j.
  * §3.1 eq. 2-4 and §3.2 "Loss Weights": per-token weight g_t / K.
  * §4.1 eq. 12: POR = 1 - N_tree / N_Xbase(root).

Readings of points the pages leave open:
  * child order in eq. 8: ascending segment id; roots ascending;
  * a forest (several roots) is several tries packed in one row, each with
    its own K (the pages' K belongs to one tree, §3.4: a batch is one
    self-contained tree);
  * every segment holds at least one token (§3.1 "each node n holds a token
    segment").
"""
from __future__ import annotations

import sys

import numpy as np


class TrieError(ValueError):
    """Invalid trie input. ``kind`` is one of 'invalid', 'cycle', 'empty', 'overflow'."""

    def __init__(self, kind: str, msg: str):
        super().__init__(msg)
        self.kind = kind


def validate(parents, lengths):
    """Check the input trie; return (parents, lengths) as Python int lists."""
    parents = [int(x) for x in parents]
    lengths = [int(x) for x in lengths]
    if len(parents) != len(lengths):
        raise TrieError("invalid", "parents and lengths differ in size")
    S = len(parents)
    for s in range(S):
        if not (-1 <= parents[s] < S) or parents[s] == s:
            raise TrieError("invalid", f"segment {s}: parent {parents[s]} out of range")
    for s in range(S):
        if lengths[s] < 1:
            raise TrieError("empty", f"segment {s} has {lengths[s]} tokens")
    # Each segment must reach a root by following parents; otherwise it is on
    # (or below) a cycle.
    for s in range(S):
        seen = set()
        x = s
        while x != -1:
            if x in seen:
                raise TrieError("cycle", f"segment {s} does not reach a root")
            seen.add(x)
            x = parents[x]
    if sum(lengths) > 2**31 - 1:
        raise TrieError("overflow", "more than 2^31-1 tokens")
    return parents, lengths


def children_of(parents):
    """children[s] in ascending id, and the roots in ascending id."""
    S = len(parents)
    children = [[] for _ in range(S)]
    roots = []
    for s in range(S):
        if parents[s] == -1:
            roots.append(s)
        else:
            children[parents[s]].append(s)
    return children, roots


def dfs_serialize(parents, lengths):
    """eq. 8 written out recursively: the list of segments in visit order.

    Returns (dfs_order, seg_start): the segments in DFS visit order and the
    token offset of each segment (indexed by segment id) in the DFS sequence.
    """
    parents, lengths = validate(parents, lengths)
    children, roots = children_of(parents)
    order = []

    def x_dfs(i):
        order.append(i)  # token(i) first ...
        for c in children[i]:  # ... then each child's subtree
            x_dfs(c)

    old = sys.getrecursionlimit()
    sys.setrecursionlimit(max(old, 4 * len(parents) + 1000))
    try:
        for r in roots:
            x_dfs(r)
    finally:
        sys.setrecursionlimit(old)
    seg_start = [0] * len(parents)
    off = 0
    for s in order:
        seg_start[s] = off
        off += lengths[s]
    return order, seg_start


def ancestors(parents, s):
    """Ancestors of s from the root down to the parent (s itself excluded)."""
    out = []
    x = parents[s]
    while x != -1:
        out.append(x)
        x = parents[x]
    return out[::-1]


def root_of(parents, s):
    while parents[s] != -1:
        s = parents[s]
    return s


def leaves(parents):
    children, _ = children_of(parents)
    return [s for s in range(len(parents)) if not children[s]]


def paths(parents):
    """All root-to-leaf paths (lists of segment ids, root first)."""
    return [ancestors(parents, leaf) + [leaf] for leaf in leaves(parents)]


def paths_through(parents):
    """g_n of §3.1: for each node, the number of root-to-leaf paths through it."""
    g = [0] * len(parents)
    for p in paths(parents):
        for n in p:
            g[n] += 1
    return g


def tries(parents):
    """Roots in ascending id; trie index of each segment."""
    _, roots = children_of(parents)
    rank = {r: i for i, r in enumerate(roots)}
    trie_id = [rank[root_of(parents, s)] for s in range(len(parents))]
    return roots, trie_id


def paths_per_trie(parents):
    """K of §3.1 for each trie (its number of root-to-leaf paths)."""
    roots, trie_id = tries(parents)
    K = [0] * len(roots)
    for leaf in leaves(parents):
        K[trie_id[leaf]] += 1
    return K


def token_segments(parents, lengths):
    """Segment id of each token of the DFS sequence."""
    order, seg_start = dfs_serialize(parents, lengths)
    tok = []
    for s in order:
        tok.extend([s] * int(lengths[s]))
    return tok


def position_ids(parents, lengths):
    """eq. 9: pos(t) = sum over ancestors n' != n of |T_n'|, plus the offset j in T_n."""
    parents, lengths = validate(parents, lengths)
    order, _ = dfs_serialize(parents, lengths)
    pos = []
    for s in order:
        base = sum(lengths[a] for a in ancestors(parents, s))
        pos.extend(base + j for j in range(lengths[s]))
    return pos


def base_serialization(parents, lengths):
    """eq. 7 / eq. 1: each root-to-leaf path laid out on its own.

    Returns a list of (leaf, token_ids) where token_ids are the DFS token
    indices of the path's tokens in path order.
    """
    parents, lengths = validate(parents, lengths)
    _, seg_start = dfs_serialize(parents, lengths)
    out = []
    for p in paths(parents):
        ids = []
        for n in p:
            ids.extend(range(seg_start[n], seg_start[n] + lengths[n]))
        out.append((p[-1], ids))
    return out


def token_weights(parents, lengths):
    """eq. 4: lambda_t = g_t / K per DFS token, rounded once to fp32.

    g_t and K are integers; the ratio is formed in fp64 and rounded to fp32.
    For integers below 2^24 this equals the correctly rounded fp32 quotient
    (a double-rounding argument: 53 >= 2*24 + 2).
    """
    parents, lengths = validate(parents, lengths)
    g = paths_through(parents)
    K = paths_per_trie(parents)
    _, trie_id = tries(parents)
    tok = token_segments(parents, lengths)
    w = np.array([g[s] / K[trie_id[s]] for s in tok], dtype=np.float64)
    return w.astype(np.float32)


def path_weight_tokens(parents, lengths, path_weights):
    """§3.1 after eq. 5: with path weights w_k, lambda_t = sum of w_k over the
    paths k that contain token t, per DFS token, summed in fp64 and rounded
    once to fp32. Paths are numbered by their leaves in DFS order (the order
    the leaves' tokens appear in the layout), each enumerated explicitly as its
    list of segments, root first."""
    parents, lengths = validate(parents, lengths)
    order, _ = dfs_serialize(parents, lengths)
    leaf_set = set(leaves(parents))
    dfs_leaves = [s for s in order if s in leaf_set]
    w = np.asarray(path_weights, dtype=np.float64)
    assert w.shape == (len(dfs_leaves),)
    lam = [0.0] * len(parents)
    for k, leaf in enumerate(dfs_leaves):
        for seg in ancestors(parents, leaf) + [leaf]:
            lam[seg] += float(w[k])
    tok = token_segments(parents, lengths)
    return np.array([lam[s] for s in tok], dtype=np.float64).astype(np.float32)


def por(n_tree: float, n_base: float) -> float:
    """eq. 12: Potential Overlap Ratio = 1 - N_tree / N_Xbase(root)."""
    return 1.0 - n_tree / n_base


def trie_por(parents, lengths) -> float:
    """POR of a trie: DFS token count against the per-path (eq. 7) token count."""
    n_tree = sum(int(x) for x in lengths)
    n_base = sum(len(ids) for _, ids in base_serialization(parents, lengths))
    return por(n_tree, n_base)
