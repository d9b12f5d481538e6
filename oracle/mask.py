"""The tree attention mask, three ways.

Follows "Tree Training" (arXiv 2511.00413):
  * §3.2 "Attention Mask": token i attends to token j iff j <= i and the
    nodes of i and j lie on a common root-to-leaf path;
  * App. A.1: i attends to j iff j is in an ancestor chunk of i (whole chunk)
    or in the same chunk with j <= i; built there as a dense bool mask from
    chunk boundaries and ancestor lists (which include the chunk itself).

``dense_mask_appendix`` restates the App. A.1 construction, ``dense_mask_paths``
restates the §3.2 wording, and ``row_intervals`` gives the same set per row as
a list of key intervals (ancestor chunks, then the own chunk up to i) for
sizes where an N x N mask is too large. The tests check the three agree.
"""
from __future__ import annotations

import numpy as np

from . import trie as T


def chunk_boundaries(parents, lengths):
    """(start, end) token range of every segment in the DFS sequence."""
    parents, lengths = T.validate(parents, lengths)
    _, seg_start = T.dfs_serialize(parents, lengths)
    return [(seg_start[s], seg_start[s] + lengths[s]) for s in range(len(parents))]


def dense_mask_appendix(parents, lengths) -> np.ndarray:
    """App. A.1: dense [N, N] bool mask from chunk boundaries and ancestor lists."""
    parents, lengths = T.validate(parents, lengths)
    N = sum(lengths)
    bounds = chunk_boundaries(parents, lengths)
    mask = np.zeros((N, N), dtype=bool)
    for c in range(len(parents)):
        c_start, c_end = bounds[c]
        for anc in T.ancestors(parents, c) + [c]:  # ancestors of c, and c itself
            a_start, a_end = bounds[anc]
            for i in range(c_start, c_end):
                if anc == c:
                    mask[i, c_start:i + 1] = True  # causal inside the own chunk
                else:
                    mask[i, a_start:a_end] = True  # the whole ancestor chunk
    return mask


def dense_mask_paths(parents, lengths) -> np.ndarray:
    """§3.2 wording: j <= i and seg(i), seg(j) lie on a common root-to-leaf path."""
    parents, lengths = T.validate(parents, lengths)
    tok = T.token_segments(parents, lengths)
    N = len(tok)
    S = len(parents)
    together = np.zeros((S, S), dtype=bool)
    for p in T.paths(parents):
        for a in p:
            for b in p:
                together[a, b] = True
    mask = np.zeros((N, N), dtype=bool)
    for i in range(N):
        for j in range(i + 1):
            mask[i, j] = together[tok[i], tok[j]]
    return mask


def segment_key_intervals(parents, lengths, s):
    """Key intervals every token of segment s sees in full: its ancestors' chunks."""
    parents, lengths = T.validate(parents, lengths)
    bounds = chunk_boundaries(parents, lengths)
    return [bounds[a] for a in T.ancestors(parents, s)]


def row_intervals(parents, lengths, i, _cache=None):
    """Visible key intervals of row i: ancestor chunks, then [own start, i+1)."""
    parents, lengths = T.validate(parents, lengths)
    tok = T.token_segments(parents, lengths)
    s = tok[i]
    bounds = chunk_boundaries(parents, lengths)
    return segment_key_intervals(parents, lengths, s) + [(bounds[s][0], i + 1)]


class TrieView:
    """Precomputed DFS layout of one trie, for the larger-than-dense oracle paths."""

    def __init__(self, parents, lengths):
        self.parents, self.lengths = T.validate(parents, lengths)
        self.order, self.seg_start = T.dfs_serialize(self.parents, self.lengths)
        self.N = sum(self.lengths)
        self.S = len(self.parents)
        self.token_seg = np.array(T.token_segments(self.parents, self.lengths), dtype=np.int64)
        self.anc = [T.ancestors(self.parents, s) for s in range(self.S)]

    def seg_range(self, s):
        return self.seg_start[s], self.seg_start[s] + self.lengths[s]

    def ancestor_keys(self, s) -> np.ndarray:
        """Indices of all ancestor tokens of segment s (root first)."""
        parts = [np.arange(*self.seg_range(a)) for a in self.anc[s]]
        return np.concatenate(parts) if parts else np.zeros(0, dtype=np.int64)

    def visible_keys(self, i) -> np.ndarray:
        """Visible key indices of row i, ascending."""
        s = int(self.token_seg[i])
        a = self.seg_start[s]
        return np.concatenate([self.ancestor_keys(s), np.arange(a, i + 1)])

    def visible_count(self) -> int:
        """Sum over rows of the number of visible keys (diagonal included)."""
        total = 0
        for s in range(self.S):
            anc_len = sum(self.lengths[a] for a in self.anc[s])
            L = self.lengths[s]
            total += L * anc_len + L * (L + 1) // 2
        return total
