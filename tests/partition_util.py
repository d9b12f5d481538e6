"""Pieces of a partitioned trie with their gateways, from the definitions of
"Tree Training" App. B.2-B.3 (helpers for the tests; CPU, plain Python).

For a partition of a trie into connected pieces (node-boundary cuts), each
piece X gets:
  * ``segs``: its segments in the trie's DFS order, and ``parents`` /
    ``lengths`` renumbered locally (a piece is a trie of its own);
  * ``tokens``: the global DFS token indices of its own DFS sequence;
  * ``gw``: the global token indices of its gateway keys, and ``vis`` their
    visibility. A root piece has none. A child piece C whose root hangs below
    the cut node n_c of its parent piece P gets gateway(P) followed by P's DFS
    tokens up to the end of n_c (B.2). P's tokens are visible where they lie
    on the chain from P's root down to n_c (B.3 eq. 15-16); P's own gateway
    keys keep the visibility they had for P (eq. 16 calls them fully visible,
    which holds when a gateway is stored with its hidden keys dropped; kept in
    place, as B.2's slice of the accumulated KV keeps them, they must stay
    hidden for the result to equal the whole trie's).
"""
from __future__ import annotations

import numpy as np

from oracle import trie as T


def pieces(parents, lengths, part_of):
    parents = [int(x) for x in parents]
    lengths = [int(x) for x in lengths]
    order, seg_start = T.dfs_serialize(parents, lengths)
    ids = []
    for s in order:
        if part_of[s] not in ids:
            ids.append(part_of[s])  # pieces in DFS order of their roots: parents first
    out = {}
    for pid in ids:
        segs = [s for s in order if part_of[s] == pid]
        local = {s: n for n, s in enumerate(segs)}
        lp = [local[parents[s]] if parents[s] >= 0 and part_of[parents[s]] == pid else -1 for s in segs]
        ll = [lengths[s] for s in segs]
        tokens = [t for s in segs for t in range(seg_start[s], seg_start[s] + lengths[s])]
        root = segs[0]
        gw, vis = [], []
        if parents[root] >= 0:
            pp = out[part_of[parents[root]]]
            nc = parents[root]
            chain = set(a for a in T.ancestors(parents, nc) if part_of[a] == part_of[nc]) | {nc}
            # P's DFS tokens up to the end of n_c
            upto = []
            for s in pp["segs"]:
                upto.extend((t, s in chain) for t in range(seg_start[s], seg_start[s] + lengths[s]))
                if s == nc:
                    break
            gw = list(pp["gw"]) + [t for t, _ in upto]
            # The parent's own gateway keeps the visibility it had for the
            # parent (eq. 16 calls it fully visible, as if it had been kept
            # filtered; with hidden keys kept in place, they stay hidden).
            vis = list(pp["vis"]) + [v for _, v in upto]
        out[pid] = {"segs": segs, "parents": lp, "lengths": ll, "tokens": tokens,
                    "gw": gw, "vis": vis}
    return [out[pid] for pid in ids]


def cut_forest(rng, parents, lengths, max_cuts=3):
    """A random node-boundary partition: cut up to max_cuts non-root segments."""
    cand = [s for s, p in enumerate(parents) if p >= 0]
    k = int(rng.integers(1, min(max_cuts, len(cand)) + 1)) if cand else 0
    cut = set(int(x) for x in rng.choice(cand, size=k, replace=False)) if k else set()
    part = list(range(len(parents)))
    for s in range(len(parents)):
        v = s
        while parents[v] >= 0 and v not in cut:
            v = parents[v]
        part[s] = v
    return part


def to_np(xs):
    return np.asarray(xs, dtype=np.int64)
