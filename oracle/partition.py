"""Redundancy-free tree partitioning, checked by brute force: test infrastructure only.

Tree Training (arXiv 2511.00413) §3.3 "Partitioning": when the tree exceeds
memory it is split into partitions, each a connected subtree cut only at node
boundaries, each holding at most C tokens, as few as possible. App. B.2 and
B.4 define what a child partition inherits from the partition above it: the
gateway past (the parent's accumulated KV up to the end of the cut node) and
the position offset of eq. 17.

Everything here follows those definitions literally and slowly: the minimum
count by trying every set of cut edges (small tries only), the partitions'
validity, eq. 17 as a recursion over the partition chain, and the peak
tokens held along any root-to-leaf path.
"""
import itertools

from . import trie as T


def pieces(parents, lengths, cut):
    """Connected pieces after cutting each segment in ``cut`` from its parent.

    Returns part_of[S] (a piece id per segment) and the piece sizes."""
    parents, lengths = T.validate(parents, lengths)
    S = len(parents)
    top = list(range(S))
    for s in range(S):  # walk up to the first cut segment or root
        v = s
        while parents[v] >= 0 and v not in cut:
            v = parents[v]
        top[s] = v
    ids = {}
    part_of = [ids.setdefault(top[s], len(ids)) for s in range(S)]
    sizes = [0] * len(ids)
    for s in range(S):
        sizes[part_of[s]] += lengths[s]
    return part_of, sizes


def min_partitions_bruteforce(parents, lengths, cap):
    """The fewest node-boundary pieces of at most cap tokens, by trying every
    subset of the S - R cuttable edges (feasible for S up to ~15)."""
    parents, lengths = T.validate(parents, lengths)
    edges = [s for s in range(len(parents)) if parents[s] >= 0]
    best = None
    for r in range(len(edges) + 1):
        for cut in itertools.combinations(edges, r):
            _, sizes = pieces(parents, lengths, set(cut))
            if max(sizes) <= cap:
                best = len(sizes) if best is None else min(best, len(sizes))
        if best is not None:  # fewer cuts give fewer pieces: stop at the first feasible size
            return best
    return None


def is_valid_partition(parents, lengths, cap, part_of):
    """Each piece connected (exactly one segment whose parent lies outside it)
    and at most cap tokens."""
    parents, lengths = T.validate(parents, lengths)
    groups = {}
    for s, p in enumerate(part_of):
        groups.setdefault(p, []).append(s)
    for p, segs in groups.items():
        tops = [s for s in segs if parents[s] < 0 or part_of[parents[s]] != p]
        if len(tops) != 1 or sum(lengths[s] for s in segs) > cap:
            return False
    return True


def partition_records(parents, lengths, part_of):
    """Per piece (keyed by piece id): root, parent piece, tokens, pos_offset
    (App. B.4 eq. 17) and past_len (App. B.2), from the definitions.

    A piece's DFS sequence is its own segments in DFS order; e of the cut
    node is the number of the parent piece's DFS tokens up to and including
    the cut node; its position within the parent piece is eq. 9 applied to
    the parent piece on its own."""
    parents, lengths = T.validate(parents, lengths)
    order, _ = T.dfs_serialize(parents, lengths)
    groups = {}
    for s in order:
        groups.setdefault(part_of[s], []).append(s)
    root = {p: segs[0] for p, segs in groups.items()}  # first in DFS order is the top
    par = {p: (part_of[parents[root[p]]] if parents[root[p]] >= 0 else -1) for p in groups}

    def within(p, node):  # (position of node's first token, e of node) inside piece p
        pos = sum(lengths[a] for a in T.ancestors(parents, node) if part_of[a] == p)
        e = 0
        for s in groups[p]:
            e += lengths[s]
            if s == node:
                return pos, e
        raise AssertionError("node not in piece")

    rec = {}
    for p in sorted(groups, key=lambda q: order.index(root[q])):  # parents before children
        if par[p] < 0:
            rec[p] = dict(root=root[p], parent=-1, pos_offset=0, past_len=0)
        else:
            nc = parents[root[p]]
            pos_nc, e_nc = within(par[p], nc)
            rec[p] = dict(root=root[p], parent=par[p],
                          pos_offset=rec[par[p]]["pos_offset"] + pos_nc + lengths[nc],  # eq. 17
                          past_len=rec[par[p]]["past_len"] + e_nc)
        rec[p]["tokens"] = sum(lengths[s] for s in groups[p])
    return rec


def peak_path_tokens(parents, lengths, part_of):
    """Largest total size of the distinct pieces met on a root-to-leaf path."""
    parents, lengths = T.validate(parents, lengths)
    size = {}
    for s, p in enumerate(part_of):
        size[p] = size.get(p, 0) + lengths[s]
    best = 0
    for path in T.paths(parents):
        best = max(best, sum(size[p] for p in {part_of[s] for s in path}))
    return best
