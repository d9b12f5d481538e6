"""Per-key visibility bound, tile visibility map, work lists: the plan fields.

The tile map is a plain count of visible (query, key) pairs per BM x BN tile of
the canonical grid, taken from the row form of the mask (ancestor chunks in
full, own chunk causally; "Tree Training" §3.2 "Attention Mask", App. A.1). A
tile is EMPTY with no visible pair, FULL when all BM*BN pairs are visible (so
it also lies entirely inside the sequence), PARTIAL otherwise. A.1 notes that
the masked blocks are skipped entirely; the map is what lets a kernel do so.

``key_end[j]`` is one past the last row that sees key j: the per-column bound
in the spirit of A.1's "per-query start/end column bounds", taken here column-wise.

Work orders and the q-tile pair lists are conventions of this library for
scheduling; the pages say nothing about them. The orders follow DFS position:
q-tiles and q-tile pairs from last to first, k-tiles from first to last.
"""
from __future__ import annotations

from collections import defaultdict

import numpy as np

from . import trie as T
from .mask import TrieView

EMPTY, PARTIAL, FULL = 0, 1, 2


def key_end(parents, lengths) -> np.ndarray:
    """key_end[j] = 1 + the largest row i that attends to key j.

    Row i attends to key j in segment s iff seg(i) == s and i >= j, or s is an
    ancestor of seg(i). The largest such row is the last token of the
    segments in s's subtree; every descendant d raises the bound of each of its
    ancestors to the end of d.
    """
    view = TrieView(parents, lengths)
    last = [view.seg_range(s)[1] for s in range(view.S)]
    for d in range(view.S):
        for a in view.anc[d]:
            last[a] = max(last[a], view.seg_range(d)[1])
    return np.array([last[s] for s in view.token_seg], dtype=np.int32)


def tile_counts(parents, lengths, bm: int = 128, bn: int = 128):
    """Number of visible pairs in each non-empty (q-tile, k-tile)."""
    view = TrieView(parents, lengths)
    counts = defaultdict(int)
    for s in range(view.S):
        a, b = view.seg_range(s)
        for qt in range(a // bm, (b - 1) // bm + 1):
            r0, r1 = max(a, qt * bm), min(b, (qt + 1) * bm)
            nrows = r1 - r0
            # ancestor chunks: every row of the segment sees all of them
            for anc in view.anc[s]:
                c, d = view.seg_range(anc)
                for kt in range(c // bn, (d - 1) // bn + 1):
                    overlap = min(d, (kt + 1) * bn) - max(c, kt * bn)
                    counts[(qt, kt)] += nrows * overlap
            # own chunk: row i sees [a, i + 1)
            rows = np.arange(r0, r1)
            for kt in range(a // bn, (r1 - 1) // bn + 1):
                lo, hi = kt * bn, (kt + 1) * bn
                overlap = np.minimum(rows + 1, hi) - max(a, lo)
                counts[(qt, kt)] += int(np.clip(overlap, 0, None).sum())
    return dict(counts)


def _unit_key_sets(view, r0, r1):
    """(keys some row of [r0, r1) sees, keys every row of [r0, r1) sees), ascending,
    from the row form of the mask: a row of segment s sees the ancestors' chunks
    and its own chunk up to itself."""
    some, every = [], None
    r = r0
    while r < r1:
        s = int(view.token_seg[r])
        a, b = view.seg_range(s)
        ra, rb = r, min(r1, b)
        anc = view.ancestor_keys(s)
        some.append(np.concatenate([anc, np.arange(a, rb)]))
        first = np.concatenate([anc, np.arange(a, ra + 1)])  # what the segment's first row sees
        every = first if every is None else np.intersect1d(every, first)
        r = rb
    if every is None:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    return np.unique(np.concatenate(some)), np.asarray(every, np.int64)


def _place_runs(seq, bn, atom):
    """Lay a key sequence into tiles of bn columns: runs of consecutive keys,
    each run from a column that is a multiple of ``atom``."""
    runs = []
    for j in seq:
        if runs and runs[-1][1] == j:
            runs[-1][1] = j + 1
        else:
            runs.append([j, j + 1])
    tiles = []
    col = bn
    for a, b in runs:
        while a < b:
            if col >= bn:
                tiles.append([None] * bn)
                col = 0
            m = min(b - a, bn - col)
            for c in range(m):
                tiles[-1][col + c] = a + c
            col += m
            a += m
        col = -(-col // atom) * atom
    return tiles


def gathered_tiles(parents, lengths, unit_rows: int, bn: int = 128, atom: int = 8,
                   past_visible=None):
    """Gathered key tiles of every unit of ``unit_rows`` query rows.

    For the unit's rows, the keys every row sees come first and the keys only
    some rows see after them, each part ascending; runs of consecutive keys
    are laid into tiles of ``bn`` columns, each run from a column that is a
    multiple of ``atom``. Per tile: the kind for each block of 128 rows (EMPTY
    no visible pair, FULL every pair visible, PARTIAL otherwise), the first
    key of each atom (-8 if the atom holds none) and the key of each column
    (None for padding), and for tiles with a PARTIAL block the key_end of each
    column (0 for padding). A layout convention of this library for loading and
    skipping keys; the pages say nothing about it.

    With ``past_visible`` (a partition's gateway, App. B.2-B.3), each unit's
    tiles start with the visible gateway keys, which every row sees, laid out
    the same way in tiles of their own (flag "gateway": atoms are rows of the
    gateway keys, bounds N, and no key-before-row condition applies)."""
    view = TrieView(parents, lengths)
    N = view.N
    kend = key_end(parents, lengths)
    gw_vis = [] if past_visible is None else [j for j, x in enumerate(past_visible) if x]
    out = []
    for r0 in range(0, N, unit_rows):
        r1 = min(N, r0 + unit_rows)
        unit = []
        for cols in _place_runs(gw_vis, bn, atom):
            kinds = []
            full_cols = all(c is not None for c in cols)
            for sa in range(r0, r0 + unit_rows, 128):
                sb = min(r1, sa + 128)
                if sa >= sb:
                    kinds.append(EMPTY)
                else:
                    kinds.append(FULL if full_cols and sb - sa == 128 else PARTIAL)
            atoms = [cols[g * atom] if cols[g * atom] is not None else -8 for g in range(bn // atom)]
            bnd = [N if c is not None else 0 for c in cols] if PARTIAL in kinds else None
            unit.append({"kinds": kinds, "atoms": atoms, "cols": cols, "bounds": bnd, "gateway": True})
        some, every = _unit_key_sets(view, r0, r1)
        seq = list(every) + sorted(set(some.tolist()) - set(every.tolist()))
        tiles = _place_runs(seq, bn, atom)
        slots = []
        for sa in range(r0, r0 + unit_rows, 128):
            sb = min(r1, sa + 128)
            slots.append(_unit_key_sets(view, sa, sb) + (sb - sa,) if sa < sb else None)
        for cols in tiles:
            kinds = []
            keys = [c for c in cols if c is not None]
            for sl in slots:
                if sl is None:
                    kinds.append(EMPTY)
                    continue
                s_some, s_every, nrows = sl
                if nrows == 128 and len(keys) == bn and np.isin(keys, s_every).all():
                    kinds.append(FULL)
                elif np.isin(keys, s_some).any():
                    kinds.append(PARTIAL)
                else:
                    kinds.append(EMPTY)
            atoms = [cols[g * atom] if cols[g * atom] is not None else -8 for g in range(bn // atom)]
            bnd = None
            if PARTIAL in kinds:
                bnd = [int(kend[c]) if c is not None else 0 for c in cols]
            unit.append({"kinds": kinds, "atoms": atoms, "cols": cols, "bounds": bnd, "gateway": False})
        out.append(unit)
    return out


def _gathered_fields(parents, lengths, past_visible=None):
    kind, atoms, bidx, bounds = [], [], [], []
    ptrs = []
    for rows in (128, 256):
        ptr = [len(kind)]
        for unit in gathered_tiles(parents, lengths, rows, past_visible=past_visible):
            for t in unit:
                kind.append(sum(k << (2 * n) for n, k in enumerate(t["kinds"])) +
                            (16 if t["gateway"] else 0))
                atoms.extend(t["atoms"])
                if t["bounds"] is None:
                    bidx.append(-1)
                else:
                    bidx.append(len(bounds) // 128)
                    bounds.extend(t["bounds"])
            ptr.append(len(kind))
        ptrs.append(ptr)
    return ptrs[0], ptrs[1], kind, atoms, bidx, bounds


def gateway_fields(N, past_visible, bn: int = 128):
    """GW_KEND (N for a visible gateway key, 0 for a hidden one, padded to whole
    tiles) and GW_KT (gateway key tiles holding a visible key)."""
    vis = [bool(x) for x in past_visible]
    tiles = -(-len(vis) // bn)
    kend = [N if x else 0 for x in vis] + [0] * (tiles * bn - len(vis))
    kt = [t for t in range(tiles) if any(vis[t * bn:(t + 1) * bn])]
    return kend, kt


def plan_fields(parents, lengths, bm: int = 128, bn: int = 128, past_visible=None,
                pos_offset: int = 0) -> dict:
    """Every plan field as int32/int64 numpy arrays, named as in the C-ABI
    (with ``past_visible``, those of a partition plan with that gateway; with
    ``pos_offset``, position ids shifted by it as App. B.4 eq. 17 starts a
    child partition's positions)."""
    parents_l, lengths_l = T.validate(parents, lengths)
    S = len(parents_l)
    N = sum(lengths_l)
    view = TrieView(parents_l, lengths_l)
    roots, trie_id = T.tries(parents_l)
    g = T.paths_through(parents_l)
    K = T.paths_per_trie(parents_l)

    depth = [len(view.anc[s]) for s in range(S)]
    # the subtree of s ends where the last of its descendants (or s) ends
    subtree_end = [view.seg_range(s)[1] for s in range(S)]
    for d in range(S):
        for a in view.anc[d]:
            subtree_end[a] = max(subtree_end[a], view.seg_range(d)[1])
    anc_ptr = [0]
    anc_idx = []
    for s in range(S):
        anc_idx.extend(view.anc[s])
        anc_ptr.append(len(anc_idx))
    cu_seqlens = [view.seg_start[r] for r in roots] + [N]

    T_q = (N + bm - 1) // bm
    T_k = (N + bn - 1) // bn
    counts = tile_counts(parents_l, lengths_l, bm, bn)
    kinds = {key: (FULL if c == bm * bn else PARTIAL) for key, c in counts.items() if c > 0}

    per_q = [[] for _ in range(T_q)]
    for (qt, kt) in kinds:
        per_q[qt].append(kt)
    per_q = [sorted(x) for x in per_q]
    qt_ptr = [0]
    qt_kt, qt_kind = [], []
    for q in range(T_q):
        for kt in per_q[q]:
            qt_kt.append(kt)
            qt_kind.append(kinds[(q, kt)])
        qt_ptr.append(len(qt_kt))

    kt_qlo = [T_q] * T_k
    kt_qhi = [0] * T_k
    for (qt, kt) in kinds:
        kt_qlo[kt] = min(kt_qlo[kt], qt)
        kt_qhi[kt] = max(kt_qhi[kt], qt + 1)

    fwd_order = list(reversed(range(T_q)))
    bwd_order = list(range(T_k))

    n_pairs = (T_q + 1) // 2
    qp_ptr = [0]
    qp_kt, qp_kind = [], []
    for p in range(n_pairs):
        slots = [2 * p, 2 * p + 1]
        union = sorted(set(kt for q in slots if q < T_q for kt in per_q[q]))
        for kt in union:
            k0 = kinds.get((slots[0], kt), EMPTY)
            k1 = kinds.get((slots[1], kt), EMPTY) if slots[1] < T_q else EMPTY
            qp_kt.append(kt)
            qp_kind.append(k0 | (k1 << 2))
        qp_ptr.append(len(qp_kt))
    qp_order = list(reversed(range(n_pairs)))

    pos_id = [p + pos_offset for p in T.position_ids(parents_l, lengths_l)]
    gq_ptr, gp_ptr, gt_kind, gt_atom, gt_bidx, gt_bounds = _gathered_fields(parents_l, lengths_l,
                                                                          past_visible)
    gw_kend, gw_kt = ([], []) if past_visible is None or len(past_visible) == 0 else \
        gateway_fields(N, past_visible, bn)
    i32 = lambda x: np.asarray(x, dtype=np.int32)  # noqa: E731
    return {
        "num_tokens": N,
        "num_segments": S,
        "num_tries": len(roots),
        "visible_pairs": view.visible_count(),
        "dfs_order": i32(view.order),
        "seg_start": i32(view.seg_start),
        "depth": i32(depth),
        "subtree_end": i32(subtree_end),
        "trie_id": i32(trie_id),
        "g": i32(g),
        "anc_ptr": i32(anc_ptr),
        "anc_idx": i32(anc_idx),
        "token_seg": i32(view.token_seg),
        "pos_id": i32(pos_id),
        "key_end": key_end(parents_l, lengths_l),
        "cu_seqlens": i32(cu_seqlens),
        "trie_paths": i32(K),
        "qt_ptr": i32(qt_ptr),
        "qt_kt": i32(qt_kt),
        "qt_kind": i32(qt_kind),
        "kt_qlo": i32(kt_qlo),
        "kt_qhi": i32(kt_qhi),
        "fwd_order": i32(fwd_order),
        "bwd_order": i32(bwd_order),
        "qp_ptr": i32(qp_ptr),
        "qp_kt": i32(qp_kt),
        "qp_kind": i32(qp_kind),
        "qp_order": i32(qp_order),
        "gq_ptr": i32(gq_ptr),
        "gp_ptr": i32(gp_ptr),
        "gt_kind": i32(gt_kind),
        "gt_atom": i32(gt_atom),
        "gt_bidx": i32(gt_bidx),
        "gt_bounds": i32(gt_bounds),
        "gw_kend": i32(gw_kend),
        "gw_kt": i32(gw_kt),
    }
