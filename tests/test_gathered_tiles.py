"""The gathered key tiles against the dense mask of App. A.1 (CPU only).

The gathered lists are a loading convention of this library, so the pages
pin them only through what they must preserve: for every unit of query rows,
the columns of its tiles (with the mask each tile carries) must cover every
visible (row, key) pair exactly once and nothing else. Checked on the C
library's plan for random forests against the dense mask built literally from
App. A.1's loop, which is itself pinned against the §3.2 statement.
"""
import numpy as np

import treegen
import tree_packed_attention_gb300 as tpa
from oracle import mask as M


def _check_plan(parents, lengths):
    plan = tpa.tree_plan_build(parents, lengths)
    f = plan.fields()
    N = plan.num_tokens
    dense = M.dense_mask_appendix(parents, lengths)
    key_end = f["key_end"]
    bounds = f["gt_bounds"].reshape(-1, 128)
    for ptr, rows in ((f["gq_ptr"], 128), (f["gp_ptr"], 256)):
        for u in range(len(ptr) - 1):
            r0, r1 = u * rows, min(N, u * rows + rows)
            covered = np.zeros((r1 - r0, N), dtype=np.int64)
            for t in range(ptr[u], ptr[u + 1]):
                atoms = f["gt_atom"][16 * t:16 * t + 16]
                kinds = [(f["gt_kind"][t] >> (2 * s)) & 3 for s in range(rows // 128)]
                b = f["gt_bidx"][t]
                # the keys each column loads: atom a holds 8 consecutive rows from atoms[a]
                loaded = np.array([atoms[c // 8] + c % 8 for c in range(128)])
                if b >= 0:
                    kidx, kend = loaded, bounds[b]
                    live = kend > 0
                    assert (kidx[live] >= 0).all() and (kidx[live] < N).all()
                    assert np.array_equal(kend[live], key_end[kidx[live]])
                for s, kd in enumerate(kinds):
                    sa, sb = r0 + 128 * s, min(r1, r0 + 128 * s + 128)
                    if sa >= sb:
                        assert kd == 0
                        continue
                    rr = np.arange(sa, sb)[:, None]
                    if kd == 2:  # FULL: every column is a distinct real key seen by every row
                        assert sb - sa == 128 and (atoms >= 0).all()
                        vis = np.ones((sb - sa, 128), dtype=bool)
                        cols = loaded
                        assert dense[sa:sb][:, cols].all()
                    elif kd == 1:
                        cols = np.where(kend > 0, kidx, 0)  # padding columns: kend 0, never seen
                        vis = (kidx[None, :] <= rr) & (rr < kend[None, :])
                    else:  # EMPTY: the tile adds nothing for these rows
                        continue
                    for c in range(128):
                        np.add.at(covered, (np.flatnonzero(vis[:, c]) + sa - r0, cols[c]), 1)
            assert covered.max(initial=0) <= 1, "a visible pair is covered twice"
            assert np.array_equal(covered.astype(bool), dense[r0:r1]), "coverage differs from the mask"


def test_gathered_tiles_cover_every_visible_pair_once():
    rng = np.random.default_rng(5)
    cases = [treegen.workload(1, s) for s in range(3)]
    cases = [(w.parents, w.lengths) for w in cases]
    cases.append(treegen.grpo_tree(2, prompt=300, n_leaves=6, lo=40, hi=260))
    cases.append(treegen.chain(700))
    for _ in range(12):
        S = int(rng.integers(2, 40))
        cases.append(treegen.random_forest(rng, S, max_len=int(rng.integers(1, 160)),
                                           n_roots=int(rng.integers(1, 4))))
    for parents, lengths in cases:
        _check_plan(parents, lengths)


def test_gathered_tiles_of_single_tokens_and_tile_edges():
    for lengths in ([1], [127], [128], [129], [1, 1, 1], [255, 1], [9, 7, 130]):
        parents = [-1] + list(range(len(lengths) - 1))
        _check_plan(parents, lengths)
    _check_plan([-1, 0, 0, 1, 1, 2, 2], [140, 60, 70, 129, 1, 127, 128])


def test_gathered_tiles_with_a_gateway_cover_the_combined_mask():
    """Partition plans: gateway tiles first, then the own tiles, cover the
    App. B.2 eq. 14 mask over [gateway keys, own keys] exactly once."""
    from oracle import gateway as GW

    rng = np.random.default_rng(31)
    for n in range(10):
        S = int(rng.integers(1, 12))
        parents = [-1] + [int(rng.integers(0, s)) for s in range(1, S)]
        lengths = [int(x) for x in rng.integers(1, 150, S)]
        vis = (rng.random(int(rng.integers(0, 400))) < [0.2, 0.6, 1.0][n % 3]).tolist()
        plan = tpa.tree_plan_build_partition(parents, lengths, vis)
        f = plan.fields()
        N, P = plan.num_tokens, len(vis)
        combined = GW.combined_mask(parents, lengths, vis)
        bounds = f["gt_bounds"].reshape(-1, 128)
        for ptr, rows in ((f["gq_ptr"], 128), (f["gp_ptr"], 256)):
            for u in range(len(ptr) - 1):
                r0, r1 = u * rows, min(N, u * rows + rows)
                covered = np.zeros((r1 - r0, P + N), dtype=np.int64)
                for t in range(ptr[u], ptr[u + 1]):
                    atoms = f["gt_atom"][16 * t:16 * t + 16]
                    word = f["gt_kind"][t]
                    gwt = (word >> 4) & 1
                    loaded = np.array([atoms[c // 8] + c % 8 for c in range(128)])
                    b = f["gt_bidx"][t]
                    for sl in range(rows // 128):
                        kd = (word >> (2 * sl)) & 3
                        sa, sb = r0 + 128 * sl, min(r1, r0 + 128 * sl + 128)
                        if sa >= sb or kd == 0:
                            continue
                        rr = np.arange(sa, sb)[:, None]
                        if kd == 2:
                            vis_m = np.ones((sb - sa, 128), dtype=bool)
                            cols = loaded
                        else:
                            kend = bounds[b]
                            cols = np.where(kend > 0, loaded, 0)
                            vis_m = (rr < kend[None, :]) & (gwt | (loaded[None, :] <= rr))
                        cols = cols if gwt else cols + P
                        for c in range(128):
                            np.add.at(covered, (np.flatnonzero(vis_m[:, c]) + sa - r0, cols[c]), 1)
                assert covered.max(initial=0) <= 1
                assert np.array_equal(covered.astype(bool), combined[r0:r1])
