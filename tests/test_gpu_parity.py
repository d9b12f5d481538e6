"""GPU parity: the CUDA path (through the C-ABI) against the fp64 CPU oracle.

Tolerances (stated for tree attention on bf16 inputs): max-abs 2e-2 and
mean-abs 2e-3 on o, lse, dq, dk, dv; fp32 inputs: max-abs 1e-4. The oracle
consumes exactly the dtype-rounded tensors the GPU gets, upcast to fp64.
"""
import numpy as np
import pytest
import torch

import treegen
import tree_packed_attention_gb300 as tpa
from oracle import attention as A
from oracle import trie as T

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN = 2e-2, 2e-3
F32_MAX = 1e-4


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _err(got, ref):
    d = (got.double().cpu() - ref).abs()
    return float(d.max()), float(d.mean())


def _check(name, got, ref, max_tol, mean_tol=None):
    mx, mn = _err(got, ref)
    assert mx <= max_tol, f"{name}: max abs err {mx:.3g} > {max_tol}"
    if mean_tol is not None:
        assert mn <= mean_tol, f"{name}: mean abs err {mn:.3g} > {mean_tol}"


def _run(parents, lengths, hq, hkv, D, dtype, seed=0, scale=0.0, grad_dtype=None):
    N = int(np.sum(lengths))
    q, k, v, do = treegen.draw_tensors(N, hq, hkv, D, dtype, seed)
    plan = tpa.tree_plan_build(parents, lengths)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = tpa.tree_attn_fwd(plan, qd, kd, vd, scale)
    dq, dk, dv = tpa.tree_attn_bwd(plan, dod, qd, kd, vd, o, lse, scale, grad_dtype=grad_dtype)
    tpa.tree_status_sync()
    return (q, k, v, do), (o, lse, dq, dk, dv)


def _full_check(parents, lengths, hq, hkv, D, dtype, seed=0, scale=0.0, grad_dtype=None):
    (q, k, v, do), (o, lse, dq, dk, dv) = _run(parents, lengths, hq, hkv, D, dtype, seed, scale, grad_dtype)
    sc = None if scale == 0.0 else scale
    ro, rlse = A.forward(q, k, v, parents, lengths, sc)
    rdq, rdk, rdv = A.backward(q, k, v, do, parents, lengths, sc)
    if dtype == "fp32":
        tol = dict(max_tol=F32_MAX)
    else:
        tol = dict(max_tol=BF16_MAX, mean_tol=BF16_MEAN)
    _check("o", o, ro, **tol)
    _check("lse", lse, rlse, **tol)
    _check("dq", dq, rdq, **tol)
    _check("dk", dk, rdk, **tol)
    _check("dv", dv, rdv, **tol)


# ---------------------------------------------------------------- fp32 path

def test_fp32_tiny_trie_all_seeds():
    _need_gpu()
    for seed in (0, 1, 2):
        w = treegen.workload(1, seed)
        _full_check(w.parents, w.lengths, 1, 1, 64, "fp32", seed=seed)


def test_fp32_forests_gqa_and_d128():
    _need_gpu()
    rng = np.random.default_rng(7)
    for n in range(6):
        p, L = treegen.random_forest(rng, int(rng.integers(2, 12)), max_len=90, n_roots=int(rng.integers(1, 3)))
        hq, hkv, D = [(2, 1, 64), (4, 2, 128), (3, 3, 64)][n % 3]
        _full_check(p, L, hq, hkv, D, "fp32", seed=n, scale=0.2 if n == 4 else 0.0)


# ---------------------------------------------------------------- bf16 path

@pytest.mark.parametrize("hq,hkv", [(4, 2), (2, 2), (3, 1), (4, 1), (6, 3)])
def test_bf16_grpo_shaped_small(hq, hkv):
    """Several tiles and a ragged tail; grouped-head pairing and q-tile pairing."""
    _need_gpu()
    p, L = treegen.grpo_tree(0, prompt=300, n_leaves=5, lo=90, hi=300)
    _full_check(p, L, hq, hkv, 128, "bf16", seed=hq)


def test_bf16_chain_equals_causal():
    _need_gpu()
    p, L = treegen.chain(777)
    _full_check(p, L, 2, 2, 128, "bf16", seed=3)


def test_bf16_random_forests():
    _need_gpu()
    rng = np.random.default_rng(11)
    for n in range(4):
        p, L = treegen.random_forest(rng, int(rng.integers(3, 30)), max_len=200,
                                     n_roots=int(rng.integers(1, 4)))
        hq, hkv = [(2, 1), (4, 4), (8, 2), (1, 1)][n]
        _full_check(p, L, hq, hkv, 128, "bf16", seed=20 + n)


def test_bf16_grad_fp32_and_scale():
    _need_gpu()
    p, L = treegen.tiny_trie(2)
    p = np.array([-1, 0, 0, 1, 1, 2, 2])
    L = np.array([140, 60, 70, 129, 1, 127, 128])
    _full_check(p, L, 4, 2, 128, "bf16", seed=5, scale=0.05, grad_dtype=torch.float32)


@pytest.mark.parametrize("lengths", [[1], [127], [128], [129], [1, 1, 1], [255, 1]])
def test_bf16_edge_sizes(lengths):
    _need_gpu()
    L = np.array(lengths)
    p = np.array([-1] + list(range(len(lengths) - 1)))  # a chain of segments
    _full_check(p, L, 2, 1, 128, "bf16", seed=len(lengths))


def test_bf16_forward_is_deterministic():
    _need_gpu()
    p, L = treegen.grpo_tree(1, prompt=256, n_leaves=4, lo=100, hi=200)
    N = int(L.sum())
    q, k, v = (x.cuda() for x in treegen.draw_tensors(N, 4, 2, 128, "bf16", 1, with_grad_out=False))
    plan = tpa.tree_plan_build(p, L)
    o1, l1 = tpa.tree_attn_fwd(plan, q, k, v)
    o2, l2 = tpa.tree_attn_fwd(plan, q, k, v)
    tpa.tree_status_sync()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_outputs_untouched_outside_their_rows():
    """Writes stay inside o/lse/dq/dk/dv: guard regions around them keep a NaN pattern."""
    _need_gpu()
    p, L = treegen.grpo_tree(2, prompt=130, n_leaves=3, lo=50, hi=140)
    N = int(L.sum())
    hq, hkv = 4, 2
    q, k, v, do = (x.cuda() for x in treegen.draw_tensors(N, hq, hkv, 128, "bf16", 2))
    plan = tpa.tree_plan_build(p, L)
    G = 4096

    def guarded(shape, dtype):
        n = int(np.prod(shape))
        buf = torch.full((n + 2 * G,), float("nan"), dtype=dtype, device="cuda")
        return buf, buf[G:G + n].view(*shape)

    ob, o = guarded((N, hq, 128), torch.bfloat16)
    lb, lse = guarded((hq, N), torch.float32)
    tpa.tree_attn_fwd(plan, q, k, v, out=o, lse=lse)
    bufs = [guarded((N, hq, 128), torch.bfloat16), guarded((N, hkv, 128), torch.bfloat16),
            guarded((N, hkv, 128), torch.bfloat16)]
    tpa.tree_attn_bwd(plan, do, q, k, v, o, lse, out=tuple(b[1] for b in bufs))
    tpa.tree_status_sync()
    for buf, inner in [(ob, o), (lb, lse)] + bufs:
        assert torch.isnan(buf[:G]).all() and torch.isnan(buf[-G:]).all()
        assert torch.isfinite(inner).all()


def test_empty_plan_is_a_no_op():
    _need_gpu()
    plan = tpa.tree_plan_build(np.zeros(0, np.int32), np.zeros(0, np.int32))
    q = torch.zeros(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    o, lse = tpa.tree_attn_fwd(plan, q, q, q)
    assert o.shape == (0, 2, 128)
    tpa.tree_status_sync()


# ------------------------------------------- full-size workloads, sampled

def _sample_rows(parents, lengths, rng, n=12):
    """Rows spread over segments: first/last token of some segments plus random ones."""
    view_starts = {}
    _, seg_start = T.dfs_serialize(parents, lengths)
    N = int(np.sum(lengths))
    rows = {0, N - 1}
    segs = rng.choice(len(parents), size=min(len(parents), n // 2), replace=False)
    for s in segs:
        rows.add(seg_start[s])
        rows.add(seg_start[s] + int(lengths[s]) - 1)
    while len(rows) < n:
        rows.add(int(rng.integers(0, N)))
    return sorted(rows)


def _leaf_tail_keys(parents, lengths, rng, n=4):
    """Keys near the end of leaf segments (few rows see them, so the oracle is cheap)."""
    _, seg_start = T.dfs_serialize(parents, lengths)
    leaves = T.leaves(list(parents))
    pick = rng.choice(len(leaves), size=min(n, len(leaves)), replace=False)
    out = []
    for idx in pick:
        s = leaves[idx]
        L = int(lengths[s])
        out.append(seg_start[s] + L - 1 - int(rng.integers(0, min(L, 40))))
    return sorted(out)


@pytest.mark.parametrize("index", [2, 3, 4, 5])
def test_full_size_workloads_sampled(index):
    _need_gpu()
    w = treegen.workload(index)
    (q, k, v, do), (o, lse, dq, dk, dv) = _run(w.parents, w.lengths, w.hq, w.hkv, w.head_dim, w.dtype, 0)
    rng = np.random.default_rng(index)
    rows = _sample_rows(w.parents, w.lengths, rng)
    ro, rlse = A.forward(q, k, v, w.parents, w.lengths, rows=rows)
    _check("o", o[rows], ro, BF16_MAX, BF16_MEAN)
    _check("lse", lse[:, rows], rlse, BF16_MAX, BF16_MEAN)
    rdq = A.backward_rows(q, k, v, do, w.parents, w.lengths, rows)
    _check("dq", dq[rows], rdq, BF16_MAX, BF16_MEAN)
    keys = _leaf_tail_keys(w.parents, w.lengths, rng)
    rdk, rdv = A.backward_keys(q, k, v, do, w.parents, w.lengths, keys)
    _check("dk", dk[keys], rdk, BF16_MAX, BF16_MEAN)
    _check("dv", dv[keys], rdv, BF16_MAX, BF16_MEAN)
    # properties at every row: finite, and lse >= the row's own logit
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()
