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
# A value stored in bf16 carries its own rounding: up to half an ulp, i.e. at
# most 2^-8 |x| (2^-9 |x| on average). For bf16-stored outputs the bound is the
# arithmetic tolerance plus that storage rounding; fp32-stored outputs (lse,
# gradients with grad_dtype=fp32) are held to the plain tolerance.
BF16_STORE_REL = 2.0 ** -8


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _check(name, got, ref, max_tol, mean_tol=None):
    got = got.double().cpu()
    d = (got - ref).abs()
    mx, mn = float(d.max()), float(d.mean())
    assert mx <= max_tol, f"{name}: max abs err {mx:.3g} > {max_tol}"
    if mean_tol is not None:
        assert mn <= mean_tol, f"{name}: mean abs err {mn:.3g} > {mean_tol}"


def _check_bf16_store(name, got, ref):
    """bf16-stored result: |err| <= 2e-2 + 2^-8 |ref| elementwise, mean <= 2e-3 + 2^-9 mean|ref|."""
    assert got.dtype == torch.bfloat16
    d = (got.double().cpu() - ref).abs()
    bound = BF16_MAX + BF16_STORE_REL * ref.abs()
    worst = float((d - bound).max())
    assert worst <= 0, f"{name}: error exceeds bf16 bound by {worst:.3g} (max err {float(d.max()):.3g})"
    mean_bound = BF16_MEAN + 0.5 * BF16_STORE_REL * float(ref.abs().mean())
    assert float(d.mean()) <= mean_bound, f"{name}: mean abs err {float(d.mean()):.3g} > {mean_bound:.3g}"


def _run(parents, lengths, hq, hkv, D, dtype, seed=0, scale=0.0):
    """Forward once; backward with fp32-stored and (bf16 inputs) bf16-stored gradients."""
    N = int(np.sum(lengths))
    q, k, v, do = treegen.draw_tensors(N, hq, hkv, D, dtype, seed)
    plan = tpa.tree_plan_build(parents, lengths)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = tpa.tree_attn_fwd(plan, qd, kd, vd, scale)
    g32 = tpa.tree_attn_bwd(plan, dod, qd, kd, vd, o, lse, scale, grad_dtype=torch.float32)
    g16 = None
    if dtype == "bf16":
        g16 = tpa.tree_attn_bwd(plan, dod, qd, kd, vd, o, lse, scale, grad_dtype=torch.bfloat16)
    tpa.tree_status_sync()
    return (q, k, v, do), (o, lse, g32, g16)


def _full_check(parents, lengths, hq, hkv, D, dtype, seed=0, scale=0.0):
    (q, k, v, do), (o, lse, g32, g16) = _run(parents, lengths, hq, hkv, D, dtype, seed, scale)
    sc = None if scale == 0.0 else scale
    ro, rlse = A.forward(q, k, v, parents, lengths, sc)
    rg = A.backward(q, k, v, do, parents, lengths, sc)
    names = ("dq", "dk", "dv")
    if dtype == "fp32":
        for name, got, ref in zip(("o", "lse") + names, (o, lse) + tuple(g32), (ro, rlse) + tuple(rg)):
            _check(name, got, ref, F32_MAX)
        return
    _check_bf16_store("o", o, ro)
    _check("lse", lse, rlse, BF16_MAX, BF16_MEAN)
    for name, got, ref in zip(names, g32, rg):
        _check(name + "(fp32)", got, ref, BF16_MAX, BF16_MEAN)
    for name, got, ref in zip(names, g16, rg):
        _check_bf16_store(name + "(bf16)", got, ref)


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


def test_bf16_scale_and_tile_edges():
    _need_gpu()
    p = np.array([-1, 0, 0, 1, 1, 2, 2])
    L = np.array([140, 60, 70, 129, 1, 127, 128])
    _full_check(p, L, 4, 2, 128, "bf16", seed=5, scale=0.05)


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


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_backward_phases_equal_whole_backward_and_repeat(dtype):
    """tree_attn_bwd_dq then tree_attn_bwd_dkdv gives tree_attn_bwd's bits; so does a rerun."""
    _need_gpu()
    p, L = treegen.grpo_tree(3, prompt=300, n_leaves=5, lo=60, hi=260)
    N = int(L.sum())
    hq, hkv, D = (8, 2, 128) if dtype == "bf16" else (4, 2, 64)
    q, k, v, do = (x.cuda() for x in treegen.draw_tensors(N, hq, hkv, D, dtype, 3))
    plan = tpa.tree_plan_build(p, L)
    o, lse = tpa.tree_attn_fwd(plan, q, k, v)
    whole = tpa.tree_attn_bwd(plan, do, q, k, v, o, lse)
    again = tpa.tree_attn_bwd(plan, do, q, k, v, o, lse)
    ws = torch.empty(tpa.tree_attn_bwd_workspace_bytes(plan, hq, D, q.dtype), dtype=torch.uint8,
                     device=q.device)
    dq = tpa.tree_attn_bwd_dq(plan, do, q, k, v, o, lse, ws)
    dk, dv = tpa.tree_attn_bwd_dkdv(plan, do, q, k, v, lse, ws)
    tpa.tree_status_sync()
    for a, b, c in zip(whole, again, (dq, dk, dv)):
        assert torch.equal(a, b) and torch.equal(a, c)


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


@pytest.mark.parametrize("grad_dtype", [torch.bfloat16, torch.float32])
def test_outputs_at_16_byte_offsets_match(grad_dtype):
    """Outputs 16- but not 32-byte aligned (the C ABI's minimum) give the same bits."""
    _need_gpu()
    p, L = treegen.grpo_tree(4, prompt=200, n_leaves=3, lo=60, hi=180)
    N = int(L.sum())
    hq, hkv = 4, 2
    q, k, v, do = (x.cuda() for x in treegen.draw_tensors(N, hq, hkv, 128, "bf16", 4))
    plan = tpa.tree_plan_build(p, L)

    def offset16(shape, dtype):
        n = int(np.prod(shape))
        pad = 16 // torch.tensor([], dtype=dtype).element_size()
        buf = torch.empty(n + 2 * pad, dtype=dtype, device="cuda")
        t = buf[pad:pad + n].view(*shape)
        assert t.data_ptr() % 16 == 0 and t.data_ptr() % 32 != 0
        return t

    o, lse = tpa.tree_attn_fwd(plan, q, k, v)
    o16 = offset16((N, hq, 128), torch.bfloat16)
    tpa.tree_attn_fwd(plan, q, k, v, out=o16, lse=torch.empty_like(lse))
    g = tpa.tree_attn_bwd(plan, do, q, k, v, o, lse, grad_dtype=grad_dtype)
    g16 = tuple(offset16(x.shape, grad_dtype) for x in g)
    tpa.tree_attn_bwd(plan, do, q, k, v, o, lse, grad_dtype=grad_dtype, out=g16)
    tpa.tree_status_sync()
    assert torch.equal(o, o16)
    for a, b in zip(g, g16):
        assert torch.equal(a, b)


def test_empty_plan_is_a_no_op():
    _need_gpu()
    plan = tpa.tree_plan_build(np.zeros(0, np.int32), np.zeros(0, np.int32))
    q = torch.zeros(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    o, lse = tpa.tree_attn_fwd(plan, q, q, q)
    assert o.shape == (0, 2, 128)
    tpa.tree_status_sync()


def test_every_call_on_an_empty_trie():
    """An N = 0 plan through every call: each returns with empty outputs and
    launches nothing that could fail on an empty grid; the conv backward's
    dweight and dbias, which it overwrites, come back zero, and the
    cross-entropy's total loss is 0."""
    _need_gpu()
    plan = tpa.tree_plan_build(np.zeros(0, np.int32), np.zeros(0, np.int32))

    def z(*shape, dtype=torch.bfloat16):
        return torch.zeros(*shape, dtype=dtype, device="cuda")

    q, k = z(0, 4, 128), z(0, 2, 128)
    o, lse = tpa.tree_attn_fwd(plan, q, k, k)
    dq, dk, dv = tpa.tree_attn_bwd(plan, q, q, k, k, o, lse)
    assert dq.shape == (0, 4, 128) and dk.shape == dv.shape == (0, 2, 128)
    tpa.tree_rope(plan, q)
    tpa.tree_rope_qk(plan, q, k)
    x = z(0, 64)
    w = torch.randn(64, 4, device="cuda")
    b = torch.randn(64, device="cuda")
    assert tpa.tree_conv_fwd(plan, x, w, b).shape == (0, 64)
    dx, dw, db = tpa.tree_conv_bwd(plan, x, w, b, x)
    assert dx.shape == (0, 64)
    assert torch.equal(dw, torch.zeros_like(w)) and torch.equal(db, torch.zeros_like(b))
    loss, row_loss, dz = tpa.tree_weighted_ce(plan, z(0, 16), torch.zeros(0, dtype=torch.int32,
                                                                      device="cuda"),
                                              z(0, dtype=torch.float32))
    assert float(loss) == 0.0 and dz.shape == (0, 16) and row_loss.shape == (0,)
    f32 = torch.float32
    og, st = tpa.tree_gdn_fwd(plan, z(0, 1, 128, dtype=f32), z(0, 1, 128, dtype=f32),
                              z(0, 2, 128, dtype=f32), z(0, 2, dtype=f32), z(0, 2, dtype=f32))
    assert og.shape == (0, 2, 128) and st.shape == (0, 2, 128, 128)
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


def _long_walk_keys(parents, lengths, max_rows):
    """First and last token of the segment whose keys are seen by the most rows,
    among segments whose subtree holds at most ``max_rows`` tokens: the longest
    walks of the key-stationary backward that the oracle can still afford (a
    key's rows are its own segment from the key on plus every descendant)."""
    parents = [int(x) for x in parents]
    lengths = [int(x) for x in lengths]
    order, seg_start = T.dfs_serialize(parents, lengths)
    sub = [0] * len(parents)
    for s in reversed(order):
        sub[s] += lengths[s]
        if parents[s] >= 0:
            sub[parents[s]] += sub[s]
    best = max((s for s in range(len(parents)) if sub[s] <= max_rows), key=lambda s: (sub[s], -s))
    return [seg_start[best], seg_start[best] + lengths[best] - 1]


# (workload, seed): seeds 1 and 2 redraw the structure and tensors of the two
# tree-shaped workloads; seed 0 also checks the longest key walks.
FULL_SIZE_CASES = [(2, 0), (3, 0), (3, 1), (3, 2), (4, 0), (5, 0), (5, 1), (5, 2)]


@pytest.mark.parametrize("index,seed", FULL_SIZE_CASES)
def test_full_size_workloads_sampled(index, seed):
    _need_gpu()
    w = treegen.workload(index, seed)
    (q, k, v, do), (o, lse, g32, g16) = _run(w.parents, w.lengths, w.hq, w.hkv, w.head_dim, w.dtype,
                                              seed)
    dq, dk, dv = g32
    rng = np.random.default_rng(index + 10 * seed)
    rows = _sample_rows(w.parents, w.lengths, rng)
    ro, rlse = A.forward(q, k, v, w.parents, w.lengths, rows=rows)
    _check_bf16_store("o", o[rows], ro)
    _check("lse", lse[:, rows], rlse, BF16_MAX, BF16_MEAN)
    rdq = A.backward_rows(q, k, v, do, w.parents, w.lengths, rows)
    _check("dq", dq[rows], rdq, BF16_MAX, BF16_MEAN)
    _check_bf16_store("dq(bf16)", g16[0][rows], rdq)
    keys = _leaf_tail_keys(w.parents, w.lengths, rng)
    if seed == 0:
        # keys seen by tens of q-tiles x every head of the group: the chain's
        # first and last key, the GRPO prompt, a depth-3 agentic subtree of 16k
        # tokens, the prompt of the largest packed trie
        keys = sorted(set(keys) | set(_long_walk_keys(w.parents, w.lengths, 23000)))
    rdk, rdv = A.backward_keys(q, k, v, do, w.parents, w.lengths, keys)
    _check("dk", dk[keys], rdk, BF16_MAX, BF16_MEAN)
    _check("dv", dv[keys], rdv, BF16_MAX, BF16_MEAN)
    _check_bf16_store("dk(bf16)", g16[1][keys], rdk)
    _check_bf16_store("dv(bf16)", g16[2][keys], rdv)
    # properties at every row and key
    for t in (o, lse, dq, dk, dv) + tuple(g16):
        assert torch.isfinite(t).all()


@pytest.mark.parametrize("index", [4, 5])
def test_full_size_every_element_written_and_repeatable(index):
    """Outputs and workspace prefilled with NaN: every element of o, lse, dq, dk
    and dv comes out finite, and a second run with fresh NaN buffers gives the
    same bits (the backward sums in a fixed order), for both gradient dtypes.
    A missed row, a read before a write or a race between the kernels' warps
    shows up here at the bench's full sizes."""
    _need_gpu()
    w = treegen.workload(index)
    N, hq, hkv, D = w.num_tokens, w.hq, w.hkv, w.head_dim
    q, k, v, do = (x.cuda() for x in treegen.draw_tensors(N, hq, hkv, D, w.dtype, 0))
    plan = tpa.tree_plan_build(w.parents, w.lengths)
    nan = float("nan")
    for gdt in (torch.float32, torch.bfloat16):
        runs = []
        for _ in range(2):
            o = torch.full_like(q, nan)
            lse = torch.full((hq, N), nan, device="cuda")
            tpa.tree_attn_fwd(plan, q, k, v, out=o, lse=lse)
            ws = torch.full((tpa.tree_attn_bwd_workspace_bytes(plan, hq, D, q.dtype) // 4 + 4,), nan,
                            device="cuda")
            grads = tuple(torch.full(x.shape, nan, dtype=gdt, device="cuda") for x in (q, k, v))
            tpa.tree_attn_bwd(plan, do, q, k, v, o, lse, grad_dtype=gdt, workspace=ws.view(torch.uint8),
                              out=grads)
            tpa.tree_status_sync()
            outs = (o, lse) + grads
            for name, t in zip(("o", "lse", "dq", "dk", "dv"), outs):
                assert torch.isfinite(t).all(), f"{name} ({gdt}): {int((~torch.isfinite(t)).sum())} elements not finite"
            runs.append(outs)
        for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), *runs):
            assert torch.equal(a, b), f"{name} ({gdt}) differs between two runs"


def test_dq_repeats_bit_for_bit_on_packed_tries():
    """Sixteen backward passes over the packed workload (seed 2) give the same
    bits. The dQ kernel keeps two S buffers; its dS arrivals are counted per
    buffer, since with one shared counter a warp that finished tile t+1 early
    could complete tile t's count before another warp had stored its dS of
    tile t, and the dQ product then read S bits as dS (non-finite rows in
    about one pass in six on this workload)."""
    _need_gpu()
    w = treegen.workload(5, 2)
    N, hq, hkv, D = w.num_tokens, w.hq, w.hkv, w.head_dim
    q, k, v, do = (x.cuda() for x in treegen.draw_tensors(N, hq, hkv, D, w.dtype, 2))
    plan = tpa.tree_plan_build(w.parents, w.lengths)
    o, lse = tpa.tree_attn_fwd(plan, q, k, v)
    for gdt in (torch.float32, torch.bfloat16):
        first = None
        for rep in range(8):
            g = tpa.tree_attn_bwd(plan, do, q, k, v, o, lse, grad_dtype=gdt)
            tpa.tree_status_sync()
            if first is None:
                first = g
                for name, t in zip(("dq", "dk", "dv"), g):
                    assert torch.isfinite(t).all(), f"{name} ({gdt}) not finite"
                continue
            for name, a, b in zip(("dq", "dk", "dv"), first, g):
                assert torch.equal(a, b), f"{name} ({gdt}) differs in pass {rep}"


@pytest.mark.parametrize("case", ["chain", "grpo"])
def test_bf16_forward_rescales_on_rising_scores(case):
    """Scores that rise by about 9 (13 in log2 units) from each 128-key block
    to the next: every query is 6u plus small noise and key j is (j // 128) u
    plus small noise, softmax scale 1.5. The forward's running row maximum
    then outgrows its lazy-rescale threshold (8 in log2 units) on almost
    every tile, so the rescale of O in tensor memory runs on nearly every
    step, which inputs drawn N(0, 1) almost never reach. o and lse against
    the oracle."""
    _need_gpu()
    if case == "chain":
        p, L = np.array([-1]), np.array([1000])
    else:
        p, L = treegen.grpo_tree(2, prompt=600, n_leaves=4, lo=100, hi=400)
        p, L = np.asarray(p), np.asarray(L)
    N, hq, hkv, D = int(np.sum(L)), 2, 1, 128
    g = torch.Generator().manual_seed(31)
    u = torch.randn(D, generator=g, dtype=torch.float64)
    u /= u.norm()
    t = (torch.arange(N, dtype=torch.float64) // 128)[:, None, None]
    q = (6.0 * u + 0.05 * torch.randn(N, hq, D, generator=g, dtype=torch.float64)).to(torch.bfloat16)
    k = (t * u + 0.05 * torch.randn(N, hkv, D, generator=g, dtype=torch.float64)).to(torch.bfloat16)
    v = torch.randn(N, hkv, D, generator=g).to(torch.bfloat16)
    plan = tpa.tree_plan_build(p, L)
    o, lse = tpa.tree_attn_fwd(plan, q.cuda(), k.cuda(), v.cuda(), 1.5)
    tpa.tree_status_sync()
    ro, rlse = A.forward(q, k, v, p, L, 1.5)
    assert float(rlse.max()) > 40.0  # the scores did rise
    _check_bf16_store("o", o, ro)
    _check("lse", lse, rlse, BF16_MAX, BF16_MEAN)
