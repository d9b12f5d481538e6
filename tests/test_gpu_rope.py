"""GPU parity of tree RoPE (the C-ABI kernel) against the fp64 oracle.

Tolerances: fp32 storage, max-abs 1e-5 (inputs ~N(0,1); the kernel rotates in
fp32 with the angle reduced in fp64). bf16 storage: each output is rounded
once, so |err| <= 2^-8 |ref| + 1e-5 elementwise.
"""
import numpy as np
import pytest
import torch

import treegen
import tree_packed_attention_gb300 as tpa
from oracle import rope as R
from oracle import trie as T

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _check(got, ref, dtype, name):
    got = got.double().cpu().numpy()
    d = np.abs(got - ref)
    if dtype == torch.float32:
        assert d.max() <= 1e-5, f"{name}: max abs err {d.max():.3g}"
    else:
        worst = float((d - (2.0 ** -8 * np.abs(ref) + 1e-5)).max())
        assert worst <= 0, f"{name}: bf16 bound exceeded by {worst:.3g}"


def _draw(N, H, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(N, H, D, generator=g).to(dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rotate_half", [False, True])
def test_rope_matches_oracle_on_small_tries(dtype, rotate_half):
    _need_gpu()
    cases = [(treegen.workload(1, 0), 64), (treegen.workload(1, 1), 128), (treegen.workload(3, 0), 128)]
    rng = np.random.default_rng(5)
    for _ in range(3):  # random forests with ragged tails
        S = int(rng.integers(2, 30))
        parents = [-1] + [int(rng.integers(-1, s)) for s in range(1, S)]
        lengths = [int(x) for x in rng.integers(1, 400, S)]
        cases.append((type("W", (), {"parents": parents, "lengths": lengths})(), 32))
    for w, D in cases:
        plan = tpa.tree_plan_build(w.parents, w.lengths)
        N = plan.num_tokens
        pos = T.position_ids(w.parents, w.lengths)
        x = _draw(N, 3, D, dtype, N)
        for base in (10000.0, 500000.0):
            for inverse in (False, True):
                got = tpa.tree_rope(plan, x.cuda(), base, rotate_half, inverse)
                tpa.tree_status_sync()
                ref = R.rope(x.double().numpy(), pos, base, rotate_half, inverse)
                _check(got, ref, dtype, f"N={N} D={D} base={base} inverse={inverse}")


@pytest.mark.parametrize("index", [4, 5])
def test_rope_full_size_sampled_rows(index):
    _need_gpu()
    w = treegen.workload(index)
    plan = tpa.tree_plan_build(w.parents, w.lengths)
    N, H, D = plan.num_tokens, w.hq, w.head_dim
    x = torch.randn(N, H, D, generator=torch.Generator(device="cuda").manual_seed(1), device="cuda")
    x = x.to(torch.bfloat16)
    x0 = x.clone()
    tpa.tree_rope(plan, x)
    tpa.tree_status_sync()
    assert torch.isfinite(x).all()
    pos = np.asarray(T.position_ids(w.parents, w.lengths))
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(index).integers(0, N, 48)]))
    ref = R.rope(x0[rows].double().cpu().numpy(), pos[rows])
    _check(x[rows], ref, torch.bfloat16, "sampled rows")


def test_rope_inverse_round_trip_and_autograd():
    _need_gpu()
    w = treegen.workload(3, 0)
    plan = tpa.tree_plan_build(w.parents, w.lengths)
    N = plan.num_tokens
    x = _draw(N, 2, 128, torch.float32, 3).cuda()
    y = tpa.tree_rope(plan, x.clone(), rotate_half=True)
    back = tpa.tree_rope(plan, y, rotate_half=True, inverse=True)
    tpa.tree_status_sync()
    assert float((back - x).abs().max()) <= 1e-5
    # the backward of the rotation is the inverse rotation of the incoming gradient
    xr = x.clone().requires_grad_(True)
    out = tpa.tree_rope_apply(xr, plan, 10000.0, True)
    gy = _draw(N, 2, 128, torch.float32, 4).cuda()
    (out * gy).sum().backward()
    pos = T.position_ids(w.parents, w.lengths)
    ref = R.rope(gy.double().cpu().numpy(), pos, 10000.0, True, inverse=True)
    _check(xr.grad, ref, torch.float32, "grad")
    assert torch.equal(x, xr.detach())  # the input is not modified in place


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rotate_half", [False, True])
@pytest.mark.parametrize("D", [128, 40])
def test_rope_qk_equals_two_calls(dtype, rotate_half, D):
    """tree_rope_qk rotates q and k in one launch exactly as two tree_rope calls
    (D = 128: the 16-byte chunk path; D = 40: the per-pair path), forward and
    inverse."""
    _need_gpu()
    parents, lengths = treegen.grpo_tree(1, prompt=150, n_leaves=3, lo=20, hi=90)
    plan = tpa.tree_plan_build(parents, lengths)
    N = plan.num_tokens
    for inverse in (False, True):
        q = _draw(N, 6, D, dtype, 1).cuda()
        k = _draw(N, 2, D, dtype, 2).cuda()
        q1, k1 = q.clone(), k.clone()
        tpa.tree_rope(plan, q1, rotate_half=rotate_half, inverse=inverse)
        tpa.tree_rope(plan, k1, rotate_half=rotate_half, inverse=inverse)
        tpa.tree_rope_qk(plan, q, k, rotate_half=rotate_half, inverse=inverse)
        tpa.tree_status_sync()
        assert torch.equal(q, q1) and torch.equal(k, k1)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_rope_at_positions_near_the_int32_limit(dtype):
    """A partition plan whose positions start at the largest offset the plan
    accepts (offset + N = 2^31 - 1): angles up to about 2.1e9 radians, formed
    and reduced modulo 2 pi in fp64, rotate at the same tolerances as small
    positions, in both pairings and both directions."""
    _need_gpu()
    w = treegen.workload(1, 0)
    N = int(np.sum(w.lengths))
    off = 2 ** 31 - 1 - N
    plan = tpa.tree_plan_build_partition(w.parents, w.lengths, [], off)
    pos = plan.field("pos_id").astype(np.int64)
    assert pos.min() == off and pos.max() > 2 ** 31 - 1 - N // 2
    assert np.array_equal(pos - off, np.asarray(T.position_ids(w.parents, w.lengths)))
    x = _draw(N, 2, 128, dtype, 9)
    for rotate_half in (False, True):
        for inverse in (False, True):
            got = tpa.tree_rope(plan, x.cuda(), 10000.0, rotate_half, inverse)
            tpa.tree_status_sync()
            ref = R.rope(x.double().numpy(), pos, 10000.0, rotate_half, inverse)
            _check(got, ref, dtype, f"rotate_half={rotate_half} inverse={inverse}")
