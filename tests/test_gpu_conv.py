"""GPU parity of the tree-correct causal conv (C-ABI kernels) against the
fp64 oracle (App. A.3), forward and backward.

Tolerances: fp32 storage max-abs 1e-5 on y and dx, 1e-4 relative to the
largest |dweight| / |dbias| (sums over every token). bf16 storage: each
stored value rounded once, |err| <= 2^-8 |ref| + 1e-3 (fp32 sums of K
products of bf16 inputs).
"""
import numpy as np
import pytest
import torch

import treegen
import tree_packed_attention_gb300 as tpa
from oracle import conv as CV

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _cases(rng):
    out = [(treegen.workload(1, 0).parents, treegen.workload(1, 0).lengths),
           (treegen.workload(3, 0).parents, treegen.workload(3, 0).lengths)]
    for _ in range(3):  # short segments: context from grandparents and beyond
        S = int(rng.integers(2, 40))
        parents = [-1] + [int(rng.integers(-1, s)) for s in range(1, S)]
        out.append((parents, [int(v) for v in rng.integers(1, 9, S)]))
    return out


def _cmp(got, ref, dtype, name, scale=None):
    got = got.double().cpu()
    d = (got - ref).abs()
    if dtype == torch.float32:
        tol = 1e-5 if scale is None else 1e-4 * max(1.0, scale)
        assert float(d.max()) <= tol, f"{name}: max abs err {float(d.max()):.3g}"
    else:
        bound = 2.0 ** -8 * ref.abs() + 1e-3
        assert float((d - bound).max()) <= 0, f"{name}: bf16 bound exceeded by {float((d - bound).max()):.3g}"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K", [1, 2, 4, 6, 8])
def test_conv_forward_and_backward_match_oracle(dtype, K):
    _need_gpu()
    rng = np.random.default_rng(K)
    for parents, lengths in _cases(rng):
        plan = tpa.tree_plan_build(parents, lengths)
        N = plan.num_tokens
        for C, act, with_bias in [(8, "silu", True), (64, "none", False)]:
            g = torch.Generator().manual_seed(N + C)
            x = torch.randn(N, C, generator=g).to(dtype)
            w = torch.randn(C, K, generator=g) * 0.5
            b = torch.randn(C, generator=g) if with_bias else None
            dy = torch.randn(N, C, generator=g).to(dtype)
            y = tpa.tree_conv_fwd(plan, x.cuda(), w.cuda(), b.cuda() if b is not None else None, act)
            dx, dw, db = tpa.tree_conv_bwd(plan, x.cuda(), w.cuda(), b.cuda() if b is not None else None,
                                           dy.cuda(), act)
            tpa.tree_status_sync()
            xr = x.double().requires_grad_(True)
            wr = w.double().requires_grad_(True)
            br = b.double().requires_grad_(True) if b is not None else None
            yr = CV.tree_conv(parents, lengths, xr, wr, br, act)
            yr.backward(dy.double())
            _cmp(y, yr.detach(), dtype, f"y K={K} C={C}")
            _cmp(dx, xr.grad, dtype, f"dx K={K} C={C}")
            _cmp(dw, wr.grad, torch.float32, "dweight", float(wr.grad.abs().max()))
            if b is not None:
                _cmp(db, br.grad, torch.float32, "dbias", float(br.grad.abs().max()))
            else:
                assert db is None


@pytest.mark.parametrize("C", [2056, 4096])
def test_conv_wide_channels_use_every_channel_group(C):
    """Channel counts past one launch row of channel groups (grid.y > 1) and,
    for C = 2056, a last group that holds only part of its channels."""
    _need_gpu()
    parents, lengths = [-1, 0, 0, 1, 2, 2], [9, 5, 3, 12, 1, 7]
    plan = tpa.tree_plan_build(parents, lengths)
    N, K = plan.num_tokens, 4
    g = torch.Generator().manual_seed(C)
    x = torch.randn(N, C, generator=g).to(torch.bfloat16)
    w = torch.randn(C, K, generator=g) * 0.5
    b = torch.randn(C, generator=g)
    dy = torch.randn(N, C, generator=g).to(torch.bfloat16)
    y = tpa.tree_conv_fwd(plan, x.cuda(), w.cuda(), b.cuda(), "silu")
    dx, dw, db = tpa.tree_conv_bwd(plan, x.cuda(), w.cuda(), b.cuda(), dy.cuda(), "silu")
    tpa.tree_status_sync()
    xr = x.double().requires_grad_(True)
    wr = w.double().requires_grad_(True)
    br = b.double().requires_grad_(True)
    yr = CV.tree_conv(parents, lengths, xr, wr, br, "silu")
    yr.backward(dy.double())
    _cmp(y, yr.detach(), torch.bfloat16, f"y C={C}")
    _cmp(dx, xr.grad, torch.bfloat16, f"dx C={C}")
    _cmp(dw, wr.grad, torch.float32, "dweight", float(wr.grad.abs().max()))
    _cmp(db, br.grad, torch.float32, "dbias", float(br.grad.abs().max()))


def test_conv_backward_repeats_bit_for_bit_and_autograd_runs_the_kernels():
    _need_gpu()
    w = treegen.workload(4)
    plan = tpa.tree_plan_build(w.parents, w.lengths)
    N, C = plan.num_tokens, 256
    g = torch.Generator(device="cuda").manual_seed(0)
    x = torch.randn(N, C, device="cuda", generator=g).to(torch.bfloat16)
    wt = torch.randn(C, 4, device="cuda", generator=g)
    b = torch.randn(C, device="cuda", generator=g)
    dy = torch.randn(N, C, device="cuda", generator=g).to(torch.bfloat16)
    r1 = tpa.tree_conv_bwd(plan, x, wt, b, dy)
    r2 = tpa.tree_conv_bwd(plan, x, wt, b, dy)
    tpa.tree_status_sync()
    for a, c in zip(r1, r2):
        assert torch.equal(a, c)
    xr = x.clone().requires_grad_(True)
    wr = wt.clone().requires_grad_(True)
    br = b.clone().requires_grad_(True)
    y = tpa.tree_conv(xr, wr, br, plan)
    y.backward(dy)
    assert torch.equal(y, tpa.tree_conv_fwd(plan, x, wt, b))
    assert torch.equal(xr.grad, r1[0]) and torch.equal(wr.grad, r1[1]) and torch.equal(br.grad, r1[2])
