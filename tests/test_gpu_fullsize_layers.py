"""Full-size GPU parity of the tree-correct causal conv (App. A.3) and the GDN
tree state routing (eq. 10, App. A.2) on the packed workload (32 tries,
131,072 tokens), and of the fused weighted cross-entropy (§3.1 eq. 3-5) on
the packed shape at 32,768 tokens with a 151,936-entry vocabulary, with the
inputs and the launch configurations that `bench.py --op conv`, `--op gdn`
and `--op ce` time.

Both layers are independent per channel (the conv is depthwise) or per value
head (each GDN value head reads only its own query/key head), so the fp64
oracle run on a sample of channels or value heads is exactly the oracle of
the whole layer restricted to them: every token, every branch point and
every segment end state of the sampled columns is compared, at the
tolerances of the small-case tests. A cross-entropy row depends only on its
own logits and the tokens that follow it on its paths, so sampled rows are
compared one by one.
"""
import numpy as np
import pytest
import torch

import treegen
import tree_packed_attention_gb300 as tpa
from oracle import conv as CV
from oracle import gdn as GD
from oracle import loss as LO

pytestmark = pytest.mark.gpu

# channels in both launch rows of channel groups (2048 channels a row), at
# the edges of 8-channel chunks and of the rows
CONV_CHANNELS = [0, 1, 7, 8, 1023, 2047, 2048, 2055, 3001, 4088, 4095]
# value heads of the 32, with their query/key heads (h // 2): the second
# head of the first pair, and the first head of the last pair
GDN_VALUE_HEADS = [1, 30]


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_conv_full_size_sampled_channels():
    """C = 4096, K = 4, SiLU, bf16 x and dy, fp32 weight and bias: y, dx,
    dweight and dbias of the sampled channels over all 131,072 tokens.
    Tolerances: y and dx stored in bf16, |err| <= 2^-8 |ref| + 1e-3;
    dweight / dbias (fp32 sums over every token) 1e-4 of the largest."""
    _need_gpu()
    w = treegen.workload(5)
    plan = tpa.tree_plan_build(w.parents, w.lengths)
    N, C, K = plan.num_tokens, 4096, 4
    gen = torch.Generator(device="cuda").manual_seed(0)
    x = torch.randn(N, C, device="cuda", generator=gen).to(torch.bfloat16)
    dy = torch.randn(N, C, device="cuda", generator=gen).to(torch.bfloat16)
    wt = torch.randn(C, K, device="cuda", generator=gen) * 0.5
    b = torch.randn(C, device="cuda", generator=gen)
    y = torch.empty_like(x)
    tpa.tree_conv_fwd(plan, x, wt, b, out=y)
    dx, dw, db = tpa.tree_conv_bwd(plan, x, wt, b, dy)
    tpa.tree_status_sync()

    cols = torch.tensor(CONV_CHANNELS, device="cuda")
    xr = x[:, cols].double().cpu().requires_grad_(True)
    wr = wt[cols].double().cpu().requires_grad_(True)
    br = b[cols].double().cpu().requires_grad_(True)
    yr = CV.tree_conv(w.parents, w.lengths, xr, wr, br, "silu")
    yr.backward(dy[:, cols].double().cpu())

    for name, got, ref in [("y", y[:, cols], yr.detach()), ("dx", dx[:, cols], xr.grad)]:
        d = (got.double().cpu() - ref).abs()
        excess = float((d - (2.0 ** -8 * ref.abs() + 1e-3)).max())
        assert excess <= 0, f"{name}: bf16 bound exceeded by {excess:.3g}"
    for name, got, ref in [("dweight", dw[cols], wr.grad), ("dbias", db[cols], br.grad)]:
        err = float((got.double().cpu() - ref).abs().max())
        assert err <= 1e-4 * max(1.0, float(ref.abs().max())), f"{name}: max abs err {err:.3g}"


def test_gdn_full_size_sampled_value_heads():
    """16 query/key heads, 32 value heads, head_dim 128, bf16 q/k/v (unit-norm
    q and k), the bench's gates: outputs and segment end states of the
    sampled value heads over all 131,072 tokens. Tolerance: fp32 arithmetic
    on the same bf16 inputs, 2e-4 + 1e-4 |ref|, plus 2^-8 |ref| for the
    bf16-stored outputs."""
    _need_gpu()
    w = treegen.workload(5)
    plan = tpa.tree_plan_build(w.parents, w.lengths)
    N, hk, hv = plan.num_tokens, 16, 32
    gen = torch.Generator(device="cuda").manual_seed(0)

    def unit(t):
        return t / t.norm(dim=-1, keepdim=True)

    q = unit(torch.randn(N, hk, 128, device="cuda", generator=gen)).to(torch.bfloat16)
    k = unit(torch.randn(N, hk, 128, device="cuda", generator=gen)).to(torch.bfloat16)
    v = torch.randn(N, hv, 128, device="cuda", generator=gen).to(torch.bfloat16)
    g = -0.5 * torch.rand(N, hv, device="cuda", generator=gen)
    beta = torch.rand(N, hv, device="cuda", generator=gen)
    o, states = tpa.tree_gdn_fwd(plan, q, k, v, g, beta)
    tpa.tree_status_sync()

    G = hv // hk
    for h in GDN_VALUE_HEADS:
        hq = h // G
        ro, rs = GD.tree_forward(q[:, hq:hq + 1].cpu(), k[:, hq:hq + 1].cpu(), v[:, h:h + 1].cpu(),
                                 g[:, h:h + 1].cpu(), beta[:, h:h + 1].cpu(), w.parents, w.lengths)
        for name, got, ref, store in [("o", o[:, h:h + 1], ro, 2.0 ** -8),
                                      ("segment states", states[:, h:h + 1], rs, 0.0)]:
            d = (got.double().cpu() - ref).abs()
            bound = 2e-4 + 1e-4 * ref.abs() + store * ref.abs()
            excess = float((d - bound).max())
            assert excess <= 0, f"{name} of value head {h}: max err {float(d.max()):.3g}"


def test_weighted_ce_full_size_sampled_rows():
    """bf16 logits [32768, 151936] drawn N(0, 9), every token predicted,
    lambda = g/K: the row losses and dlogits of the rows before branch points
    (several predictions each), of leaf ends (none), of the first and last
    rows and of random rows, against the oracle; the total is the
    fixed-order sum of all row losses. Tolerances as the small-case tests:
    row losses 1e-5 relative + 1e-5, dlogits 1e-6 + (1e-5 + 2^-8) |ref|."""
    _need_gpu()
    w = treegen.workload(6)
    plan = tpa.tree_plan_build(w.parents, w.lengths)
    N, V = plan.num_tokens, 151936
    gen = torch.Generator(device="cuda").manual_seed(0)
    z = torch.empty(N, V, dtype=torch.bfloat16, device="cuda")
    for r0 in range(0, N, 4096):
        r1 = min(N, r0 + 4096)
        z[r0:r1] = (torch.randn(r1 - r0, V, device="cuda", generator=gen) * 3).to(torch.bfloat16)
    tokens = torch.randint(0, V, (N,), device="cuda", generator=gen, dtype=torch.int32)
    lam = torch.as_tensor(tpa.tree_weights(plan), device="cuda")
    loss, row_loss, dz = tpa.tree_weighted_ce(plan, z, tokens, lam)
    tpa.tree_status_sync()

    succ = LO.path_successors(w.parents, w.lengths)
    branch = [r for r in range(N) if len(succ[r]) > 1]
    ends = [r for r in range(N) if not succ[r]]
    rng = np.random.default_rng(0)
    rows = sorted(set(branch[:96] + ends[:16] + [0, N - 1] + rng.integers(0, N, 64).tolist()))
    # the oracle reads only the sampled rows' logits
    zc = torch.empty(N, V, dtype=torch.bfloat16)
    zc[rows] = z[rows].cpu()
    _, rrow, rdz = LO.weighted_ce(zc, tokens.cpu().numpy(), lam.cpu().numpy().astype(np.float64),
                                  w.parents, w.lengths, 1.0, rows=rows)
    got_rows = row_loss.cpu().double()[rows]
    assert torch.allclose(got_rows, rrow, rtol=1e-5, atol=1e-5), float((got_rows - rrow).abs().max())
    got_dz = dz[rows].cpu().double()
    bound = 1e-6 + (1e-5 + 2.0 ** -8) * rdz.abs()
    assert float(((got_dz - rdz).abs() - bound).max()) <= 0, float((got_dz - rdz).abs().max())
    assert abs(float(loss) - float(row_loss.double().sum())) <= 1e-6 * max(1.0, abs(float(loss)))
