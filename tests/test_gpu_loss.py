"""GPU parity of the fused weighted tree cross-entropy (§3.1 eq. 3-5, §3.2
"Loss Weights") through the C-ABI, against the fp64 oracle.

Tolerances: fp32 logits: dlogits max-abs 1e-6 + 1e-5 relative, row losses
1e-5 relative + 1e-5 absolute; bf16 logits (the oracle reads the same bf16
values): dlogits add the bf16 storage rounding, 2^-8 |ref|. The total loss
is compared with the fp64 sum of the oracle's row losses at 1e-5 relative.
"""
import numpy as np
import pytest
import torch

import treegen
import tree_packed_attention_gb300 as tpa
from oracle import loss as LO
from oracle import trie as T

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _inputs(parents, lengths, V, dtype, seed, ignore=0.1, lam_kind="g/K"):
    N = int(np.sum(lengths))
    g = torch.Generator().manual_seed(seed)
    z = (torch.randn(N, V, generator=g) * 4).to(dtype)
    tokens = torch.randint(0, V, (N,), generator=g, dtype=torch.int32)
    drop = torch.rand(N, generator=g) < ignore
    tokens[drop] = -1
    if lam_kind == "g/K":
        lam = torch.as_tensor(T.token_weights(parents, lengths))
    else:  # any sign, some zero
        lam = torch.randn(N, generator=g, dtype=torch.float32)
        lam[torch.rand(N, generator=g) < 0.1] = 0.0
    return z, tokens, lam


def _check(z, tokens, lam, parents, lengths, gs, rows=None):
    plan = tpa.tree_plan_build(parents, lengths)
    zd, td, ld = z.cuda(), tokens.cuda(), lam.cuda()
    loss, row_loss, dz = tpa.tree_weighted_ce(plan, zd, td, ld, grad_scale=gs)
    tpa.tree_status_sync()
    rl, rrow, rdz = LO.weighted_ce(z, tokens.numpy(), lam.numpy().astype(np.float64), parents, lengths,
                                   gs, rows=rows)
    got_rows = row_loss.cpu().double() if rows is None else row_loss.cpu().double()[rows]
    got_dz = dz.cpu().double() if rows is None else dz.cpu().double()[rows]
    assert torch.allclose(got_rows, rrow, rtol=1e-5, atol=1e-5), float((got_rows - rrow).abs().max())
    bound = 1e-6 + 1e-5 * rdz.abs() + (2.0 ** -8 * rdz.abs() if z.dtype == torch.bfloat16 else 0.0)
    err = (got_dz - rdz).abs() - bound
    assert float(err.max()) <= 0, float((got_dz - rdz).abs().max())
    if rows is None:
        assert abs(float(loss) - rl) <= 1e-5 * max(1.0, abs(rl))
    return loss, row_loss, dz


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("seed", range(3))
def test_weighted_ce_matches_the_oracle_on_tries_and_forests(dtype, seed):
    _need_gpu()
    cases = [treegen.tiny_trie(seed), treegen.grpo_tree(seed, prompt=60, n_leaves=5, lo=5, hi=40),
             tuple(np.asarray(x) for x in treegen.random_forest(np.random.default_rng(seed), 30, 9))]
    for k, (parents, lengths) in enumerate(cases):
        for V in (8, 1000, 4104):
            z, tokens, lam = _inputs(parents, lengths, V, dtype, seed * 10 + k,
                                     lam_kind="g/K" if k % 2 == 0 else "any")
            _check(z, tokens, lam, parents, lengths, gs=1.0 if k != 1 else 0.37)


def test_weighted_ce_in_place_repeats_and_token_checks():
    _need_gpu()
    parents, lengths = treegen.grpo_tree(3, prompt=100, n_leaves=4, lo=20, hi=60)
    z, tokens, lam = _inputs(parents, lengths, 2048, torch.bfloat16, 5)
    plan = tpa.tree_plan_build(parents, lengths)
    zd, td, ld = z.cuda(), tokens.cuda(), lam.cuda()
    l1, r1, d1 = tpa.tree_weighted_ce(plan, zd, td, ld)
    l2, r2, d2 = tpa.tree_weighted_ce(plan, zd, td, ld)
    z2 = zd.clone()
    l3, r3, d3 = tpa.tree_weighted_ce(plan, z2, td, ld, in_place=True)
    tpa.tree_status_sync()
    assert d3.data_ptr() == z2.data_ptr()
    for a, b in ((l1, l2), (r1, r2), (d1, d2), (l1, l3), (r1, r3), (d1, d3)):
        assert torch.equal(a, b)
    # a token id past the vocabulary: its prediction is skipped and reported
    bad = td.clone()
    bad[3] = 5000
    tpa.tree_weighted_ce(plan, zd, bad, ld)
    with pytest.raises(tpa.TreeAttnError, match="vocab"):
        tpa.tree_status_sync()
    tpa.tree_status_sync()  # cleared


def test_weighted_ce_sampled_rows_on_the_grpo_workload():
    """Workload 3's trie (22,637 tokens; a 2048-token prompt with 16 leaves),
    V = 32,000 bf16 logits: sampled rows, including the prompt's last row
    (16 predictions) and leaf ends (none), against the oracle."""
    _need_gpu()
    w = treegen.workload(3)
    N = w.num_tokens
    z, tokens, lam = _inputs(w.parents, w.lengths, 32000, torch.bfloat16, 9)
    succ = LO.path_successors(w.parents, w.lengths)
    branch = [r for r in range(N) if len(succ[r]) > 1]
    ends = [r for r in range(N) if not succ[r]][:3]
    rng = np.random.default_rng(0)
    rows = sorted(set(branch + ends + [0, N - 1] + rng.integers(0, N, 12).tolist()))
    loss, row_loss, _ = _check(z, tokens, lam, w.parents, w.lengths, 1.0, rows=rows)
    # the total is the fixed-order sum of the row losses
    assert abs(float(loss) - float(row_loss.double().sum())) <= 1e-6 * max(1.0, abs(float(loss)))


@pytest.mark.parametrize("V,dtype", [(8, torch.bfloat16), (151936, torch.bfloat16),
                                     (151936, torch.float32), (262144, torch.float32)])
def test_weighted_ce_short_and_long_rows(V, dtype):
    """The smallest vocabulary (8) and long rows (bf16 and fp32 V = 151,936, fp32
    V = 262,144: a 1 MB row, far past what the kernel's second pass finds in
    L2): every row against the oracle, and a second call bit for bit the same."""
    _need_gpu()
    parents, lengths = treegen.tiny_trie(2)
    z, tokens, lam = _inputs(parents, lengths, V, dtype, 17, lam_kind="any")
    _check(z, tokens, lam, parents, lengths, 0.5)
    plan = tpa.tree_plan_build(parents, lengths)
    zd, td, ld = z.cuda(), tokens.cuda(), lam.cuda()
    a = tpa.tree_weighted_ce(plan, zd, td, ld, grad_scale=0.5)
    b = tpa.tree_weighted_ce(plan, zd, td, ld, grad_scale=0.5)
    tpa.tree_status_sync()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_weighted_ce_extreme_and_flat_rows(dtype):
    """Logits up to about 1e5 in magnitude (each row's softmax all but
    one-hot, every other exponential underflowing), rows whose logits are
    all equal (a uniform softmax), and rows with one spike of 3e4 over zeros,
    with the g/K weights: against the oracle in fp64 at the same tolerances
    as ordinary logits, since the kernel subtracts the row maximum before the
    exponent (an error that grew with |z| would fail here)."""
    _need_gpu()
    parents, lengths = treegen.tiny_trie(1)
    z, tokens, lam = _inputs(parents, lengths, 4096, torch.float32, 23)
    z = z * 5e3
    z[1::5] = 7.0
    z[2::5] = 0.0
    z[2::5, 11] = 3e4
    z = z.to(dtype)
    loss, row_loss, dz = _check(z, tokens, lam, parents, lengths, 1.0)
    assert torch.isfinite(dz).all() and torch.isfinite(row_loss).all()
