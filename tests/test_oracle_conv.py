"""Pins for the tree-correct causal conv oracle (CPU, no GPU).

App. A.3's claim is the pin: the segment-by-segment convolution with parent
context equals a plain causal conv1d run on each root-to-leaf path on its own.
The plain conv is itself pinned against numpy's convolution."""
import numpy as np
import pytest
import torch

import treegen
from oracle import conv as CV
from oracle import trie as T


def _rand(shape, seed):
    return torch.from_numpy(np.random.default_rng(seed).standard_normal(shape))


@pytest.mark.parametrize("K", [1, 2, 4, 7])
def test_plain_causal_conv_matches_numpy_convolution(K):
    x, w, b = _rand((23, 5), K), _rand((5, K), K + 1), _rand((5,), K + 2)
    y = CV.causal_conv(x, w, b, act="none").numpy()
    for c in range(5):
        # np.convolve flips its kernel: weight index K-1 meets the current token
        ref = np.convolve(x[:, c].numpy(), w[c].numpy()[::-1])[:23] + b[c].item()
        assert np.allclose(y[:, c], ref, atol=1e-12)
    assert torch.allclose(CV.causal_conv(x, w, b, act="silu"), torch.nn.functional.silu(torch.from_numpy(y)))


@pytest.mark.parametrize("K", [1, 3, 4, 8])
@pytest.mark.parametrize("act", ["none", "silu"])
def test_tree_conv_equals_conv_on_every_path(K, act):
    rng = np.random.default_rng(K)
    cases = [treegen.workload(1, 0), treegen.workload(1, 3)]
    for _ in range(4):  # forests with segments shorter than K-1: context from grandparents
        S = int(rng.integers(2, 16))
        parents = [-1] + [int(rng.integers(-1, s)) for s in range(1, S)]
        lengths = [int(v) for v in rng.integers(1, 6, S)]
        cases.append(type("W", (), {"parents": parents, "lengths": lengths})())
    for w in cases:
        N = int(np.sum(w.lengths))
        x, wt, b = _rand((N, 6), N), _rand((6, K), N + 1), _rand((6,), N + 2)
        y = CV.tree_conv(w.parents, w.lengths, x, wt, b, act)
        for _, ids in T.base_serialization(w.parents, w.lengths):
            ref = CV.causal_conv(x[ids], wt, b, act)
            assert torch.allclose(y[ids], ref, atol=1e-12)


def test_delta_kernel_is_the_identity_and_one_tap_is_pointwise():
    w = treegen.workload(1, 0)
    N = int(np.sum(w.lengths))
    x = _rand((N, 4), 0)
    delta = torch.zeros(4, 4, dtype=torch.float64)
    delta[:, 3] = 1.0  # the current token only
    assert torch.equal(CV.tree_conv(w.parents, w.lengths, x, delta, None, "none"), x)
    one = _rand((4, 1), 1)
    assert torch.allclose(CV.tree_conv(w.parents, w.lengths, x, one, None, "none"), x * one[:, 0])
