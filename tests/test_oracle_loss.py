"""Pins for the weighted tree cross-entropy oracle (§3.1 eq. 3-5), CPU only.

The pin is the pages' identity itself: with lambda_t = g_t / K, the tree loss
over unique tokens equals the average over root-to-leaf paths of each path's
own next-token loss, computed here by laying every path out on its own and
calling torch's cross_entropy on it; its gradient, by autograd through those
per-path losses, equals the oracle's closed form.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import loss as LO
from oracle import trie as T


def _forest(seed):
    rng = np.random.default_rng(seed)
    S = int(rng.integers(1, 12))
    parents = [-1] + [int(rng.integers(-1, s)) if rng.random() < 0.15 else int(rng.integers(0, s))
                      for s in range(1, S)]
    lengths = [int(x) for x in rng.integers(1, 9, S)]
    return parents, lengths


def _per_path_objective(z, tokens, parents, lengths):
    """(1/K_trie) * sum over paths of the path's summed next-token NLL, the
    paths laid out on their own (eq. 1-3)."""
    K = T.paths_per_trie(parents)
    _, trie_id = T.tries(parents)
    total = z.new_zeros(())
    for leaf, ids in T.base_serialization(parents, lengths):
        if len(ids) < 2:
            continue
        idx = torch.as_tensor(ids)
        nll = F.cross_entropy(z[idx[:-1]], torch.as_tensor(np.asarray(tokens)[ids[1:]]), reduction="sum")
        total = total + nll / K[trie_id[leaf]]
    return total


@pytest.mark.parametrize("seed", range(12))
def test_tree_loss_equals_the_average_of_per_path_losses(seed):
    parents, lengths = _forest(seed)
    N = sum(lengths)
    V = 37
    g = torch.Generator().manual_seed(seed)
    z = torch.randn(N, V, generator=g, dtype=torch.float64) * 3
    tokens = torch.randint(0, V, (N,), generator=g).numpy()
    lam = T.token_weights(parents, lengths).astype(np.float64)
    # the fp32-rounded g/K differ from g/K by under 2^-24 relative
    exact = np.array([T.paths_through(parents)[s] / T.paths_per_trie(parents)[T.tries(parents)[1][s]]
                      for s in T.token_segments(parents, lengths)])
    loss, row_loss, dz = LO.weighted_ce(z, tokens, exact, parents, lengths)
    zz = z.clone().requires_grad_(True)
    ref = _per_path_objective(zz, tokens, parents, lengths)
    ref.backward()
    assert abs(loss - float(ref)) <= 1e-10 * max(1.0, abs(float(ref)))
    assert torch.allclose(dz, zz.grad, atol=1e-12)
    assert abs(float(row_loss.sum()) - loss) <= 1e-12 * max(1.0, abs(loss))
    # and with the fp32 weights the library uses: within their rounding
    loss32, _, _ = LO.weighted_ce(z, tokens, lam, parents, lengths)
    assert abs(loss32 - loss) <= 2 ** -23 * sum(abs(float(x)) for x in row_loss) + 1e-12


def test_chain_is_plain_shifted_cross_entropy_and_special_cases():
    N, V = 50, 20
    g = torch.Generator().manual_seed(1)
    z = torch.randn(N, V, generator=g, dtype=torch.float64)
    tokens = torch.randint(0, V, (N,), generator=g)
    loss, row_loss, dz = LO.weighted_ce(z, tokens.numpy(), np.ones(N), [-1], [N], grad_scale=0.5)
    ref = F.cross_entropy(z[:-1], tokens[1:], reduction="sum")
    assert abs(loss - float(ref)) < 1e-10
    assert float(row_loss[-1]) == 0.0 and torch.all(dz[-1] == 0)  # the last token predicts nothing
    # dz rows of predicting positions sum to zero (softmax minus one-hot), times the weight
    assert torch.allclose(dz[:-1].sum(dim=1), torch.zeros(N - 1, dtype=torch.float64), atol=1e-12)
    # uniform logits: every prediction costs log V
    loss_u, _, _ = LO.weighted_ce(torch.zeros(N, V), tokens.numpy(), np.ones(N), [-1], [N])
    assert abs(loss_u - (N - 1) * np.log(V)) < 1e-9
    # zero weights: nothing
    loss_0, _, dz0 = LO.weighted_ce(z, tokens.numpy(), np.zeros(N), [-1], [N])
    assert loss_0 == 0.0 and torch.all(dz0 == 0)


def test_successors_of_a_branching_trie():
    # root (segment 0) holds DFS tokens 0-2; its children a (segment 1) and
    # b (segment 2) follow in ascending id, a's child c (segment 3) before b:
    # a = [3, 4], c = [5], b = [6]
    parents, lengths = [-1, 0, 0, 1], [3, 2, 1, 1]
    succ = LO.path_successors(parents, lengths)
    assert succ == [[1], [2], [3, 6], [4], [5], [], []]
