"""Seeded synthetic inputs for tree-packed attention.

This module only draws random trie structures and random tensors. It holds
none of the method's arithmetic (no DFS layout, no mask, no weights, no
attention), so that both the CPU oracle and the CUDA path can take their
inputs from it without sharing any computation.

Workload shapes follow the tree-training paper ("Tree Training: Accelerating
Agentic LLMs Training via Shared Prefix Reuse", arXiv 2511.00413): RL rollouts
with one prompt and many completions, and sparse, unbalanced multi-turn
agentic trees (§4.4, Fig. 6). The real trajectories of §4.4 are not
available; these generators stand in for their stated shapes.

A trie is returned as ``(parents, lengths)``: ``parents[s]`` is the parent
segment id of segment ``s`` (``-1`` for a root) and ``lengths[s]`` is the
number of tokens of segment ``s``. Several roots make a packed forest.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass

import numpy as np

__all__ = [
    "Workload",
    "tiny_trie",
    "chain",
    "grpo_tree",
    "agentic_tree",
    "packed_tries",
    "random_forest",
    "workload",
    "WORKLOADS",
    "draw_tensors",
]


@dataclass(frozen=True)
class Workload:
    """A named synthetic workload: trie structure plus head configuration."""

    name: str
    parents: np.ndarray  # int32 [S]
    lengths: np.ndarray  # int32 [S]
    hq: int
    hkv: int
    head_dim: int
    dtype: str  # "fp32" or "bf16"

    @property
    def num_tokens(self) -> int:
        return int(self.lengths.sum())


def _i32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def tiny_trie(seed: int = 0):
    """Root -> 2 children -> 4 grandchildren, lengths uniform in [8, 32]."""
    rng = np.random.default_rng(seed)
    parents = [-1, 0, 0, 1, 1, 2, 2]
    lengths = rng.integers(8, 33, size=7)
    return _i32(parents), _i32(lengths)


def chain(n_tokens: int = 4096):
    """A branchless trie: one segment of ``n_tokens`` tokens."""
    return _i32([-1]), _i32([n_tokens])


def grpo_tree(seed: int = 0, rng: np.random.Generator | None = None,
              prompt: int = 2048, n_leaves: int = 16, lo: int = 512, hi: int = 2048):
    """One prompt root with ``n_leaves`` completion leaves of length U{lo..hi}."""
    if rng is None:
        rng = np.random.default_rng(seed)
    leaves = rng.integers(lo, hi + 1, size=n_leaves)
    parents = [-1] + [0] * n_leaves
    lengths = [prompt] + [int(x) for x in leaves]
    return _i32(parents), _i32(lengths)


def agentic_tree(seed: int = 0, total: int = 65536, max_depth: int = 6,
                 lo: int = 256, hi: int = 4096):
    """Multi-turn agentic tree.

    The root has depth 1. Breadth-first growth: every node of depth below
    ``max_depth`` draws b ~ U{1,2,3} children; segment lengths are
    round(exp(U[ln lo, ln hi])). Growth stops when the token total reaches
    ``total``; the last segment is cut so the total is exact. If the tree of
    depth ``max_depth`` runs out of nodes first, it is drawn again with the
    next generator state.
    """
    rng = np.random.default_rng(seed)
    lnlo, lnhi = np.log(lo), np.log(hi)

    def draw_len() -> int:
        return int(np.round(np.exp(rng.uniform(lnlo, lnhi))))

    while True:
        parents = [-1]
        lengths = [min(draw_len(), total)]
        depth = [1]
        tot = lengths[0]
        queue = deque([0])
        while queue and tot < total:
            n = queue.popleft()
            if depth[n] >= max_depth:
                continue
            b = int(rng.integers(1, 4))
            for _ in range(b):
                L = draw_len()
                if tot + L >= total:
                    L = total - tot
                parents.append(n)
                lengths.append(L)
                depth.append(depth[n] + 1)
                tot += L
                queue.append(len(parents) - 1)
                if tot >= total:
                    break
        if tot == total:
            return _i32(parents), _i32(lengths)


def packed_tries(seed: int = 0, n_tries: int = 32, total: int = 131072,
                 cap_lo: int = 2048):
    """``n_tries`` GRPO-shaped tries packed into one row (a forest).

    Caps: c_t = cap_lo + round(u_t * (total - n_tries*cap_lo) / sum(u)), u ~ U[0,1),
    the rounding residual going to the largest cap so the caps sum to
    ``total``. Each trie is drawn in the GRPO shape (prompt 2048, 16 leaves
    U{512..2048}), every length is scaled by c_t / (its drawn total) and
    rounded (at least 1), and the last leaf takes the residual.
    """
    rng = np.random.default_rng(seed)
    u = rng.uniform(0.0, 1.0, size=n_tries)
    spare = total - n_tries * cap_lo
    caps = cap_lo + np.round(u * spare / u.sum()).astype(np.int64)
    caps[int(np.argmax(caps))] += total - int(caps.sum())
    parents: list[int] = []
    lengths: list[int] = []
    for t in range(n_tries):
        p, L = grpo_tree(rng=rng)
        L = L.astype(np.float64)
        scaled = np.maximum(1, np.round(L * caps[t] / L.sum())).astype(np.int64)
        scaled[-1] = caps[t] - int(scaled[:-1].sum())
        assert scaled[-1] >= 1
        base = len(parents)
        parents.extend([-1 if x < 0 else int(x) + base for x in p])
        lengths.extend(int(x) for x in scaled)
    return _i32(parents), _i32(lengths)


def random_forest(rng: np.random.Generator, n_segments: int, max_len: int = 40,
                  n_roots: int = 1, shuffle: bool = True):
    """A random forest for property tests.

    Segment ids are optionally shuffled so that parents may follow their
    children in the id order.
    """
    n_roots = max(1, min(n_roots, n_segments))
    parents = np.full(n_segments, -1, dtype=np.int64)
    for s in range(n_roots, n_segments):
        parents[s] = int(rng.integers(0, s))
    lengths = rng.integers(1, max_len + 1, size=n_segments)
    if shuffle and n_segments > 1:
        perm = rng.permutation(n_segments)  # new id of old segment s is perm[s]
        new_parents = np.full(n_segments, -1, dtype=np.int64)
        new_lengths = np.zeros(n_segments, dtype=np.int64)
        for s in range(n_segments):
            new_parents[perm[s]] = -1 if parents[s] < 0 else perm[parents[s]]
            new_lengths[perm[s]] = lengths[s]
        parents, lengths = new_parents, new_lengths
    return _i32(parents), _i32(lengths)


def workload(index: int, seed: int = 0) -> Workload:
    """The five synthetic workloads, numbered 1..5."""
    if index == 1:
        p, L = tiny_trie(seed)
        return Workload("tiny-trie-7seg-fp32-h1-d64", p, L, 1, 1, 64, "fp32")
    if index == 2:
        p, L = chain(4096)
        return Workload("chain-4096-bf16-h16-d128", p, L, 16, 16, 128, "bf16")
    if index == 3:
        p, L = grpo_tree(seed)
        return Workload("grpo-1x2048+16leaves-bf16-hq32-hkv8-d128", p, L, 32, 8, 128, "bf16")
    if index == 4:
        p, L = agentic_tree(seed)
        return Workload("agentic-depth6-64k-bf16-h16-d128", p, L, 16, 16, 128, "bf16")
    if index == 5:
        p, L = packed_tries(seed)
        return Workload("packed-32-tries-128k-bf16-hq64-hkv8-d128", p, L, 64, 8, 128, "bf16")
    if index == 6:  # workload 5's shape at a quarter of the size (profiling captures)
        p, L = packed_tries(seed, n_tries=8, total=32768)
        return Workload("packed-8-tries-32k-bf16-hq64-hkv8-d128", p, L, 64, 8, 128, "bf16")
    raise ValueError(f"unknown workload {index}")


WORKLOADS = (1, 2, 3, 4, 5)


def draw_tensors(n_tokens: int, hq: int, hkv: int, head_dim: int, dtype: str = "bf16",
                 seed: int = 0, with_grad_out: bool = True):
    """q, k, v (and dO) drawn as fp32 N(0,1) from one seeded CPU generator.

    Draw order is q [N,hq,D], k [N,hkv,D], v [N,hkv,D], dO [N,hq,D]; each is
    then rounded to ``dtype``. The CPU tensors returned are the exact values
    both sides consume (the oracle upcasts them to fp64).
    """
    import torch

    g = torch.Generator(device="cpu").manual_seed(seed)
    tdt = {"bf16": torch.bfloat16, "fp32": torch.float32}[dtype]
    q = torch.randn(n_tokens, hq, head_dim, generator=g, dtype=torch.float32).to(tdt)
    k = torch.randn(n_tokens, hkv, head_dim, generator=g, dtype=torch.float32).to(tdt)
    v = torch.randn(n_tokens, hkv, head_dim, generator=g, dtype=torch.float32).to(tdt)
    if not with_grad_out:
        return q, k, v
    do = torch.randn(n_tokens, hq, head_dim, generator=g, dtype=torch.float32).to(tdt)
    return q, k, v, do


def draw_gdn(n_tokens: int, hk: int, hv: int, head_dim: int = 128, dtype: str = "bf16", seed: int = 0,
             with_state: bool = True):
    """Inputs of a Gated DeltaNet layer, as its kernel receives them.

    From one seeded CPU generator, in this order: q, k [N, hk, D] drawn N(0,1)
    and scaled to unit L2 norm per head (the layer normalises them), v
    [N, hv, D] N(0,1), g [N, hv] = -U(0, 0.5) (log decays, per-token decay
    exp(g) in (0.6, 1]), beta [N, hv] U(0, 1), and the initial state
    [hv, D, D] N(0, 0.3^2). q, k, v are rounded to ``dtype``; g, beta and the
    state stay fp32.
    """
    import torch

    g = torch.Generator(device="cpu").manual_seed(seed)
    tdt = {"bf16": torch.bfloat16, "fp32": torch.float32}[dtype]

    def unit(x):
        return x / x.norm(dim=-1, keepdim=True)

    q = unit(torch.randn(n_tokens, hk, head_dim, generator=g)).to(tdt)
    k = unit(torch.randn(n_tokens, hk, head_dim, generator=g)).to(tdt)
    v = torch.randn(n_tokens, hv, head_dim, generator=g).to(tdt)
    lg = -0.5 * torch.rand(n_tokens, hv, generator=g)
    beta = torch.rand(n_tokens, hv, generator=g)
    s0 = 0.3 * torch.randn(hv, head_dim, head_dim, generator=g) if with_state else None
    return q, k, v, lg, beta, s0
