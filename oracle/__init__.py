"""CPU oracle for tree-packed attention: test infrastructure only.

A plain, slow, fp64 restatement of what tree-packed attention computes, written
from "Tree Training: Accelerating Agentic LLMs Training via Shared Prefix Reuse"
(arXiv 2511.00413): the trie and DFS serialization (§3.1, eq. 7-8), the tree
attention mask (§3.2 "Attention Mask"; App. A.1), tree position ids (§3.2
eq. 9) and RoPE at them, the per-token loss weight g_n/K (§3.1 eq. 2-4; §3.2
"Loss Weights") and its general form for any path weights, and plain
masked-softmax attention with its analytic backward.

Only the test suite, the package's smoke check and the benchmark's CPU
baseline leg may import this package. It shares no code with the CUDA path
(``tree_packed_attention_gb300``) and imports nothing from it; inputs come
from the separate seeded generator module ``treegen``.

Modules:
  trie      -- validation, children, DFS layout (eq. 8), ancestors, g_n, K,
               position ids (eq. 9), weights g_n/K, POR (eq. 12)
  mask      -- the dense mask built literally as in App. A.1, the
               common-path mask of §3.2, per-row visible intervals
  tiles     -- tile visibility map by brute-force counting, the backward
               row ranges, work lists and orders
  attention -- fp64 forward (o, lse) and analytic backward (dq, dk, dv)
  conv      -- the tree-correct causal depthwise conv of App. A.3 (eq. 11),
               written per token over its root-to-leaf path predecessors,
               in torch fp64 so autograd gives its backward
  partition -- node-boundary partitions under a token cap by brute force,
               their validity, App. B.2 gateway lengths and B.4 eq. 17
               position offsets, peak tokens along a path (§3.3)
  rope      -- rotary position embedding at the eq. 9 position ids
               (§3.2 "Position Embedding"); trie.path_weight_tokens gives the
               general per-token weights lambda_t of §3.1 for any path weights

Parity pins: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py`` against the pages' worked numbers, closed forms,
library routines (torch SDPA, autograd, gradcheck) or brute force. The tile
work orders (``fwd_order``, ``bwd_order``, ``qp_order`` in ``tiles.plan_fields``)
and the q-tile pair lists are scheduling conventions of this library, not of
the pages; they are pinned only by invariants (permutation, ordering, union)
-- parity unpinned by the pages.
"""
