"""Rotary position embedding at tree position ids (fp64, numpy): test infrastructure only.

Tree Training (arXiv 2511.00413) §3.2 "Position Embedding": every token takes
the position id of eq. 9 (``trie.position_ids``), the one it has in each
standalone root-to-leaf sequence, so that RoPE gives the per-path result. The
rotation is RoFormer's rotary matrix (Su et al. 2023): in each head, dimension
pair i turns by the angle pos * theta_i with theta_i = base^(-2i/D).

Two pairings of the D dimensions are in use; the pages name neither, so both
are offered: (2i, 2i+1), RoFormer's own, and (i, i + D/2), the split-halves
layout. ``inverse`` turns by the opposite angle (the transpose of the
rotation, which is its backward and its inverse).
"""
import numpy as np


def rope(x, pos, base=10000.0, rotate_half=False, inverse=False):
    """x[N, H, D] rotated at positions pos[N]; fp64 result."""
    x = np.asarray(x, dtype=np.float64)
    N, H, D = x.shape
    assert D % 2 == 0
    i = np.arange(D // 2, dtype=np.float64)
    theta = float(base) ** (-2.0 * i / D)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * theta[None, :]  # [N, D/2]
    if inverse:
        ang = -ang
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    if rotate_half:
        a, b = x[..., : D // 2], x[..., D // 2:]
    else:
        a, b = x[..., 0::2], x[..., 1::2]
    ya = a * c - b * s
    yb = a * s + b * c
    out = np.empty_like(x)
    if rotate_half:
        out[..., : D // 2], out[..., D // 2:] = ya, yb
    else:
        out[..., 0::2], out[..., 1::2] = ya, yb
    return out
