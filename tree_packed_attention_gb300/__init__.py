"""Tree-packed attention on one GB300: Python binding of libtreeattn.

The calls mirror the C-ABI in ``include/treeattn.h``:

* ``tree_plan_build(segment_parents, segment_lengths) -> Plan`` -- DFS layout,
  ancestor lists, per-key visibility bounds and the tile visibility map of a
  trie (or forest) of token segments ("Tree Training", arXiv 2511.00413,
  §3.1 eq. 8, §3.2 eq. 9, App. A.1);
* ``tree_attn_fwd(plan, q, k, v) -> (o, lse)``;
* ``tree_attn_bwd(plan, do, q, k, v, o, lse) -> (dq, dk, dv)``;
* ``tree_weights(plan) -> w`` with w_t = g_t / K (§3.1 eq. 4).

Tensors are torch CUDA tensors in DFS token order: q/o/do [N, hq, D], k/v
[N, hkv, D], lse [hq, N] fp32. torch provides device memory and the current
stream; every step of the computation runs in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from ._lib import (ACT_NONE, ACT_SILU, DTYPE_BF16, DTYPE_F32, EXPORTS, FIELDS, LIB_PATH,
                   PartitionRec, PlanInfo, TreeAttnError, check, lib)

__all__ = [
    "Plan", "tree_plan_build", "tree_plan_build_partition", "tree_attn_fwd_gateway",
    "tree_attn_bwd_gateway", "tree_attn_fwd", "tree_attn_bwd", "tree_attn_bwd_dq",
    "tree_attn_bwd_dkdv", "tree_attn_bwd_workspace_bytes",
    "tree_weights", "tree_weights_paths", "tree_partition", "tree_rope", "tree_rope_qk", "tree_rope_apply",
    "TreeRopeFn", "tree_conv_fwd", "tree_conv_bwd", "tree_conv", "TreeConvFn",
    "tree_weighted_ce", "tree_gdn_fwd", "tree_status_sync", "tree_diag_wait_timeout", "TreeAttnFn", "tree_attention", "TreeAttnError",
    "FIELDS", "EXPORTS", "LIB_PATH",
]


class Plan:
    """Owns a ``tree_plan_t``: the host plan and, once uploaded, its device copy."""

    def __init__(self, segment_parents, segment_lengths, past_visible=None, pos_offset=0):
        parents = np.ascontiguousarray(np.asarray(segment_parents, dtype=np.int32))
        lengths = np.ascontiguousarray(np.asarray(segment_lengths, dtype=np.int32))
        if parents.shape != lengths.shape or parents.ndim != 1:
            raise ValueError("segment_parents and segment_lengths must be 1-D and of equal length")
        h = C.c_void_p()
        if past_visible is None and pos_offset == 0:
            check(lib.tree_plan_build(parents.ctypes.data, lengths.ctypes.data, int(parents.size),
                                      C.byref(h)))
        else:
            vis = np.ascontiguousarray(np.asarray([] if past_visible is None else past_visible,
                                                  dtype=bool).astype(np.uint8))
            if vis.ndim != 1:
                raise ValueError("past_visible must be 1-D")
            check(lib.tree_plan_build_partition(parents.ctypes.data, lengths.ctypes.data,
                                                int(parents.size),
                                                vis.ctypes.data if vis.size else None,
                                                int(vis.size), int(pos_offset), C.byref(h)))
        self._h = h
        info = PlanInfo()
        check(lib.tree_plan_info(self._h, C.byref(info)))
        self.info = {name: int(getattr(info, name)) for name, _ in PlanInfo._fields_}
        self.num_tokens = self.info["num_tokens"]

    @property
    def handle(self):
        return self._h

    def field(self, name: str) -> np.ndarray:
        idx = FIELDS.index(name)
        n = C.c_int64()
        check(lib.tree_plan_field_len(self._h, idx, C.byref(n)))
        out = np.empty(n.value, dtype=np.int32)
        check(lib.tree_plan_get(self._h, idx, out.ctypes.data, out.nbytes))
        return out

    def fields(self) -> dict:
        return {name: self.field(name) for name in FIELDS}

    def to_device(self, stream=None) -> "Plan":
        check(lib.tree_plan_to_device(self._h, _stream_ptr(stream)))
        return self

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            lib.tree_plan_destroy(h)
            self._h = None


def tree_plan_build(segment_parents, segment_lengths) -> Plan:
    return Plan(segment_parents, segment_lengths)


def tree_plan_build_partition(segment_parents, segment_lengths, past_visible, pos_offset=0) -> Plan:
    """Plan of one partition (§3.3; App. B): its own segments plus a gateway of
    len(past_visible) cached keys, key j visible to every row iff past_visible[j]
    (App. B.3 eq. 16); position ids start at pos_offset (App. B.4 eq. 17)."""
    return Plan(segment_parents, segment_lengths, past_visible, pos_offset)


def _stream_ptr(stream):
    if isinstance(stream, C.c_void_p):
        return stream
    if stream is None:
        import torch

        if not torch.cuda.is_available():
            return None
        stream = torch.cuda.current_stream()
    return C.c_void_p(int(getattr(stream, "cuda_stream", stream)))


def _dtype_code(t):
    import torch

    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _check_tensor(name, t, shape, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")


def tree_attn_fwd(plan: Plan, q, k, v, softmax_scale: float = 0.0, out=None, lse=None, stream=None):
    """(o, lse) of tree attention. ``softmax_scale`` 0 means 1/sqrt(D)."""
    import torch

    N, hq, D = q.shape
    hkv = k.shape[1]
    if N != plan.num_tokens:
        raise ValueError(f"q has {N} tokens, the plan {plan.num_tokens}")
    _check_tensor("q", q, (N, hq, D))
    _check_tensor("k", k, (N, hkv, D), q.dtype)
    _check_tensor("v", v, (N, hkv, D), q.dtype)
    o = torch.empty_like(q) if out is None else out
    lse_t = torch.empty(hq, N, dtype=torch.float32, device=q.device) if lse is None else lse
    _check_tensor("o", o, (N, hq, D), q.dtype)
    _check_tensor("lse", lse_t, (hq, N), torch.float32)
    s = _stream_ptr(stream)
    plan.to_device(s)
    check(lib.tree_attn_fwd(plan.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            lse_t.data_ptr(), hq, hkv, D, _dtype_code(q), float(softmax_scale), s))
    return o, lse_t


def tree_attn_bwd_workspace_bytes(plan: Plan, hq: int, head_dim: int, dtype) -> int:
    import torch

    code = DTYPE_BF16 if dtype == torch.bfloat16 else DTYPE_F32
    return int(lib.tree_attn_bwd_workspace_bytes(plan.handle, hq, head_dim, code))


def _bwd_prepare(plan: Plan, do, q, k, v, o, lse, grad_dtype, workspace, stream):
    import torch

    N, hq, D = q.shape
    hkv = k.shape[1]
    if N != plan.num_tokens:
        raise ValueError(f"q has {N} tokens, the plan {plan.num_tokens}")
    checks = [("do", do, (N, hq, D)), ("q", q, (N, hq, D)), ("k", k, (N, hkv, D)),
              ("v", v, (N, hkv, D))]
    if o is not None:
        checks.append(("o", o, (N, hq, D)))
    for name, t, shp in checks:
        _check_tensor(name, t, shp, q.dtype)
    _check_tensor("lse", lse, (hq, N), torch.float32)
    gdt = q.dtype if grad_dtype is None else grad_dtype
    nbytes = tree_attn_bwd_workspace_bytes(plan, hq, D, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    s = _stream_ptr(stream)
    plan.to_device(s)
    gcode = DTYPE_BF16 if gdt == torch.bfloat16 else DTYPE_F32
    return N, hq, hkv, D, gdt, gcode, workspace, s


def tree_attn_bwd(plan: Plan, do, q, k, v, o, lse, softmax_scale: float = 0.0, grad_dtype=None,
                  workspace=None, out=None, stream=None):
    """(dq, dk, dv) of tree attention. ``grad_dtype`` defaults to q's dtype."""
    import torch

    N, hq, hkv, D, gdt, gcode, workspace, s = _bwd_prepare(plan, do, q, k, v, o, lse, grad_dtype,
                                                           workspace, stream)
    if out is None:
        dq = torch.empty(N, hq, D, dtype=gdt, device=q.device)
        dk = torch.empty(N, hkv, D, dtype=gdt, device=q.device)
        dv = torch.empty(N, hkv, D, dtype=gdt, device=q.device)
    else:
        dq, dk, dv = out
    check(lib.tree_attn_bwd(plan.handle, do.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                            o.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                            dv.data_ptr(), hq, hkv, D, _dtype_code(q), gcode,
                            float(softmax_scale), workspace.data_ptr(), workspace.numel(), s))
    return dq, dk, dv


def tree_attn_bwd_dq(plan: Plan, do, q, k, v, o, lse, workspace, softmax_scale: float = 0.0,
                     grad_dtype=None, out=None, stream=None):
    """First phase of the backward: Delta into ``workspace``, then dq."""
    import torch

    N, hq, hkv, D, gdt, gcode, workspace, s = _bwd_prepare(plan, do, q, k, v, o, lse, grad_dtype,
                                                           workspace, stream)
    dq = torch.empty(N, hq, D, dtype=gdt, device=q.device) if out is None else out
    check(lib.tree_attn_bwd_dq(plan.handle, do.data_ptr(), q.data_ptr(), k.data_ptr(),
                               v.data_ptr(), o.data_ptr(), lse.data_ptr(), dq.data_ptr(), hq, hkv,
                               D, _dtype_code(q), gcode, float(softmax_scale),
                               workspace.data_ptr(), workspace.numel(), s))
    return dq


def tree_attn_bwd_dkdv(plan: Plan, do, q, k, v, lse, workspace, softmax_scale: float = 0.0,
                       grad_dtype=None, out=None, stream=None):
    """Second phase of the backward: (dk, dv) from the workspace tree_attn_bwd_dq filled."""
    import torch

    N, hq, hkv, D, gdt, gcode, workspace, s = _bwd_prepare(plan, do, q, k, v, None, lse,
                                                           grad_dtype, workspace, stream)
    if out is None:
        dk = torch.empty(N, hkv, D, dtype=gdt, device=q.device)
        dv = torch.empty(N, hkv, D, dtype=gdt, device=q.device)
    else:
        dk, dv = out
    check(lib.tree_attn_bwd_dkdv(plan.handle, do.data_ptr(), q.data_ptr(), k.data_ptr(),
                                 v.data_ptr(), lse.data_ptr(), dk.data_ptr(), dv.data_ptr(), hq,
                                 hkv, D, _dtype_code(q), gcode, float(softmax_scale),
                                 workspace.data_ptr(), workspace.numel(), s))
    return dk, dv


def tree_attn_fwd_gateway(plan: Plan, q, k, v, past_k, past_v, softmax_scale: float = 0.0,
                          out=None, lse=None, stream=None):
    """(o, lse) of a partition with its gateway (App. B.2 eq. 14): past_k, past_v
    [past_len, hkv, D] hold the gateway keys and values. bf16 only."""
    import torch

    N, hq, D = q.shape
    hkv = k.shape[1]
    P = plan.info["past_len"]
    if N != plan.num_tokens:
        raise ValueError(f"q has {N} tokens, the plan {plan.num_tokens}")
    _check_tensor("q", q, (N, hq, D))
    _check_tensor("k", k, (N, hkv, D), q.dtype)
    _check_tensor("v", v, (N, hkv, D), q.dtype)
    _check_tensor("past_k", past_k, (P, hkv, D), q.dtype)
    _check_tensor("past_v", past_v, (P, hkv, D), q.dtype)
    o = torch.empty_like(q) if out is None else out
    lse_t = torch.empty(hq, N, dtype=torch.float32, device=q.device) if lse is None else lse
    _check_tensor("o", o, (N, hq, D), q.dtype)
    _check_tensor("lse", lse_t, (hq, N), torch.float32)
    s = _stream_ptr(stream)
    plan.to_device(s)
    check(lib.tree_attn_fwd_gateway(plan.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                    past_k.data_ptr(), past_v.data_ptr(), o.data_ptr(),
                                    lse_t.data_ptr(), hq, hkv, D, _dtype_code(q),
                                    float(softmax_scale), s))
    return o, lse_t


def tree_attn_bwd_gateway(plan: Plan, do, q, k, v, past_k, past_v, o, lse, past_dk_acc=None,
                          past_dv_acc=None, softmax_scale: float = 0.0, grad_dtype=None,
                          workspace=None, stream=None):
    """(dq, dk, dv, past_dk_acc, past_dv_acc) of tree_attn_fwd_gateway. The gateway
    gradients are added in fp32 to past_dk_acc / past_dv_acc (created as zeros when
    None), as several children sharing a cut node accumulate them (App. B.5)."""
    import torch

    N, hq, hkv, D, gdt, gcode, workspace, s = _bwd_prepare(plan, do, q, k, v, o, lse, grad_dtype,
                                                           workspace, stream)
    P = plan.info["past_len"]
    _check_tensor("past_k", past_k, (P, hkv, D), q.dtype)
    _check_tensor("past_v", past_v, (P, hkv, D), q.dtype)
    if past_dk_acc is None:
        past_dk_acc = torch.zeros(P, hkv, D, dtype=torch.float32, device=q.device)
    if past_dv_acc is None:
        past_dv_acc = torch.zeros(P, hkv, D, dtype=torch.float32, device=q.device)
    _check_tensor("past_dk_acc", past_dk_acc, (P, hkv, D), torch.float32)
    _check_tensor("past_dv_acc", past_dv_acc, (P, hkv, D), torch.float32)
    dq = torch.empty(N, hq, D, dtype=gdt, device=q.device)
    dk = torch.empty(N, hkv, D, dtype=gdt, device=q.device)
    dv = torch.empty(N, hkv, D, dtype=gdt, device=q.device)
    check(lib.tree_attn_bwd_gateway(plan.handle, do.data_ptr(), q.data_ptr(), k.data_ptr(),
                                    v.data_ptr(), past_k.data_ptr(), past_v.data_ptr(), o.data_ptr(),
                                    lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                    past_dk_acc.data_ptr(), past_dv_acc.data_ptr(), hq, hkv, D,
                                    _dtype_code(q), gcode, float(softmax_scale),
                                    workspace.data_ptr(), workspace.numel(), s))
    return dq, dk, dv, past_dk_acc, past_dv_acc


def tree_weights(plan: Plan) -> np.ndarray:
    """Per-token loss weights g_t / K as fp32 (host)."""
    out = np.empty(plan.num_tokens, dtype=np.float32)
    check(lib.tree_weights(plan.handle, out.ctypes.data))
    return out


def tree_weights_paths(plan: Plan, path_weights) -> np.ndarray:
    """Per-token weights lambda_t = sum of the weights of the paths through t (fp32, host).

    ``path_weights`` holds one weight per root-to-leaf path of the forest, the
    paths numbered by their leaves in DFS order."""
    w = np.ascontiguousarray(path_weights, dtype=np.float64)
    out = np.empty(plan.num_tokens, dtype=np.float32)
    check(lib.tree_weights_paths(plan.handle, w.ctypes.data, int(w.size), out.ctypes.data))
    return out


def tree_partition(plan: Plan, cap_tokens: int) -> dict:
    """Fewest node-boundary partitions of at most ``cap_tokens`` tokens (§3.3).

    Returns part_of_segment [S], and per partition (parents first) root,
    parent, tokens, pos_offset and past_len, plus num_parts and
    peak_path_tokens."""
    S = plan.info["num_segments"]
    part = np.empty(max(S, 1), dtype=np.int32)
    recs = (PartitionRec * max(S, 1))()
    n = C.c_int32()
    peak = C.c_int64()
    check(lib.tree_partition(plan.handle, int(cap_tokens), part.ctypes.data, recs, C.byref(n),
                             C.byref(peak)))
    k = n.value
    out = {"part_of_segment": part[:S].copy(), "num_parts": k, "peak_path_tokens": peak.value}
    for name in ("root", "parent", "tokens", "pos_offset", "past_len"):
        out[name] = np.array([getattr(recs[i], name) for i in range(k)], dtype=np.int64)
    return out


def _conv_prepare(plan: Plan, kernel_size: int, stream):
    s = _stream_ptr(stream)
    plan.to_device(s)
    check(lib.tree_conv_prepare(plan.handle, int(kernel_size), s))
    return s


def _conv_check(plan: Plan, x, weight, bias):
    import torch

    if x.dim() != 2 or x.shape[0] != plan.num_tokens:
        raise ValueError(f"x must be [N={plan.num_tokens}, C], got {tuple(x.shape)}")
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError(f"x must be bf16 or fp32, got {x.dtype}")
    C = x.shape[1]
    _check_tensor("x", x, (plan.num_tokens, C))
    if weight.dim() != 2 or weight.shape[0] != C:
        raise ValueError(f"weight must be fp32 [C={C}, K], got {tuple(weight.shape)}")
    _check_tensor("weight", weight, (C, weight.shape[1]), torch.float32)
    if weight.device != x.device:
        raise ValueError("weight must be on x's device")
    if bias is not None:
        _check_tensor("bias", bias, (C,), torch.float32)
        if bias.device != x.device:
            raise ValueError("bias must be on x's device")
    return C, weight.shape[1]


def _act_code(activation: str) -> int:
    if activation == "silu":
        return ACT_SILU
    if activation == "none":
        return ACT_NONE
    raise ValueError(f"activation must be 'silu' or 'none', got {activation!r}")


def tree_conv_fwd(plan: Plan, x, weight, bias=None, activation: str = "silu", out=None, stream=None):
    """Tree-correct causal depthwise conv of x[N, C] (App. A.3): y[N, C]."""
    import torch

    act = _act_code(activation)
    C, K = _conv_check(plan, x, weight, bias)
    y = torch.empty_like(x) if out is None else out
    _check_tensor("out", y, tuple(x.shape), x.dtype)
    if y.device != x.device:
        raise ValueError("out must be on x's device")
    s = _conv_prepare(plan, K, stream)
    check(lib.tree_conv_fwd(plan.handle, x.data_ptr(), weight.data_ptr(),
                            bias.data_ptr() if bias is not None else None, y.data_ptr(), C,
                            _dtype_code(x), act, s))
    return y


def tree_conv_bwd(plan: Plan, x, weight, bias, dy, activation: str = "silu", stream=None):
    """(dx, dweight, dbias) of tree_conv_fwd; dbias is None when bias is None."""
    import torch

    act = _act_code(activation)
    C, K = _conv_check(plan, x, weight, bias)
    _check_tensor("dy", dy, tuple(x.shape), x.dtype)
    if dy.device != x.device:
        raise ValueError("dy must be on x's device")
    s = _conv_prepare(plan, K, stream)
    dx = torch.empty_like(x)
    dw = torch.empty_like(weight)
    db = torch.empty_like(bias) if bias is not None else None
    nbytes = lib.tree_conv_bwd_workspace_bytes(plan.handle, C)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=x.device)
    check(lib.tree_conv_bwd(plan.handle, x.data_ptr(), weight.data_ptr(),
                            bias.data_ptr() if bias is not None else None, dy.data_ptr(),
                            dx.data_ptr(), dw.data_ptr(), db.data_ptr() if db is not None else None,
                            C, _dtype_code(x), act, ws.data_ptr(), ws.numel(), s))
    return dx, dw, db


def tree_rope(plan: Plan, x, base: float = 10000.0, rotate_half: bool = False,
              inverse: bool = False, stream=None):
    """Rotary embedding of x[N, H, D] (bf16 or fp32, on the GPU) at the plan's
    tree position ids, in place; returns x. ``inverse`` applies the backward."""
    import torch

    if x.dim() != 3 or x.shape[0] != plan.num_tokens:
        raise ValueError(f"x must be [N={plan.num_tokens}, H, D], got {tuple(x.shape)}")
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError(f"x must be bf16 or fp32, got {x.dtype}")
    _check_tensor("x", x, tuple(x.shape))
    s = _stream_ptr(stream)
    plan.to_device(s)
    check(lib.tree_rope(plan.handle, x.data_ptr(), x.shape[1], x.shape[2], _dtype_code(x),
                        float(base), int(bool(rotate_half)), int(bool(inverse)), s))
    return x


def tree_rope_qk(plan: Plan, q, k, base: float = 10000.0, rotate_half: bool = False,
                 inverse: bool = False, stream=None):
    """tree_rope on q [N, Hq, D] and k [N, Hk, D] (same dtype) in one launch, in
    place, bit for bit as two tree_rope calls; returns (q, k)."""
    import torch

    for name, x in (("q", q), ("k", k)):
        if x.dim() != 3 or x.shape[0] != plan.num_tokens:
            raise ValueError(f"{name} must be [N={plan.num_tokens}, H, D], got {tuple(x.shape)}")
        if x.dtype not in (torch.bfloat16, torch.float32):
            raise TypeError(f"{name} must be bf16 or fp32, got {x.dtype}")
        _check_tensor(name, x, tuple(x.shape), q.dtype)
    if k.shape[2] != q.shape[2]:
        raise ValueError(f"q and k head_dim differ: {q.shape[2]} and {k.shape[2]}")
    s = _stream_ptr(stream)
    plan.to_device(s)
    check(lib.tree_rope_qk(plan.handle, q.data_ptr(), q.shape[1], k.data_ptr(), k.shape[1], q.shape[2],
                           _dtype_code(q), float(base), int(bool(rotate_half)), int(bool(inverse)), s))
    return q, k


def tree_weighted_ce(plan: Plan, logits, tokens, lam, grad_scale: float = 1.0, in_place: bool = False,
                     stream=None):
    """Fused weighted next-token cross-entropy over the trie (§3.1 eq. 3-5, §3.2
    "Loss Weights"); returns (loss fp64 scalar tensor, row_loss [N] fp32, dlogits).

    logits [N, V] (bf16 or fp32, V a multiple of 8); tokens [N] int32 token ids of
    the DFS sequence (< 0: that token is not predicted); lam [N] fp32 weight of the
    prediction of each token (e.g. tree_weights: g_t / K). dlogits is the gradient
    of grad_scale * loss; with ``in_place`` it overwrites logits."""
    import torch

    N = plan.num_tokens
    if logits.dim() != 2 or logits.shape[0] != N:
        raise ValueError(f"logits must be [N={N}, V], got {tuple(logits.shape)}")
    if logits.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError(f"logits must be bf16 or fp32, got {logits.dtype}")
    V = logits.shape[1]
    _check_tensor("logits", logits, (N, V))
    if tokens.dtype != torch.int32 or tuple(tokens.shape) != (N,):
        raise ValueError("tokens must be int32 [N]")
    if lam.dtype != torch.float32 or tuple(lam.shape) != (N,):
        raise ValueError("lam must be fp32 [N]")
    _check_tensor("tokens", tokens, (N,))
    _check_tensor("lam", lam, (N,))
    dlogits = logits if in_place else torch.empty_like(logits)
    row_loss = torch.empty(N, dtype=torch.float32, device=logits.device)
    loss = torch.empty((), dtype=torch.float64, device=logits.device)
    s = _stream_ptr(stream)
    plan.to_device(s)
    check(lib.tree_weighted_ce(plan.handle, logits.data_ptr(), dlogits.data_ptr(), tokens.data_ptr(),
                               lam.data_ptr(), V, _dtype_code(logits), float(grad_scale),
                               row_loss.data_ptr(), loss.data_ptr(), s))
    return loss, row_loss, dlogits


def tree_gdn_fwd(plan: Plan, q, k, v, g, beta, initial_state=None, stream=None):
    """Gated DeltaNet forward with tree state routing (eq. 10, App. A.2); returns
    (o [N, hv, 128], segment_states [S, hv, 128, 128] fp32, by segment id).

    q, k [N, hk, 128] and v [N, hv, 128] (bf16 or fp32, one dtype), g and beta
    [N, hv] fp32, initial_state [hv, 128, 128] fp32 or None (zeros)."""
    import torch

    N = plan.num_tokens
    if q.dim() != 3 or q.shape[0] != N or q.shape[2] != 128:
        raise ValueError(f"q must be [N={N}, hk, 128], got {tuple(q.shape)}")
    hk, hv = q.shape[1], v.shape[1]
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError(f"q must be bf16 or fp32, got {q.dtype}")
    _check_tensor("q", q, (N, hk, 128))
    _check_tensor("k", k, (N, hk, 128), q.dtype)
    _check_tensor("v", v, (N, hv, 128), q.dtype)
    _check_tensor("g", g, (N, hv), torch.float32)
    _check_tensor("beta", beta, (N, hv), torch.float32)
    if initial_state is not None:
        _check_tensor("initial_state", initial_state, (hv, 128, 128), torch.float32)
    o = torch.empty_like(v)
    S = plan.info["num_segments"]
    states = torch.empty(S, hv, 128, 128, dtype=torch.float32, device=q.device)
    s = _stream_ptr(stream)
    plan.to_device(s)
    check(lib.tree_gdn_fwd(plan.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(),
                           beta.data_ptr(), None if initial_state is None else initial_state.data_ptr(),
                           o.data_ptr(), states.data_ptr(), hk, hv, 128, _dtype_code(q), s))
    return o, states


def tree_status_sync(stream=None) -> None:
    """Wait for the stream; raise if a kernel gave up a bounded wait."""
    check(lib.tree_status_sync(_stream_ptr(stream)))


def tree_diag_wait_timeout(limit_ns: int = 20_000_000, stream=None) -> None:
    """Launch the diagnostic wait that gives up after ``limit_ns``; the next
    ``tree_status_sync`` raises TREE_ERR_TIMEOUT naming wait site 50000."""
    check(lib.tree_diag_wait_timeout(int(limit_ns), _stream_ptr(stream)))


def _make_autograd():
    import torch

    class TreeAttnFn(torch.autograd.Function):
        """Autograd wrapper: forward/backward both run the library's kernels."""

        @staticmethod
        def forward(ctx, q, k, v, plan, softmax_scale=0.0):
            o, lse = tree_attn_fwd(plan, q, k, v, softmax_scale)
            ctx.save_for_backward(q, k, v, o, lse)
            ctx.plan = plan
            ctx.scale = softmax_scale
            return o

        @staticmethod
        def backward(ctx, do):
            q, k, v, o, lse = ctx.saved_tensors
            dq, dk, dv = tree_attn_bwd(ctx.plan, do.contiguous(), q, k, v, o, lse, ctx.scale)
            return dq, dk, dv, None, None

    return TreeAttnFn


TreeAttnFn = _make_autograd()


def _make_rope_autograd():
    import torch

    class TreeRopeFn(torch.autograd.Function):
        """Autograd wrapper: the forward rotates a copy of x, the backward applies
        the inverse rotation to the incoming gradient; both run the library's kernel."""

        @staticmethod
        def forward(ctx, x, plan, base=10000.0, rotate_half=False):
            ctx.plan, ctx.base, ctx.rotate_half = plan, base, rotate_half
            return tree_rope(plan, x.contiguous().clone(), base, rotate_half)

        @staticmethod
        def backward(ctx, gy):
            gx = tree_rope(ctx.plan, gy.contiguous().clone(), ctx.base, ctx.rotate_half, inverse=True)
            return gx, None, None, None

    return TreeRopeFn


TreeRopeFn = _make_rope_autograd()


def _make_conv_autograd():
    import torch

    class TreeConvFn(torch.autograd.Function):
        """Autograd wrapper: forward and backward both run the library's kernels."""

        @staticmethod
        def forward(ctx, x, weight, bias, plan, activation="silu"):
            x = x.contiguous()
            ctx.save_for_backward(x, weight, bias)
            ctx.plan, ctx.activation = plan, activation
            return tree_conv_fwd(plan, x, weight, bias, activation)

        @staticmethod
        def backward(ctx, dy):
            x, weight, bias = ctx.saved_tensors
            dx, dw, db = tree_conv_bwd(ctx.plan, x, weight, bias, dy.contiguous().to(x.dtype),
                                       ctx.activation)
            return dx, dw, db, None, None

    return TreeConvFn


TreeConvFn = _make_conv_autograd()


def tree_conv(x, weight, bias, plan: Plan, activation: str = "silu"):
    """Differentiable tree-correct causal conv (App. A.3)."""
    return TreeConvFn.apply(x, weight, bias, plan, activation)


def tree_rope_apply(x, plan: Plan, base: float = 10000.0, rotate_half: bool = False):
    """Differentiable tree RoPE (returns a rotated copy of x)."""
    return TreeRopeFn.apply(x, plan, base, rotate_half)


def tree_attention(q, k, v, plan: Plan, softmax_scale: float = 0.0):
    """Differentiable tree attention (o only)."""
    return TreeAttnFn.apply(q, k, v, plan, softmax_scale)
