"""ctypes loader for libtreeattn.so: argument marshalling only.

Importing this module fails loudly if the library has not been built; there
is no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtreeattn.so")

TREE_OK = 0
STATUS_NAMES = {
    0: "TREE_OK",
    1: "TREE_ERR_INVALID_ARG",
    2: "TREE_ERR_CYCLE",
    3: "TREE_ERR_EMPTY_SEGMENT",
    4: "TREE_ERR_OVERFLOW",
    5: "TREE_ERR_UNSUPPORTED",
    6: "TREE_ERR_CUDA",
    7: "TREE_ERR_TIMEOUT",
    8: "TREE_ERR_OOM",
    9: "TREE_ERR_NOT_ON_DEVICE",
}
DTYPE_F32, DTYPE_BF16 = 0, 1
ACT_NONE, ACT_SILU = 0, 1

FIELDS = [
    "dfs_order", "seg_start", "depth", "subtree_end", "trie_id", "g", "anc_ptr", "anc_idx",
    "token_seg", "pos_id", "key_end", "cu_seqlens", "trie_paths", "qt_ptr", "qt_kt", "qt_kind",
    "kt_qlo", "kt_qhi", "fwd_order", "bwd_order", "qp_ptr", "qp_kt", "qp_kind", "qp_order",
    "gq_ptr", "gp_ptr", "gt_kind", "gt_atom", "gt_bidx", "gt_bounds", "gw_kend", "gw_kt",
]

# Every symbol the public header declares.
EXPORTS = [
    "tree_plan_build", "tree_plan_info", "tree_plan_get", "tree_plan_field_len",
    "tree_plan_to_device", "tree_plan_destroy", "tree_attn_fwd", "tree_attn_bwd_workspace_bytes",
    "tree_attn_bwd", "tree_attn_bwd_dq", "tree_attn_bwd_dkdv", "tree_attn_bwd_static_scratch",
    "tree_weights", "tree_weights_paths", "tree_partition", "tree_conv_prepare", "tree_conv_fwd",
    "tree_conv_bwd_workspace_bytes", "tree_conv_bwd", "tree_rope", "tree_rope_qk", "tree_status_sync",
    "tree_last_error", "tree_plan_build_partition", "tree_attn_fwd_gateway", "tree_attn_bwd_gateway",
    "tree_weighted_ce", "tree_gdn_fwd", "tree_diag_wait_timeout",
]


class PlanInfo(C.Structure):
    _fields_ = [(name, C.c_int64) for name in (
        "num_tokens", "num_segments", "num_tries", "block_m", "block_n", "num_q_tiles",
        "num_k_tiles", "nnz_tiles", "num_pairs", "nnz_pair_tiles", "num_ancestors",
        "visible_pairs", "num_gathered_tiles", "past_len", "past_visible", "gdn_levels")]


class TreeAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.status_name = STATUS_NAMES.get(status, str(status))


class PartitionRec(C.Structure):
    _fields_ = [("root", C.c_int32), ("parent", C.c_int32), ("tokens", C.c_int64),
                ("pos_offset", C.c_int64), ("past_len", C.c_int64)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()' "
            "or python -m tree_packed_attention_gb300._build)")
    lib = C.CDLL(LIB_PATH)
    vp, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
    sig = {
        "tree_plan_build": (i32, [vp, vp, i32, C.POINTER(vp)]),
        "tree_plan_info": (i32, [vp, C.POINTER(PlanInfo)]),
        "tree_plan_get": (i32, [vp, i32, vp, sz]),
        "tree_plan_field_len": (i32, [vp, i32, C.POINTER(i64)]),
        "tree_plan_to_device": (i32, [vp, vp]),
        "tree_plan_destroy": (None, [vp]),
        "tree_attn_fwd": (i32, [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, C.c_float, vp]),
        "tree_attn_bwd_workspace_bytes": (sz, [vp, i32, i32, i32]),
        "tree_attn_bwd": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                C.c_float, vp, sz, vp]),
        "tree_attn_bwd_dq": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                   C.c_float, vp, sz, vp]),
        "tree_attn_bwd_dkdv": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                     C.c_float, vp, sz, vp]),
        "tree_attn_bwd_static_scratch": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                               i32, i32, C.c_float, vp]),
        "tree_weights": (i32, [vp, vp]),
        "tree_weights_paths": (i32, [vp, vp, i32, vp]),
        "tree_partition": (i32, [vp, i64, vp, vp, C.POINTER(i32), C.POINTER(i64)]),
        "tree_rope": (i32, [vp, vp, i32, i32, i32, C.c_float, i32, i32, vp]),
        "tree_rope_qk": (i32, [vp, vp, i32, vp, i32, i32, i32, C.c_float, i32, i32, vp]),
        "tree_conv_prepare": (i32, [vp, i32, vp]),
        "tree_conv_fwd": (i32, [vp, vp, vp, vp, vp, i32, i32, i32, vp]),
        "tree_conv_bwd_workspace_bytes": (sz, [vp, i32]),
        "tree_conv_bwd": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, sz, vp]),
        "tree_status_sync": (i32, [vp]),
        "tree_diag_wait_timeout": (i32, [C.c_int64, vp]),
        "tree_last_error": (C.c_char_p, []),
        "tree_plan_build_partition": (i32, [vp, vp, i32, vp, i32, i32, C.POINTER(vp)]),
        "tree_attn_fwd_gateway": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, C.c_float,
                                        vp]),
        "tree_attn_bwd_gateway": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                        i32, i32, i32, i32, C.c_float, vp, sz, vp]),
        "tree_weighted_ce": (i32, [vp, vp, vp, vp, vp, i32, i32, C.c_float, vp, vp, vp]),
        "tree_gdn_fwd": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def check(status: int) -> None:
    if status != TREE_OK:
        msg = lib.tree_last_error()
        raise TreeAttnError(status, msg.decode() if msg else "")
