"""The allocation-free backward entry point, called through the C-ABI.

tree_attn_bwd_static_scratch serves callers that cannot allocate device
memory when they run the backward (a memory pool that owns the whole device,
a latency-critical loop where cudaMalloc would synchronize). It must give the
same gradients as tree_attn_bwd with a caller workspace, call after call,
since every call reuses one scratch array built into the library.
This file is collected last so that a stop-at-first-failure run has already
run every other test when it gets here.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import treegen
import tree_packed_attention_gb300 as tpa
from tree_packed_attention_gb300._lib import DTYPE_BF16, DTYPE_F32

pytestmark = pytest.mark.gpu


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_static_scratch_backward_matches_workspace_backward():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    parents, lengths = treegen.grpo_tree(4, prompt=260, n_leaves=4, lo=70, hi=200)
    N = int(lengths.sum())
    hq, hkv, D = 4, 2, 128
    q, k, v, do = (x.cuda() for x in treegen.draw_tensors(N, hq, hkv, D, "bf16", seed=11))
    plan = tpa.tree_plan_build(parents, lengths)
    o, lse = tpa.tree_attn_fwd(plan, q, k, v)
    ref = tpa.tree_attn_bwd(plan, do, q, k, v, o, lse, grad_dtype=torch.float32)
    for _ in range(2):  # the second call reuses the scratch the first one left behind
        got = [torch.full_like(x, float("nan")) for x in ref]
        st = tpa.lib.tree_attn_bwd_static_scratch(
            plan.handle, do.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
            lse.data_ptr(), got[0].data_ptr(), got[1].data_ptr(), got[2].data_ptr(), hq, hkv, D,
            DTYPE_BF16, DTYPE_F32, 0.0, _stream())
        assert st == 0, tpa.lib.tree_last_error()
        tpa.tree_status_sync()
        # the same kernels in the same fixed order: equal bit for bit
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            assert torch.equal(a, b), name


def test_static_scratch_rejects_oversized_requests():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    plan = tpa.tree_plan_build([-1], [200])
    hq = 40000  # 2 rows of hq x 256 fp32 = 81,920,000 bytes > TREE_STATIC_SCRATCH_BYTES
    # Every tensor pointer is NULL: the size check must answer first, and were
    # it ever skipped the NULL checks behind it would still refuse the call
    # before any launch.
    st = tpa.lib.tree_attn_bwd_static_scratch(plan.handle, None, None, None, None, None, None,
                                              None, None, None, hq, hq, 128, DTYPE_BF16,
                                              DTYPE_BF16, 0.0, None)
    assert tpa._lib.STATUS_NAMES[st] == "TREE_ERR_UNSUPPORTED"
    assert b"scratch" in tpa.lib.tree_last_error()


def test_static_scratch_at_its_size_limit():
    """The packed 131,072-token workload with 64 q heads needs exactly
    TREE_STATIC_SCRATCH_BYTES (two rows of 64 x 131,072 fp32): the largest
    request the entry point takes runs bit for bit as tree_attn_bwd, and the
    same trie with one token more is refused before any launch."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = treegen.workload(5)
    plan = tpa.tree_plan_build(w.parents, w.lengths)
    N, hq, hkv, D = w.num_tokens, w.hq, w.hkv, w.head_dim
    assert tpa.tree_attn_bwd_workspace_bytes(plan, hq, D, torch.bfloat16) == 64 << 20
    g = torch.Generator(device="cuda").manual_seed(5)
    q, do = (torch.randn(N, hq, D, device="cuda", generator=g).to(torch.bfloat16) for _ in range(2))
    k, v = (torch.randn(N, hkv, D, device="cuda", generator=g).to(torch.bfloat16) for _ in range(2))
    o, lse = tpa.tree_attn_fwd(plan, q, k, v)
    ref = tpa.tree_attn_bwd(plan, do, q, k, v, o, lse)
    got = [torch.full_like(x, float("nan")) for x in ref]
    st = tpa.lib.tree_attn_bwd_static_scratch(
        plan.handle, do.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
        lse.data_ptr(), got[0].data_ptr(), got[1].data_ptr(), got[2].data_ptr(), hq, hkv, D,
        DTYPE_BF16, DTYPE_BF16, 0.0, _stream())
    assert st == 0, tpa.lib.tree_last_error()
    tpa.tree_status_sync()
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        assert torch.equal(a, b), name
    lengths = np.array(w.lengths).copy()
    lengths[0] += 1
    bigger = tpa.tree_plan_build(w.parents, lengths)
    st = tpa.lib.tree_attn_bwd_static_scratch(bigger.handle, None, None, None, None, None, None,
                                              None, None, None, hq, hkv, D, DTYPE_BF16, DTYPE_BF16,
                                              0.0, None)
    assert tpa._lib.STATUS_NAMES[st] == "TREE_ERR_UNSUPPORTED"
