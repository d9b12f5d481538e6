"""The failure path on the GPU without a fault: a bounded wait that nothing
completes gives up after its limit, the device status word names the wait,
tree_status_sync reports TREE_ERR_TIMEOUT and clears the word, and the
context keeps running the library's kernels."""
import time

import numpy as np
import pytest
import torch

import treegen
import tree_packed_attention_gb300 as tpa
from oracle import attention as A

pytestmark = pytest.mark.gpu


def test_a_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.synchronize()
    tpa.tree_status_sync()  # start from a clear status word
    t0 = time.perf_counter()
    tpa.tree_diag_wait_timeout(20_000_000)  # 20 ms
    with pytest.raises(tpa.TreeAttnError) as e:
        tpa.tree_status_sync()
    waited = time.perf_counter() - t0
    assert e.value.status_name == "TREE_ERR_TIMEOUT" and "50000" in str(e.value)
    assert waited >= 0.015
    tpa.tree_status_sync()  # the word was cleared
    parents, lengths = [-1, 0, 0], [40, 20, 30]
    q, k, v, _ = treegen.draw_tensors(int(np.sum(lengths)), 2, 1, 128, "bf16", 0)
    plan = tpa.tree_plan_build(parents, lengths)
    o, lse = tpa.tree_attn_fwd(plan, q.cuda(), k.cuda(), v.cuda())
    tpa.tree_status_sync()
    ro, rlse = A.forward(q, k, v, parents, lengths)
    assert float((o.double().cpu() - ro).abs().max()) <= 2e-2 + 2.0 ** -8 * float(ro.abs().max())
    assert float((lse.double().cpu() - rlse).abs().max()) <= 2e-2
