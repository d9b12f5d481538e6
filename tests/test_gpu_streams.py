"""The attention calls under concurrency: persistent launches of two
different tries overlapping on two streams (each launch draws its work items
from its own counter of the library's ring), and a forward and backward
captured in a CUDA graph and replayed. The kernels sum in a fixed order, so
every output must equal, bit for bit, the same calls run eagerly one after
another."""
import numpy as np
import pytest
import torch

import treegen
import tree_packed_attention_gb300 as tpa

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _case(parents, lengths, hq, hkv, seed):
    N = int(np.sum(lengths))
    q, k, v, do = (x.cuda() for x in treegen.draw_tensors(N, hq, hkv, 128, "bf16", seed))
    plan = tpa.tree_plan_build(parents, lengths)
    o, lse = tpa.tree_attn_fwd(plan, q, k, v)
    g = tpa.tree_attn_bwd(plan, do, q, k, v, o, lse, grad_dtype=torch.float32)
    return plan, (q, k, v, do), (o, lse) + tuple(g)


def test_launches_overlapping_on_two_streams_repeat_the_sequential_bits():
    _need_gpu()
    w = treegen.workload(3)
    parents, lengths = treegen.random_forest(np.random.default_rng(8), 40, 300, n_roots=3)
    cases = [_case(w.parents, w.lengths, w.hq, w.hkv, 60), _case(parents, lengths, 8, 2, 61)]
    torch.cuda.synchronize()
    tpa.tree_status_sync()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for _ in range(3):
        fwd, got = [None, None], [None, None]
        for n in range(2):  # both forwards in flight, then both backwards
            with torch.cuda.stream(streams[n]):
                plan, (q, k, v, _), _ = cases[n]
                fwd[n] = tpa.tree_attn_fwd(plan, q, k, v)
        for n in range(2):
            with torch.cuda.stream(streams[n]):
                plan, (q, k, v, do), _ = cases[n]
                o, lse = fwd[n]
                got[n] = (o, lse) + tuple(tpa.tree_attn_bwd(plan, do, q, k, v, o, lse,
                                                            grad_dtype=torch.float32))
        torch.cuda.synchronize()
        tpa.tree_status_sync()
        for n in range(2):
            for a, b in zip(got[n], cases[n][2]):
                assert torch.equal(a, b)


def test_forward_and_backward_replay_from_a_cuda_graph():
    _need_gpu()
    parents, lengths = treegen.grpo_tree(3, prompt=300, n_leaves=5, lo=50, hi=200)
    hq, hkv = 4, 2
    plan, (q, k, v, do), ref = _case(parents, lengths, hq, hkv, 62)  # uploads the plan
    N = q.shape[0]
    ws = torch.empty(tpa.tree_attn_bwd_workspace_bytes(plan, hq, 128, torch.bfloat16), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(hq, N, dtype=torch.float32, device="cuda")
    dq = torch.empty(N, hq, 128, dtype=torch.float32, device="cuda")
    dk = torch.empty(N, hkv, 128, dtype=torch.float32, device="cuda")
    dv = torch.empty(N, hkv, 128, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        tpa.tree_attn_fwd(plan, q, k, v, out=o, lse=lse)
        tpa.tree_attn_bwd(plan, do, q, k, v, o, lse, grad_dtype=torch.float32, workspace=ws,
                          out=(dq, dk, dv))
    for _ in range(2):
        for t in (o, lse, dq, dk, dv):
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        tpa.tree_status_sync()
        for a, b in zip((o, lse, dq, dk, dv), ref):
            assert torch.equal(a, b)
