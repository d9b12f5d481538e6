"""The Python binding rejects bad conv / RoPE calls before anything reaches the
library (CPU only, no GPU).

Each bad argument is a stand-in that reports itself as a CUDA tensor but
fails the test if its device address is ever taken: a call that raises
before asking for an address cannot have launched a kernel.
"""
import pytest
import torch

import tree_packed_attention_gb300 as tpa


class FakeCuda:
    """Shape, dtype and layout of a CPU tensor, presented as a CUDA tensor."""

    def __init__(self, t, device="cuda:0"):
        self._t = t
        self.is_cuda = True
        self.device = torch.device(device)
        self.shape = t.shape
        self.dtype = t.dtype

    def dim(self):
        return self._t.dim()

    def is_contiguous(self):
        return self._t.is_contiguous()

    def data_ptr(self):
        raise AssertionError("a device address was requested: the call got past the checks")


PARENTS, LENGTHS = [-1, 0, 0], [5, 3, 4]
N, CH, K = 12, 16, 4


def _ok():
    x = FakeCuda(torch.zeros(N, CH, dtype=torch.bfloat16))
    w = FakeCuda(torch.zeros(CH, K))
    b = FakeCuda(torch.zeros(CH))
    dy = FakeCuda(torch.zeros(N, CH, dtype=torch.bfloat16))
    return x, w, b, dy


@pytest.fixture(scope="module")
def plan():
    return tpa.tree_plan_build(PARENTS, LENGTHS)


def test_conv_rejects_unknown_activation(plan):
    x, w, b, dy = _ok()
    for act in ("SiLU", "gelu", ""):
        with pytest.raises(ValueError, match="activation"):
            tpa.tree_conv_fwd(plan, x, w, b, act)
        with pytest.raises(ValueError, match="activation"):
            tpa.tree_conv_bwd(plan, x, w, b, dy, act)


def test_conv_rejects_host_tensors(plan):
    x, w, b, dy = _ok()
    with pytest.raises(ValueError, match="CUDA"):
        tpa.tree_conv_fwd(plan, torch.zeros(N, CH, dtype=torch.bfloat16), w, b)
    with pytest.raises(ValueError, match="CUDA"):
        tpa.tree_conv_fwd(plan, x, torch.zeros(CH, K), b)
    with pytest.raises(ValueError, match="CUDA"):
        tpa.tree_conv_bwd(plan, x, w, b, torch.zeros(N, CH, dtype=torch.bfloat16))


@pytest.mark.parametrize("bad", ["dy_dtype", "dy_shape", "dy_strided", "out_dtype", "out_shape",
                                 "w_dtype", "w_shape", "b_shape", "x_dtype", "x_rows", "w_device"])
def test_conv_rejects_mismatched_tensors(plan, bad):
    x, w, b, dy = _ok()
    out = None
    if bad == "dy_dtype":
        dy = FakeCuda(torch.zeros(N, CH, dtype=torch.float32))
    elif bad == "dy_shape":
        dy = FakeCuda(torch.zeros(N - 1, CH, dtype=torch.bfloat16))
    elif bad == "dy_strided":
        dy = FakeCuda(torch.zeros(CH, N, dtype=torch.bfloat16).t())
    elif bad == "out_dtype":
        out = FakeCuda(torch.zeros(N, CH, dtype=torch.float32))
    elif bad == "out_shape":
        out = FakeCuda(torch.zeros(N, CH // 2, dtype=torch.bfloat16))
    elif bad == "w_dtype":
        w = FakeCuda(torch.zeros(CH, K, dtype=torch.bfloat16))
    elif bad == "w_shape":
        w = FakeCuda(torch.zeros(CH + 8, K))
    elif bad == "b_shape":
        b = FakeCuda(torch.zeros(CH + 1))
    elif bad == "x_dtype":
        x = FakeCuda(torch.zeros(N, CH, dtype=torch.float16))
    elif bad == "x_rows":
        x = FakeCuda(torch.zeros(N + 3, CH, dtype=torch.bfloat16))
    elif bad == "w_device":
        w = FakeCuda(torch.zeros(CH, K), device="cuda:1")
    with pytest.raises((ValueError, TypeError)):
        if bad.startswith("out"):
            tpa.tree_conv_fwd(plan, x, w, b, out=out)
        elif bad.startswith("dy"):
            tpa.tree_conv_bwd(plan, x, w, b, dy)
        else:
            tpa.tree_conv_fwd(plan, x, w, b)
            tpa.tree_conv_bwd(plan, x, w, b, dy)


def test_rope_rejects_bad_tensors(plan):
    with pytest.raises(ValueError, match="CUDA"):
        tpa.tree_rope(plan, torch.zeros(N, 2, 64, dtype=torch.bfloat16))
    with pytest.raises(TypeError):
        tpa.tree_rope(plan, FakeCuda(torch.zeros(N, 2, 64, dtype=torch.float16)))
    with pytest.raises(ValueError):
        tpa.tree_rope(plan, FakeCuda(torch.zeros(N + 1, 2, 64, dtype=torch.bfloat16)))
    with pytest.raises(ValueError, match="contiguous"):
        tpa.tree_rope(plan, FakeCuda(torch.zeros(N, 64, 2, dtype=torch.bfloat16).transpose(1, 2)))
