import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _build_library():
    """Compile libtreeattn.so in-tree if it is missing or stale (no GPU needed)."""
    path = os.path.join(ROOT, "tree_packed_attention_gb300", "_build.py")
    spec = importlib.util.spec_from_file_location("_tpa_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    _build_library()


def cuda_ok():
    import torch

    return torch.cuda.is_available()
