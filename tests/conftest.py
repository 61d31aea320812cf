import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a)")


def pytest_sessionstart(session):
    # A fresh checkout has no library yet: build it (nvcc cross-compiles
    # without a GPU).  The tests then load the real library; without nvcc the
    # library tests fail loudly, as the product does (no fallback).
    lib = os.path.join(ROOT, "tree_structured_decode_gb300", "lib", "libtreeattn.so")
    if not os.path.exists(lib) and shutil.which("nvcc"):
        from tree_structured_decode_gb300 import build

        build.build()


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
