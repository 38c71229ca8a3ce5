import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    # Build libpagedkv.so in-tree when it is missing or older than its sources.
    import importlib.util
    path = os.path.join(ROOT, "paged_kv_cache_118_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("pkv_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: large inputs; minutes of host work")


def pytest_collection_modifyitems(config, items):
    """Run GPU tests only where a GPU exists: on a CPU-only host they are skipped
    (the driver selects them with -m gpu on the GPU machine)."""
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device on this host")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
