import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running oracle work")


def _build_library():
    """Build libverify_attn.so in-tree before collection (nvcc cross-compiles
    without a GPU), so test modules can import the binding."""
    import importlib.util
    path = os.path.join(ROOT, "speculative_decoding_verify_kv_gb300", "_build.py")
    spec = importlib.util.spec_from_file_location("_va_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()


_build_library()
