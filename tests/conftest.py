import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes of host-side input generation)")


def _ensure_built():
    """Compile the CUDA library (nvcc, sm_103a) and the C oracle if they are missing or stale."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("_lora_build", os.path.join(ROOT, "adapter_serving_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    import oracle
    oracle.build()


_ensure_built()
