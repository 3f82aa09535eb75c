import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload (runs on the GPU box)")


def _lib_built():
    return os.path.exists(os.path.join(ROOT, "paged_hybrid_attention_gb300", "libgw.so"))


def _cuda():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


# On a machine without a GPU and without the built library, GPU test modules
# cannot even be imported; leave them out of collection there.  With a GPU
# they are always collected, so a missing library fails loudly.
collect_ignore_glob = [] if (_lib_built() or _cuda()) else ["test_gpu_*.py", "test_zz_*.py"]
