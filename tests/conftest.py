import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(scope="session")
def se_lib():
    """The built library (built here if missing or older than its sources)."""
    import glob
    from sparse_decode_attention_quest_gb300 import build as b
    path = b.lib_path()
    srcs = glob.glob(os.path.join(b.CSRC, "*")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    if not os.path.exists(path) or os.path.getmtime(path) < max(os.path.getmtime(s) for s in srcs):
        b.build()
    import sparse_decode_attention_quest_gb300 as se
    return se.load_library()
