import os
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

GOLDEN = Path(__file__).resolve().parent / "golden"


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and runs the CUDA kernels")
    config.addinivalue_line("markers", "slow: full-size configurations")


def golden_lines(name: str):
    """Non-comment, non-empty lines of a golden fixture."""
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.strip()
        if line and not line.startswith("#"):
            yield line


@pytest.fixture(scope="session")
def libtq():
    """The C-ABI library, built in-tree if it is missing or stale."""
    from kv_cache_quantization_store_gb300 import build, lib

    build.build()
    return lib()


@pytest.fixture(scope="session")
def cuda_device(libtq):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", int(os.environ.get("TQ_TEST_DEVICE", "0")))
