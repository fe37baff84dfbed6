import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large CPU oracle work")


def golden_path(name: str) -> str:
    return os.path.join(GOLDEN, name)


def read_golden(name: str) -> dict:
    """Parse a `key: values` fixture (lines starting with # are comments)."""
    out = {}
    with open(golden_path(name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                k, v = line.split(":", 1)
                out[k.strip()] = v.strip()
    return out


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library (skips when no GPU is present; fails if a GPU is present but
    the library cannot be loaded -- there is no fallback)."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_w4a4_moe_quantize_gb300 as lib
    lib.load()
    return lib
