import os
import sys
from pathlib import Path

import numpy as np
import pytest

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

LUT_PATH = ROOT / "trellis_row_decode_gb300" / "data" / "cp_lut_v2_l16_512.bin"


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libcp")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def lut() -> np.ndarray:
    """The shared fp16 LUT as bit patterns, shape (512, 2)."""
    return np.fromfile(LUT_PATH, dtype="<u2").reshape(512, 2)


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle


def n_threads() -> int:
    return max(1, os.cpu_count() or 1)
