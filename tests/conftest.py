import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def read_golden(name):
    """Rows of a '|'-separated golden file, comments dropped, fields stripped."""
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([c.strip() for c in line.split("|")])
    return rows


@pytest.fixture(scope="session")
def oracle():
    """The oracle on every host core (its threads only spread independent
    output rows; the results equal the single-thread ones bit for bit)."""
    from oracle import Oracle
    o = Oracle()
    o.set_threads(o.max_threads())
    return o


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, loaded through its binding.  A GPU test that reaches
    this fixture on a machine with a GPU fails (never skips) when the
    library is missing, so a silent fallback cannot pass."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_74_gb300 as pa
    pa.load_library()  # raises if the shared library is absent
    return pa
