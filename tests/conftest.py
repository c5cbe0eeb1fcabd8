import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def read_golden(name):
    """Parse a `key value...` fixture; '#' starts a comment line."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


def read_golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle


@pytest.fixture(scope="session")
def dev():
    """cuda:0 with libi8q.so built and loaded (GPU tests only)."""
    import torch
    from int8_quantized_gb300 import _lib, build
    build.build()
    _lib.load()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def bf16_ulp_distance(a_bits, b_bits):
    """Distance in units in the last place between two arrays of bf16 bit
    patterns (uint16), on the ordered integer line of the format."""
    import numpy as np

    def ordered(b):
        v = b.astype(np.int32)
        return np.where(v & 0x8000, 0x8000 - (v & 0x7FFF), 0x8000 + (v & 0x7FFF)).astype(np.int64)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def max_rel_err(got, ref):
    import numpy as np
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1e-30))) if ref.size else 0.0
