import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session", autouse=True)
def _host_libs():
    """Build the CPU-side libraries (oracle, generator twin) once per session."""
    import oracle
    import synth
    if not os.path.exists(os.path.join(ROOT, "oracle", "liboracle.so")):
        oracle.build()
    if not os.path.exists(os.path.join(ROOT, "synth", "libsynth.so")):
        synth.build(gpu=False)
    if not os.path.exists(os.path.join(ROOT, "bit_exact_xor_gb300", "libdcr.so")):
        from bit_exact_xor_gb300 import build as dcr_build
        dcr_build.build()
    yield


GOLDEN = os.path.join(ROOT, "tests", "golden")


def read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([c.strip() for c in line.split("|")])
    return rows
