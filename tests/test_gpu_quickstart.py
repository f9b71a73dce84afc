"""examples/quickstart.py runs as shipped: on the GPU its own asserts check
the receiver against the new weights in the checkpoint layout."""
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
EXAMPLE = os.path.join(ROOT, "examples", "quickstart.py")


def test_quickstart_parses():
    compile(open(EXAMPLE).read(), EXAMPLE, "exec")


@pytest.mark.gpu
def test_quickstart_runs():
    pytest.importorskip("torch")
    out = subprocess.run([sys.executable, EXAMPLE], stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr.decode()[-2000:]
    m = re.search(r"(\d+) values changed; payload (\d+) bytes for (\d+) weight bytes", out.stdout.decode())
    assert m, out.stdout.decode()
    changed, size, n = map(int, m.groups())
    assert n == 1024 * 1024 * 2 + 1024 * 2
    assert 0 < changed and 0 < size < n
