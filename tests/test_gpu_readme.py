"""The quickstart in README.md runs as printed: its Python block is
executed on the GPU (its own asserts check the receiver against the new
weights in the checkpoint layout)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _quickstart():
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert blocks, "README.md has no python block"
    return blocks[0]


def test_quickstart_block_parses():
    compile(_quickstart(), "README.md", "exec")


@pytest.mark.gpu
def test_readme_quickstart_runs(capsys):
    pytest.importorskip("torch")
    exec(compile(_quickstart(), "README.md", "exec"), {"__name__": "readme"})
    out = capsys.readouterr().out
    m = re.search(r"(\d+) values changed; payload (\d+) bytes for (\d+) weight bytes", out)
    assert m, out
    changed, size, n = map(int, m.groups())
    assert n == 1024 * 1024 * 2 + 1024 * 2
    assert 0 < changed and 0 < size < n
