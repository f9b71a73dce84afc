"""The C-ABI library loads on a machine without a GPU and exports every
entry point declared in include/*.h (no compute calls)."""
import glob
import os
import re
import subprocess

import bit_exact_xor_gb300 as dcr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(dcr_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported():
    names = declared()
    assert {"dcr_plan_build", "dcr_encode", "dcr_apply", "dcr_apply_retry"} <= names
    L = dcr.lib()
    for n in sorted(names):
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", dcr.LIB_PATH], stdout=subprocess.PIPE).stdout.decode()
    exported = set(re.findall(r"\bT (dcr_\w+)", out))
    assert names <= exported, names - exported
    assert set(dcr.EXPORTS) <= exported


def test_last_error_without_gpu_work():
    rc = dcr.lib().dcr_plan_build(None, 0, None, None)
    assert rc == dcr.ERR_INVALID
    assert "NULL" in dcr.last_error() or "no tensors" in dcr.last_error()
