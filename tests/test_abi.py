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


def _build(descs, window_bytes=0):
    """dcr_plan_build on descriptors that fail validation (rejected before
    any CUDA call, so this runs without a GPU)."""
    import ctypes
    arr = (dcr.TensorDesc * len(descs))(*descs)
    opts = dcr.PlanOpts(window_bytes)
    h = ctypes.c_void_p()
    rc = dcr.lib().dcr_plan_build(arr, len(descs), ctypes.byref(opts), ctypes.byref(h))
    return rc, dcr.last_error(), h.value


def test_plan_rejects_degenerate_tensors():
    ok = dict(split=dcr.REPLICATED, tp=1, shard_offset=[0], recv_offset=0)
    cases = [
        (dcr.make_desc("empty_rows", 16, 0, 64, **ok), "empty tensor"),
        (dcr.make_desc("empty_cols", 16, 64, 0, **ok), "empty tensor"),
        (dcr.make_desc("bits", 12, 64, 64, **ok), "elem_bits"),
        (dcr.make_desc("odd_e2m1", 4, 64, 63, **ok), "even column"),
        (dcr.make_desc("tp0", 16, 64, 64, dcr.REPLICATED, 0, [0], 0), "tp must be"),
        (dcr.make_desc("tp17", 16, 64, 64, dcr.REPLICATED, 17, [0] * 16, 0), "tp must be"),
        (dcr.make_desc("rows", 16, 65, 64, dcr.SPLIT_ROWS, 2, [0, 0], 0), "rows not divisible"),
        (dcr.make_desc("cols", 16, 64, 65, dcr.SPLIT_COLS, 2, [0, 0], 0), "cols not divisible"),
        (dcr.make_desc("qkv0", 16, 64, 64, dcr.RESIDUAL_QKV_INTERLEAVED, 2, [0, 0], 0), "head counts"),
        (dcr.make_desc("qkv_rows", 16, 100, 64, dcr.RESIDUAL_QKV_INTERLEAVED, 2, [0, 0], 0, q_heads=4, kv_heads=2,
                       head_dim=8), "qkv rows"),
        (dcr.make_desc("qkv_div", 16, (3 + 2) * 8, 64, dcr.RESIDUAL_QKV_INTERLEAVED, 1, [0], 0, q_heads=3, kv_heads=1,
                       head_dim=8, recv_layout=dcr.LAYOUT_ROWGROUP_INTERLEAVE, recv_group=8), "receiver layout"),
        (dcr.make_desc("group", 16, 60, 64, dcr.REPLICATED, 1, [0], 0, recv_layout=dcr.LAYOUT_ROWGROUP_INTERLEAVE,
                       recv_group=8), "row-group"),
        (dcr.make_desc("slot2", 16, 64, 64, dcr.REPLICATED, 1, [0], 0, recv_layout=dcr.LAYOUT_ROWGROUP_INTERLEAVE,
                       recv_group=8, recv_slot=2), "row-group"),
        (dcr.make_desc("e2m1_shard", 4, 64, 66, dcr.SPLIT_COLS, 2, [0, 0], 0), "shard columns must be even"),
        (dcr.make_desc("split7", 16, 64, 64, 7, 1, [0], 0), "unknown split"),
        (dcr.make_desc("layout5", 16, 64, 64, dcr.REPLICATED, 1, [0], 0, recv_layout=5), "unknown receiver layout"),
    ]
    for d, why in cases:
        rc, msg, h = _build([d])
        assert rc == dcr.ERR_INVALID and h is None, (d.name, rc)
        assert why in msg and d.name.decode() in msg, (why, msg)


def test_plan_rejects_window_sizes_out_of_range():
    d = dcr.make_desc("t", 16, 64, 64, dcr.REPLICATED, 1, [0], 0)
    for w in (1, 65535, (256 << 30) + 1):
        rc, msg, h = _build([d], window_bytes=w)
        assert rc == dcr.ERR_INVALID and "window_bytes" in msg and h is None


def test_calls_reject_null_handles():
    import ctypes
    L = dcr.lib()
    size = ctypes.c_size_t()
    assert L.dcr_encode(None, 0, 0, None, None, 0, 1, None, 0, ctypes.byref(size), None, None) == dcr.ERR_INVALID
    assert L.dcr_apply(None, None, None, 0, None, None, None, None) == dcr.ERR_INVALID
    assert L.dcr_apply_retry(None, None, None, 0, None, None, None) == dcr.ERR_INVALID
    assert L.dcr_apply_noalloc(None, None, None, 0, None, None, None) == dcr.ERR_INVALID
    assert L.dcr_dense_refit(None, None, None, None) == dcr.ERR_INVALID
    h = ctypes.c_void_p()
    assert L.dcr_recv_state_create(None, 0, ctypes.byref(h)) == dcr.ERR_INVALID
    assert L.dcr_plan_set_profiling(None, 1) == dcr.ERR_INVALID
    dev, host = ctypes.c_size_t(), ctypes.c_size_t()
    assert L.dcr_pipeline_sizes(None, ctypes.byref(dev), ctypes.byref(host)) == dcr.ERR_INVALID
    assert L.dcr_refit_pipelined(None, None, 0, None, None, 0, 1, None, None, 0, None, 0, None, None,
                                 None) == dcr.ERR_INVALID
    assert "NULL" in dcr.last_error()


def test_plan_rejects_unknown_encoder_variant():
    import ctypes
    d = dcr.make_desc("t", 16, 64, 64, dcr.REPLICATED, 1, [0], 0)
    arr = (dcr.TensorDesc * 1)(d)
    opts = dcr.PlanOpts(0, dcr.ENCODER_CTA + 1)
    h = ctypes.c_void_p()
    rc = dcr.lib().dcr_plan_build(arr, 1, ctypes.byref(opts), ctypes.byref(h))
    assert rc == dcr.ERR_INVALID and "encoder" in dcr.last_error() and h.value is None
    opts = dcr.PlanOpts(0, 0, 0, 0, dcr.APPLY_SPLIT + 1)
    rc = dcr.lib().dcr_plan_build(arr, 1, ctypes.byref(opts), ctypes.byref(h))
    assert rc == dcr.ERR_INVALID and "apply" in dcr.last_error() and h.value is None
    opts = dcr.PlanOpts(0, 0, 0, 4)   # unknown plan flag
    rc = dcr.lib().dcr_plan_build(arr, 1, ctypes.byref(opts), ctypes.byref(h))
    assert rc == dcr.ERR_INVALID and "flags" in dcr.last_error() and h.value is None


def header_constants():
    """Every DCR_* constant of include/dcr.h: enumerators (implicit values
    count on from the previous one) and integer #defines."""
    src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "dcr.h")).read(), flags=re.S)
    out = {}
    for body in re.findall(r"enum\s*\{(.*?)\}", src, flags=re.S):
        nxt = 0
        for item in body.split(","):
            m = re.match(r"\s*(DCR_\w+)\s*(?:=\s*(-?\w+))?\s*$", item)
            if not m:
                continue
            nxt = int(m.group(2), 0) if m.group(2) else nxt
            out[m.group(1)] = nxt
            nxt += 1
    for name, val in re.findall(r"#define\s+(DCR_\w+)\s+(0x[0-9A-Fa-f]+|\d+)u?\s*$", src, flags=re.M):
        out[name] = int(val, 0)
    return out


def test_header_constants_match_binding_and_bench():
    h = header_constants()
    # the binding's names are the header's without the DCR_ prefix
    for name, val in h.items():
        py = name[len("DCR_"):]
        if py in ("CHUNK_BYTES", "STREAM_HEADER_BYTES", "FRAME_HEADER_BYTES", "H"):
            continue
        assert hasattr(dcr, py), name
        assert getattr(dcr, py) == val, (name, val, getattr(dcr, py))
    for v in ("AUTO", "WARP", "CTA", "LANE", "SPLIT"):
        assert "DCR_APPLY_" + v in h
    assert h["DCR_CHUNK_BYTES"] == dcr.CHUNK_BYTES
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.APPLY_VARIANTS == {k.lower()[len("DCR_APPLY_"):]: v for k, v in h.items() if k.startswith("DCR_APPLY_")}
    assert bench.ENCODER_VARIANTS == {k.lower()[len("DCR_ENCODER_"):]: v for k, v in h.items()
                                      if k.startswith("DCR_ENCODER_")}
