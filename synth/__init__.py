"""Seeded synthetic weight generator (test and benchmark infrastructure).

Produces the raw old/new weight bit buffers that both the CPU oracle and the
CUDA path consume.  Holds none of the refit method's arithmetic.  The C twin
(``synth.c``) fills host buffers, the CUDA twin (``synth_gpu.cu``) fills
device buffers with the same bytes.
"""
import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
_CPU_SO = os.path.join(HERE, "libsynth.so")
_GPU_SO = os.path.join(HERE, "libsynth_gpu.so")

VAL_BF16_NORMAL, VAL_BYTES, VAL_E4M3_SCALE = 0, 1, 2
RULE_NONE, RULE_PM4, RULE_LOW3, RULE_NIBBLE, RULE_BPM4, RULE_RANDOM = 0, 1, 2, 3, 4, 5


class Params(ctypes.Structure):
    _fields_ = [
        ("seed", ctypes.c_uint64),
        ("stream", ctypes.c_uint64),
        ("elem_base", ctypes.c_uint64),
        ("threshold", ctypes.c_uint64),
        ("zero_threshold", ctypes.c_uint64),
        ("value_kind", ctypes.c_uint32),
        ("rule", ctypes.c_uint32),
    ]


def frac_threshold(f):
    """Selection threshold for a change fraction f (select iff hash < thr)."""
    if f <= 0:
        return 0
    return min(int(f * 2.0**64), 2**64 - 1)


def build(gpu=True):
    """Compile the CPU twin with gcc and (optionally) the GPU twin with nvcc."""
    cmds = [["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
             os.path.join(HERE, "synth.c"), "-o", _CPU_SO]]
    if gpu:
        cmds.append(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
                     "-Xcompiler", "-fPIC", "-shared", "-fmad=false",
                     os.path.join(HERE, "synth_gpu.cu"), "-o", _GPU_SO])
    procs = [subprocess.Popen(c, stdout=subprocess.PIPE, stderr=subprocess.STDOUT) for c in cmds]
    for c, p in zip(cmds, procs):
        out, _ = p.communicate()
        if p.returncode != 0:
            raise RuntimeError("synth build failed: %s\n%s" % (" ".join(c), out.decode()))


_cpu = None
_gpu = None


def _cpu_lib():
    global _cpu
    if _cpu is None:
        if not os.path.exists(_CPU_SO):
            build(gpu=False)
        _cpu = ctypes.CDLL(_CPU_SO)
        _cpu.syn_fill.argtypes = [ctypes.POINTER(Params), ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p]
        _cpu.syn_fill.restype = None
        _cpu.syn_count_selected.argtypes = [ctypes.POINTER(Params), ctypes.c_uint64]
        _cpu.syn_count_selected.restype = ctypes.c_uint64
    return _cpu


def _gpu_lib():
    global _gpu
    if _gpu is None:
        if not os.path.exists(_GPU_SO):
            raise RuntimeError("libsynth_gpu.so is not built: run __graft_entry__.build()")
        _gpu = ctypes.CDLL(_GPU_SO)
        _gpu.syn_fill_gpu.argtypes = [ctypes.POINTER(Params), ctypes.c_uint64, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p]
        _gpu.syn_fill_gpu.restype = ctypes.c_int
    return _gpu


def make_params(seed, stream, value_kind, rule, frac=0.0, zero_frac=0.0, elem_base=0):
    return Params(seed, stream, elem_base, frac_threshold(frac), frac_threshold(zero_frac),
                  value_kind, rule)


def elem_bytes(value_kind):
    return 2 if value_kind == VAL_BF16_NORMAL else 1


def fill_cpu(p, n_elems):
    """Return (old, new) as uint8 arrays of n_elems elements' bytes."""
    eb = elem_bytes(p.value_kind)
    old = np.empty(n_elems * eb, dtype=np.uint8)
    new = np.empty(n_elems * eb, dtype=np.uint8)
    _cpu_lib().syn_fill(ctypes.byref(p), n_elems, old.ctypes.data, new.ctypes.data)
    return old, new


def fill_cpu_into(p, n_elems, old_view, new_view):
    """Fill caller-provided contiguous uint8 numpy views (either may be None)."""
    optr = old_view.ctypes.data if old_view is not None else None
    nptr = new_view.ctypes.data if new_view is not None else None
    _cpu_lib().syn_fill(ctypes.byref(p), n_elems, optr, nptr)


def count_selected(p, n_elems):
    return int(_cpu_lib().syn_count_selected(ctypes.byref(p), n_elems))


def fill_gpu(p, n_elems, old_ptr, new_ptr, stream_ptr=0):
    """Fill device buffers (raw pointers) on the given CUDA stream."""
    rc = _gpu_lib().syn_fill_gpu(ctypes.byref(p), n_elems, old_ptr or None, new_ptr or None,
                                 stream_ptr or None)
    if rc != 0:
        raise RuntimeError("syn_fill_gpu failed")
