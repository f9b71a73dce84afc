"""CPU oracle for bit-exact delta-compressed refit (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  It shares no code with ``bit_exact_xor_gb300`` and neither imports
the other.  See ``oracle.c`` for what each function computes and which
passage of the pages it follows.
"""
import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(HERE, "liboracle.so")
MAX_TP = 16
CHUNK = 65536

OK, E_INVALID, E_CAPACITY, E_CORRUPT, E_VERSION, E_ABORTED, E_NOMEM, E_INCOMPLETE = (
    0, -1, -2, -3, -4, -5, -7, -8)
MODE_HYBRID, MODE_OVERWRITE_ONLY = 0, 1
K_XOR_LZ4, K_XOR_RAW, K_OVERWRITE, K_OVERWRITE_DENSE, K_XOR_SNAPPY = 1, 2, 3, 4, 5
CODEC_LZ4, CODEC_SNAPPY = 0, 1
NO_FAULT = 2**64 - 1


class OrcTensor(ctypes.Structure):
    _fields_ = [
        ("elem_bits", ctypes.c_uint32), ("split", ctypes.c_uint32), ("tp", ctypes.c_uint32),
        ("q_heads", ctypes.c_uint32), ("kv_heads", ctypes.c_uint32), ("head_dim", ctypes.c_uint32),
        ("rows", ctypes.c_uint64), ("cols", ctypes.c_uint64),
        ("shard_off", ctypes.c_uint64 * MAX_TP),
        ("recv_layout", ctypes.c_uint32), ("recv_group", ctypes.c_uint32),
        ("recv_slot", ctypes.c_uint32), ("pad_", ctypes.c_uint32),
        ("recv_off", ctypes.c_uint64),
    ]


class OrcInfo(ctypes.Structure):
    _fields_ = [("n_parts", ctypes.c_uint64), ("n_chunks", ctypes.c_uint64),
                ("n_windows", ctypes.c_uint64), ("canonical_bytes", ctypes.c_uint64),
                ("plan_hash", ctypes.c_uint64)]


def build():
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           os.path.join(HERE, "oracle.c"), "-o", _SO]
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if p.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + p.stdout.decode())


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_SO):
            build()
        L = ctypes.CDLL(_SO)
        P, U32, U64, VP = ctypes.POINTER, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_void_p
        T = P(OrcTensor)
        L.orc_info_get.argtypes = [T, U32, U64, P(OrcInfo)]
        L.orc_window_range.argtypes = [T, U32, U64, U32, P(U64), P(U64)]
        L.orc_chunk_info.argtypes = [T, U32, U64, P(U32), P(U32), P(U64), P(U32)]
        L.orc_canonical.argtypes = [T, U32, VP, VP]
        L.orc_receiver_dense.argtypes = [T, U32, VP, VP]
        L.orc_xor.argtypes = [VP, VP, VP, U64]
        L.orc_xor.restype = None
        L.orc_count_changed.argtypes = [VP, U64, U32]
        L.orc_count_changed.restype = U64
        L.orc_fnv1a64.argtypes = [VP, U64]
        L.orc_fnv1a64.restype = U64
        L.orc_lz4_encode.argtypes = [VP, U64, VP, U64]
        L.orc_lz4_encode.restype = U64
        L.orc_lz4_decode.argtypes = [VP, U64, VP, U64, U32]
        L.orc_snappy_encode.argtypes = [VP, U64, VP, U64]
        L.orc_snappy_encode.restype = U64
        L.orc_snappy_decode.argtypes = [VP, U64, VP, U64, U32]
        L.orc_encode.argtypes = [T, U32, U64, VP, VP, U32, U32, U32, U64, U64, U32, VP, U64, P(U64), VP]
        L.orc_state_new.argtypes = [T, U32, U64, U64]
        L.orc_state_new.restype = VP
        L.orc_state_free.argtypes = [VP]
        L.orc_state_free.restype = None
        L.orc_state_version.argtypes = [VP]
        L.orc_state_version.restype = U64
        L.orc_apply.argtypes = [T, U32, U64, VP, VP, U64, VP, U32, U64, U32, U32, U32]
        _lib = L
    return _lib


def _ptr(a):
    return a.ctypes.data if a is not None else None


def tensors_of(workload):
    """orc_tensor array for a synth workload (its own copy of the layout)."""
    arr = (OrcTensor * len(workload.tensors))()
    for k, t in enumerate(workload.tensors):
        o = arr[k]
        o.elem_bits, o.split, o.tp = t.elem_bits, t.split, workload.tp
        o.q_heads, o.kv_heads, o.head_dim = t.q_heads, t.kv_heads, t.head_dim
        o.rows, o.cols = t.rows, t.cols
        for r in range(workload.tp):
            o.shard_off[r] = t.shard_offset[r]
        o.recv_layout, o.recv_group, o.recv_slot = t.recv_layout, t.recv_group, t.recv_slot
        o.recv_off = t.recv_offset
    return arr


class Oracle:
    """The oracle bound to one workload's tensor list."""

    def __init__(self, workload, window_bytes=None):
        self.wl = workload
        self.t = tensors_of(workload)
        self.n = len(workload.tensors)
        self.W = window_bytes if window_bytes is not None else workload.window_bytes
        info = OrcInfo()
        rc = lib().orc_info_get(self.t, self.n, self.W, ctypes.byref(info))
        if rc:
            raise ValueError("oracle rejected the tensor list (%d)" % rc)
        self.info = info

    @property
    def n_windows(self):
        return self.info.n_windows

    @property
    def n_chunks(self):
        return self.info.n_chunks

    @property
    def plan_hash(self):
        return self.info.plan_hash

    def window_range(self, w):
        b, c = ctypes.c_uint64(), ctypes.c_uint64()
        rc = lib().orc_window_range(self.t, self.n, self.W, w, ctypes.byref(b), ctypes.byref(c))
        if rc:
            raise ValueError(rc)
        return b.value, c.value

    def chunk_info(self, c):
        d, s, o, ln = ctypes.c_uint32(), ctypes.c_uint32(), ctypes.c_uint64(), ctypes.c_uint32()
        rc = lib().orc_chunk_info(self.t, self.n, c, ctypes.byref(d), ctypes.byref(s),
                                  ctypes.byref(o), ctypes.byref(ln))
        if rc:
            raise ValueError(rc)
        return d.value, s.value, o.value, ln.value

    @staticmethod
    def _shard_ptrs(shards):
        arr = (ctypes.c_void_p * MAX_TP)()
        for i, s in enumerate(shards):
            arr[i] = s.ctypes.data
        return arr

    def canonical(self, k, sub, shards):
        t = self.wl.tensors[k]
        rows = t.rows
        if t.split == 3:
            rows = (t.q_heads if sub == 0 else t.kv_heads) * t.head_dim
        out = np.zeros(rows * t.cols * t.elem_bits // 8, dtype=np.uint8)
        rc = lib().orc_canonical(ctypes.byref(self.t[k]), sub, self._shard_ptrs(shards), _ptr(out))
        if rc:
            raise ValueError(rc)
        return out

    def receiver_dense(self, shards):
        out = np.zeros(max(self.wl.recv_bytes, 16), dtype=np.uint8)
        rc = lib().orc_receiver_dense(self.t, self.n, self._shard_ptrs(shards), _ptr(out))
        if rc:
            raise ValueError(rc)
        return out

    def encode(self, olds, news, window=0, mode=MODE_HYBRID, base_version=0, target_version=1,
               threads=4, cap=None, codec=CODEC_LZ4):
        size = ctypes.c_uint64()
        changed = np.zeros(self.n, dtype=np.uint64)
        if cap is None:
            rc = lib().orc_encode(self.t, self.n, self.W, self._shard_ptrs(olds),
                                  self._shard_ptrs(news), mode, codec, window, base_version,
                                  target_version, threads, None, 0, ctypes.byref(size),
                                  _ptr(changed))
            if rc not in (OK, E_CAPACITY):
                raise ValueError("oracle encode failed (%d)" % rc)
            cap = size.value
        out = np.zeros(max(cap, 1), dtype=np.uint8)
        rc = lib().orc_encode(self.t, self.n, self.W, self._shard_ptrs(olds), self._shard_ptrs(news),
                              mode, codec, window, base_version, target_version, threads, _ptr(out), cap,
                              ctypes.byref(size), _ptr(changed))
        if rc:
            raise ValueError("oracle encode failed (%d)" % rc)
        return out[:size.value].copy(), changed

    def state(self, version=0):
        return OracleState(self, version)

    def apply(self, state, payload, target, retry_only=False, abort_at=NO_FAULT, split=0,
              dedup=True, threads=4):
        payload = np.ascontiguousarray(payload, dtype=np.uint8)
        return lib().orc_apply(self.t, self.n, self.W, state.h, _ptr(payload), payload.size,
                               _ptr(target), int(retry_only), abort_at, split, int(dedup), threads)


class OracleState:
    def __init__(self, orc, version):
        self.h = lib().orc_state_new(orc.t, orc.n, orc.W, version)
        if not self.h:
            raise ValueError("orc_state_new failed")

    @property
    def version(self):
        return lib().orc_state_version(self.h)

    def __del__(self):
        if getattr(self, "h", None):
            lib().orc_state_free(self.h)
            self.h = None


# ---- primitives -----------------------------------------------------------
def xor(a, b):
    out = np.empty_like(a)
    lib().orc_xor(_ptr(a), _ptr(b), _ptr(out), a.size)
    return out


def count_changed(mask, elem_bits):
    return int(lib().orc_count_changed(_ptr(mask), mask.size, elem_bits))


def fnv1a64(data):
    """FNV-1a 64 of a bytes object (the plan hash's step)."""
    buf = np.frombuffer(bytes(data), dtype=np.uint8) if len(data) else np.zeros(1, dtype=np.uint8)
    return int(lib().orc_fnv1a64(_ptr(buf), len(data)))


def lz4_encode(data):
    data = np.ascontiguousarray(data, dtype=np.uint8)
    cap = data.size + data.size // 255 + 16
    out = np.zeros(cap, dtype=np.uint8)
    n = lib().orc_lz4_encode(_ptr(data), data.size, _ptr(out), cap)
    if n == 0:
        raise ValueError("lz4 encode overflow")
    return out[:n].copy()


def lz4_decode(block, raw_len, zsrc=False):
    """Decoded bytes, or None if the block is malformed."""
    block = np.ascontiguousarray(block, dtype=np.uint8)
    out = np.zeros(max(raw_len, 1), dtype=np.uint8)
    rc = lib().orc_lz4_decode(_ptr(block), block.size, _ptr(out), raw_len, int(zsrc))
    return out[:raw_len] if rc == OK else None


def snappy_encode(data):
    data = np.ascontiguousarray(data, dtype=np.uint8)
    cap = data.size + data.size // 60 + 16
    out = np.zeros(cap, dtype=np.uint8)
    n = lib().orc_snappy_encode(_ptr(data), data.size, _ptr(out), cap)
    if n == 0:
        raise ValueError("snappy encode overflow")
    return out[:n].copy()


def snappy_decode(block, raw_len, zsrc=False):
    """Decoded bytes, or None if the block is malformed."""
    block = np.ascontiguousarray(block, dtype=np.uint8)
    out = np.zeros(max(raw_len, 1), dtype=np.uint8)
    rc = lib().orc_snappy_decode(_ptr(block), block.size, _ptr(out), raw_len, int(zsrc))
    return out[:raw_len] if rc == OK else None
