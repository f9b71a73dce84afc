"""Python binding of libdcr (bit-exact delta-compressed refit on GB300).

Argument marshalling only: every step of the refit runs in the library's CUDA
kernels.  Device buffers are passed as torch CUDA tensors (or raw integer
device pointers); PyTorch is used for device memory and streams only.  The
library must be built (``__graft_entry__.build()``); importing this package
without it raises.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdcr.so")

MAX_TP = 16
CHUNK_BYTES = 65536
NO_FAULT = 2**64 - 1

OK = 0
ERR_INVALID, ERR_CAPACITY, ERR_CORRUPT, ERR_VERSION, ERR_ABORTED = -1, -2, -3, -4, -5
ERR_CUDA, ERR_NOMEM, ERR_INCOMPLETE, ERR_TIMEOUT = -6, -7, -8, -9
STATUS_NAMES = {0: "OK", -1: "INVALID", -2: "CAPACITY", -3: "CORRUPT", -4: "VERSION", -5: "ABORTED",
                -6: "CUDA", -7: "NOMEM", -8: "INCOMPLETE", -9: "TIMEOUT"}

REPLICATED, SPLIT_ROWS, SPLIT_COLS, RESIDUAL_QKV_INTERLEAVED = 0, 1, 2, 3
LAYOUT_CANONICAL, LAYOUT_ROWGROUP_INTERLEAVE = 0, 1
MODE_HYBRID, MODE_OVERWRITE_ONLY = 0, 1
ENCODER_AUTO, ENCODER_WIDE, ENCODER_DEEP, ENCODER_CTA = 0, 1, 2, 3
APPLY_AUTO, APPLY_WARP, APPLY_CTA, APPLY_LANE, APPLY_SPLIT = 0, 1, 2, 3, 4
CODEC_LZ4, CODEC_SNAPPY = 0, 1
PLAN_HOST_ONLY = 1
PLAN_TEST_STALL_SCAN = 2   # test only: the encoder's offset scan waits out its limit
NO_OVERFLOW = 0xFFFFFFFF
MAX_PARTS = 65536


class DcrError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("%s (%d): %s" % (STATUS_NAMES.get(code, "?"), code, msg))
        self.code = code


class TensorDesc(ctypes.Structure):
    _fields_ = [
        ("name", ctypes.c_char_p),
        ("elem_bits", ctypes.c_uint32), ("split", ctypes.c_uint32), ("tp", ctypes.c_uint32),
        ("q_heads", ctypes.c_uint32), ("kv_heads", ctypes.c_uint32), ("head_dim", ctypes.c_uint32),
        ("rows", ctypes.c_uint64), ("cols", ctypes.c_uint64),
        ("shard_offset", ctypes.c_uint64 * MAX_TP),
        ("recv_layout", ctypes.c_uint32), ("recv_group", ctypes.c_uint32),
        ("recv_slot", ctypes.c_uint32), ("reserved", ctypes.c_uint32),
        ("recv_offset", ctypes.c_uint64),
    ]


class PlanOpts(ctypes.Structure):
    _fields_ = [("window_bytes", ctypes.c_uint64), ("encoder", ctypes.c_uint32), ("codec", ctypes.c_uint32),
                ("flags", ctypes.c_uint32), ("apply", ctypes.c_uint32), ("overflow_kib", ctypes.c_uint32),
                ("reserved", ctypes.c_uint32)]


class PartInfo(ctypes.Structure):
    _fields_ = [("chunk_begin", ctypes.c_uint64), ("chunk_count", ctypes.c_uint64),
                ("canonical_bytes", ctypes.c_uint64), ("shard_mask", ctypes.c_uint32),
                ("reserved", ctypes.c_uint32)]


class PartSize(ctypes.Structure):
    _fields_ = [("frame_bytes", ctypes.c_uint64), ("n_frames", ctypes.c_uint64)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("n_tensors", ctypes.c_uint64), ("n_parts", ctypes.c_uint64),
                ("n_chunks", ctypes.c_uint64), ("n_windows", ctypes.c_uint64),
                ("canonical_bytes", ctypes.c_uint64), ("plan_hash", ctypes.c_uint64),
                ("recv_bytes", ctypes.c_uint64), ("shard_bytes", ctypes.c_uint64 * MAX_TP),
                ("tp", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


class WindowInfo(ctypes.Structure):
    _fields_ = [("chunk_begin", ctypes.c_uint64), ("chunk_count", ctypes.c_uint64),
                ("canonical_bytes", ctypes.c_uint64), ("payload_bound", ctypes.c_uint64)]


class Fault(ctypes.Structure):
    _fields_ = [("abort_after_frames", ctypes.c_uint64), ("abort_split", ctypes.c_uint32),
                ("reserved", ctypes.c_uint32)]


class ApplyResult(ctypes.Structure):
    _fields_ = [("target_version", ctypes.c_uint64), ("n_frames", ctypes.c_uint64),
                ("frames_applied", ctypes.c_uint64), ("frames_skipped", ctypes.c_uint64),
                ("pending", ctypes.c_uint64), ("window", ctypes.c_uint32),
                ("committed", ctypes.c_uint32)]


class Profile(ctypes.Structure):
    _fields_ = [("encode_ms", ctypes.c_float), ("finalize_ms", ctypes.c_float),
                ("apply_ms", ctypes.c_float), ("defer_ms", ctypes.c_float),
                ("pending_ms", ctypes.c_float), ("encode_valid", ctypes.c_uint32),
                ("apply_valid", ctypes.c_uint32), ("encode_kernels", ctypes.c_uint32),
                ("apply_kernels", ctypes.c_uint32)]


class PipelineStats(ctypes.Structure):
    _fields_ = [("windows", ctypes.c_uint64), ("payload_bytes", ctypes.c_uint64),
                ("max_window_payload", ctypes.c_uint64), ("committed", ctypes.c_uint32),
                ("reserved", ctypes.c_uint32)]


EXPORTS = ["dcr_last_error", "dcr_plan_build", "dcr_plan_info_get", "dcr_window_info_get",
           "dcr_plan_destroy", "dcr_recv_state_create", "dcr_recv_state_destroy",
           "dcr_recv_state_version", "dcr_encode", "dcr_apply", "dcr_apply_retry",
           "dcr_dense_refit", "dcr_plan_set_profiling", "dcr_plan_last_profile", "dcr_apply_noalloc",
           "dcr_pipeline_sizes", "dcr_refit_pipelined", "dcr_part_info_get", "dcr_encode_part",
           "dcr_encode_part_write", "dcr_stream_layout", "dcr_stream_header", "dcr_encode_retry"]

_lib = None


def lib():
    """Load libdcr.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libdcr.so is not built; run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, VP, U32, U64, SZ = ctypes.POINTER, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_size_t
        L.dcr_last_error.restype = ctypes.c_char_p
        L.dcr_plan_build.argtypes = [P(TensorDesc), SZ, P(PlanOpts), P(VP)]
        L.dcr_plan_info_get.argtypes = [VP, P(PlanInfo)]
        L.dcr_window_info_get.argtypes = [VP, U32, P(WindowInfo)]
        L.dcr_plan_destroy.argtypes = [VP]
        L.dcr_plan_destroy.restype = None
        L.dcr_recv_state_create.argtypes = [VP, U64, P(VP)]
        L.dcr_recv_state_destroy.argtypes = [VP]
        L.dcr_recv_state_destroy.restype = None
        L.dcr_recv_state_version.argtypes = [VP, P(U64)]
        L.dcr_encode.argtypes = [VP, U32, U32, P(VP), P(VP), U64, U64, VP, SZ, P(SZ), P(U64), VP]
        L.dcr_apply.argtypes = [VP, VP, VP, SZ, VP, P(Fault), P(ApplyResult), VP]
        L.dcr_apply_retry.argtypes = [VP, VP, VP, SZ, VP, P(ApplyResult), VP]
        L.dcr_apply_noalloc.argtypes = [VP, VP, VP, SZ, VP, P(ApplyResult), VP]
        L.dcr_dense_refit.argtypes = [VP, P(VP), VP, VP]
        L.dcr_plan_set_profiling.argtypes = [VP, ctypes.c_int]
        L.dcr_plan_last_profile.argtypes = [VP, P(Profile)]
        L.dcr_pipeline_sizes.argtypes = [VP, P(SZ), P(SZ)]
        L.dcr_refit_pipelined.argtypes = [VP, VP, U32, P(VP), P(VP), U64, U64, VP, VP, SZ, VP, SZ, P(U64),
                                          P(PipelineStats), VP]
        L.dcr_part_info_get.argtypes = [VP, U32, U32, U32, P(PartInfo)]
        L.dcr_encode_part.argtypes = [VP, U32, U32, U32, U32, P(VP), P(VP), P(PartSize), P(U64), VP]
        L.dcr_encode_part_write.argtypes = [VP, U64, VP, SZ, VP, VP]
        L.dcr_stream_layout.argtypes = [U32, P(PartSize), P(U64), P(U64), P(U64)]
        L.dcr_stream_header.argtypes = [VP, U32, U32, U64, U64, U64, U64, VP]
        L.dcr_encode_retry.argtypes = [VP, VP, SZ, P(VP), VP, SZ, P(SZ), VP]
        _lib = L
    return _lib


def last_error():
    return lib().dcr_last_error().decode()


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr_array(xs):
    arr = (ctypes.c_void_p * MAX_TP)()
    for i, x in enumerate(xs):
        arr[i] = _ptr(x)
    return arr


def check(rc):
    if rc != OK:
        raise DcrError(rc, last_error())
    return rc


class Plan:
    """dcr_plan_build over a list of TensorDesc."""

    def __init__(self, descs, window_bytes=0, encoder=0, codec=0, host_only=False, apply=0, overflow_kib=0,
                 flags=0):
        arr = (TensorDesc * len(descs))(*descs)
        self._names = [d.name for d in descs]
        flags |= PLAN_HOST_ONLY if host_only else 0
        opts = PlanOpts(window_bytes, encoder, codec, flags, apply, overflow_kib)
        h = ctypes.c_void_p()
        check(lib().dcr_plan_build(arr, len(descs), ctypes.byref(opts), ctypes.byref(h)))
        self.h = h
        self.info = PlanInfo()
        check(lib().dcr_plan_info_get(self.h, ctypes.byref(self.info)))

    @property
    def n_windows(self):
        return self.info.n_windows

    def window(self, w):
        wi = WindowInfo()
        check(lib().dcr_window_info_get(self.h, w, ctypes.byref(wi)))
        return wi

    def part(self, window, part, n_parts):
        """dcr_part_info_get (host only)."""
        pi = PartInfo()
        check(lib().dcr_part_info_get(self.h, window, part, n_parts, ctypes.byref(pi)))
        return pi

    def set_profiling(self, on=True):
        check(lib().dcr_plan_set_profiling(self.h, int(on)))

    def last_profile(self):
        p = Profile()
        check(lib().dcr_plan_last_profile(self.h, ctypes.byref(p)))
        return p

    def close(self):
        if getattr(self, "h", None):
            lib().dcr_plan_destroy(self.h)
            self.h = None

    __del__ = close


class RecvState:
    def __init__(self, plan, version=0):
        self.plan = plan
        h = ctypes.c_void_p()
        check(lib().dcr_recv_state_create(plan.h, version, ctypes.byref(h)))
        self.h = h

    @property
    def version(self):
        v = ctypes.c_uint64()
        check(lib().dcr_recv_state_version(self.h, ctypes.byref(v)))
        return v.value

    def close(self):
        if getattr(self, "h", None):
            lib().dcr_recv_state_destroy(self.h)
            self.h = None

    __del__ = close


def encode(plan, olds, news, payload, cap=None, window=0, mode=MODE_HYBRID, base_version=0,
           target_version=1, counts=True, stream=None):
    """dcr_encode.  Returns (status, payload_size, per-tensor changed counts)."""
    size = ctypes.c_size_t()
    n = plan.info.n_tensors
    cnt = (ctypes.c_uint64 * n)() if counts else None
    if cap is None:
        cap = payload.numel() if payload is not None and not isinstance(payload, int) else 0
    rc = lib().dcr_encode(plan.h, mode, window, _ptr_array(olds), _ptr_array(news), base_version,
                          target_version, _ptr(payload), cap, ctypes.byref(size), cnt,
                          _stream(stream))
    return rc, size.value, (list(cnt) if counts else None)


def apply(plan, state, payload, size, target, fault=None, stream=None):
    """dcr_apply.  fault = (abort_after_frames, abort_split) or None.
    Returns (status, ApplyResult)."""
    res = ApplyResult()
    f = None
    if fault is not None:
        f = ctypes.byref(Fault(fault[0], fault[1], 0))
    rc = lib().dcr_apply(plan.h, state.h, _ptr(payload), size, _ptr(target), f, ctypes.byref(res),
                         _stream(stream))
    return rc, res


def apply_retry(plan, state, payload, size, target, stream=None):
    res = ApplyResult()
    rc = lib().dcr_apply_retry(plan.h, state.h, _ptr(payload), size, _ptr(target), ctypes.byref(res),
                               _stream(stream))
    return rc, res


def apply_noalloc(plan, state, payload, size, target, stream=None):
    """dcr_apply without allocation: scratch in the library's static device array."""
    res = ApplyResult()
    rc = lib().dcr_apply_noalloc(plan.h, state.h, _ptr(payload), size, _ptr(target), ctypes.byref(res),
                                 _stream(stream))
    return rc, res


def pipeline_sizes(plan):
    """dcr_pipeline_sizes: (device bytes, pinned host bytes) dcr_refit_pipelined needs."""
    dev, host = ctypes.c_size_t(), ctypes.c_size_t()
    check(lib().dcr_pipeline_sizes(plan.h, ctypes.byref(dev), ctypes.byref(host)))
    return dev.value, host.value


def refit_pipelined(plan, state, olds, news, target, device_buf, host_buf, mode=MODE_HYBRID, base_version=0,
                    target_version=1, counts=True, stream=None):
    """dcr_refit_pipelined.  device_buf: a device tensor, host_buf: a pinned
    host tensor (pipeline_sizes bytes each).  Returns (status, PipelineStats,
    per-tensor changed counts)."""
    n = plan.info.n_tensors
    cnt = (ctypes.c_uint64 * n)() if counts else None
    st = PipelineStats()
    rc = lib().dcr_refit_pipelined(plan.h, state.h, mode, _ptr_array(olds), _ptr_array(news), base_version,
                                   target_version, _ptr(target), _ptr(device_buf), device_buf.numel(),
                                   _ptr(host_buf), host_buf.numel(), cnt, ctypes.byref(st), _stream(stream))
    return rc, st, (list(cnt) if counts else None)


def encode_retry(plan, xor_payload, xor_size, news, payload, cap=None, stream=None):
    """dcr_encode_retry.  Returns (status, payload_size)."""
    size = ctypes.c_size_t()
    if cap is None:
        cap = payload.numel() if payload is not None and not isinstance(payload, int) else 0
    rc = lib().dcr_encode_retry(plan.h, _ptr(xor_payload), xor_size, _ptr_array(news), _ptr(payload), cap,
                                ctypes.byref(size), _stream(stream))
    return rc, size.value


def encode_part(plan, olds, news, part, n_parts, window=0, mode=MODE_HYBRID, counts=True, stream=None):
    """dcr_encode_part.  Returns (status, (frame_bytes, n_frames), per-tensor changed counts)."""
    size = PartSize()
    n = plan.info.n_tensors
    cnt = (ctypes.c_uint64 * n)() if counts else None
    rc = lib().dcr_encode_part(plan.h, mode, window, part, n_parts, _ptr_array(olds), _ptr_array(news),
                               ctypes.byref(size), cnt, _stream(stream))
    return rc, (size.frame_bytes, size.n_frames), (list(cnt) if counts else None)


def encode_part_write(plan, frame_offset, frames, frames_cap, index, stream=None):
    """dcr_encode_part_write: frames / index are device tensors or raw device addresses."""
    return lib().dcr_encode_part_write(plan.h, frame_offset, _ptr(frames), frames_cap, _ptr(index),
                                       _stream(stream))


def stream_layout(sizes):
    """dcr_stream_layout over [(frame_bytes, n_frames), ...] in part order.
    Returns (frame_offsets, index_offsets, total)."""
    n = len(sizes)
    arr = (PartSize * n)(*[PartSize(int(f), int(k)) for f, k in sizes])
    fo, io, tot = (ctypes.c_uint64 * n)(), (ctypes.c_uint64 * n)(), ctypes.c_uint64()
    check(lib().dcr_stream_layout(n, arr, fo, io, ctypes.byref(tot)))
    return list(fo), list(io), tot.value


def stream_header(plan, window, base_version, target_version, n_frames, frame_bytes, mode=MODE_HYBRID):
    """dcr_stream_header: the 64 header bytes (host)."""
    buf = (ctypes.c_uint8 * 64)()
    check(lib().dcr_stream_header(plan.h, mode, window, base_version, target_version, n_frames, frame_bytes,
                                  buf))
    return bytes(buf)


def gather_stream(plan, window, part, n_parts, size, write, base_version=0, target_version=1,
                  mode=MODE_HYBRID, group=None, dst=0, device="cpu"):
    """The exchange step of the ownership-sharded encode, one call per rank.

    Every rank owns part `part` (its rank in `group`) of `n_parts` parts of
    the window and has sized it: `size` = (frame_bytes, n_frames), as
    encode_part returns.  The ranks all-gather their sizes, take the stream
    layout from dcr_stream_layout, and each rank calls
    write(frame_offset, frames, index) to fill a staging tensor with its
    frames and index entries (on the GPU: encode_part_write).  The staging
    tensors are gathered to rank `dst`, which places them and the header
    (dcr_stream_header) into the window's stream.  Returns the stream (a
    uint8 tensor on `device`) on `dst`, None on the other ranks.  Only
    compressed frames cross between ranks."""
    import torch
    import torch.distributed as dist
    ws = dist.get_world_size(group)
    assert ws == n_parts and 0 <= part < n_parts
    mine = torch.tensor([int(size[0]), int(size[1])], dtype=torch.int64, device=device)
    allsz = [torch.empty_like(mine) for _ in range(ws)]
    dist.all_gather(allsz, mine, group=group)
    sizes = [(int(t[0]), int(t[1])) for t in allsz]
    fo, io, total = stream_layout(sizes)
    blob_bytes = [f + 8 * k for f, k in sizes]
    cap = max(max(blob_bytes), 16)
    blob = torch.zeros(cap, dtype=torch.uint8, device=device)
    fb, nf = sizes[part]
    write(fo[part], blob[:fb], blob[fb:fb + 8 * nf])
    rank = dist.get_rank(group) if group is not None else dist.get_rank()
    blobs = [torch.empty_like(blob) for _ in range(ws)] if rank == dst else None
    dist.gather(blob, blobs, dst=dst, group=group)
    if rank != dst:
        return None
    fbytes, nframes = sum(f for f, _ in sizes), sum(k for _, k in sizes)
    out = torch.empty(total, dtype=torch.uint8, device=device)
    hdr = stream_header(plan, window, base_version, target_version, nframes, fbytes, mode)
    out[:64] = torch.frombuffer(bytearray(hdr), dtype=torch.uint8).to(device)
    for q, (f, k) in enumerate(sizes):
        out[fo[q]:fo[q] + f] = blobs[q][:f]
        out[io[q]:io[q] + 8 * k] = blobs[q][f:f + 8 * k]
    return out


def dense_refit(plan, shards, target, stream=None):
    return lib().dcr_dense_refit(plan.h, _ptr_array(shards), _ptr(target), _stream(stream))


def make_desc(name, elem_bits, rows, cols, split, tp, shard_offset, recv_offset, q_heads=0, kv_heads=0,
              head_dim=0, recv_layout=LAYOUT_CANONICAL, recv_group=0, recv_slot=0):
    d = TensorDesc()
    d.name = name.encode() if isinstance(name, str) else name
    d.elem_bits, d.split, d.tp = elem_bits, split, tp
    d.q_heads, d.kv_heads, d.head_dim = q_heads, kv_heads, head_dim
    d.rows, d.cols = rows, cols
    for i, o in enumerate(shard_offset):
        d.shard_offset[i] = o
    d.recv_layout, d.recv_group, d.recv_slot = recv_layout, recv_group, recv_slot
    d.recv_offset = recv_offset
    return d
