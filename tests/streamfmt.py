"""Independent reader of the refit stream wire format, for tests only.

Layout (little-endian): a 64-byte stream header, 16-byte-aligned frames in
ascending chunk order (each a 32-byte frame header plus body), then an index
of u64 frame offsets.  Written from the format description alone; shares no
code with the oracle or the CUDA library.
"""
import struct

import numpy as np

STREAM_MAGIC = b"DCRS"
FRAME_MAGIC = b"DCRF"
K_XOR_LZ4, K_XOR_RAW, K_OVERWRITE, K_OVERWRITE_DENSE, K_XOR_SNAPPY = 1, 2, 3, 4, 5
FLAG_OVERWRITE_ONLY = 1
FRAME_ZSRC = 1


def parse(payload):
    b = bytes(np.asarray(payload, dtype=np.uint8))
    assert len(b) >= 64
    (magic, fmt, plan_hash, base_v, target_v, window, flags, cb, cc, nf, total) = struct.unpack_from(
        "<4sIQQQIIIIQQ", b, 0)
    hdr = dict(magic=magic, format=fmt, plan_hash=plan_hash, base_version=base_v,
               target_version=target_v, window=window, flags=flags, chunk_begin=cb,
               chunk_count=cc, n_frames=nf, total=total)
    idx_off = total - 8 * nf
    offs = list(struct.unpack_from("<%dQ" % nf, b, idx_off)) if nf else []
    frames = []
    for o in offs:
        fm, kind, bits, fflags, chunk, raw, bl, changed, res = struct.unpack_from("<4sBBHIIIIQ", b, o)
        frames.append(dict(offset=o, magic=fm, kind=kind, elem_bits=bits, flags=fflags, chunk=chunk,
                           raw_len=raw, body_len=bl, changed=changed, reserved=res,
                           body=np.frombuffer(b[o + 32:o + 32 + bl], dtype=np.uint8)))
    return hdr, frames, idx_off


def check_structure(payload):
    """Structural invariants every well-formed stream meets."""
    hdr, frames, idx_off = parse(payload)
    assert hdr["magic"] == STREAM_MAGIC and hdr["format"] == 1
    assert hdr["total"] == len(payload)
    pos = 64
    prev = -1
    for f in frames:
        assert f["magic"] == FRAME_MAGIC
        assert f["offset"] == pos, "frames are contiguous and in index order"
        assert f["offset"] % 16 == 0
        assert hdr["chunk_begin"] <= f["chunk"] < hdr["chunk_begin"] + hdr["chunk_count"]
        assert f["chunk"] > prev, "ascending chunk order"
        prev = f["chunk"]
        assert f["kind"] in (1, 2, 3, 4, 5) and f["reserved"] == 0 and f["changed"] > 0
        flen = (32 + f["body_len"] + 15) // 16 * 16
        pad = np.asarray(payload[f["offset"] + 32 + f["body_len"]:f["offset"] + flen])
        assert not pad.any(), "frame padding is zero"
        pos += flen
    assert pos == idx_off
    return hdr, frames


def overwrite_records(f):
    """(unit offsets, values as uint8 rows) of an OVERWRITE frame body."""
    body = f["body"]
    ub = 2 if f["elem_bits"] == 16 else 1
    n = int(struct.unpack_from("<I", body.tobytes(), 0)[0])
    offs = np.frombuffer(body[4:4 + 2 * n].tobytes(), dtype="<u2").astype(np.int64)
    pad = (4 - (2 * n) % 4) % 4
    vals = body[4 + 2 * n + pad:4 + 2 * n + pad + n * ub].reshape(n, ub)
    return offs, vals


def build_stream(plan_hash, window, chunk_begin, chunk_count, frames, base_version=0, target_version=1,
                 flags=0):
    """A stream assembled by hand from the format description: frames is a
    list of (kind, elem_bits, frame_flags, chunk, raw_len, changed, body)."""
    out = bytearray(64)
    offs = []
    for kind, bits, fflags, chunk, raw, changed, body in frames:
        body = bytes(body)
        offs.append(len(out))
        out += struct.pack("<4sBBHIIIIQ", FRAME_MAGIC, kind, bits, fflags, chunk, raw, len(body), changed, 0)
        out += body + bytes((-(32 + len(body))) % 16)
    for o in offs:
        out += struct.pack("<Q", o)
    struct.pack_into("<4sIQQQIIIIQQ", out, 0, STREAM_MAGIC, 1, plan_hash, base_version, target_version,
                     window, flags, chunk_begin, chunk_count, len(offs), len(out))
    return np.frombuffer(bytes(out), dtype=np.uint8).copy()


def overwrite_body(offsets, values, unit):
    """OVERWRITE body: u32 count, u16 unit offsets, pad to 4, the new units."""
    n = len(offsets)
    b = struct.pack("<I", n) + struct.pack("<%dH" % n, *offsets)
    b += bytes((4 - (2 * n) % 4) % 4)
    assert len(values) == n * unit
    return b + bytes(values)
