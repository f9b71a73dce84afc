"""Helpers that compare the CUDA path with the CPU oracle frame by frame."""
import numpy as np

import oracle
from streamfmt import K_OVERWRITE, K_OVERWRITE_DENSE, K_XOR_LZ4, K_XOR_RAW, K_XOR_SNAPPY, FRAME_ZSRC, parse


def frame_content(f):
    """What a frame says about its chunk, in a form independent of the
    encoder: ('mask', bytes) for XOR frames, ('put', offsets, values) for
    overwrite records, ('dense', bytes) for dense overwrites."""
    if f["kind"] == K_XOR_LZ4:
        m = oracle.lz4_decode(f["body"], f["raw_len"], zsrc=bool(f["flags"] & FRAME_ZSRC))
        assert m is not None, "oracle decoder rejected frame of chunk %d" % f["chunk"]
        return ("mask", m)
    if f["kind"] == K_XOR_SNAPPY:
        m = oracle.snappy_decode(f["body"], f["raw_len"], zsrc=bool(f["flags"] & FRAME_ZSRC))
        assert m is not None, "oracle decoder rejected frame of chunk %d" % f["chunk"]
        return ("mask", m)
    if f["kind"] == K_XOR_RAW:
        return ("mask", np.asarray(f["body"]))
    if f["kind"] == K_OVERWRITE:
        return ("put", np.asarray(f["body"]))
    return ("dense", np.asarray(f["body"]))


def frames_by_chunk(payload):
    hdr, frames, _ = parse(payload)
    return hdr, {f["chunk"]: f for f in frames}


def assert_same_frames(gpu_payload, orc_payload, chunks=None):
    """Same chunk set, same changed counts, same masks / overwrite records."""
    gh, gf = frames_by_chunk(gpu_payload)
    oh, of = frames_by_chunk(orc_payload)
    for k in ("plan_hash", "base_version", "target_version", "window", "flags", "chunk_begin",
              "chunk_count"):
        assert gh[k] == oh[k], k
    keys = set(of) if chunks is None else set(chunks) & (set(of) | set(gf))
    if chunks is None:
        assert set(gf) == set(of), "frame set differs"
    for c in sorted(keys):
        a, b = gf.get(c), of.get(c)
        assert (a is None) == (b is None), "chunk %d framed on one side only" % c
        if a is None:
            continue
        assert a["changed"] == b["changed"], "chunk %d changed count" % c
        assert a["raw_len"] == b["raw_len"] and a["elem_bits"] == b["elem_bits"]
        ca, cb = frame_content(a), frame_content(b)
        assert ca[0] == cb[0], "chunk %d kind family %s vs %s" % (c, a["kind"], b["kind"])
        assert np.array_equal(ca[1], cb[1]), "chunk %d content differs" % c
        if ca[0] != "mask":
            assert a["kind"] == b["kind"]
    return gh, gf, of
