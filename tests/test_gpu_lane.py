"""ZSRC frames through the walks that take large or Snappy frames: one
thread per frame (the LANE apply variant), the split walk (big_kernel on
plans of the Snappy codec) and the windowed walk (big_kernel on plans of the
LZ4 codec).  Hand-made LZ4 and Snappy blocks are checked byte for byte
against the oracle's apply of the same stream.

The thread proves a match copies zeros only when its source lies after the
last non-zero output byte or between the last two.  The blocks below also
hold valid matches whose source lies in an older zero stretch (the walk must
undo its XORs and hand the frame to the bitmap walk, which applies it), a
match that copies a non-zero byte late in the block and one whose source
starts before the chunk (rejected, the chunk left as it was), and truncated
bodies.  Each block opens with 3200 random literal bytes, so the split
walk's lanes start their stretches inside literal data and must be joined;
random single-byte corruptions of the blocks check every walk against the
oracle's verdict."""
import numpy as np
import pytest

import oracle
from synth import configs
from streamfmt import FRAME_ZSRC, K_XOR_LZ4, K_XOR_SNAPPY, build_stream

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_exact_xor_gb300 as dcr  # noqa: E402
from wl import descs_of, to_device  # noqa: E402

CHUNK = 65536
N_CHUNKS = 4


def _ext(out, v):
    while v >= 255:
        out.append(255)
        v -= 255
    out.append(v)


def lz4_block(seqs):
    """LZ4 block from (literals, offset, match length) sequences (block
    format: token, length bytes, literals, 2-byte offset, length bytes); the
    last sequence has offset None and no match."""
    out = bytearray()
    for lit, off, ml in seqs:
        ll = len(lit)
        m = 0 if off is None else ml - 4
        out.append((min(ll, 15) << 4) | min(m, 15))
        if ll >= 15:
            _ext(out, ll - 15)
        out += bytes(lit)
        if off is None:
            break
        out += int(off).to_bytes(2, "little")
        if m >= 15:
            _ext(out, m - 15)
    return bytes(out)


def snappy_block(raw, elems):
    """Snappy block: varint output length, then ("lit", bytes) and ("copy",
    offset, length) elements (copies of at most 64 bytes, 2-byte offset)."""
    out = bytearray()
    v = raw
    while v >= 128:
        out.append((v & 127) | 128)
        v >>= 7
    out.append(v)
    for e in elems:
        if e[0] == "lit":
            b = bytes(e[1])
            n = len(b) - 1
            if n < 60:
                out.append(n << 2)
            else:
                nb = 1 if n < 256 else 2
                out.append((59 + nb) << 2)
                out += n.to_bytes(nb, "little")
            out += b
        else:
            _, off, ln = e
            while ln:
                k = min(ln, 64)
                out.append(((k - 1) << 2) | 2)
                out += int(off).to_bytes(2, "little")
                ln -= k
    return bytes(out)


def _rand_lit(rng, n):
    return rng.randint(1, 256, size=n).astype(np.uint8).tobytes()


# the match or copy after the 7 that ends the hand-made prefix, per case:
# (distance back from the position after the 7 to the source start, length)
#   old_gap  source in the zeros behind the last two non-zero bytes: valid,
#            not provable by the thread walk
#   lying    source covers the 5: copies a non-zero byte
#   recent   source between the 6 and the 7: provable
#   plain    the zero literal after the 7 (offset 1): provable
#   far      source starts 10 bytes before the chunk: malformed


def lz4_case(kind, rng):
    """Sequences of one 64 KiB chunk: 3200 random literal bytes (a body above
    the warp kernel's cache), zeros copied from just behind, non-zero bytes
    5, 6 and 7 at 3308, 3363 and 3385, the case's match, then zeros to the
    chunk's end."""
    seqs = [(_rand_lit(rng, 3200) + bytes(8), 8, 100),   # zeros [3200, 3308)
            (b"\x05" + bytes(4), 4, 50),                 # 5 at 3308, zeros to 3363
            (b"\x06\x00", 1, 20)]                        # 6 at 3363, zeros to 3385
    op = 3385
    if kind == "plain":
        seqs.append((b"\x07\x00", 1, 40))
        op += 2 + 40
    else:
        back, ml = {"old_gap": (3386 - 3205, 40), "lying": (3386 - 3300, 40), "recent": (3386 - 3370, 10),
                    "far": (3386 + 10, 40)}[kind]
        seqs.append((b"\x07", back, ml))
        op += 1 + ml
    seqs.append((b"\x00", 1, CHUNK - op - 1 - 5))
    seqs.append((bytes(5), None, 0))
    return lz4_block(seqs)


def snappy_case(kind, rng):
    """The same shape in Snappy elements: 300 random literal bytes, then
    non-zero bytes 5, 6 and 7 at 408, 460 and 482."""
    el = [("lit", _rand_lit(rng, 300) + bytes(8)), ("copy", 8, 100),   # zeros [300, 408)
          ("lit", b"\x05\x00"), ("copy", 1, 50),                        # 5 at 408
          ("lit", b"\x06\x00"), ("copy", 1, 20)]                        # 6 at 460
    op = 482
    if kind == "plain":
        el += [("lit", b"\x07\x00"), ("copy", 1, 40)]
        op += 2 + 40
    else:
        back, ln = {"old_gap": (483 - 305, 40), "lying": (483 - 400, 40), "recent": (483 - 476, 4),
                    "far": (483 + 10, 40)}[kind]
        el += [("lit", b"\x07"), ("copy", back, ln)]
        op += 1 + ln
    el += [("lit", b"\x00"), ("copy", 1, CHUNK - op - 1)]
    return snappy_block(CHUNK, el)


@pytest.fixture(scope="module")
def setup():
    t0 = configs.Tensor("z", elem_bits=8, rows=N_CHUNKS, cols=CHUNK, split=configs.REPLICATED, value_kind=1,
                        rule=0, frac=0)
    wl = configs.Workload("lane", 3, 1, [t0]).layout()
    orc = oracle.Oracle(wl)
    assert orc.n_chunks == N_CHUNKS and all(orc.chunk_info(c)[3] == CHUNK for c in range(N_CHUNKS))
    rng = np.random.RandomState(5)
    old = rng.randint(0, 256, size=wl.shard_bytes[0]).astype(np.uint8)
    # walk -> (plan codec, apply variant) whose big_kernel (or lane_kernel) takes the frames
    plans = {
        "lane-lz4": dcr.Plan(descs_of(wl), apply=dcr.APPLY_LANE, codec=dcr.CODEC_LZ4),
        "lane-snappy": dcr.Plan(descs_of(wl), apply=dcr.APPLY_LANE, codec=dcr.CODEC_SNAPPY),
        "split": dcr.Plan(descs_of(wl), apply=dcr.APPLY_WARP, codec=dcr.CODEC_SNAPPY),
        "split-all": dcr.Plan(descs_of(wl), apply=dcr.APPLY_SPLIT, codec=dcr.CODEC_LZ4),
        "window": dcr.Plan(descs_of(wl), apply=dcr.APPLY_WARP, codec=dcr.CODEC_LZ4),
    }
    return wl, orc, old, plans


WALKS = ["lane", "split", "split-all", "window"]


def _plan(plans, walk, codec):
    return plans["%s-%s" % (walk, codec)] if walk == "lane" else plans[walk]


def _blocks(codec, kinds):
    rng = np.random.RandomState(11)
    out = []
    for kind in kinds:
        body = lz4_case(kind, rng) if codec == "lz4" else snappy_case(kind, rng)
        dec = oracle.lz4_decode if codec == "lz4" else oracle.snappy_decode
        m = dec(np.frombuffer(body, np.uint8), CHUNK)
        assert (m is None) == (kind == "far")                      # a well-formed block, but in "far"
        if m is not None:
            assert m.size == CHUNK
            zs = dec(np.frombuffer(body, np.uint8), CHUNK, zsrc=True)
            assert (zs is None) == (kind == "lying")               # every match copies zeros, but in "lying"
        if codec == "lz4":
            assert len(body) > 3072                                # above the warp kernel's body cache
        out.append((body, 0 if m is None else int(np.count_nonzero(m))))
    return out


def _apply_both(setup, walk, codec, bodies):
    wl, orc, old, plans = setup
    frames = [(K_XOR_LZ4 if codec == "lz4" else K_XOR_SNAPPY, 8, FRAME_ZSRC, c, CHUNK, chg, body)
              for c, (body, chg) in enumerate(bodies)]
    stream = np.frombuffer(build_stream(orc.plan_hash, 0, 0, N_CHUNKS, frames), np.uint8).copy()
    start = orc.receiver_dense([old])
    ref = start.copy()
    orc_rc = orc.apply(orc.state(0), stream, ref)
    plan = _plan(plans, walk, codec)
    t = to_device([start])[0]
    rc, _ = dcr.apply(plan, dcr.RecvState(plan, 0), torch.from_numpy(stream).cuda(), stream.size, t)
    got = t.cpu().numpy()[:start.size]
    return orc_rc, rc, got, ref, start


def _run(setup, walk, codec, kinds, truncate=None):
    bodies = _blocks(codec, kinds)
    if truncate is not None:
        bodies[truncate] = (bodies[truncate][0][:-3], bodies[truncate][1])
    return _apply_both(setup, walk, codec, bodies)


@pytest.mark.parametrize("walk", WALKS)
@pytest.mark.parametrize("codec", ["lz4", "snappy"])
def test_valid_frames_proven_or_handed_on(setup, walk, codec):
    orc_rc, rc, got, ref, start = _run(setup, walk, codec, ["recent", "old_gap", "plain", "old_gap"])
    assert orc_rc == oracle.OK and rc == dcr.OK
    assert np.array_equal(got, ref) and not np.array_equal(got, start)


@pytest.mark.parametrize("walk", WALKS)
@pytest.mark.parametrize("codec", ["lz4", "snappy"])
@pytest.mark.parametrize("bad", ["lying", "far"])
def test_lying_frame_rejected_and_undone(setup, walk, codec, bad):
    orc_rc, rc, got, ref, start = _run(setup, walk, codec, ["recent", bad, "old_gap", "plain"])
    assert orc_rc == oracle.E_CORRUPT and rc == dcr.ERR_CORRUPT
    # the other frames applied, the rejected one's chunk exactly as it was
    assert np.array_equal(got[CHUNK:2 * CHUNK], start[CHUNK:2 * CHUNK])
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("walk", WALKS)
@pytest.mark.parametrize("codec", ["lz4", "snappy"])
def test_truncated_frame_rejected_and_undone(setup, walk, codec):
    orc_rc, rc, got, ref, start = _run(setup, walk, codec, ["plain", "recent", "old_gap", "plain"], truncate=2)
    assert orc_rc == oracle.E_CORRUPT and rc == dcr.ERR_CORRUPT
    assert np.array_equal(got[2 * CHUNK:3 * CHUNK], start[2 * CHUNK:3 * CHUNK])
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("walk", WALKS)
@pytest.mark.parametrize("codec", ["lz4", "snappy"])
def test_corrupted_bytes_follow_the_oracle(setup, walk, codec):
    # one byte of one frame replaced, 48 times: whether the frame is still a
    # valid ZSRC block (then applied) or not (then rejected, its chunk as it
    # was) is the oracle's call; the receiver bytes must agree either way
    base = _blocks(codec, ["recent", "old_gap", "plain", "old_gap"])
    rng = np.random.RandomState(1000 + 10 * WALKS.index(walk) + (codec == "snappy"))
    verdicts = set()
    for _ in range(48):
        bodies = list(base)
        f = int(rng.randint(len(bodies)))
        b = bytearray(bodies[f][0])
        # half of the hits on the structure after the random literal prefix
        i = int(rng.randint(len(b))) if rng.rand() < 0.5 else int(rng.randint(len(b) - 120, len(b)))
        b[i] = (b[i] + int(rng.randint(1, 256))) % 256
        bodies[f] = (bytes(b), bodies[f][1])
        orc_rc, rc, got, ref, _ = _apply_both(setup, walk, codec, bodies)
        assert (orc_rc == oracle.OK) == (rc == dcr.OK), (f, i, orc_rc, rc)
        assert np.array_equal(got, ref), (f, i)
        verdicts.add(rc)
    assert verdicts == {dcr.OK, dcr.ERR_CORRUPT}


@pytest.mark.parametrize("codec", ["lz4", "snappy"])
def test_retry_stream_from_hand_made_xor_stream(setup, codec):
    # dcr_encode_retry walks ZSRC frames one thread each too: a valid match it
    # cannot prove hands the frame to the full decode, which must build the
    # same records; the retry stream then equals the oracle's overwrite-only
    # encode of (old, old ^ mask) byte for byte.  A lying frame is rejected.
    wl, orc, old, plans = setup
    plan = _plan(plans, "lane", codec)
    for kinds, ok in ((["recent", "old_gap", "plain", "old_gap"], True), (["recent", "lying", "plain", "plain"], False)):
        rng = np.random.RandomState(11)
        frames, new = [], old.copy()
        for c, kind in enumerate(kinds):
            body = lz4_case(kind, rng) if codec == "lz4" else snappy_case(kind, rng)
            dec = oracle.lz4_decode if codec == "lz4" else oracle.snappy_decode
            m = dec(np.frombuffer(body, np.uint8), CHUNK)
            new[c * CHUNK:(c + 1) * CHUNK] ^= m
            frames.append((K_XOR_LZ4 if codec == "lz4" else K_XOR_SNAPPY, 8, FRAME_ZSRC, c, CHUNK,
                           int(np.count_nonzero(m)), body))
        stream = np.frombuffer(build_stream(orc.plan_hash, 0, 0, N_CHUNKS, frames), np.uint8).copy()
        d_new = to_device([new])
        out = torch.zeros(plan.window(0).payload_bound, dtype=torch.uint8, device="cuda")
        rc, size = dcr.encode_retry(plan, torch.from_numpy(stream).cuda(), stream.size, d_new, out)
        if not ok:
            assert rc == dcr.ERR_CORRUPT
            continue
        assert rc == dcr.OK, dcr.last_error()
        ref, _ = orc.encode([old], [new], mode=oracle.MODE_OVERWRITE_ONLY)
        assert size == ref.size and np.array_equal(out[:size].cpu().numpy(), ref)
