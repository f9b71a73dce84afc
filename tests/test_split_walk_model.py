"""A model, in plain Python, of how the split walk finds a block's chain of
elements (LZ4 sequences or Snappy elements): the body after the preamble is
cut into 32 stretches, each stretch is walked from its first few bytes as
though an element started there, and the stretches are joined in order by
following the true chain into each stretch until it meets a start that one
of that stretch's walks passed.  A chain of elements depends only on where
it starts, so the joined chain must be the one a serial parse finds, and a
body the serial parse rejects must be rejected.  The blocks are the
oracle's LZ4 and Snappy encodings of sparse masks, hand-corrupted copies of
them, and random bytes.  This checks the method; the GPU tests check the
kernel against the oracle."""
import numpy as np
import pytest

import oracle

BAD = 0x7FFFFFFF
FIN = 0x80000000
STRETCHES = 32


def lz4_end(src, n, p):
    """Where the LZ4 sequence at p ends (| FIN for the block's last), or BAD."""
    if p >= n:
        return BAD
    tok = src[p]
    q, ll = p + 1, tok >> 4
    if ll == 15:
        while True:
            if q >= n:
                return BAD
            b = src[q]
            q += 1
            ll += b
            if b != 255:
                break
    if ll > n - q:
        return BAD
    q += ll
    if q == n:
        return q | FIN
    if n - q < 2:
        return BAD
    q += 2
    if tok & 15 == 15:
        while True:
            if q >= n:
                return BAD
            b = src[q]
            q += 1
            if b != 255:
                break
    return q


def snappy_end(src, n, p):
    """Where the Snappy element at p ends (| FIN at the body's end), or BAD."""
    if p >= n:
        return BAD
    tag = src[p]
    t = tag & 3
    if t == 0:
        ln, nb = (tag >> 2) + 1, 0
        if tag >> 2 >= 60:
            nb = (tag >> 2) - 59
            if p + 1 + nb > n:
                return BAD
            ln = int.from_bytes(bytes(src[p + 1:p + 1 + nb]), "little") + 1
        e = p + 1 + nb + ln
    else:
        e = p + (2, 3, 5)[t - 1]
    if e > n:
        return BAD
    return e | FIN if e == n else e


def snappy_first(src, n):
    """End of the varint preamble, or BAD."""
    for i in range(min(5, n)):
        if not src[i] & 128:
            return i + 1
    return BAD


def bad_end(x, n):
    return x == BAD or (not x & FIN and x >= n)


def serial_chain(end, src, n, ip0):
    """The element starts of a serial parse, or None for a malformed body."""
    starts, p = [], ip0
    while True:
        x = end(src, n, p)
        if bad_end(x, n):
            return None
        starts.append(p)
        if x & FIN:
            return starts
        p = x


def split_chain(end, src, n, ip0, walks):
    """The split walk's chain: (element starts or None, elements the join
    re-walked)."""
    span = n - ip0
    S = (span + STRETCHES - 1) // STRETCHES
    edge = [ip0 + min(i * S, span) for i in range(STRETCHES + 1)]
    walker = {}   # start -> which walk of its stretch passed it
    ex = {}
    for i in range(STRETCHES):
        s0, s1 = edge[i], edge[i + 1]
        for c in range(walks):
            e, p = s1, s0 + c
            while p < s1:
                if p in walker:
                    e = ex[i, walker[p]]
                    break
                walker[p] = c
                x = end(src, n, p)
                if bad_end(x, n):
                    e = BAD
                    break
                if x & FIN or x >= s1:
                    e = x
                    break
                p = x
            ex[i, c] = e
    T, t, rework = [ip0], ex[0, 0], 0
    for i in range(1, STRETCHES):
        T.append(t)
        b = edge[i + 1]
        if t == BAD or t & FIN or t >= b:
            continue
        q = t
        while True:
            if q in walker:
                t = ex[i, walker[q]]
                break
            rework += 1
            x = end(src, n, q)
            if bad_end(x, n):
                t = BAD
                break
            if x & FIN or x >= b:
                t = x
                break
            q = x
    if t != (n | FIN):
        return None, rework
    starts = []
    for i in range(STRETCHES):
        p = T[i]
        while not p & FIN and p < edge[i + 1]:
            starts.append(p)
            p = end(src, n, p)
    return starts, rework


def sparse_mask(rng, frac, bits16=True):
    m = np.zeros(65536, np.uint8)
    step = 2 if bits16 else 1
    pos = np.flatnonzero(rng.random_sample(65536 // step) < frac) * step
    m[pos] = rng.randint(1, 8, size=pos.size)
    return m


CODECS = {"lz4": (oracle.lz4_encode, lz4_end, lambda s, n: 0),
          "snappy": (oracle.snappy_encode, snappy_end, snappy_first)}


@pytest.mark.parametrize("codec", ["lz4", "snappy"])
def test_joined_chain_is_the_serial_chain(codec):
    enc, end, first = CODECS[codec]
    rng = np.random.RandomState(7)
    worst = 0
    for frac in (0.001, 0.01, 0.03, 0.1):
        for _ in range(6):
            body = [int(v) for v in enc(sparse_mask(rng, frac))]
            n = len(body)
            ip0 = first(body, n)
            ref = serial_chain(end, body, n, ip0)
            assert ref is not None
            got, rework = split_chain(end, body, n, ip0, walks=4)
            assert got == ref
            if len(ref) >= 4 * STRETCHES:   # stretches of several elements
                worst = max(worst, rework)
    # four walks per stretch: the true chain meets one of them within an
    # element or two (sparser LZ4 blocks, whose stretches are shorter than a
    # sequence, re-walk more, and are right all the same)
    assert worst <= 8


@pytest.mark.parametrize("codec", ["lz4", "snappy"])
def test_one_walk_per_stretch_is_right_but_rewalks(codec):
    enc, end, first = CODECS[codec]
    rng = np.random.RandomState(8)
    body = [int(v) for v in enc(sparse_mask(rng, 0.01))]
    n = len(body)
    ip0 = first(body, n)
    got, rework = split_chain(end, body, n, ip0, walks=1)
    assert got == serial_chain(end, body, n, ip0)
    _, rework4 = split_chain(end, body, n, ip0, walks=4)
    assert rework > 8 * max(rework4, 1)   # out-of-step walks: the join walks much of the body again


@pytest.mark.parametrize("codec", ["lz4", "snappy"])
def test_corrupt_and_random_bodies_rejected_exactly_when_serially_malformed(codec):
    enc, end, first = CODECS[codec]
    rng = np.random.RandomState(9)
    base = [int(v) for v in enc(sparse_mask(rng, 0.01))]
    cases = []
    for _ in range(60):   # one byte replaced
        b = list(base)
        i = int(rng.randint(len(b)))
        b[i] = (b[i] + int(rng.randint(1, 256))) % 256
        cases.append(b)
    for _ in range(10):   # cut short or extended
        k = int(rng.randint(1, 20))
        cases.append(base[:-k])
        cases.append(base + [int(v) for v in rng.randint(0, 256, size=k)])
    for _ in range(20):   # random bytes
        cases.append([int(v) for v in rng.randint(0, 256, size=int(rng.randint(2, 3000)))])
    verdicts = set()
    for b in cases:
        n = len(b)
        ip0 = first(b, n)
        if ip0 == BAD or ip0 >= n:
            continue
        ref = serial_chain(end, b, n, ip0)
        got, _ = split_chain(end, b, n, ip0, walks=4)
        assert got == ref
        verdicts.add(ref is None)
    assert verdicts == {True, False}
