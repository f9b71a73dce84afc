"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: closed-form
identities of the XOR delta algebra, brute-force numpy counts, hand-derived
LZ4 block vectors, exhaustive round trips, numpy reshapes/concatenations of
the shard layouts, and the recovery semantics (retry after any abort point,
dedup, idempotent overwrite).
"""
import itertools

import numpy as np
import pytest

import oracle
import synth
from synth import configs

from conftest import read_table
import lowbit_vectors
from streamfmt import check_structure, overwrite_records, parse

pytestmark = pytest.mark.filterwarnings("ignore")


# --------------------------------------------------------------------------
# delta algebra ("GPU-accelerated weight teleportation", Delta update algebra)
# --------------------------------------------------------------------------
def test_xor_algebra_identities():
    rng = np.random.default_rng(1)
    old = rng.integers(0, 256, 100003, dtype=np.uint8)
    new = rng.integers(0, 256, 100003, dtype=np.uint8)
    mask = oracle.xor(old, new)
    assert np.array_equal(oracle.xor(old, mask), new)          # old ^ (old ^ new) == new
    assert np.array_equal(oracle.xor(oracle.xor(old, mask), mask), old)  # XOR twice = identity
    assert np.array_equal(mask, old ^ new)
    assert not oracle.xor(old, old).any()


@pytest.mark.parametrize("bits", [16, 8, 4])
def test_count_matches_brute_force(bits):
    rng = np.random.default_rng(bits)
    m = np.zeros(4096, dtype=np.uint8)
    pos = rng.choice(m.size, 300, replace=False)
    m[pos] = rng.integers(1, 256, pos.size, dtype=np.uint8)
    if bits == 16:
        ref = int((m.view("<u2") != 0).sum())
    elif bits == 8:
        ref = int((m != 0).sum())
    else:
        ref = int(((m & 15) != 0).sum() + ((m >> 4) != 0).sum())
    assert oracle.count_changed(m, bits) == ref


def test_signed_zero_is_a_change():
    # popular write-up, shard owners: +0 and -0 compare equal as values but
    # differ in stored bits, so the change test must see them
    old = np.array([0x00, 0x00, 0x01, 0x3C], dtype=np.uint8)   # bf16 +0, bf16 0x3C01
    new = np.array([0x00, 0x80, 0x01, 0x3C], dtype=np.uint8)   # bf16 -0, unchanged
    assert np.float32(0.0) == np.float32(-0.0)
    assert oracle.count_changed(oracle.xor(old, new), 16) == 1


def test_planted_counts_equal_generator_selection():
    wl = configs.mini(1)
    o = oracle.Oracle(wl)
    olds, news = wl.host_arenas()
    _, changed = o.encode(olds, news)
    t = wl.tensors[0]
    sel = synth.count_selected(wl.params(t, 0), t.rows * t.cols)
    assert int(changed[0]) == sel > 0


# --------------------------------------------------------------------------
# LZ4 block format (blog footnote 4 names the block format)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("row", read_table("lz4_block_vectors.txt"), ids=lambda r: r[0])
def test_lz4_decoder_hand_vectors(row):
    name, blk, raw, exp = row
    out = oracle.lz4_decode(np.frombuffer(bytes.fromhex(blk), dtype=np.uint8), int(raw))
    if exp == "ERR":
        assert out is None
    else:
        assert out is not None and bytes(out) == bytes.fromhex(exp)


@pytest.mark.parametrize("row", read_table("lz4_greedy_vectors.txt"), ids=lambda r: r[0])
def test_lz4_greedy_encoder_hand_vectors(row):
    name, data, exp = row
    blk = oracle.lz4_encode(np.frombuffer(bytes.fromhex(data), dtype=np.uint8))
    assert bytes(blk) == bytes.fromhex(exp)


def parse_block(blk):
    """Independent block walker: list of (lit_len, offset, match_len) and the
    output length; asserts the format's encoder-side end-of-block rules."""
    b = bytes(blk)
    ip, op, seqs = 0, 0, []
    while True:
        tok = b[ip]; ip += 1
        ll = tok >> 4
        if ll == 15:
            while True:
                x = b[ip]; ip += 1; ll += x
                if x != 255:
                    break
        ip += ll; op += ll
        if ip == len(b):
            seqs.append((ll, 0, 0))
            return seqs, op
        off = b[ip] | (b[ip + 1] << 8); ip += 2
        ml = tok & 15
        if ml == 15:
            while True:
                x = b[ip]; ip += 1; ml += x
                if x != 255:
                    break
        ml += 4
        seqs.append((ll, off, ml))
        op += ml


def assert_conformant(blk, n):
    seqs, out_len = parse_block(blk)
    assert out_len == n
    pos = 0
    for ll, off, ml in seqs[:-1]:
        pos += ll
        assert 1 <= off <= 65535 and off <= pos and ml >= 4
        assert pos <= n - 12, "no match starts in the last 12 bytes"
        pos += ml
        assert pos <= n - 5, "the last 5 bytes are literals"
    assert seqs[-1][1] == 0 and seqs[-1][2] == 0


def test_lz4_exhaustive_small_round_trips():
    count = 0
    for n in range(0, 7):
        for tup in itertools.product((0x00, 0x01, 0xFF), repeat=n):
            d = np.array(tup, dtype=np.uint8)
            blk = oracle.lz4_encode(d)
            assert_conformant(blk, n)
            out = oracle.lz4_decode(blk, n)
            assert out is not None and np.array_equal(out, d)
            count += 1
    assert count == sum(3 ** n for n in range(7))


@pytest.mark.parametrize("density", [0.0, 0.001, 0.01, 0.1, 0.5, 1.0])
def test_lz4_random_round_trips(density):
    rng = np.random.default_rng(int(density * 1000) + 7)
    for n in list(rng.integers(0, 301, 40)) + [65536]:
        d = np.zeros(int(n), dtype=np.uint8)
        k = rng.random(int(n)) < density
        d[k] = rng.integers(1, 256, int(k.sum()), dtype=np.uint8)
        blk = oracle.lz4_encode(d)
        assert_conformant(blk, int(n))
        out = oracle.lz4_decode(blk, int(n))
        assert np.array_equal(out, d)


def test_lz4_decoder_rejects_truncations_of_valid_blocks():
    d = np.zeros(4000, dtype=np.uint8)
    d[::97] = 3
    blk = oracle.lz4_encode(d)
    for cut in range(1, blk.size):
        assert oracle.lz4_decode(blk[:cut], d.size) is None or cut == blk.size


# --------------------------------------------------------------------------
# Snappy block format (same footnote: the other byte-oriented LZ77 codec; one
# copy covers at most 64 bytes)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("row", read_table("snappy_block_vectors.txt"), ids=lambda r: r[0])
def test_snappy_decoder_hand_vectors(row):
    name, blk, raw, exp = row
    out = oracle.snappy_decode(np.frombuffer(bytes.fromhex(blk), dtype=np.uint8), int(raw))
    if exp == "ERR":
        assert out is None
    else:
        assert out is not None and bytes(out) == bytes.fromhex(exp)


def test_snappy_greedy_encoder_hand_vectors():
    enc = lambda b: bytes(oracle.snappy_encode(np.frombuffer(b, dtype=np.uint8)))
    # shorter than a 4-byte word: one literal element
    assert enc(b"xyz") == bytes([0x03, 0x08]) + b"xyz"
    # "abcd" then a 4-byte copy at offset 4: a 1-byte-offset copy (tag 0x01)
    assert enc(b"abcdabcd") == bytes([0x08, 0x0C]) + b"abcd" + bytes([0x01, 0x04])
    # 11 x 'a': literal 'a', then 10 bytes at offset 1 (tag 1 | 6 << 2)
    assert enc(b"a" * 11) == bytes([0x0B, 0x00, 0x61, 0x19, 0x01])
    # 64 KiB of zeros: preamble 80 80 04, literal 00, then the 65535-byte
    # match at offset 1 as 1023 copies of 64 (tag 2 | 63 << 2) and one of 63
    z = enc(bytes(65536))
    assert z == bytes([0x80, 0x80, 0x04, 0x00, 0x00]) + bytes([0xFE, 0x01, 0x00]) * 1023 + bytes([0xFA, 0x01, 0x00])


def walk_snappy(blk):
    """Independent element walker: (preamble, [(kind, length, offset)])."""
    b = bytes(blk)
    ip, v, shift = 0, 0, 0
    while True:
        x = b[ip]; ip += 1
        v |= (x & 127) << shift
        shift += 7
        if not x & 128:
            break
    els = []
    while ip < len(b):
        tag = b[ip]; ip += 1
        t = tag & 3
        if t == 0:
            n = (tag >> 2) + 1
            if (tag >> 2) >= 60:
                nb = (tag >> 2) - 59
                n = int.from_bytes(b[ip:ip + nb], "little") + 1
                ip += nb
            els.append(("lit", n, 0))
            ip += n
        elif t == 1:
            els.append(("copy", ((tag >> 2) & 7) + 4, ((tag >> 5) << 8) | b[ip]))
            ip += 1
        else:
            nb = 2 if t == 2 else 4
            els.append(("copy", (tag >> 2) + 1, int.from_bytes(b[ip:ip + nb], "little")))
            ip += nb
    return v, els


def test_snappy_exhaustive_small_round_trips():
    count = 0
    for n in range(0, 7):
        for tup in itertools.product((0x00, 0x01, 0xFF), repeat=n):
            d = np.array(tup, dtype=np.uint8)
            blk = oracle.snappy_encode(d)
            pre, els = walk_snappy(blk)
            assert pre == n and sum(e[1] for e in els) == n
            out = oracle.snappy_decode(blk, n)
            assert out is not None and np.array_equal(out, d)
            count += 1
    assert count == sum(3 ** n for n in range(7))


@pytest.mark.parametrize("density", [0.0, 0.001, 0.01, 0.1, 0.5, 1.0])
def test_snappy_random_round_trips(density):
    rng = np.random.default_rng(int(density * 1000) + 11)
    for n in list(rng.integers(0, 301, 40)) + [65536]:
        d = np.zeros(int(n), dtype=np.uint8)
        k = rng.random(int(n)) < density
        d[k] = rng.integers(1, 256, int(k.sum()), dtype=np.uint8)
        blk = oracle.snappy_encode(d)
        pre, els = walk_snappy(blk)
        assert pre == n and sum(e[1] for e in els) == n
        assert all(1 <= e[1] <= 64 and e[2] >= 1 for e in els if e[0] == "copy")
        out = oracle.snappy_decode(blk, int(n))
        assert np.array_equal(out, d)


def test_snappy_decoder_rejects_truncations_and_nonzero_copies_under_zsrc():
    d = np.zeros(4000, dtype=np.uint8)
    d[::97] = 3
    blk = oracle.snappy_encode(d)
    for cut in range(1, blk.size):
        assert oracle.snappy_decode(blk[:cut], d.size) is None
    e = np.zeros(200, dtype=np.uint8)
    e[10] = 7
    e[110] = 7  # the greedy encoder copies "07 00 00 .." from position 10
    blk = oracle.snappy_encode(e)
    assert oracle.snappy_decode(blk, 200) is not None
    assert oracle.snappy_decode(blk, 200, zsrc=True) is None


def test_lz4_is_smaller_than_snappy_on_zero_run_masks():
    # the pages' reading: masks are mostly long zero runs, which one LZ4 match
    # covers while Snappy needs a copy per 64 bytes.  (At a few percent of
    # non-zero bytes the runs are short and Snappy's 2-byte copies win.)
    rng = np.random.default_rng(3)
    for density in (0.00085, 0.01):
        d = np.zeros(65536, dtype=np.uint8)
        k = rng.random(65536) < density
        d[k] = rng.integers(1, 256, int(k.sum()), dtype=np.uint8)
        assert oracle.lz4_encode(d).size < oracle.snappy_encode(d).size


def test_zsrc_decoder_flag_rejects_nonzero_copies():
    d = np.zeros(200, dtype=np.uint8)
    d[10] = 7
    d[110] = 7  # a greedy encoder copies "07 00 00 .." from position 10
    blk = oracle.lz4_encode(d)
    assert oracle.lz4_decode(blk, 200) is not None
    assert oracle.lz4_decode(blk, 200, zsrc=True) is None
    z = np.zeros(200, dtype=np.uint8)
    z[0] = 9
    assert np.array_equal(oracle.lz4_decode(oracle.lz4_encode(z), 200, zsrc=True), z)


# --------------------------------------------------------------------------
# projection into canonical coordinates (paper summary, Direct Projection;
# popular write-up, canonical coordinates and fused Q/K/V)
# --------------------------------------------------------------------------
def _u16(a):
    return a.view("<u2")


def test_tp1_projection_is_identity():
    wl = configs.single(rows=40, cols=70)
    o = oracle.Oracle(wl)
    olds, _ = wl.host_arenas()
    t = wl.tensors[0]
    assert np.array_equal(o.canonical(0, 0, olds), olds[0][t.shard_offset[0]:][:t.nbytes])


def test_split_projection_equals_numpy_concatenate():
    wl = configs.mini(2)
    o = oracle.Oracle(wl)
    olds, _ = wl.host_arenas()
    seen = {0: 0, 1: 0, 2: 0}
    for k, t in enumerate(wl.tensors):
        if t.split == configs.RESIDUAL_QKV:
            continue
        rl, cl = t.local_shape(wl.tp)
        parts = []
        for r in t.holders(wl.tp):
            off = t.shard_offset[r]
            parts.append(_u16(olds[r][off:off + rl * cl * 2]).reshape(rl, cl))
        if t.split == configs.SPLIT_ROWS:
            ref = np.concatenate(parts, axis=0)
        elif t.split == configs.SPLIT_COLS:
            ref = np.concatenate(parts, axis=1)
        else:
            ref = parts[0]
        assert np.array_equal(_u16(o.canonical(k, 0, olds)).reshape(t.rows, t.cols), ref), t.name
        seen[t.split] += 1
    assert all(seen.values())


def test_tp16_projection_equals_numpy_and_round_trips():
    # the largest shard count: every split kind against numpy stacking of the
    # 16 shards (fused QKV: one kv group per shard), then a whole refit
    wl = configs.tp16()
    o = oracle.Oracle(wl)
    olds, news = wl.host_arenas()
    for k, t in enumerate(wl.tensors):
        eb = t.elem_bits // 8
        rl, cl = t.local_shape(wl.tp)
        parts = [olds[r][t.shard_offset[r]:t.shard_offset[r] + rl * cl * eb].reshape(rl, cl * eb)
                 for r in t.holders(wl.tp)]
        if t.split == configs.RESIDUAL_QKV:
            qpg, D = t.q_heads // t.kv_heads, t.head_dim
            g = np.concatenate(parts, axis=0).reshape(t.kv_heads, qpg + 2, D, cl * eb)
            refs = [g[:, :qpg].reshape(-1, cl * eb), g[:, qpg].reshape(-1, cl * eb), g[:, qpg + 1].reshape(-1, cl * eb)]
        elif t.split == configs.SPLIT_COLS:
            refs = [np.concatenate(parts, axis=1)]
        else:
            refs = [np.concatenate(parts, axis=0)]
        assert len(parts) == (1 if t.split == configs.REPLICATED else 16)
        for sub, ref in enumerate(refs):
            assert np.array_equal(o.canonical(k, sub, olds), ref.reshape(-1)), (t.name, sub)
    tgt, exp = o.receiver_dense(olds), o.receiver_dense(news)
    st = o.state(0)
    pl, ch = o.encode(olds, news)
    assert int(ch.sum()) > 0
    assert o.apply(st, pl, tgt) == oracle.OK and st.version == 1
    assert np.array_equal(tgt, exp)


def test_qkv_deinterleave_equals_numpy_reshape():
    wl = configs.mini(3)
    o = oracle.Oracle(wl)
    olds, _ = wl.host_arenas()
    t = [x for x in wl.tensors if x.split == configs.RESIDUAL_QKV][0]
    k = wl.tensors.index(t)
    G, D, H, tp = t.kv_heads, t.head_dim, t.cols, wl.tp
    qpg = t.q_heads // G
    fused = []
    for r in range(tp):
        off = t.shard_offset[r]
        n = (G // tp) * (qpg + 2) * D * H
        fused.append(_u16(olds[r][off:off + 2 * n]).reshape(G // tp, qpg + 2, D, H))
    allg = np.concatenate(fused, axis=0)              # [G, qpg + 2, D, H]
    q_ref = allg[:, :qpg].reshape(G * qpg * D, H)
    k_ref = allg[:, qpg].reshape(G * D, H)
    v_ref = allg[:, qpg + 1].reshape(G * D, H)
    for sub, ref in enumerate((q_ref, k_ref, v_ref)):
        assert np.array_equal(_u16(o.canonical(k, sub, olds)).reshape(ref.shape), ref)


@pytest.mark.parametrize("split", [configs.SPLIT_ROWS, configs.SPLIT_COLS, configs.RESIDUAL_QKV])
def test_projection_is_a_bijection(split):
    # every shard element lands in exactly one canonical place: fill the shard
    # arenas with distinct 16-bit ids and look for each one
    if split == configs.RESIDUAL_QKV:
        t = configs.Tensor("x", elem_bits=16, rows=(4 + 2 * 2) * 8, cols=12, split=split,
                           value_kind=0, rule=0, frac=0, q_heads=4, kv_heads=2, head_dim=8)
    else:
        t = configs.Tensor("x", elem_bits=16, rows=24, cols=36, split=split, value_kind=0, rule=0,
                           frac=0)
    wl = configs.Workload("bij", 1, 2, [t]).layout()
    o = oracle.Oracle(wl)
    shards = []
    base = 0
    for r in range(2):
        a = np.zeros(max(wl.shard_bytes[r], 16), dtype=np.uint8)
        n = t.local_bytes(2) // 2
        a[t.shard_offset[r]:t.shard_offset[r] + 2 * n] = np.arange(base, base + n, dtype="<u2").view(np.uint8)
        base += n
        shards.append(a)
    subs = 3 if split == configs.RESIDUAL_QKV else 1
    got = np.concatenate([_u16(o.canonical(0, s, shards)) for s in range(subs)])
    assert np.array_equal(np.sort(got), np.arange(base))


def test_rowgroup_receiver_layout_equals_numpy():
    # blog, Working with low-precision RL: gate and up rows paired in groups of 64
    wl = configs.mini(5)
    o = oracle.Oracle(wl)
    olds, _ = wl.host_arenas()
    tgt = o.receiver_dense(olds)
    gate = [t for t in wl.tensors if t.name.endswith(".gate")][0]
    up = [t for t in wl.tensors if t.recv_offset == gate.recv_offset and t.recv_slot == 1][0]
    rb = gate.cols // 2
    g = np.frombuffer(olds[0][gate.shard_offset[0]:gate.shard_offset[0] + gate.nbytes], np.uint8).reshape(gate.rows, rb)
    u = np.frombuffer(olds[0][up.shard_offset[0]:up.shard_offset[0] + up.nbytes], np.uint8).reshape(up.rows, rb)
    grp = gate.recv_group
    ref = np.concatenate([g.reshape(-1, grp, rb), u.reshape(-1, grp, rb)], axis=1).reshape(-1, rb)
    got = tgt[gate.recv_offset:gate.recv_offset + 2 * gate.nbytes].reshape(-1, rb)
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------------
# stream, apply, dedup, retry (paper summary, Recoverable in-place apply;
# popular write-up, dedup by unique IDs and overwrite-only retry)
# --------------------------------------------------------------------------
def _setup(n, **kw):
    wl = configs.mini(n)
    o = oracle.Oracle(wl, **kw)
    olds, news = wl.host_arenas()
    return wl, o, olds, news, o.receiver_dense(olds), o.receiver_dense(news)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_refit_reaches_new_bit_exact(n):
    wl, o, olds, news, tgt, exp = _setup(n)
    st = o.state(7)
    total_changed = 0
    for w in range(o.n_windows):
        pl, ch = o.encode(olds, news, window=w, base_version=7, target_version=8)
        hdr, frames = check_structure(pl)
        assert hdr["plan_hash"] == o.plan_hash and hdr["window"] == w
        assert (hdr["base_version"], hdr["target_version"]) == (7, 8)
        assert sum(f["changed"] for f in frames) == int(ch.sum())
        total_changed += int(ch.sum())
        rc = o.apply(st, pl, tgt)
        assert rc == oracle.OK
        assert st.version == (8 if w == o.n_windows - 1 else 7)
    assert np.array_equal(tgt, exp)
    assert total_changed > 0


def test_frame_kinds_follow_the_hybrid_rule():
    wl, o, olds, news, tgt, exp = _setup(3)
    pl, _ = o.encode(olds, news)
    _, frames = check_structure(pl)
    kinds = {}
    for f in frames:
        d, sub, _, _ = o.chunk_info(f["chunk"])
        residual = wl.tensors[d].split == configs.RESIDUAL_QKV
        kinds.setdefault(residual, set()).add(f["kind"])
    assert kinds[True] <= {3, 4} and kinds[False] <= {1, 2}


def test_overwrite_records_hold_exactly_the_changed_units():
    wl, o, olds, news, tgt, exp = _setup(1)
    pl, _ = o.encode(olds, news, mode=oracle.MODE_OVERWRITE_ONLY)
    _, frames = check_structure(pl)
    t = wl.tensors[0]
    cold = o.canonical(0, 0, olds).view("<u2")
    cnew = o.canonical(0, 0, news).view("<u2")
    for f in frames:
        assert f["kind"] == 3
        offs, vals = overwrite_records(f)
        base = (f["chunk"]) * 32768
        ref = np.flatnonzero(cold[base:base + f["raw_len"] // 2] != cnew[base:base + f["raw_len"] // 2])
        assert np.array_equal(offs, ref)
        assert np.array_equal(vals.view("<u2").ravel(), cnew[base + ref])


def test_no_change_sends_header_only():
    wl = configs.mini(2)
    o = oracle.Oracle(wl)
    olds, _ = wl.host_arenas()
    pl, ch = o.encode(olds, olds)
    hdr, frames = check_structure(pl)
    assert pl.size == 64 and hdr["n_frames"] == 0 and not ch.any()
    tgt = o.receiver_dense(olds)
    before = tgt.copy()
    st = o.state(0)
    assert o.apply(st, pl, tgt) == oracle.OK and np.array_equal(tgt, before) and st.version == 1


def test_signed_zero_travels_through_the_stream():
    t = configs.Tensor("z", elem_bits=16, rows=1, cols=64, split=configs.REPLICATED, value_kind=0,
                       rule=0, frac=0)
    wl = configs.Workload("z", 1, 1, [t]).layout()
    o = oracle.Oracle(wl)
    old = np.zeros(128, dtype=np.uint8)
    new = old.copy()
    new[41] = 0x80     # element 20: +0 -> -0
    pl, ch = o.encode([old], [new])
    assert int(ch[0]) == 1
    tgt = old.copy()
    assert o.apply(o.state(0), pl, tgt) == oracle.OK and np.array_equal(tgt, new)


def test_version_and_hash_checks_reject_without_mutation():
    wl, o, olds, news, tgt, exp = _setup(1)
    pl, _ = o.encode(olds, news, base_version=3, target_version=4)
    before = tgt.copy()
    assert o.apply(o.state(2), pl, tgt) == oracle.E_VERSION
    bad = pl.copy()
    bad[8] ^= 1   # plan hash
    assert o.apply(o.state(3), bad, tgt) == oracle.E_INVALID
    assert np.array_equal(tgt, before)
    st = o.state(3)
    assert o.apply(st, pl, tgt) == oracle.OK and st.version == 4
    assert o.apply(st, pl, tgt) == oracle.E_VERSION     # the same delta never lands twice
    assert np.array_equal(tgt, exp)


def _with_index(pl, order):
    """Stream whose index lists the given frame ordinals (duplicates allowed)."""
    hdr, frames, idx_off = parse(pl)
    offs = np.array([frames[i]["offset"] for i in order], dtype="<u8")
    out = np.concatenate([pl[:idx_off], offs.view(np.uint8)])
    out[48:56] = np.array([len(order)], dtype="<u8").view(np.uint8)
    out[56:64] = np.array([out.size], dtype="<u8").view(np.uint8)
    return out


def test_duplicate_frames_are_applied_once():
    wl, o, olds, news, tgt, exp = _setup(2)
    pl, _ = o.encode(olds, news)
    nf = parse(pl)[0]["n_frames"]
    dup = _with_index(pl, list(range(nf)) + list(range(nf)) + [0, 0])
    st = o.state(0)
    assert o.apply(st, dup, tgt) == oracle.OK and np.array_equal(tgt, exp) and st.version == 1


def test_negative_control_without_dedup_breaks():
    wl, o, olds, news, tgt, exp = _setup(2)
    pl, _ = o.encode(olds, news)
    nf = parse(pl)[0]["n_frames"]
    dup = _with_index(pl, list(range(nf)) + [0])
    o.apply(o.state(0), dup, tgt, dedup=False)
    assert not np.array_equal(tgt, exp)


def test_xor_payload_applied_twice_without_dedup_is_identity():
    wl, o, olds, news, tgt, exp = _setup(1)
    pl, _ = o.encode(olds, news)
    before = tgt.copy()
    o.apply(o.state(0), pl, tgt, dedup=False)
    assert np.array_equal(tgt, exp)
    o.apply(o.state(0), pl, tgt, dedup=False)
    assert np.array_equal(tgt, before)


def test_overwrite_is_idempotent():
    wl, o, olds, news, tgt, exp = _setup(3)
    pl, _ = o.encode(olds, news, mode=oracle.MODE_OVERWRITE_ONLY)
    for _ in range(3):
        st = o.state(0)
        assert o.apply(st, pl, tgt, retry_only=True) == oracle.OK
        assert np.array_equal(tgt, exp)


def test_retry_only_refuses_xor_streams():
    wl, o, olds, news, tgt, exp = _setup(1)
    pl, _ = o.encode(olds, news)
    before = tgt.copy()
    assert o.apply(o.state(0), pl, tgt, retry_only=True) == oracle.E_INVALID
    assert np.array_equal(tgt, before)


@pytest.mark.parametrize("n", [1, 3])
def test_abort_at_every_frame_then_overwrite_retry(n):
    wl, o, olds, news, tgt0, exp = _setup(n)
    pl, _ = o.encode(olds, news)
    retry, _ = o.encode(olds, news, mode=oracle.MODE_OVERWRITE_ONLY)
    nf = parse(pl)[0]["n_frames"]
    for k in range(nf):
        for split in (0, 777, 65536):
            tgt = tgt0.copy()
            st = o.state(0)
            rc = o.apply(st, pl, tgt, abort_at=k, split=split)
            assert rc == oracle.E_ABORTED and st.version == 0
            if split < 65536 and k < nf - 1:
                assert not np.array_equal(tgt, exp), "the weights are mixed after an abort"
            # a re-sent XOR stream must not corrupt claimed chunks
            rc = o.apply(st, pl, tgt)
            assert rc in (oracle.OK, oracle.E_INCOMPLETE)
            if rc == oracle.OK:
                # the cut frame was an (idempotent) overwrite: the re-send completes
                assert st.version == 1 and np.array_equal(tgt, exp)
                continue
            rc = o.apply(st, retry, tgt, retry_only=True)
            assert rc == oracle.OK and st.version == 1
            assert np.array_equal(tgt, exp)


# ---- overwrite apply on 8- and 4-bit units, through the row-group remap ----
# (popular write-up, XOR or overwrite: both reach the new bits exactly;
# blog, Working with low-precision RL: packed FP4 with fp8 scales, gate/up
# rows paired in groups)
@pytest.mark.parametrize("make", [lambda: configs.mini(5), configs.tp16, configs.lowbit_pair],
                         ids=["mini-moe", "tp16", "lowbit-pair"])
def test_overwrite_only_stream_reaches_new_on_low_bit_layouts(make):
    wl = make()
    o = oracle.Oracle(wl)
    olds, news = wl.host_arenas()
    tgt, exp = o.receiver_dense(olds), o.receiver_dense(news)
    assert not np.array_equal(tgt, exp)
    st = o.state(0)
    kinds = set()
    for w in range(o.n_windows):
        pl, ch = o.encode(olds, news, window=w, mode=oracle.MODE_OVERWRITE_ONLY)
        _, frames = check_structure(pl)
        kinds |= {(f["kind"], f["elem_bits"]) for f in frames}
        assert o.apply(st, pl, tgt, retry_only=True) == oracle.OK
    assert np.array_equal(tgt, exp) and st.version == 1
    assert {b for _, b in kinds} >= ({4, 8} if make is not configs.tp16 else {8, 16})


def test_abort_at_every_frame_then_overwrite_retry_low_bit_windows():
    wl, o, olds, news, tgt0, exp = _setup(5)
    for w in range(o.n_windows):
        pl, _ = o.encode(olds, news, window=w)
        retry, _ = o.encode(olds, news, window=w, mode=oracle.MODE_OVERWRITE_ONLY)
        nf = parse(pl)[0]["n_frames"]
        for k in range(0, nf, max(1, nf // 7)):
            for split in (0, 301, 65536):
                tgt = tgt0.copy()
                st = o.state(0)
                # the other windows applied cleanly, this one aborted at frame k
                for v in range(o.n_windows):
                    if v != w:
                        assert o.apply(st, o.encode(olds, news, window=v)[0], tgt) == oracle.OK
                assert o.apply(st, pl, tgt, abort_at=k, split=split) == oracle.E_ABORTED
                assert st.version == 0
                assert o.apply(st, retry, tgt, retry_only=True) == oracle.OK
                assert st.version == 1 and np.array_equal(tgt, exp)


def _lowbit_apply(pl):
    wl = configs.lowbit_pair()
    o = oracle.Oracle(wl)
    tgt = np.zeros(wl.recv_bytes, dtype=np.uint8)
    assert o.apply(o.state(0), pl, tgt, retry_only=True) == oracle.OK
    again = tgt.copy()
    assert o.apply(o.state(0), pl, again, retry_only=True) == oracle.OK
    assert np.array_equal(again, tgt), "overwrite is idempotent"
    return tgt


@pytest.mark.parametrize("make", [lowbit_vectors.dense_gate_stream, lowbit_vectors.record_stream],
                         ids=["dense-e2m1", "records-e2m1-e4m3"])
def test_overwrite_through_rowgroup_remap_hand_vectors(make):
    pl, want = make(oracle.Oracle(configs.lowbit_pair()).plan_hash)
    assert np.array_equal(_lowbit_apply(pl), want)


def test_corrupt_frame_is_reported_and_retry_recovers():
    wl, o, olds, news, tgt, exp = _setup(1)
    pl, _ = o.encode(olds, news)
    hdr, frames, _ = parse(pl)
    bad = pl.copy()
    f = [f for f in frames if f["kind"] == 1][0]
    bad[f["offset"] + 32:f["offset"] + 32 + 8] = 0xFF
    st = o.state(0)
    assert o.apply(st, bad, tgt) == oracle.E_CORRUPT and st.version == 0
    retry, _ = o.encode(olds, news, mode=oracle.MODE_OVERWRITE_ONLY)
    assert o.apply(st, retry, tgt, retry_only=True) == oracle.OK
    assert np.array_equal(tgt, exp)


def test_windows_partition_at_tensor_boundaries():
    wl = configs.mini(5)
    o = oracle.Oracle(wl)
    assert o.n_windows > 1
    starts = [o.window_range(w)[0] for w in range(o.n_windows)]
    sizes = []
    for w in range(o.n_windows):
        b, c = o.window_range(w)
        tot = sum(o.chunk_info(k)[3] for k in range(b, b + c))
        sizes.append(tot)
        assert tot <= wl.window_bytes
        d, sub, off, _ = o.chunk_info(b)
        assert off == 0 and sub == 0, "windows start on a tensor boundary"
    assert sum(sizes) == wl.canonical_bytes
    assert starts == sorted(starts)


def test_tensor_larger_than_a_window_is_cut_at_chunks():
    # windows pack whole tensors while they fit; a larger tensor is cut at
    # 64 KiB chunk boundaries (700 KiB holds 10 chunks): by hand, chunks
    # [0, 10), [10, 20), [20, 30) of the 32-chunk tensor, then its last two
    # with the 2 chunks (64 + 36 KiB) of the 100 KiB tensor after it
    wl = configs.oversized_window()
    o = oracle.Oracle(wl)
    assert o.n_windows == 4
    assert [tuple(o.window_range(w)) for w in range(4)] == [(0, 10), (10, 10), (20, 10), (30, 4)]
    assert [o.chunk_info(k)[0] for k in range(30, 34)] == [0, 0, 1, 1]
    assert o.chunk_info(33)[3] == 100 * 1024 - 65536
    olds, news = wl.host_arenas()
    tgt, exp = o.receiver_dense(olds), o.receiver_dense(news)
    st = o.state(0)
    for i, w in enumerate([2, 0, 3, 1]):   # any window order; commit after the last
        pl, _ = o.encode(olds, news, window=w)
        assert check_structure(pl)[0]["window"] == w
        assert o.apply(st, pl, tgt) == oracle.OK
        assert st.version == (1 if i == 3 else 0)
    assert np.array_equal(tgt, exp)


def test_plan_hash_depends_only_on_canonical_description():
    a = configs.mini(2)
    b = configs.mini(2)
    for t in b.tensors:      # a different trainer arena layout
        t.shard_offset = [x + 4096 for x in t.shard_offset]
        t.recv_offset += 512
    assert oracle.Oracle(a).plan_hash == oracle.Oracle(b).plan_hash
    c = configs.dense(hidden=96, layers=2, ffn=320, vocab=1002)
    assert oracle.Oracle(c).plan_hash != oracle.Oracle(a).plan_hash


# The plan hash is FNV-1a 64 (Fowler, Noll and Vo's published definition:
# offset basis 0xcbf29ce484222325, prime 0x100000001b3, xor then multiply per
# byte); pinned to the reference values of that definition's test suite.
def test_fnv1a64_reference_values():
    assert oracle.fnv1a64(b"") == 0xCBF29CE484222325
    assert oracle.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert oracle.fnv1a64(b"foobar") == 0x85944171F73967E8
    # xor-then-multiply order: FNV-1 (multiply first) gives another value
    assert oracle.fnv1a64(b"a") != 0xAF63BD4C8601B7BE
