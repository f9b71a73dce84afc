"""Every route a frame body can take through the encoder, on one crafted
workload: bodies that fit the per-chunk slot, LZ4 bodies that outgrow it
(written by the second, restream pass), LZ4 chunks whose literal runs are
longer than the event ring (the shared-memory pass), raw and dense frames,
overwrite records past the slot, on 16-bit, 8-bit, unaligned and fused-QKV
chunks, in both encode modes.  The CPU test pins what the oracle makes of
the workload, so the GPU test is known to reach each route."""
import numpy as np
import pytest

import oracle
import synth
from synth import configs
from parity import assert_same_frames
from streamfmt import K_OVERWRITE, K_OVERWRITE_DENSE, K_XOR_LZ4, K_XOR_RAW, check_structure, parse

CHUNK = 65536
SLOT_BODY = 6144 - 32   # frame body bytes the encoder's per-chunk slot holds


def crafted():
    """Workload (TP 2) and its old/new shard arenas.  Per chunk of tensor a
    (bf16, replicated): 5 % of units changed, a 3000-byte run of changed
    bytes, random, three changes, 30 %, then unchanged.  Tensor b (8-bit):
    10 %, a 2000-byte run, one change.  Tensor c: bf16 split by columns into
    666-byte pieces (not 16-byte aligned), 5 %.  Tensor d: fused QKV
    residual, 10 % (more overwrite records than a slot holds)."""
    ts = [
        configs.Tensor("a", rows=64, cols=4096, split=configs.REPLICATED, rule=synth.RULE_PM4, frac=0.0,
                       **configs.BF),
        configs.Tensor("b", elem_bits=8, rows=256, cols=1024, split=configs.REPLICATED,
                       value_kind=synth.VAL_E4M3_SCALE, rule=synth.RULE_BPM4, frac=0.0),
        configs.Tensor("c", rows=100, cols=666, split=configs.SPLIT_COLS, rule=synth.RULE_PM4, frac=0.0,
                       **configs.BF),
        configs.Tensor("d", rows=(4 + 2 * 2) * 32, cols=512, split=configs.RESIDUAL_QKV, rule=synth.RULE_PM4,
                       frac=0.0, q_heads=4, kv_heads=2, head_dim=32, **configs.BF),
    ]
    wl = configs.Workload("routes", 0xDC5EED77, 2, ts).layout()
    olds, news = wl.host_arenas()
    rng = np.random.RandomState(77)

    def units(r, t, lo, hi, frac, ub):
        """Flip a random nonzero value into the low byte of `frac` of the
        units of shard r's bytes [lo, hi) of tensor t."""
        base = t.shard_offset[r]
        n = (hi - lo) // ub
        pick = np.flatnonzero(rng.random_sample(n) < frac)
        at = base + lo + pick * ub
        news[r][at] ^= rng.randint(1, 256, size=pick.size).astype(np.uint8)

    a, b, c, d = ts
    units(0, a, 0, CHUNK, 0.05, 2)
    o = a.shard_offset[0] + CHUNK + 100
    news[0][o:o + 3000] ^= 0xFF
    o = a.shard_offset[0] + 2 * CHUNK
    news[0][o:o + CHUNK] = rng.randint(0, 256, size=CHUNK).astype(np.uint8)
    for x in (5, 777, 40001):
        news[0][a.shard_offset[0] + 3 * CHUNK + 2 * x] ^= 0x01
    units(0, a, 4 * CHUNK, 5 * CHUNK, 0.3, 2)
    units(0, b, 0, CHUNK, 0.1, 1)
    o = b.shard_offset[0] + CHUNK
    news[0][o:o + 2000] ^= 0x5A
    news[0][b.shard_offset[0] + 2 * CHUNK + 12345] ^= 0x10
    for r in (0, 1):
        units(r, c, 0, c.local_bytes(2), 0.05, 2)
        units(r, d, 0, d.local_bytes(2), 0.1, 2)
    return wl, olds, news


def _frames(payload):
    _, frames, _ = parse(payload)
    return {f["chunk"]: f for f in frames}


def test_crafted_workload_reaches_every_route():
    wl, olds, news = crafted()
    orc = oracle.Oracle(wl)
    o, _ = orc.encode(olds, news)
    f = _frames(o)
    a0 = 0   # tensor a's chunks come first in canonical order
    assert f[a0]["kind"] == K_XOR_LZ4 and len(f[a0]["body"]) > SLOT_BODY
    assert f[a0 + 1]["kind"] == K_XOR_LZ4 and len(f[a0 + 1]["body"]) < CHUNK
    m = oracle.lz4_decode(f[a0 + 1]["body"], f[a0 + 1]["raw_len"])
    assert np.count_nonzero(m) == 3000                  # one literal run of 3000 events
    assert f[a0 + 2]["kind"] == K_XOR_RAW
    assert f[a0 + 3]["kind"] == K_XOR_LZ4 and len(f[a0 + 3]["body"]) < SLOT_BODY
    assert f[a0 + 4]["kind"] == K_XOR_LZ4 and len(f[a0 + 4]["body"]) > SLOT_BODY
    b0 = 8
    assert f[b0]["kind"] == K_XOR_LZ4 and len(f[b0]["body"]) > SLOT_BODY
    assert f[b0 + 1]["kind"] == K_XOR_LZ4
    kinds = [f[k]["kind"] for k in f]
    assert kinds.count(K_OVERWRITE) >= 4
    assert max(len(f[k]["body"]) for k in f if f[k]["kind"] == K_OVERWRITE) > SLOT_BODY
    ow, _ = orc.encode(olds, news, mode=oracle.MODE_OVERWRITE_ONLY)
    fo = _frames(ow)
    assert fo[a0 + 2]["kind"] == K_OVERWRITE_DENSE
    assert fo[a0]["kind"] == K_OVERWRITE and len(fo[a0]["body"]) > SLOT_BODY


# overflow heap: the default (bodies past their slot move to the heap), none
# (the write pass derives them again from old and new), and 16 KiB, which
# runs out part way through the window (both routes in one encode)
@pytest.mark.gpu
@pytest.mark.parametrize("overflow", ["heap", "none", "16kib"])
@pytest.mark.parametrize("encoder", ["wide", "deep", "cta"])
@pytest.mark.parametrize("mode", ["hybrid", "overwrite"])
def test_every_route_matches_oracle(mode, encoder, overflow):
    torch = pytest.importorskip("torch")
    import bit_exact_xor_gb300 as dcr
    from wl import descs_of, to_device

    wl, olds, news = crafted()
    orc = oracle.Oracle(wl)
    plan = dcr.Plan(descs_of(wl), window_bytes=wl.window_bytes,
                    encoder={"wide": dcr.ENCODER_WIDE, "deep": dcr.ENCODER_DEEP, "cta": dcr.ENCODER_CTA}[encoder],
                    # every apply kernel on every route: warp per frame after the wide encoder,
                    # CTA per frame after the deep one, thread per ZSRC frame after the CTA one
                    apply={"wide": dcr.APPLY_WARP, "deep": dcr.APPLY_CTA, "cta": dcr.APPLY_LANE}[encoder],
                    overflow_kib={"heap": 0, "none": dcr.NO_OVERFLOW, "16kib": 16}[overflow])
    assert plan.info.plan_hash == orc.plan_hash
    d_old, d_new = to_device(olds), to_device(news)
    dm = dcr.MODE_HYBRID if mode == "hybrid" else dcr.MODE_OVERWRITE_ONLY
    om = oracle.MODE_HYBRID if mode == "hybrid" else oracle.MODE_OVERWRITE_ONLY
    pl = torch.zeros(plan.window(0).payload_bound, dtype=torch.uint8, device="cuda")
    for _ in range(2):   # the second call reuses the scratch of the first
        rc, size, counts = dcr.encode(plan, d_old, d_new, pl, mode=dm)
        assert rc == dcr.OK, dcr.last_error()
        g = pl[:size].cpu().numpy()
        o, oc = orc.encode(olds, news, mode=om)
        check_structure(g)
        assert counts == [int(x) for x in oc]
        assert_same_frames(g, o)
        assert g.size <= 1.15 * o.size + 64
    exp = orc.receiver_dense(news)
    t = torch.zeros(max(plan.info.recv_bytes, wl.recv_bytes, 16), dtype=torch.uint8, device="cuda")
    dcr.check(dcr.dense_refit(plan, d_old, t))
    st = dcr.RecvState(plan, 0)
    if mode == "hybrid":
        rc, _ = dcr.apply(plan, st, pl, size, t)
    else:
        rc, _ = dcr.apply_retry(plan, st, pl, size, t)
    assert rc == dcr.OK, dcr.last_error()
    assert np.array_equal(t.cpu().numpy()[:exp.size], exp)
