"""The Snappy variant of the mask codec (plan option codec = Snappy, frame
kind 5) against the CPU oracle's Snappy encoder and decoder, through the C
ABI: same masks and counts, each side's stream applied by the other, every
encoder route, and a lying ZSRC flag rejected.  Payload: within 1.15x of the
oracle's greedy Snappy on sparse masks (<= 1 % change).  Denser masks are
held to bit-exactness only, with 1.25x at 3 %: the greedy matcher also
copies repeated non-zero patterns ("00 00 00 03"), which Snappy's 2-byte
copies make cheap, while the GPU parse copies zero bytes only (its frames
carry the ZSRC promise)."""
import numpy as np
import pytest

import oracle
from synth import configs
from parity import assert_same_frames, frames_by_chunk
from streamfmt import K_XOR_SNAPPY, check_structure

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_exact_xor_gb300 as dcr  # noqa: E402
from wl import descs_of, to_device  # noqa: E402
from test_gpu_random import random_workload  # noqa: E402
from test_gpu_routes import crafted  # noqa: E402


def _check(wl, olds, news, encoder=dcr.ENCODER_AUTO, size_bar=1.15):
    orc = oracle.Oracle(wl)
    # the thread-per-frame apply after the CTA encoder, the default after the others
    plan = dcr.Plan(descs_of(wl), window_bytes=wl.window_bytes, encoder=encoder, codec=dcr.CODEC_SNAPPY,
                    apply=dcr.APPLY_LANE if encoder == dcr.ENCODER_CTA else dcr.APPLY_AUTO)
    d_old, d_new = to_device(olds), to_device(news)
    exp = orc.receiver_dense(news)
    t = torch.zeros(max(plan.info.recv_bytes, wl.recv_bytes, 16), dtype=torch.uint8, device="cuda")
    dcr.check(dcr.dense_refit(plan, d_old, t))
    t2 = t.clone()
    st, st2 = dcr.RecvState(plan, 0), dcr.RecvState(plan, 0)
    ost, otgt = orc.state(0), orc.receiver_dense(olds)
    kinds = set()
    for w in range(plan.n_windows):
        pl = torch.zeros(plan.window(w).payload_bound, dtype=torch.uint8, device="cuda")
        rc, size, counts = dcr.encode(plan, d_old, d_new, pl, window=w)
        assert rc == dcr.OK, dcr.last_error()
        g = pl[:size].cpu().numpy()
        o, oc = orc.encode(olds, news, window=w, codec=oracle.CODEC_SNAPPY)
        check_structure(g)
        assert counts == [int(x) for x in oc]
        assert_same_frames(g, o)
        if size_bar:
            assert g.size <= size_bar * o.size + 64, (g.size, o.size)
        kinds |= {f["kind"] for f in frames_by_chunk(g)[1].values()}
        rc, _ = dcr.apply(plan, st, pl, size, t)                       # GPU stream on the GPU
        assert rc == dcr.OK, dcr.last_error()
        rc, _ = dcr.apply(plan, st2, torch.from_numpy(o).cuda(), o.size, t2)   # oracle stream on the GPU
        assert rc == dcr.OK, dcr.last_error()
        assert orc.apply(ost, g, otgt) == oracle.OK                    # GPU stream on the oracle
    assert np.array_equal(t.cpu().numpy()[:exp.size], exp)
    assert np.array_equal(t2.cpu().numpy()[:exp.size], exp)
    assert np.array_equal(otgt, exp)
    assert st.version == 1 and st2.version == 1
    return kinds


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_snappy_twins(n):
    wl = configs.mini(n)
    olds, news = wl.host_arenas()
    dense = max(t.frac for t in wl.tensors) > 0.011
    kinds = _check(wl, olds, news, size_bar=1.25 if dense else 1.15)
    assert K_XOR_SNAPPY in kinds


@pytest.mark.parametrize("seed", [0, 3, 6, 9, 13, 17])
def test_snappy_random_workloads(seed):
    wl = random_workload(seed)
    olds, news = wl.host_arenas()
    sparse = max(t.frac for t in wl.tensors) <= 0.011
    _check(wl, olds, news, size_bar=1.15 if sparse else None)


@pytest.mark.parametrize("encoder", [dcr.ENCODER_WIDE, dcr.ENCODER_DEEP, dcr.ENCODER_CTA])
def test_snappy_every_route(encoder):
    wl, olds, news = crafted()
    _check(wl, olds, news, encoder=encoder, size_bar=None)   # crafted dense chunks


def test_snappy_lying_zsrc_flag_is_rejected():
    # a chunk whose mask repeats "07 00 00 ..": the greedy Snappy encoder
    # copies non-zero bytes; with the ZSRC flag set on that frame the GPU must
    # reject it and leave the chunk as it was
    t0 = configs.Tensor("z", elem_bits=8, rows=1, cols=65536, split=configs.REPLICATED, value_kind=1,
                        rule=0, frac=0)
    wl = configs.Workload("zs", 1, 1, [t0]).layout()
    old = np.zeros(wl.shard_bytes[0], dtype=np.uint8)
    new = old.copy()
    new[10] = 7
    new[5000] = 7
    new[5003] = 9
    new[9000] = 7
    new[9003] = 9
    orc = oracle.Oracle(wl)
    o, _ = orc.encode([old], [new], codec=oracle.CODEC_SNAPPY)
    hdr, frames = frames_by_chunk(o)
    f = frames[0]
    assert f["kind"] == K_XOR_SNAPPY
    assert oracle.snappy_decode(f["body"], f["raw_len"], zsrc=True) is None   # it does copy non-zero bytes
    lied = o.copy()
    lied[f["offset"] + 6] |= 1   # frame flags: ZSRC
    plan = dcr.Plan(descs_of(wl), codec=dcr.CODEC_SNAPPY)
    t = to_device([old])[0]
    rc, _ = dcr.apply(plan, dcr.RecvState(plan, 0), torch.from_numpy(lied).cuda(), lied.size, t)
    assert rc == dcr.ERR_CORRUPT
    assert not t.cpu().numpy().any()
    # the honest frame applies
    rc, _ = dcr.apply(plan, dcr.RecvState(plan, 0), torch.from_numpy(o).cuda(), o.size, t)
    assert rc == dcr.OK and np.array_equal(t.cpu().numpy(), new)
