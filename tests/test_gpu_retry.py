"""Overwrite-only retry streams built from the XOR stream and new, without
old (paper summary, Recoverable in-place apply; popular write-up, in-place
apply without a backup copy): byte for byte the stream dcr_encode writes in
overwrite-only mode, equal to the oracle's, and a retry after an abort
reaches new.  Inputs cover every frame kind: LZ4 and Snappy masks (ZSRC
from the GPU encoder, general blocks from the oracle), raw masks, residual
overwrite records, dense chunks, records past the 6 KiB slot."""
import numpy as np
import pytest

import oracle
from synth import configs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_exact_xor_gb300 as dcr  # noqa: E402
from wl import descs_of, to_device  # noqa: E402

CASES = [("mini", 1, 0), ("mini", 2, 0), ("mini", 3, 0), ("mini", 4, 0), ("mini", 5, 0), ("mini", 3, 1),
         ("tp16", 0, 0), ("routes", 0, 0), ("dense30", 0, 0)]


def _workload(kind, n):
    if kind == "mini":
        wl = configs.mini(n)
        return wl, wl.host_arenas()
    if kind == "tp16":
        wl = configs.tp16()
        return wl, wl.host_arenas()
    if kind == "routes":
        from test_gpu_routes import crafted
        wl, olds, news = crafted()
        return wl, (olds, news)
    wl = configs.mini(4)   # 30 % of the values changed: dense chunks and records past the slot
    return wl, wl.host_arenas(frac_override=0.3)


@pytest.mark.parametrize("kind,n,codec", CASES, ids=["%s%d-c%d" % c for c in CASES])
def test_retry_from_xor_stream_equals_overwrite_only_encode(kind, n, codec):
    wl, (olds, news) = _workload(kind, n)
    orc = oracle.Oracle(wl)
    plan = dcr.Plan(descs_of(wl), window_bytes=wl.window_bytes, codec=codec)
    d_old, d_new = to_device(olds), to_device(news)
    tgt = torch.zeros(max(plan.info.recv_bytes, wl.recv_bytes, 16), dtype=torch.uint8, device="cuda")
    dcr.check(dcr.dense_refit(plan, d_old, tgt))
    st = dcr.RecvState(plan, 3)
    for w in range(plan.n_windows):
        bound = plan.window(w).payload_bound
        xor = torch.zeros(bound, dtype=torch.uint8, device="cuda")
        rc, xsize, _ = dcr.encode(plan, d_old, d_new, xor, window=w, base_version=3, target_version=4)
        dcr.check(rc)
        ref = torch.zeros(bound, dtype=torch.uint8, device="cuda")
        rc, rsize, _ = dcr.encode(plan, d_old, d_new, ref, window=w, mode=dcr.MODE_OVERWRITE_ONLY,
                                  base_version=3, target_version=4)
        dcr.check(rc)
        got = torch.zeros(bound, dtype=torch.uint8, device="cuda")
        rc, gsize = dcr.encode_retry(plan, xor, xsize, d_new, got)
        assert rc == dcr.OK, dcr.last_error()
        assert gsize == rsize and torch.equal(got[:gsize], ref[:rsize])
        o, _ = orc.encode(olds, news, window=w, mode=oracle.MODE_OVERWRITE_ONLY, base_version=3,
                          target_version=4)
        assert np.array_equal(got[:gsize].cpu().numpy(), o)
        # the oracle's XOR stream (general LZ4 / Snappy blocks) gives the same retry stream
        ox, _ = orc.encode(olds, news, window=w, base_version=3, target_version=4,
                           codec=oracle.CODEC_SNAPPY if codec else oracle.CODEC_LZ4)
        d_ox = torch.from_numpy(ox).cuda()
        got2 = torch.zeros(bound, dtype=torch.uint8, device="cuda")
        rc, gsize2 = dcr.encode_retry(plan, d_ox, ox.size, d_new, got2)
        assert rc == dcr.OK, dcr.last_error()
        assert torch.equal(got2[:gsize2], ref[:rsize])
        # abort the XOR stream half way, then retry with the stream built from it
        nf = int(xor[48:56].cpu().numpy().view("<u8")[0])
        rc, _ = dcr.apply(plan, st, xor, xsize, tgt, fault=(nf // 2, 333))
        assert rc in (dcr.ERR_ABORTED, dcr.OK)
        rc, _ = dcr.apply_retry(plan, st, got, gsize, tgt)
        dcr.check(rc)
    assert st.version == 4
    exp = orc.receiver_dense(news)
    assert np.array_equal(tgt.cpu().numpy()[:exp.size], exp)


def test_retry_rejects_foreign_corrupt_and_short_input():
    wl = configs.mini(2)
    olds, news = wl.host_arenas()
    plan = dcr.Plan(descs_of(wl))
    other = dcr.Plan(descs_of(configs.mini(1)))
    d_old, d_new = to_device(olds), to_device(news)
    bound = plan.window(0).payload_bound
    xor = torch.zeros(bound, dtype=torch.uint8, device="cuda")
    rc, xsize, _ = dcr.encode(plan, d_old, d_new, xor)
    dcr.check(rc)
    out = torch.zeros(bound, dtype=torch.uint8, device="cuda")
    assert dcr.encode_retry(other, xor, xsize, d_new, out)[0] == dcr.ERR_INVALID
    assert dcr.encode_retry(plan, xor, 32, d_new, out)[0] == dcr.ERR_CORRUPT
    rc, need = dcr.encode_retry(plan, xor, xsize, d_new, out, cap=64)
    assert rc == dcr.ERR_CAPACITY and need > 64
    bad = xor.clone()
    fo = int(xor[xsize - 8 * 1:xsize].cpu().numpy().view("<u8")[0])   # the last frame
    bad[fo + 32:fo + 40] = 0xFF   # its block's first bytes
    rc, _ = dcr.encode_retry(plan, bad, xsize, d_new, out)
    assert rc == dcr.ERR_CORRUPT
    # a chunk framed twice
    from test_oracle import _with_index
    dup = _with_index(xor[:xsize].cpu().numpy(), [0, 0])
    rc, _ = dcr.encode_retry(plan, torch.from_numpy(dup).cuda(), dup.size, d_new, out)
    assert rc == dcr.ERR_CORRUPT
