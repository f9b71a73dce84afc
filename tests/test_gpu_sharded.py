"""Ownership-sharded encode on one GPU: each emulated rank holds its own plan
(its own scratch) and encodes its part of every window with dcr_encode_part;
the parts' frames and index entries are written at the offsets
dcr_stream_layout gives, under the header dcr_stream_header writes.  The
assembled stream must equal dcr_encode's single-rank stream byte for byte
and refit the receiver to `new` (checked against the oracle).  Blog, "A
strong baseline with the Blackwell-native DE": the ranks cover the
checkpoint exactly once and only compressed payloads are gathered."""
import numpy as np
import pytest

import oracle
from synth import configs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_exact_xor_gb300 as dcr  # noqa: E402
from wl import descs_of, to_device  # noqa: E402


def _assemble(plans, d_old, d_new, w, mode, base=0, target=1, staging=False):
    n = len(plans)
    sizes, counts = [], []
    for q, p in enumerate(plans):
        rc, sz, cnt = dcr.encode_part(p, d_old, d_new, q, n, window=w, mode=mode)
        dcr.check(rc)
        sizes.append(sz)
        counts.append(cnt)
    fo, io, total = dcr.stream_layout(sizes)
    out = torch.zeros(total, dtype=torch.uint8, device="cuda")
    for q, p in enumerate(plans):
        fb, nf = sizes[q]
        if staging:   # the rank's own buffer, then copied (the gather) into the stream
            blob = torch.zeros(max(fb + 8 * nf, 16), dtype=torch.uint8, device="cuda")
            dcr.check(dcr.encode_part_write(p, fo[q], blob, fb, blob.data_ptr() + fb))
            out[fo[q]:fo[q] + fb] = blob[:fb]
            out[io[q]:io[q] + 8 * nf] = blob[fb:fb + 8 * nf]
        else:
            dcr.check(dcr.encode_part_write(p, fo[q], out.data_ptr() + fo[q], fb, out.data_ptr() + io[q]))
    hdr = dcr.stream_header(plans[0], w, base, target, sum(k for _, k in sizes), sum(f for f, _ in sizes), mode)
    out[:64] = torch.frombuffer(bytearray(hdr), dtype=torch.uint8).cuda()
    tot_counts = [sum(c) for c in zip(*counts)]
    return out, tot_counts


CASES = [(1, 0, 0), (2, 0, 0), (3, 0, 0), (3, 1, 0), (4, 0, 0), (5, 0, 0), (5, 0, 1), (16, 0, 0)]


@pytest.mark.parametrize("n,mode,codec", CASES, ids=["%s-%s-%s" % c for c in CASES])
@pytest.mark.parametrize("n_parts", [1, 2, 3, 8])
def test_sharded_stream_equals_single_rank_stream(n, mode, codec, n_parts):
    wl = configs.tp16() if n == 16 else configs.mini(n)
    descs = descs_of(wl)
    ref_plan = dcr.Plan(descs, window_bytes=wl.window_bytes, codec=codec)
    plans = [dcr.Plan(descs, window_bytes=wl.window_bytes, codec=codec) for _ in range(n_parts)]
    orc = oracle.Oracle(wl)
    olds, news = wl.host_arenas()
    d_old, d_new = to_device(olds), to_device(news)
    tgt = torch.zeros(max(ref_plan.info.recv_bytes, wl.recv_bytes, 16), dtype=torch.uint8, device="cuda")
    dcr.check(dcr.dense_refit(ref_plan, d_old, tgt))
    st = dcr.RecvState(ref_plan, 0)
    for w in range(ref_plan.n_windows):
        ref = torch.zeros(ref_plan.window(w).payload_bound, dtype=torch.uint8, device="cuda")
        rc, size, ref_counts = dcr.encode(ref_plan, d_old, d_new, ref, window=w, mode=mode)
        dcr.check(rc)
        got, counts = _assemble(plans, d_old, d_new, w, mode, staging=(w % 2 == 1))
        assert got.numel() == size
        assert torch.equal(got, ref[:size]), "assembled stream differs from the single-rank stream"
        assert counts == ref_counts
        apply = dcr.apply_retry if mode else dcr.apply
        rc, res = apply(ref_plan, st, got, got.numel(), tgt)
        dcr.check(rc)
    assert st.version == 1
    exp = orc.receiver_dense(news)
    assert np.array_equal(tgt.cpu().numpy()[:exp.size], exp)


def test_sharded_write_errors_and_rewrite():
    wl = configs.mini(2)
    plan = dcr.Plan(descs_of(wl))
    olds, news = wl.host_arenas()
    d_old, d_new = to_device(olds), to_device(news)
    buf = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    # nothing sized on this plan yet
    assert dcr.encode_part_write(plan, 64, buf, buf.numel(), buf) == dcr.ERR_INVALID
    rc, (fb, nf), _ = dcr.encode_part(plan, d_old, d_new, 1, 2)
    dcr.check(rc)
    assert fb > 0 and nf > 0
    assert dcr.encode_part_write(plan, 64, buf, fb - 16, buf.data_ptr() + fb) == dcr.ERR_CAPACITY
    assert dcr.encode_part_write(plan, 72, buf, fb, buf.data_ptr() + fb) == dcr.ERR_INVALID
    assert dcr.encode_part_write(plan, 64, buf.data_ptr() + 8, fb, buf.data_ptr() + fb + 8) == dcr.ERR_INVALID
    # written twice: the same bytes (the write pass may be repeated)
    dcr.check(dcr.encode_part_write(plan, 4096, buf, fb, buf.data_ptr() + fb))
    first = buf[:fb + 8 * nf].clone()
    buf.zero_()
    dcr.check(dcr.encode_part_write(plan, 4096, buf, fb, buf.data_ptr() + fb))
    assert torch.equal(buf[:fb + 8 * nf], first)
    idx = first[fb:fb + 8 * nf].cpu().numpy().view("<u8")
    assert idx[0] == 4096 and np.all(np.diff(idx.astype(np.int64)) > 0) and np.all(idx % 16 == 0)
    # a full encode in between invalidates the sized part
    pl = torch.zeros(plan.window(0).payload_bound, dtype=torch.uint8, device="cuda")
    dcr.check(dcr.encode(plan, d_old, d_new, pl)[0])
    assert dcr.encode_part_write(plan, 64, buf, fb, buf.data_ptr() + fb) == dcr.ERR_INVALID
    # a part only reads the shards in its mask: the other arenas may be NULL
    pi = plan.part(0, 63, 64)
    if pi.shard_mask == 1:
        rc, _, _ = dcr.encode_part(plan, [d_old[0], None], [d_new[0], None], 63, 64)
        dcr.check(rc)
    rc, _, _ = dcr.encode_part(plan, [d_old[0], None], [d_new[0], None], 0, 1)
    assert rc == dcr.ERR_INVALID
