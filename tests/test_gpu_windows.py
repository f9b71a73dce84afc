"""A tensor larger than the window: the library cuts it at the same chunk
boundaries as the CPU oracle, each window's stream carries the oracle's
frames, windows apply in any order, and the receiver's version moves only
when the last one lands (through the C ABI)."""
import numpy as np
import pytest

import oracle
from synth import configs
from parity import assert_same_frames
from streamfmt import check_structure, parse

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_exact_xor_gb300 as dcr  # noqa: E402
from wl import descs_of, to_device  # noqa: E402


@pytest.mark.parametrize("encoder", [dcr.ENCODER_WIDE, dcr.ENCODER_DEEP, dcr.ENCODER_CTA])
def test_oversized_tensor_windows(encoder):
    wl = configs.oversized_window()
    orc = oracle.Oracle(wl)
    olds, news = wl.host_arenas()
    plan = dcr.Plan(descs_of(wl), window_bytes=wl.window_bytes, encoder=encoder,
                    apply=dcr.APPLY_LANE if encoder == dcr.ENCODER_CTA else dcr.APPLY_AUTO)
    assert plan.info.plan_hash == orc.plan_hash
    assert plan.n_windows == orc.n_windows == 4
    for w in range(plan.n_windows):
        wi = plan.window(w)
        assert (wi.chunk_begin, wi.chunk_count) == tuple(orc.window_range(w))
    d_old, d_new = to_device(olds), to_device(news)
    t = torch.zeros(max(plan.info.recv_bytes, wl.recv_bytes, 16), dtype=torch.uint8, device="cuda")
    dcr.check(dcr.dense_refit(plan, d_old, t))
    st = dcr.RecvState(plan, 0)
    counts = np.zeros(len(wl.tensors), dtype=np.int64)
    ocounts = np.zeros(len(wl.tensors), dtype=np.int64)
    for i, w in enumerate([3, 1, 0, 2]):
        pl = torch.zeros(plan.window(w).payload_bound, dtype=torch.uint8, device="cuda")
        rc, size, cnt = dcr.encode(plan, d_old, d_new, pl, window=w)
        assert rc == dcr.OK, dcr.last_error()
        g = pl[:size].cpu().numpy()
        o, oc = orc.encode(olds, news, window=w)
        hdr, _ = check_structure(g)
        assert hdr["window"] == w
        assert_same_frames(g, o)
        assert g.size <= 1.15 * o.size + 64
        b, c = orc.window_range(w)
        assert all(b <= f["chunk"] < b + c for f in parse(g)[1])
        counts += cnt
        ocounts += np.asarray(oc, dtype=np.int64)
        rc, res = dcr.apply(plan, st, pl, size, t)
        assert rc == dcr.OK, dcr.last_error()
        assert st.version == (1 if i == 3 else 0) and res.committed == (1 if i == 3 else 0)
    assert np.array_equal(counts, ocounts)
    exp = orc.receiver_dense(news)
    assert np.array_equal(t.cpu().numpy()[:exp.size], exp)
