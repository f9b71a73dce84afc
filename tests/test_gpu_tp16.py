"""The largest shard count (TP=16) through the C ABI: every split kind
(row-split, column-split with 64-column pieces, fused QKV with one kv group
per shard, replicated, e4m3) against the CPU oracle, in both encode modes
and with both encoder variants."""
import numpy as np
import pytest

import oracle
from synth import configs
from parity import assert_same_frames
from streamfmt import check_structure

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_exact_xor_gb300 as dcr  # noqa: E402
from wl import descs_of, to_device  # noqa: E402


@pytest.mark.parametrize("encoder", [dcr.ENCODER_WIDE, dcr.ENCODER_DEEP, dcr.ENCODER_CTA])
@pytest.mark.parametrize("mode", ["hybrid", "overwrite"])
def test_tp16_matches_oracle(mode, encoder):
    wl = configs.tp16()
    assert wl.tp == dcr.MAX_TP
    orc = oracle.Oracle(wl)
    olds, news = wl.host_arenas()
    plan = dcr.Plan(descs_of(wl), window_bytes=wl.window_bytes, encoder=encoder,
                    apply=dcr.APPLY_LANE if encoder == dcr.ENCODER_CTA else dcr.APPLY_AUTO)
    assert plan.info.plan_hash == orc.plan_hash and plan.info.tp == 16
    d_old, d_new = to_device(olds), to_device(news)
    dm = dcr.MODE_HYBRID if mode == "hybrid" else dcr.MODE_OVERWRITE_ONLY
    om = oracle.MODE_HYBRID if mode == "hybrid" else oracle.MODE_OVERWRITE_ONLY
    pl = torch.zeros(plan.window(0).payload_bound, dtype=torch.uint8, device="cuda")
    rc, size, counts = dcr.encode(plan, d_old, d_new, pl, mode=dm)
    assert rc == dcr.OK, dcr.last_error()
    g = pl[:size].cpu().numpy()
    o, oc = orc.encode(olds, news, mode=om)
    check_structure(g)
    assert counts == [int(x) for x in oc] and all(c > 0 for c in counts)
    assert_same_frames(g, o)
    assert g.size <= 1.15 * o.size + 64
    t = torch.zeros(max(plan.info.recv_bytes, wl.recv_bytes, 16), dtype=torch.uint8, device="cuda")
    dcr.check(dcr.dense_refit(plan, d_old, t))
    assert np.array_equal(t.cpu().numpy()[:wl.recv_bytes], orc.receiver_dense(olds)[:wl.recv_bytes])
    st = dcr.RecvState(plan, 0)
    rc, _ = (dcr.apply if mode == "hybrid" else dcr.apply_retry)(plan, st, pl, size, t)
    assert rc == dcr.OK, dcr.last_error()
    exp = orc.receiver_dense(news)
    assert np.array_equal(t.cpu().numpy()[:exp.size], exp) and st.version == 1
    tgt = orc.receiver_dense(olds)   # the oracle applies the GPU stream too
    assert orc.apply(orc.state(0), g, tgt, retry_only=mode != "hybrid") == oracle.OK
    assert np.array_equal(tgt, exp)
