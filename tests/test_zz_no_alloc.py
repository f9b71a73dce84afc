"""dcr_apply_noalloc (dcr_apply with the library's static device scratch)
against dcr_apply on the same streams, two refits in a row, through the C
ABI; and its window limit.  Kept in a file of its own, collected last, so it
also runs after every other GPU test in the same process."""
import numpy as np
import pytest

import oracle
from synth import configs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_exact_xor_gb300 as dcr  # noqa: E402
from wl import descs_of, to_device  # noqa: E402


def _target(plan, wl, shards):
    t = torch.zeros(max(plan.info.recv_bytes, wl.recv_bytes, 16), dtype=torch.uint8, device="cuda")
    dcr.check(dcr.dense_refit(plan, shards, t))
    return t


@pytest.mark.parametrize("n,codec,apply", [(1, 0, 0), (2, 0, 0), (3, 0, 0), (3, 1, 0), (2, 0, 3), (3, 1, 3)])
def test_noalloc_matches_apply_two_calls_in_a_row(n, codec, apply):
    wl = configs.mini(n)
    orc = oracle.Oracle(wl)
    olds, news = wl.host_arenas()
    plan = dcr.Plan(descs_of(wl), window_bytes=wl.window_bytes, codec=codec, apply=apply)
    d_old, d_new = to_device(olds), to_device(news)
    ref_t, got_t = _target(plan, wl, d_old), _target(plan, wl, d_old)
    ref_st, got_st = dcr.RecvState(plan, 0), dcr.RecvState(plan, 0)
    # refit 0 -> 1 (old -> new), then 1 -> 2 (new -> old)
    for v, (a, b, host_b) in enumerate([(d_old, d_new, news), (d_new, d_old, olds)]):
        for w in range(plan.info.n_windows):
            pl = torch.zeros(plan.window(w).payload_bound, dtype=torch.uint8, device="cuda")
            rc, size, _ = dcr.encode(plan, a, b, pl, window=w, base_version=v, target_version=v + 1)
            dcr.check(rc)
            rc1, r1 = dcr.apply(plan, ref_st, pl, size, ref_t)
            rc2, r2 = dcr.apply_noalloc(plan, got_st, pl, size, got_t)
            assert rc1 == dcr.OK and rc2 == dcr.OK, (rc1, rc2, dcr.last_error())
            fields = ("target_version", "n_frames", "frames_applied", "frames_skipped", "pending", "window",
                      "committed")
            assert [getattr(r2, f) for f in fields] == [getattr(r1, f) for f in fields]
        torch.cuda.synchronize()
        assert torch.equal(ref_t, got_t)
        assert ref_st.version == got_st.version == v + 1
        exp = orc.receiver_dense(host_b)
        assert np.array_equal(got_t.cpu().numpy()[:exp.size], exp)


def test_noalloc_rejects_windows_beyond_its_limit():
    # one 4 GiB + 64 KiB tensor: a window of 65537 chunks, one more than the
    # static scratch holds; rejected before any kernel runs
    d = dcr.make_desc("big", 8, 65537, 65536, dcr.REPLICATED, 1, [0], 0)
    plan = dcr.Plan([d])
    assert plan.window(0).chunk_count == 65537
    st = dcr.RecvState(plan, 0)
    pl = torch.zeros(64, dtype=torch.uint8, device="cuda")
    t = torch.full((64,), 7, dtype=torch.uint8, device="cuda")
    rc, _ = dcr.apply_noalloc(plan, st, pl, 64, t)
    assert rc == dcr.ERR_CAPACITY
    assert "static scratch limit" in dcr.last_error()
    assert st.version == 0 and bool((t == 7).all())


def test_noalloc_after_state_creation_allocates_no_device_memory():
    # the receiver state's creation looks up the static scratch and the plan
    # build loads the apply kernels, so the first dcr_apply_noalloc call (and
    # every later one) leaves the device's free memory exactly as it was
    wl = configs.mini(2)
    olds, news = wl.host_arenas()
    plan = dcr.Plan(descs_of(wl), window_bytes=wl.window_bytes)
    d_old, d_new = to_device(olds), to_device(news)
    tgt = _target(plan, wl, d_old)
    st = dcr.RecvState(plan, 0)
    pls = []
    for v, (a, b) in enumerate([(d_old, d_new), (d_new, d_old)]):
        pl = torch.zeros(plan.window(0).payload_bound, dtype=torch.uint8, device="cuda")
        rc, size, _ = dcr.encode(plan, a, b, pl, base_version=v, target_version=v + 1)
        dcr.check(rc)
        pls.append((pl, size))
    torch.cuda.synchronize()
    for pl, size in pls:
        free0 = torch.cuda.mem_get_info()[0]
        rc, res = dcr.apply_noalloc(plan, st, pl, size, tgt)
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        assert rc == dcr.OK, dcr.last_error()
        assert free1 == free0, "dcr_apply_noalloc changed the device's free memory by %d bytes" % (free0 - free1)
    assert st.version == 2
    assert np.array_equal(tgt.cpu().numpy()[:wl.recv_bytes], oracle.Oracle(wl).receiver_dense(olds)[:wl.recv_bytes])
