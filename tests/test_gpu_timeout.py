"""Bounded device waits.  The encoder's offset scan runs one CTA per tile of
8192 chunks, each waiting for the running total of the tiles before it; a
test-only plan flag keeps tile 0 from ever publishing its total, so every
later tile's wait runs out.  The call must return DCR_ERR_TIMEOUT after
about a second, write no stream byte, and leave the context and the plans'
scratch usable: the same inputs then encode to the oracle's frames through
a plan without the flag.  Nothing faults or hangs the GPU."""
import time

import numpy as np
import pytest

import oracle
import synth
from synth import configs
from parity import assert_same_frames
from streamfmt import K_XOR_RAW, check_structure, parse

import bit_exact_xor_gb300 as dcr
from wl import descs_of

SCAN_TILE = 8192


def workload():
    """Two 64 KiB chunks of random bytes (raw frames, written by the spill
    pass from offsets the stalled scan never makes final) ahead of 8300
    bf16 tensors of 256 bytes with 5 % of their values changed: 8302 chunks,
    two scan tiles in one window."""
    ts = [configs.Tensor("big%d" % i, elem_bits=8, rows=1, cols=65536, split=configs.REPLICATED,
                         value_kind=synth.VAL_BYTES, rule=synth.RULE_RANDOM, frac=1.0) for i in range(2)]
    ts += [configs.Tensor("t%d" % i, rows=1, cols=128, split=configs.REPLICATED, rule=synth.RULE_PM4,
                          frac=0.05, **configs.BF) for i in range(8300)]
    return configs.Workload("stall", 0x5CA7, 1, ts).layout()


def test_stall_workload_spans_two_scan_tiles():
    wl = workload()
    plan = dcr.Plan(descs_of(wl), window_bytes=wl.window_bytes, host_only=True, flags=dcr.PLAN_TEST_STALL_SCAN)
    assert plan.n_windows == 1
    n = plan.window(0).chunk_count
    assert SCAN_TILE < n <= 2 * SCAN_TILE
    orc = oracle.Oracle(wl)
    assert orc.plan_hash == plan.info.plan_hash   # the flag is no part of the plan's identity
    olds, news = wl.host_arenas()
    o, _ = orc.encode(olds, news)
    _, frames, _ = parse(o)
    assert [f["kind"] for f in frames[:2]] == [K_XOR_RAW, K_XOR_RAW]
    assert len(frames) > SCAN_TILE


@pytest.mark.gpu
def test_scan_wait_runs_out_and_context_stays_usable():
    torch = pytest.importorskip("torch")
    from wl import to_device

    wl = workload()
    orc = oracle.Oracle(wl)
    olds, news = wl.host_arenas()
    d_old, d_new = to_device(olds), to_device(news)
    stalled = dcr.Plan(descs_of(wl), window_bytes=wl.window_bytes, flags=dcr.PLAN_TEST_STALL_SCAN)
    plan = dcr.Plan(descs_of(wl), window_bytes=wl.window_bytes)
    bound = plan.window(0).payload_bound
    pl = torch.full((bound,), 0xAB, dtype=torch.uint8, device="cuda")

    for _ in range(2):   # the second call reuses the scratch the first left behind
        t0 = time.monotonic()
        rc, _, _ = dcr.encode(stalled, d_old, d_new, pl)
        dt = time.monotonic() - t0
        assert rc == dcr.ERR_TIMEOUT, dcr.last_error()
        assert 0.5 < dt < 30.0, dt
        assert bool((pl == 0xAB).all())   # no stream byte written
    rc, _, _ = dcr.encode_part(stalled, d_old, d_new, 0, 1)
    assert rc == dcr.ERR_TIMEOUT

    # the context goes on: the plan without the flag encodes the same inputs
    rc, size, counts = dcr.encode(plan, d_old, d_new, pl)
    assert rc == dcr.OK, dcr.last_error()
    g = pl[:size].cpu().numpy()
    o, oc = orc.encode(olds, news)
    check_structure(g)
    assert counts == [int(x) for x in oc]
    assert_same_frames(g, o)

    # the retry encoder shares the scan: the stalled plan gives up, the plan
    # without the flag rebuilds the overwrite-only stream
    out = torch.full((bound,), 0xAB, dtype=torch.uint8, device="cuda")
    rc, _ = dcr.encode_retry(stalled, pl, size, d_new, out)
    assert rc == dcr.ERR_TIMEOUT
    assert bool((out == 0xAB).all())
    rc, rsize = dcr.encode_retry(plan, pl, size, d_new, out)
    assert rc == dcr.OK, dcr.last_error()
    ref, _ = orc.encode(olds, news, mode=oracle.MODE_OVERWRITE_ONLY)
    assert rsize == ref.size and np.array_equal(out[:rsize].cpu().numpy(), ref)

    # and the stream applies
    exp = orc.receiver_dense(news)
    t = torch.zeros(max(plan.info.recv_bytes, 16), dtype=torch.uint8, device="cuda")
    dcr.check(dcr.dense_refit(plan, d_old, t))
    rc, _ = dcr.apply(plan, dcr.RecvState(plan, 0), pl, size, t)
    assert rc == dcr.OK, dcr.last_error()
    assert np.array_equal(t.cpu().numpy()[:exp.size], exp)
