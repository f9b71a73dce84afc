"""dcr_refit_pipelined (every window encoded, sent through pinned host memory
and applied, the transfer of one window overlapping its neighbours'
compute) against the CPU oracle and against the same windows done one call
at a time, through the C ABI."""
import numpy as np
import pytest

import oracle
from synth import configs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_exact_xor_gb300 as dcr  # noqa: E402
from wl import descs_of, to_device  # noqa: E402
from test_gpu_random import random_workload  # noqa: E402


def _buffers(plan):
    dev, host = dcr.pipeline_sizes(plan)
    return (torch.empty(dev, dtype=torch.uint8, device="cuda"),
            torch.empty(host, dtype=torch.uint8).pin_memory())


def _target(plan, wl, shards):
    t = torch.zeros(max(plan.info.recv_bytes, wl.recv_bytes, 16), dtype=torch.uint8, device="cuda")
    dcr.check(dcr.dense_refit(plan, shards, t))
    return t


def _sequential_sizes(plan, olds, news, mode=dcr.MODE_HYBRID):
    sizes = []
    for w in range(plan.n_windows):
        pl = torch.empty(plan.window(w).payload_bound, dtype=torch.uint8, device="cuda")
        rc, size, _ = dcr.encode(plan, olds, news, pl, window=w, mode=mode)
        dcr.check(rc)
        sizes.append(size)
    return sizes


WORKLOADS = [("mini-moe", lambda: configs.mini(5)), ("mini-gqa", lambda: configs.mini(3)),
             ("mini-dense", lambda: configs.mini(2))] + \
            [("random-%d" % s, (lambda s=s: random_workload(s))) for s in (1, 4, 7, 12)]


# the apply kernels AUTO picks for these small windows (one CTA per frame), and
# the route + warp + thread-per-frame kernels with every deferred kernel
CASES = [(w, a) for w in WORKLOADS for a in ("auto", "lane")]


@pytest.mark.parametrize("name,make,apply", [(w[0], w[1], a) for w, a in CASES],
                         ids=["%s-%s" % (w[0], a) for w, a in CASES])
def test_pipelined_refit_matches_oracle_and_sequential(name, make, apply):
    wl = make()
    orc = oracle.Oracle(wl)
    olds, news = wl.host_arenas()
    plan = dcr.Plan(descs_of(wl), window_bytes=wl.window_bytes,
                    apply=dcr.APPLY_LANE if apply == "lane" else dcr.APPLY_AUTO)
    d_old, d_new = to_device(olds), to_device(news)
    dev, host = _buffers(plan)
    t = _target(plan, wl, d_old)
    st = dcr.RecvState(plan, 0)
    rc, stats, counts = dcr.refit_pipelined(plan, st, d_old, d_new, t, dev, host)
    assert rc == dcr.OK, dcr.last_error()
    exp = orc.receiver_dense(news)
    assert np.array_equal(t.cpu().numpy()[:exp.size], exp)
    assert st.version == 1 and stats.committed == 1 and stats.windows == plan.n_windows
    oc = np.zeros(len(wl.tensors), dtype=np.int64)
    for w in range(orc.n_windows):
        oc += np.asarray(orc.encode(olds, news, window=w)[1], dtype=np.int64)
    assert counts == [int(x) for x in oc]
    sizes = _sequential_sizes(plan, d_old, d_new)
    assert stats.payload_bytes == sum(sizes) and stats.max_window_payload == max(sizes)
    # and back (version 1 -> 2), overwrite-only, from the state just committed
    rc, stats2, _ = dcr.refit_pipelined(plan, st, d_new, d_old, t, dev, host, mode=dcr.MODE_OVERWRITE_ONLY,
                                        base_version=1, target_version=2)
    assert rc == dcr.OK, dcr.last_error()
    assert st.version == 2 and stats2.committed == 1
    assert np.array_equal(t.cpu().numpy()[:exp.size], orc.receiver_dense(olds))


def test_pipelined_refit_snappy_codec():
    wl = configs.mini(5)
    orc = oracle.Oracle(wl)
    olds, news = wl.host_arenas()
    plan = dcr.Plan(descs_of(wl), window_bytes=wl.window_bytes, codec=dcr.CODEC_SNAPPY)
    d_old, d_new = to_device(olds), to_device(news)
    dev, host = _buffers(plan)
    t = _target(plan, wl, d_old)
    st = dcr.RecvState(plan, 0)
    rc, stats, _ = dcr.refit_pipelined(plan, st, d_old, d_new, t, dev, host)
    assert rc == dcr.OK, dcr.last_error()
    exp = orc.receiver_dense(news)
    assert np.array_equal(t.cpu().numpy()[:exp.size], exp)
    assert st.version == 1 and stats.windows == plan.n_windows
    assert stats.payload_bytes == sum(_sequential_sizes(plan, d_old, d_new))


def test_pipelined_refit_rejections_leave_target_untouched():
    wl = configs.mini(5)
    olds, news = wl.host_arenas()
    plan = dcr.Plan(descs_of(wl), window_bytes=wl.window_bytes)
    d_old, d_new = to_device(olds), to_device(news)
    dev, host = _buffers(plan)
    t = _target(plan, wl, d_old)
    before = t.clone()
    st = dcr.RecvState(plan, 0)
    # pageable host memory
    rc, _, _ = dcr.refit_pipelined(plan, st, d_old, d_new, t, dev, torch.empty(host.numel(), dtype=torch.uint8))
    assert rc == dcr.ERR_INVALID and "pinned" in dcr.last_error()
    # buffers one byte short
    rc, _, _ = dcr.refit_pipelined(plan, st, d_old, d_new, t, dev[:dev.numel() - 1], host)
    assert rc == dcr.ERR_INVALID and "too small" in dcr.last_error()
    # a stream built on a version the receiver is not at
    rc, stats, _ = dcr.refit_pipelined(plan, st, d_old, d_new, t, dev, host, base_version=5, target_version=6)
    assert rc == dcr.ERR_VERSION
    assert stats.committed == 0 and st.version == 0
    torch.cuda.synchronize()
    assert torch.equal(t, before)
    # the state is still usable
    rc, stats, _ = dcr.refit_pipelined(plan, st, d_old, d_new, t, dev, host)
    assert rc == dcr.OK and st.version == 1
