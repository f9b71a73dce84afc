"""GPU parity on the small structural twins of the five workloads: the CUDA
path, called through the C ABI, against the CPU oracle on the same seeded
inputs.  Sizes span several 64 KiB chunks and ragged tails."""
import numpy as np
import pytest

import oracle
import synth
from synth import configs
from parity import assert_same_frames, frames_by_chunk
from streamfmt import check_structure, parse

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_exact_xor_gb300 as dcr  # noqa: E402
from wl import descs_of, to_device  # noqa: E402


class Case:
    def __init__(self, wl, rule=None, frac=None, apply=dcr.APPLY_AUTO):
        self.wl = wl
        self.orc = oracle.Oracle(wl)
        self.olds, self.news = wl.host_arenas(rule_override=rule, frac_override=frac)
        self.plan = dcr.Plan(descs_of(wl), window_bytes=wl.window_bytes, apply=apply)
        self.d_old, self.d_new = to_device(self.olds), to_device(self.news)
        self.exp = self.orc.receiver_dense(self.news)
        self.start = self.orc.receiver_dense(self.olds)

    def target(self):
        t = torch.zeros(max(self.plan.info.recv_bytes, self.wl.recv_bytes, 16), dtype=torch.uint8,
                        device="cuda")
        dcr.check(dcr.dense_refit(self.plan, self.d_old, t))
        return t

    def encode(self, w=0, mode=dcr.MODE_HYBRID, base=0, target=1, olds=None, news=None):
        wi = self.plan.window(w)
        pl = torch.zeros(wi.payload_bound, dtype=torch.uint8, device="cuda")
        rc, size, counts = dcr.encode(self.plan, olds or self.d_old, news or self.d_new, pl, window=w,
                                      mode=mode, base_version=base, target_version=target)
        dcr.check(rc)
        return pl, size, counts

    def host(self, t):
        return t.cpu().numpy()[:self.exp.size]


# every small twin with each apply kernel: one warp per frame, one CTA per
# frame, one thread per ZSRC frame, the split walk of every ZSRC frame
APPLY = {"warp": dcr.APPLY_WARP, "cta": dcr.APPLY_CTA, "lane": dcr.APPLY_LANE, "split": dcr.APPLY_SPLIT}


@pytest.fixture(scope="module", params=[(n, a) for n in (1, 2, 3, 4, 5) for a in APPLY],
                ids=lambda p: "%d-%s" % p)
def case(request):
    n, a = request.param
    return Case(configs.mini(n), apply=APPLY[a])


def test_generator_twins_agree():
    for vk, rule, fr, zf in [(synth.VAL_BF16_NORMAL, synth.RULE_PM4, 0.01, 0.0001),
                             (synth.VAL_BF16_NORMAL, synth.RULE_LOW3, 0.05, 0.0),
                             (synth.VAL_BF16_NORMAL, synth.RULE_RANDOM, 0.0, 0.0),
                             (synth.VAL_BYTES, synth.RULE_NIBBLE, 0.01, 0.0),
                             (synth.VAL_E4M3_SCALE, synth.RULE_BPM4, 0.01, 0.0)]:
        p = synth.make_params(0xABC, 77, vk, rule, fr, zf, elem_base=123457)
        n = 300001
        o, w = synth.fill_cpu(p, n)
        eb = synth.elem_bytes(vk)
        go = torch.zeros(n * eb, dtype=torch.uint8, device="cuda")
        gw = torch.zeros(n * eb, dtype=torch.uint8, device="cuda")
        synth.fill_gpu(p, n, go.data_ptr(), gw.data_ptr(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert np.array_equal(go.cpu().numpy(), o) and np.array_equal(gw.cpu().numpy(), w)


def test_plan_matches_oracle_layout(case):
    assert case.plan.info.plan_hash == case.orc.plan_hash
    assert case.plan.n_windows == case.orc.n_windows
    assert case.plan.info.n_chunks == case.orc.n_chunks
    assert case.plan.info.canonical_bytes == case.wl.canonical_bytes
    for w in range(case.plan.n_windows):
        wi = case.plan.window(w)
        assert (wi.chunk_begin, wi.chunk_count) == case.orc.window_range(w)


def test_dense_refit_matches_oracle(case):
    assert np.array_equal(case.host(case.target()), case.start)


@pytest.mark.parametrize("mode", [dcr.MODE_HYBRID, dcr.MODE_OVERWRITE_ONLY])
def test_encode_parity(case, mode):
    tot_g = tot_o = 0
    for w in range(case.plan.n_windows):
        pl, size, counts = case.encode(w, mode, base=3, target=4)
        g = pl[:size].cpu().numpy()
        o, oc = case.orc.encode(case.olds, case.news, window=w, mode=mode, base_version=3,
                                target_version=4)
        check_structure(g)
        assert counts == [int(x) for x in oc]
        hdr, gf, of = assert_same_frames(g, o)
        if mode == dcr.MODE_OVERWRITE_ONLY:
            assert np.array_equal(g, o), "overwrite streams are deterministic: byte-identical"
        tot_g += g.size
        tot_o += o.size
    assert tot_g <= 1.15 * tot_o, (tot_g, tot_o)


def test_gpu_stream_applies_on_gpu_and_oracle(case):
    t = case.target()
    st = dcr.RecvState(case.plan, 0)
    ost = case.orc.state(0)
    otgt = case.start.copy()
    for w in range(case.plan.n_windows):
        pl, size, _ = case.encode(w)
        rc, res = dcr.apply(case.plan, st, pl, size, t)
        assert rc == dcr.OK, dcr.last_error()
        assert res.committed == (w == case.plan.n_windows - 1)
        assert case.orc.apply(ost, pl[:size].cpu().numpy(), otgt) == oracle.OK
    assert np.array_equal(case.host(t), case.exp)
    assert np.array_equal(otgt, case.exp)
    assert st.version == 1 and ost.version == 1


def test_oracle_stream_applies_on_gpu(case):
    t = case.target()
    st = dcr.RecvState(case.plan, 5)
    for w in range(case.plan.n_windows):
        o, _ = case.orc.encode(case.olds, case.news, window=w, base_version=5, target_version=6)
        d = torch.from_numpy(o).cuda()
        rc, res = dcr.apply(case.plan, st, d, o.size, t)
        assert rc == dcr.OK, dcr.last_error()
    assert np.array_equal(case.host(t), case.exp) and st.version == 6


def test_overwrite_retry_stream_reaches_new(case):
    t = case.target()
    st = dcr.RecvState(case.plan, 0)
    for w in range(case.plan.n_windows):
        pl, size, _ = case.encode(w, dcr.MODE_OVERWRITE_ONLY)
        rc, _ = dcr.apply_retry(case.plan, st, pl, size, t)
        assert rc == dcr.OK, dcr.last_error()
    assert np.array_equal(case.host(t), case.exp)


@pytest.mark.parametrize("apply", ["auto", "lane", "split"])
@pytest.mark.parametrize("n", [1, 3])
def test_abort_state_matches_oracle_then_retry(n, apply):
    c = Case(configs.mini(n), apply=dcr.APPLY_AUTO if apply == "auto" else APPLY[apply])
    pl, size, _ = c.encode()
    rp, rsize, _ = c.encode(mode=dcr.MODE_OVERWRITE_ONLY)
    nf = parse(pl[:size].cpu().numpy())[0]["n_frames"]
    g_pl = pl[:size].cpu().numpy()
    for k in sorted(set([0, 1, nf // 2, nf - 1])):
        for split in (0, 1001, 65536):
            t = c.target()
            st = dcr.RecvState(c.plan, 0)
            rc, res = dcr.apply(c.plan, st, pl, size, t, fault=(k, split))
            assert rc == dcr.ERR_ABORTED and st.version == 0
            otgt = c.start.copy()
            ost = c.orc.state(0)
            assert c.orc.apply(ost, g_pl, otgt, abort_at=k, split=split) == oracle.E_ABORTED
            assert np.array_equal(c.host(t), otgt), "mixed state after abort differs from oracle"
            rc, _ = dcr.apply(c.plan, st, pl, size, t)           # re-sent XOR stream
            assert rc in (dcr.OK, dcr.ERR_INCOMPLETE)
            if rc == dcr.OK:
                assert st.version == 1
            else:
                rc, _ = dcr.apply_retry(c.plan, st, rp, rsize, t)
                assert rc == dcr.OK and st.version == 1
            assert np.array_equal(c.host(t), c.exp)


def _reindexed(pl_np, order):
    hdr, frames, idx = parse(pl_np)
    offs = np.array([frames[i]["offset"] for i in order], dtype="<u8")
    out = np.concatenate([pl_np[:idx], offs.view(np.uint8)])
    out[48:56] = np.array([len(order)], dtype="<u8").view(np.uint8)
    out[56:64] = np.array([out.size], dtype="<u8").view(np.uint8)
    return out


@pytest.mark.parametrize("apply", ["auto", "warp", "lane", "split"])
def test_duplicate_frames_applied_once(apply):
    c = Case(configs.mini(2), apply=dcr.APPLY_AUTO if apply == "auto" else APPLY[apply])
    pl, size, _ = c.encode()
    g = pl[:size].cpu().numpy()
    nf = parse(g)[0]["n_frames"]
    dup = _reindexed(g, list(range(nf)) * 3 + [0, nf - 1])
    t = c.target()
    st = dcr.RecvState(c.plan, 0)
    rc, res = dcr.apply(c.plan, st, torch.from_numpy(dup).cuda(), dup.size, t)
    assert rc == dcr.OK and res.frames_skipped == 2 * nf + 2 and st.version == 1
    assert np.array_equal(c.host(t), c.exp)


@pytest.mark.parametrize("apply", ["cta", "warp", "lane", "split"])
def test_repeated_overwrite_frames(apply):
    # overwrite frames are applied unclaimed (idempotent): a stream that
    # repeats them is applied while they fit route_kernel's frame list (one
    # entry per chunk and one more), and rejected there, with nothing written
    # out of bounds, once they outnumber it; the CTA kernel and apply_kernel
    # routing frames itself keep no such list
    c = Case(configs.mini(1), apply=APPLY[apply])
    rp, rsize, _ = c.encode(mode=dcr.MODE_OVERWRITE_ONLY)
    g = rp[:rsize].cpu().numpy()
    nf = parse(g)[0]["n_frames"]
    chunks = c.plan.window(0).chunk_count
    assert 0 < nf <= chunks
    fits = _reindexed(g, list(range(nf)) + [0] * (chunks + 1 - nf))
    t = c.target()
    st = dcr.RecvState(c.plan, 0)
    rc, _ = dcr.apply_retry(c.plan, st, torch.from_numpy(fits).cuda(), fits.size, t)
    assert rc == dcr.OK and st.version == 1 and np.array_equal(c.host(t), c.exp)
    over = _reindexed(g, list(range(nf)) * 3 + [0] * (chunks + 1))
    t = c.target()
    st = dcr.RecvState(c.plan, 0)
    rc, _ = dcr.apply_retry(c.plan, st, torch.from_numpy(over).cuda(), over.size, t)
    if apply != "lane":
        assert rc == dcr.OK and st.version == 1 and np.array_equal(c.host(t), c.exp)
    else:
        assert rc == dcr.ERR_CORRUPT and st.version == 0


@pytest.mark.parametrize("apply", ["auto", "warp", "lane", "split"])
def test_duplicate_oracle_frames_applied_once(apply):
    c = Case(configs.mini(1), apply=dcr.APPLY_AUTO if apply == "auto" else APPLY[apply])
    o, _ = c.orc.encode(c.olds, c.news)
    nf = parse(o)[0]["n_frames"]
    dup = _reindexed(o, list(range(nf)) + list(range(nf)))
    t = c.target()
    st = dcr.RecvState(c.plan, 0)
    rc, res = dcr.apply(c.plan, st, torch.from_numpy(dup).cuda(), dup.size, t)
    assert rc == dcr.OK and res.frames_skipped == nf
    assert np.array_equal(c.host(t), c.exp)


@pytest.mark.parametrize("apply", ["auto", "warp", "lane", "split"])
def test_rejections_leave_target_untouched(apply):
    c = Case(configs.mini(1), apply=dcr.APPLY_AUTO if apply == "auto" else APPLY[apply])
    pl, size, _ = c.encode(base=3, target=4)
    t = c.target()
    before = c.host(t).copy()
    rc, _ = dcr.apply(c.plan, dcr.RecvState(c.plan, 2), pl, size, t)
    assert rc == dcr.ERR_VERSION
    bad = pl.clone()
    bad[8] ^= 1
    rc, _ = dcr.apply(c.plan, dcr.RecvState(c.plan, 3), bad, size, t)
    assert rc == dcr.ERR_INVALID
    rc, _ = dcr.apply_retry(c.plan, dcr.RecvState(c.plan, 3), pl, size, t)
    assert rc == dcr.ERR_INVALID
    bad = pl.clone()
    bad[0] ^= 1
    rc, _ = dcr.apply(c.plan, dcr.RecvState(c.plan, 3), bad, size, t)
    assert rc == dcr.ERR_CORRUPT
    assert np.array_equal(c.host(t), before)
    st = dcr.RecvState(c.plan, 3)
    rc, _ = dcr.apply(c.plan, st, pl, size, t)
    assert rc == dcr.OK and st.version == 4
    rc, _ = dcr.apply(c.plan, st, pl, size, t)
    assert rc == dcr.ERR_VERSION
    assert np.array_equal(c.host(t), c.exp)


@pytest.mark.parametrize("apply", ["auto", "warp", "lane", "split"])
def test_corrupt_lz4_frame_reported_and_retry_recovers(apply):
    c = Case(configs.mini(1), apply=dcr.APPLY_AUTO if apply == "auto" else APPLY[apply])
    pl, size, _ = c.encode()
    g = pl[:size].cpu().numpy()
    _, frames, _ = parse(g)
    f = [f for f in frames if f["kind"] == 1][0]
    bad = g.copy()
    bad[f["offset"] + 32:f["offset"] + 40] = 0xFF
    t = c.target()
    st = dcr.RecvState(c.plan, 0)
    rc, _ = dcr.apply(c.plan, st, torch.from_numpy(bad).cuda(), size, t)
    assert rc == dcr.ERR_CORRUPT and st.version == 0
    rp, rsize, _ = c.encode(mode=dcr.MODE_OVERWRITE_ONLY)
    rc, _ = dcr.apply_retry(c.plan, st, rp, rsize, t)
    assert rc == dcr.OK and np.array_equal(c.host(t), c.exp)


def _last_match_offset(body):
    """Byte position of the offset field of the last match in an LZ4 block."""
    ip, last = 0, None
    while True:
        tok = int(body[ip]); ip += 1
        ll = tok >> 4
        if ll == 15:
            while True:
                b = int(body[ip]); ip += 1; ll += b
                if b != 255:
                    break
        ip += ll
        if ip == body.size:
            return last
        last = ip
        ip += 2
        if tok & 15 == 15:
            while int(body[ip]) == 255:
                ip += 1
            ip += 1


@pytest.mark.parametrize("apply", ["auto", "lane", "split"])
def test_frame_failing_late_leaves_its_chunk_untouched(apply):
    # a ZSRC frame whose last match offset is zeroed fails only after most of
    # its literals were XOR-ed in; the chunk must come back exactly as it was,
    # otherwise the overwrite-only retry (changed units only) cannot repair it
    c = Case(configs.mini(1), apply=dcr.APPLY_AUTO if apply == "auto" else APPLY[apply])
    pl, size, _ = c.encode()
    g = pl[:size].cpu().numpy()
    _, frames, _ = parse(g)
    k = next(i for i, f in enumerate(frames)
             if f["kind"] == 1 and f["flags"] & 1 and _last_match_offset(f["body"]) not in (None, 0))
    f = frames[k]
    bad = g.copy()
    at = f["offset"] + 32 + _last_match_offset(f["body"])
    bad[at:at + 2] = 0
    t = c.target()
    st = dcr.RecvState(c.plan, 0)
    rc, _ = dcr.apply(c.plan, st, torch.from_numpy(bad).cuda(), size, t)
    assert rc == dcr.ERR_CORRUPT and st.version == 0
    # the oracle applying every other frame gives the expected bytes
    rest = _reindexed(g, [i for i in range(len(frames)) if i != k])
    ref = c.start.copy()
    assert c.orc.apply(c.orc.state(0), rest, ref) == oracle.OK
    assert np.array_equal(c.host(t), ref)
    rp, rsize, _ = c.encode(mode=dcr.MODE_OVERWRITE_ONLY)
    rc, _ = dcr.apply_retry(c.plan, st, rp, rsize, t)
    assert rc == dcr.OK and st.version == 1 and np.array_equal(c.host(t), c.exp)


@pytest.mark.parametrize("apply", ["auto", "lane", "split"])
@pytest.mark.parametrize("frac", [None, 0.05])
def test_zsrc_flag_is_verified(frac, apply):
    # a greedy (oracle) block whose matches copy non-zero bytes, relabelled
    # as ZSRC, must be rejected rather than applied as zeros; at 5 % change the
    # bodies are larger than the warp path's cache (the large-frame kernel)
    c = Case(configs.mini(1) if frac is None else configs.mini(4), frac=frac,
             apply=dcr.APPLY_AUTO if apply == "auto" else APPLY[apply])
    o, _ = c.orc.encode(c.olds, c.news)
    _, frames, _ = parse(o)
    lied = o.copy()
    n = 0
    for f in frames:
        if f["kind"] == 1:
            m = oracle.lz4_decode(f["body"], f["raw_len"])
            if oracle.lz4_decode(f["body"], f["raw_len"], zsrc=True) is None and m is not None:
                lied[f["offset"] + 6] = 1
                n += 1
                big = f["body_len"] > 3072 if frac else False
    assert n > 0
    if frac:
        assert big
    t = c.target()
    rc, _ = dcr.apply(c.plan, dcr.RecvState(c.plan, 0), torch.from_numpy(lied).cuda(), o.size, t)
    assert rc == dcr.ERR_CORRUPT


def test_no_change_and_capacity():
    c = Case(configs.mini(2))
    wi = c.plan.window(0)
    pl = torch.zeros(wi.payload_bound, dtype=torch.uint8, device="cuda")
    rc, size, counts = dcr.encode(c.plan, c.d_old, c.d_old, pl)
    assert rc == dcr.OK and size == 64 and not any(counts)
    t = c.target()
    st = dcr.RecvState(c.plan, 0)
    rc, _ = dcr.apply(c.plan, st, pl, size, t)
    assert rc == dcr.OK and st.version == 1 and np.array_equal(c.host(t), c.start)
    _, need, _ = dcr.encode(c.plan, c.d_old, c.d_new, pl)
    small = torch.zeros(need - 1, dtype=torch.uint8, device="cuda")
    rc, size2, _ = dcr.encode(c.plan, c.d_old, c.d_new, small)
    assert rc == dcr.ERR_CAPACITY and size2 == need
    rc, size3, _ = dcr.encode(c.plan, c.d_old, c.d_new, pl, cap=need)
    assert rc == dcr.OK and size3 == need


@pytest.mark.parametrize("apply", ["auto", "lane", "split"])
@pytest.mark.parametrize("frac", [0.0, 0.00085, 0.05, 0.3, "random"])
def test_change_rates_parity(frac, apply):
    wl = configs.mini(4)
    c = Case(wl, rule=synth.RULE_RANDOM if frac == "random" else None,
             frac=None if frac == "random" else frac,
             apply=dcr.APPLY_AUTO if apply == "auto" else APPLY[apply])
    pl, size, counts = c.encode()
    g = pl[:size].cpu().numpy()
    o, oc = c.orc.encode(c.olds, c.news)
    assert counts == [int(x) for x in oc]
    assert_same_frames(g, o)
    assert g.size <= 1.15 * o.size + 64
    t = c.target()
    rc, _ = dcr.apply(c.plan, dcr.RecvState(c.plan, 0), pl, size, t)
    assert rc == dcr.OK and np.array_equal(c.host(t), c.exp)


def test_signed_zero_on_gpu():
    t0 = configs.Tensor("z", elem_bits=16, rows=64, cols=1024, split=configs.REPLICATED,
                        value_kind=0, rule=0, frac=0)
    wl = configs.Workload("z", 1, 1, [t0]).layout()
    old = np.zeros(wl.shard_bytes[0], dtype=np.uint8)
    new = old.copy()
    new[2 * 777 + 1] = 0x80
    plan = dcr.Plan(descs_of(wl))
    d_old, d_new = to_device([old]), to_device([new])
    pl = torch.zeros(plan.window(0).payload_bound, dtype=torch.uint8, device="cuda")
    rc, size, counts = dcr.encode(plan, d_old, d_new, pl)
    assert rc == dcr.OK and counts == [1]
    tgt = to_device([old])[0]
    rc, _ = dcr.apply(plan, dcr.RecvState(plan, 0), pl, size, tgt)
    assert rc == dcr.OK and np.array_equal(tgt.cpu().numpy(), new)


# kernels of one apply: the first phase (CTA kernel; apply_kernel routing
# itself; route, warp and thread kernels) and the commit check, and with
# deferred frames the defer and big kernels and the commit check again
FIRST_PHASE = {"auto": 1, "warp": 1, "lane": 3, "split": 1}


@pytest.mark.parametrize("apply", ["auto", "warp", "lane", "split"])
def test_kernel_timing_profile(apply):
    c = Case(configs.mini(2), apply=dcr.APPLY_AUTO if apply == "auto" else APPLY[apply])
    p0 = c.plan.last_profile()
    assert p0.encode_valid == 0 and p0.apply_valid == 0
    c.plan.set_profiling(True)
    pl, size, _ = c.encode()
    t = c.target()
    rc, _ = dcr.apply(c.plan, dcr.RecvState(c.plan, 0), pl, size, t)
    assert rc == dcr.OK
    p = c.plan.last_profile()   # one read after encode and apply returns both
    assert p.encode_valid == 1 and p.apply_valid == 1
    assert p.encode_ms > 0 and p.apply_ms > 0 and p.finalize_ms >= 0 and p.pending_ms >= 0
    assert p.encode_ms < 1000 and p.apply_ms < 1000
    assert p.encode_kernels == 5
    assert p.apply_kernels in (FIRST_PHASE[apply] + 1, FIRST_PHASE[apply] + 4)
    c.plan.set_profiling(False)
    q = c.plan.last_profile()
    assert q.encode_valid == 0 and q.apply_valid == 0


def _flip_case(elem_bits, rows, cols, flips, seed=5, encoder=0):
    """One replicated tensor, old random, new = old XOR a non-zero byte at
    each canonical byte offset in `flips`; encode, compare with the oracle
    and apply both streams on the GPU."""
    t0 = configs.Tensor("e", elem_bits=elem_bits, rows=rows, cols=cols, split=configs.REPLICATED,
                        value_kind=synth.VAL_BYTES, rule=0, frac=0)
    wl = configs.Workload("edge", 1, 1, [t0]).layout()
    rng = np.random.RandomState(seed)
    old = rng.randint(0, 256, size=wl.shard_bytes[0]).astype(np.uint8)
    new = old.copy()
    for x in flips:
        new[x] ^= np.uint8(rng.randint(1, 256))
    orc = oracle.Oracle(wl)
    plan = dcr.Plan(descs_of(wl), encoder=encoder)
    d_old, d_new = to_device([old]), to_device([new])
    pl = torch.zeros(plan.window(0).payload_bound, dtype=torch.uint8, device="cuda")
    rc, size, counts = dcr.encode(plan, d_old, d_new, pl)
    assert rc == dcr.OK, dcr.last_error()
    g = pl[:size].cpu().numpy()
    o, oc = orc.encode([old], [new])
    check_structure(g)
    assert counts == [int(x) for x in oc]
    assert_same_frames(g, o)
    exp = orc.receiver_dense([new])
    for stream in (g, o):
        t = torch.zeros(max(exp.size, 16), dtype=torch.uint8, device="cuda")
        t[:exp.size] = torch.from_numpy(orc.receiver_dense([old])).cuda()
        rc, _ = dcr.apply(plan, dcr.RecvState(plan, 0), torch.from_numpy(stream).cuda(), stream.size, t)
        assert rc == dcr.OK, dcr.last_error()
        assert np.array_equal(t.cpu().numpy()[:exp.size], exp)
    return g, o


@pytest.mark.parametrize("shape", [(16, 1, 1, [0]), (16, 1, 1, [1]), (8, 1, 13, [0, 5, 12]),
                                   (8, 1, 13, list(range(13))), (16, 1, 32769, [7, 65536, 65537]),
                                   (8, 1, 65536, [65535]), (8, 1, 65537, [65536])])
def test_tiny_and_ragged_tensors(shape):
    bits, rows, cols, flips = shape
    _flip_case(bits, rows, cols, flips)


@pytest.mark.parametrize("encoder", [dcr.ENCODER_WIDE, dcr.ENCODER_DEEP, dcr.ENCODER_CTA])
def test_changes_near_the_end_of_a_chunk(encoder):
    # chunk i: one change i + 1 bytes before its end (the block's end rules:
    # last five bytes literal, no match starting in the last twelve), chunks
    # 20..39 the same after an early change (a long zero run to copy from),
    # chunk 40 its last five bytes changed, chunk 41 its last thirteen
    flips = []
    for i in range(20):
        flips.append(i * 65536 + 65536 - 1 - i)
    for i in range(20):
        flips += [(20 + i) * 65536 + 3, (20 + i) * 65536 + 65536 - 1 - i]
    flips += [40 * 65536 + 65536 - 1 - k for k in range(5)]
    flips += [41 * 65536 + 65536 - 1 - k for k in range(13)]
    g, o = _flip_case(8, 42, 65536, flips, encoder=encoder)
    assert len(frames_by_chunk(g)[1]) == 42


@pytest.mark.parametrize("make", ["dense_gate_stream", "record_stream"])
def test_overwrite_low_bit_rowgroup_hand_vectors(make):
    # the same hand-built overwrite streams the oracle is pinned with, applied
    # by the GPU retry path: 4- and 8-bit units land through the row-group remap
    import lowbit_vectors
    wl = configs.lowbit_pair()
    plan = dcr.Plan(descs_of(wl))
    pl, want = getattr(lowbit_vectors, make)(plan.info.plan_hash)
    d_pl = torch.from_numpy(pl).to("cuda")
    for _ in range(2):   # idempotent: a second apply leaves the same bytes
        tgt = torch.zeros(max(plan.info.recv_bytes, wl.recv_bytes), dtype=torch.uint8, device="cuda")
        st = dcr.RecvState(plan, 0)
        rc, res = dcr.apply_retry(plan, st, d_pl, pl.size, tgt)
        dcr.check(rc)
        rc, res = dcr.apply_retry(plan, dcr.RecvState(plan, 0), d_pl, pl.size, tgt)
        dcr.check(rc)
        assert np.array_equal(tgt.cpu().numpy()[:want.size], want)
