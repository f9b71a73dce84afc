"""The benchmark's multi-rank path (one replica per GPU, max-over-ranks
timing) exercised on CPU with the gloo backend, world size 2."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, ws, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    env = bench.dist_env()
    bench.dist_barrier(ws)
    m = bench.dist_max(10.0 * (rank + 1) + 0.5, ws)
    q.put((rank, env, m))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(ws)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, m in out:
        assert env == (ws, rank, rank)
        assert m == 20.5


def test_single_rank_helpers_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_max(3.25, 1) == 3.25
    bench.dist_barrier(1)


# --------------------------------------------------------------------------
# ownership-sharded encode: partition, size exchange, layout, gather and
# header, with the oracle standing in for each rank's GPU encoder (blog, "A
# strong baseline with the Blackwell-native DE": ranks cover the checkpoint
# exactly once and only their compressed payloads are gathered)
# --------------------------------------------------------------------------
SHARD_CASES = [("mini", 2, 0), ("mini", 5, 0), ("mini", 3, 1), ("tp16", 0, 0)]


def _shard_worker(rank, ws, port, q):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import numpy as np
    import bit_exact_xor_gb300 as dcr
    import oracle
    from synth import configs
    from streamfmt import parse
    from wl import descs_of
    results = []
    try:
        for kind, n, mode in SHARD_CASES:
            wl = configs.mini(n) if kind == "mini" else configs.tp16()
            plan = dcr.Plan(descs_of(wl), window_bytes=wl.window_bytes, host_only=True)
            orc = oracle.Oracle(wl)
            assert plan.info.plan_hash == orc.plan_hash
            olds, news = wl.host_arenas()
            tgt = orc.receiver_dense(olds) if rank == 0 else None
            st = orc.state(0)
            omode = oracle.MODE_OVERWRITE_ONLY if mode else oracle.MODE_HYBRID
            for w in range(plan.n_windows):
                ref, _ = orc.encode(olds, news, window=w, mode=omode)
                hdr, frames, _ = parse(ref)
                pi = plan.part(w, rank, ws)
                mine = [f for f in frames if pi.chunk_begin <= f["chunk"] < pi.chunk_begin + pi.chunk_count]
                lens = [(32 + f["body_len"] + 15) // 16 * 16 for f in mine]
                size = (sum(lens), len(mine))

                def write(frame_offset, fr, ix):
                    # this rank's frames, position-independent, and their
                    # stream offsets (what dcr_encode_part_write does on a GPU)
                    o, offs = 0, []
                    for f, L in zip(mine, lens):
                        fr[o:o + L] = torch.from_numpy(ref[f["offset"]:f["offset"] + L].copy())
                        offs.append(frame_offset + o)
                        o += L
                    ix[:] = torch.from_numpy(np.array(offs, dtype="<u8").view(np.uint8))

                out = dcr.gather_stream(plan, w, rank, ws, size, write, 0, 1, mode=mode)
                if rank == 0:
                    got = out.numpy()
                    same = got.size == ref.size and bool(np.array_equal(got, ref))
                    rc = orc.apply(st, got, tgt, retry_only=bool(mode))
                    results.append((kind, n, w, same, rc))
            if rank == 0:
                results.append((kind, n, "final", bool(np.array_equal(tgt, orc.receiver_dense(news))), st.version))
        q.put((rank, results, None))
    except Exception as e:  # reported to the test process
        import traceback
        q.put((rank, None, traceback.format_exc()))
    dist.destroy_process_group()


def test_sharded_stream_assembled_by_gloo_equals_single_rank_stream():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_shard_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    out = {}
    for _ in range(ws):
        rank, res, err = q.get(timeout=300)
        assert err is None, err
        out[rank] = res
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res = out[0]
    assert res and out[1] == []
    for kind, n, w, a, b in res:
        if w == "final":
            assert a and b == 1, (kind, n)     # the assembled streams refit the receiver to `new`
        else:
            assert a, (kind, n, w)             # byte-identical to the oracle's single-rank stream
            assert b == 0, (kind, n, w, b)


def test_parts_cover_each_window_exactly_once_in_order():
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import bit_exact_xor_gb300 as dcr
    from synth import configs
    from wl import descs_of
    for wl in (configs.mini(2), configs.mini(5), configs.tp16(), configs.dense()):
        plan = dcr.Plan(descs_of(wl), window_bytes=wl.window_bytes, host_only=True)
        for w in range(plan.n_windows):
            wi = plan.window(w)
            for n in (1, 2, 3, 8, 64, 1000):
                parts = [plan.part(w, q, n) for q in range(n)]
                c = wi.chunk_begin
                for p in parts:
                    assert p.chunk_begin == c
                    c += p.chunk_count
                assert c == wi.chunk_begin + wi.chunk_count
                assert sum(p.canonical_bytes for p in parts) == wi.canonical_bytes
                nonempty = [p.canonical_bytes for p in parts if p.chunk_count]
                if n <= wi.chunk_count:   # balanced to within one chunk of the even share
                    assert max(nonempty) - min(nonempty) <= 2 * 65536
    # a TP=2 part reads only the shards its chunks need: the replicated tail
    # (norms, owned by shard 0) reads shard 0 alone
    plan = dcr.Plan(descs_of(configs.mini(2)), host_only=True)
    masks = {plan.part(0, q, 64).shard_mask for q in range(64)}
    assert masks <= {0, 1, 2, 3} and 3 in masks
    with pytest.raises(dcr.DcrError):
        plan.part(0, 2, 2)
    with pytest.raises(dcr.DcrError):
        plan.part(0, 0, dcr.MAX_PARTS + 1)


def test_stream_layout_and_header_follow_the_format():
    import struct
    import bit_exact_xor_gb300 as dcr
    fo, io, total = dcr.stream_layout([(48, 1), (0, 0), (96, 3)])
    assert fo == [64, 112, 112] and io == [208, 216, 216] and total == 240
    with pytest.raises(dcr.DcrError):
        dcr.stream_layout([(40, 1)])   # frames are 16-byte multiples
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from synth import configs
    from wl import descs_of
    plan = dcr.Plan(descs_of(configs.mini(5)), window_bytes=configs.mini(5).window_bytes, host_only=True)
    h = dcr.stream_header(plan, 2, 7, 8, 4, 160, mode=dcr.MODE_OVERWRITE_ONLY)
    magic, fmt, ph, bv, tv, win, flags, cb, cc, nf, tot = struct.unpack("<4sIQQQIIIIQQ", h)
    wi = plan.window(2)
    assert (magic, fmt, ph, bv, tv, win, flags) == (b"DCRS", 1, plan.info.plan_hash, 7, 8, 2, 1)
    assert (cb, cc, nf, tot) == (wi.chunk_begin, wi.chunk_count, 4, 64 + 160 + 32)
