"""Benchmark: bit-exact delta-compressed refit (encode + apply) on GB300.

One step = one full refit of the NVFP4 MoE block stack (hidden 6144, 64
experts, expert FFN 2048, 16 layers; e2m1 values packed two per byte with
e4m3 scales per 16; 20.25 GiB canonical, streamed in two windows of at most
16 GiB; 0.085 % of bytes changed; the receiver pairs gate/up rows in groups
of 64): per window dcr_encode (gather + XOR + count + LZ4 + frame
compaction) then dcr_apply on the receiver arena (decode + XOR in place
through the row-group remap + dedup + commit).  This is the largest of the
five workloads that fits one GPU.  Steps alternate direction (old->new,
new->old) so the receiver never needs a restore.  Inputs (2N = 43.5 GB read
per refit) are larger than L2; workloads small enough to stay in L2 get a
512 MiB buffer written before each timed step, outside that step's events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--workload moe|dense|single|gqa|sweep] [--frac F]
                  [--moe-layers L] [--window-mb M] [--codec lz4|snappy] [--overflow-kib K]
                  [--encoder auto|wide|deep|cta] [--apply auto|warp|cta|lane|split]
                  [--pipeline] [--abort-retry] [--shard] [--no-e2e] [--no-cpu-baseline]

Prints one JSON line.  --impl reference times the CPU oracle (the
benchmark's reference arm) on the same workload: each of its steps refits a
bounded sample of it (at most 640 MiB of the workload's own bytes), as does
the cpu_baseline leg of the GPU arm.  --moe-layers builds a shorter MoE stack
(the same tensors per layer) for profiler captures.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

METRIC = "encode & apply GB/s of weight bytes on 1 GB300 (% HBM peak); payload bytes"
UNIT = "GB/s"
L2_BYTES = 129 << 20        # GB300 L2
FLUSH_BYTES = 512 << 20


def l2_resident(n):
    """Whether an encode's inputs (old + new, 2n bytes) could still sit in L2
    from the previous step."""
    return 2 * n < 4 * L2_BYTES


WORKLOAD_NAMES = {
    "dense": "dense-tp2: bf16 transformer h1024 l24 ffn4096 v32768, TP=2 shards, 1% low-3-bit changes",
    "single": "single-bf16: one 4096x4096 bf16 tensor, 1% +-1..4 changes + 0.01% signed zeros",
    "gqa": "gqa-tp4: Llama GQA h4096 l32 32q/8kv hd128 ffn14336 v128256, TP=4, fused QKV residual, 3%",
    "sweep": "sweep: one 8 GiB bf16 buffer, +-1..4 changes",
    "moe": "nvfp4-moe: h6144 64 experts ffn2048 %d layers, e2m1 + e4m3 scales, 0.085%%, 16 GiB windows, "
           "receiver gate/up row groups of 64",
}


DEFAULT_FRAC = {"dense": 0.01, "single": 0.01, "gqa": 0.03, "sweep": 0.01, "moe": 0.00085}


def change_rate(args):
    """The changed fraction the run uses ("random" for the fully random new
    buffer of the sweep)."""
    if args.workload == "sweep" and args.frac is not None and args.frac >= 1.0:
        return "random"
    return args.frac if args.frac is not None else DEFAULT_FRAC[args.workload]


def build_workload(name, frac=None, moe_layers=16):
    from synth import configs
    if name == "dense":
        return configs.dense(frac=frac if frac is not None else 0.01)
    if name == "single":
        return configs.single(frac=frac if frac is not None else 0.01)
    if name == "gqa":
        return configs.gqa(frac=frac if frac is not None else 0.03)
    if name == "sweep":
        if frac is not None and frac >= 1.0:   # the incompressible case: a fully random new buffer
            return configs.sweep(random_new=True)
        return configs.sweep(frac=frac if frac is not None else 0.01)
    if name == "moe":
        return configs.nvfp4_moe(frac=frac if frac is not None else 0.00085, layers=moe_layers)
    raise SystemExit("unknown workload " + name)


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


PROFILED = {"dense": "encode_kernel_dense_tp2.md", "moe": "encode_kernel_nvfp4_moe.md"}
APPLY_VARIANTS = {"auto": 0, "warp": 1, "cta": 2, "lane": 3, "split": 4}   # dcr_plan_opts.apply
ENCODER_VARIANTS = {"auto": 0, "wide": 1, "deep": 2, "cta": 3}   # dcr_plan_opts.encoder


def ncu_traffic(args, bytes_per_launch):
    """Per-launch DRAM bytes (read + write) of the encode kernel from a
    committed ncu summary, or None.  Only for a workload that has one (its own
    change rate, LZ4, its own windows) and only while encode.cu is the source
    that was profiled.  A capture taken on a shorter stack of the same
    tensors (same dtype mix and change rate) is scaled to this run's
    canonical bytes per launch."""
    if args.workload not in PROFILED or (args.frac, args.codec, args.window_mb) != (None, "lz4", 0):
        return None
    path = os.path.join(ROOT, "profiles", PROFILED[args.workload])
    src = os.path.join(ROOT, "bit_exact_xor_gb300", "csrc", "encode.cu")
    try:
        text = open(path).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        keys = ("traffic_bytes_per_launch", "canonical_bytes_per_launch", "encode_cu_sha256_16")
        fields = {k.strip(): v.strip() for k, v in (l.split(":", 1) for l in text.splitlines()
                                                    if l.startswith(keys))}
        if fields.get("encode_cu_sha256_16") != sha:
            return None
        t = int(fields["traffic_bytes_per_launch"])
        c = int(fields.get("canonical_bytes_per_launch", bytes_per_launch))
        return int(round(t * bytes_per_launch / c))
    except Exception:
        return None


class Clocks:
    """nvidia-smi sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
        return self

    def __exit__(self, *a):
        self.rows = []
        if self.p is None:
            return
        time.sleep(0.25)
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except Exception:
            self.p.kill()
            out = ""
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def summary(self):
        if not getattr(self, "rows", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# --------------------------------------------------------------------------
# multi-process helpers (one rank per GPU, replicas of the single-GPU refit)
# --------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_max(value, ws):
    """Maximum of a float over ranks (identity for one rank)."""
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------
# CPU oracle leg (baseline and reference arm)
# --------------------------------------------------------------------------
def oracle_runner(wl, threads, codec="lz4"):
    import numpy as np
    import oracle
    orc = oracle.Oracle(wl)
    oc = oracle.CODEC_SNAPPY if codec == "snappy" else oracle.CODEC_LZ4
    olds, news = wl.host_arenas()
    tgt = orc.receiver_dense(olds)
    state = {"st": orc.state(0), "dir": 0, "v": 0}

    def step():
        a, b = (olds, news) if state["dir"] == 0 else (news, olds)
        total = 0
        for w in range(orc.n_windows):
            pl, _ = orc.encode(a, b, window=w, base_version=state["v"], target_version=state["v"] + 1,
                               threads=threads, codec=oc)
            rc = orc.apply(state["st"], pl, tgt, threads=threads)
            assert rc == oracle.OK, rc
            total += pl.size
        state["v"] += 1
        state["dir"] ^= 1
        return total

    return step


ORACLE_SAMPLE_BYTES = 640 << 20    # bytes of the workload one oracle step refits at most


def oracle_sample(wl):
    """(sample workload, description): the workload itself if it is small,
    else a bounded sample of its own bytes (same generator streams)."""
    from synth import configs
    return configs.sample(wl, ORACLE_SAMPLE_BYTES)


def cpu_baseline(wl, budget_s=12.0, codec="lz4"):
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    swl, what = oracle_sample(wl)
    step = oracle_runner(swl, threads, codec)
    n, t0, payload = 0, time.perf_counter(), 0
    while True:
        payload = step()
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    out = {"value": round(swl.canonical_bytes * n / dt / 1e9, 4), "unit": UNIT, "cores": threads,
           "kind": "oracle", "sample": "%d full refit steps (encode+apply) of %s, %.1f s" % (n, what, dt),
           "payload_bytes": payload, "sample_bytes": swl.canonical_bytes, "sample_workload": swl,
           "sample_what": what}
    # the same oracle on one thread, for one step, when that stays bounded
    est = dt / n * threads
    if threads == 1:
        out["value_1_thread"] = out["value"]
    elif est <= 30.0:
        one = oracle_runner(swl, 1, codec)
        t0 = time.perf_counter()
        one()
        d1 = time.perf_counter() - t0
        out["value_1_thread"] = round(swl.canonical_bytes / d1 / 1e9, 4)
        out["sample_1_thread"] = "1 full refit step of the same sample on one thread, %.1f s" % d1
    else:
        out["value_1_thread"] = None
        out["sample_1_thread"] = "not run: one step on one thread would take about %.0f s" % est
    return out


def run_config(args, wl, nw, ws):
    """The workload description both arms print."""
    N = wl.canonical_bytes
    name = WORKLOAD_NAMES[args.workload]
    if args.workload == "moe":
        name = name % args.moe_layers
    if args.frac is not None:
        name += " [change rate set to %s]" % ("a fully random new buffer" if change_rate(args) == "random"
                                             else "%g%%" % (100 * args.frac))
    return {"workload": name, "change_rate": change_rate(args), "canonical_bytes": N, "codec": getattr(args, "codec", "lz4"),
            "encoder": getattr(args, "encoder", "auto"), "apply": getattr(args, "apply", "auto"),
            "tp": wl.tp, "windows": nw, "parallelism": "replicas" if ws > 1 else "single GPU",
            "l2": "L2 flushed before each timed step (%d MiB written outside the step's events)" % (FLUSH_BYTES >> 20)
            if l2_resident(N) else "inputs larger than L2 (2N = %.2f GB read per encode)" % (2 * N / 1e9)}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    wl = build_workload(args.workload, args.frac, args.moe_layers)
    swl, what = oracle_sample(wl)
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    step = oracle_runner(swl, threads, args.codec)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = swl.canonical_bytes * args.steps / dt / 1e9
    sample = "each step one full oracle refit (encode+apply) of %s" % what
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": run_config(args, wl, oracle.Oracle(wl).n_windows, 1),
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": "%d timed steps; %s" % (args.steps, sample)},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    line["config"]["oracle_sample"] = sample
    line["config"]["oracle_sample_bytes"] = swl.canonical_bytes
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------
def run_gpu(args):
    import torch

    import bit_exact_xor_gb300 as dcr
    from wl import descs_of

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()

    wl = build_workload(args.workload, args.frac, args.moe_layers)
    N = wl.canonical_bytes
    plan = dcr.Plan(descs_of(wl), window_bytes=(args.window_mb << 20) or wl.window_bytes,
                    codec=dcr.CODEC_SNAPPY if args.codec == "snappy" else dcr.CODEC_LZ4,
                    overflow_kib=dcr.NO_OVERFLOW if args.overflow_kib < 0 else args.overflow_kib,
                    apply=APPLY_VARIANTS[args.apply], encoder=ENCODER_VARIANTS[args.encoder])
    plan.set_profiling(True)
    olds, news = wl.device_arenas(torch)
    target = torch.empty(max(plan.info.recv_bytes, wl.recv_bytes), dtype=torch.uint8, device=dev)
    dcr.check(dcr.dense_refit(plan, olds, target))
    nw = plan.n_windows
    caps = [plan.window(w).payload_bound for w in range(nw)]
    # payload buffers sized from a first encode (grown to the reported size)
    payloads = []
    for w in range(nw):
        guess = max(plan.window(w).canonical_bytes // 8, 1 << 20)
        buf = torch.empty(guess, dtype=torch.uint8, device=dev)
        rc, size, _ = dcr.encode(plan, olds, news, buf, window=w)
        if rc == dcr.ERR_CAPACITY:
            buf = torch.empty(min(int(size * 1.25), caps[w]), dtype=torch.uint8, device=dev)
        payloads.append(buf)
    st = dcr.RecvState(plan, 0)
    ver = [0]
    d = [0]
    enc_ms, app_ms, rest_ms, sizes, changed, launches = [], [], [], [], [], []
    parts_ms = {"encode_kernel": [], "encode_write_pass": [], "apply_first_kernel": [], "apply_deferred_kernels": [],
                "commit_check": []}

    sh = stream.cuda_stream

    def step(record, counts=False):
        a, b = (olds, news) if d[0] == 0 else (news, olds)
        for w in range(nw):
            rc, size, cnt = dcr.encode(plan, a, b, payloads[w], window=w, base_version=ver[0],
                                       target_version=ver[0] + 1, counts=counts, stream=sh)
            dcr.check(rc)
            rc, res = dcr.apply(plan, st, payloads[w], size, target, stream=sh)
            dcr.check(rc)
            if record:
                p = plan.last_profile()   # this window's encode and apply kernels
                enc_ms.append(p.encode_ms)
                app_ms.append(p.apply_ms + p.defer_ms)
                rest_ms.append(p.finalize_ms + p.pending_ms)
                for k, v in zip(parts_ms, (p.encode_ms, p.finalize_ms, p.apply_ms, p.defer_ms, p.pending_ms)):
                    parts_ms[k].append(v)
                launches.append(p.encode_kernels + p.apply_kernels)
                sizes.append(size)
            if counts:
                changed.append(sum(cnt))
        ver[0] += 1
        d[0] ^= 1

    # per-tensor changed counts from the last warm-up step (the same in both
    # directions), so the timed steps do not read them back
    for i in range(args.warmup):
        step(False, counts=i == args.warmup - 1)
    # inputs that could stay in L2 between steps: write a 512 MiB buffer
    # before each timed step, outside that step's events
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if l2_resident(N) else None
    torch.cuda.synchronize()
    dist_barrier(ws)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    spans = []
    with Clocks(local) as clk:
        torch.cuda.synchronize()
        ev0.record(stream)
        for i in range(args.steps):
            if flush is not None:
                flush.fill_(i & 0xFF)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                step(True)
                b.record(stream)
                spans.append((a, b))
            else:
                step(True)
        ev1.record(stream)
        torch.cuda.synchronize()
    dist_barrier(ws)
    ms = sum(a.elapsed_time(b) for a, b in spans) if spans else ev0.elapsed_time(ev1)
    del flush
    ms_max = dist_max(ms, ws)
    value = N * args.steps * ws / (ms_max / 1e3) / 1e9

    # end to end through the public API with host buffers: H2D of old/new,
    # encode, D2H of the payload, H2D of the payload, apply (status read
    # inside).  Each step's inputs are copied on a second stream while the
    # previous step computes (two device input buffers); every copy of every
    # timed step, the first one included, is inside the timed region.
    e2e = None
    if not args.no_e2e:
        def pinned_copy(x):   # straight into pinned memory: no pageable staging copy
            h = torch.empty(x.numel(), dtype=torch.uint8, pin_memory=True)
            h.copy_(x)
            return h

        h_old = [pinned_copy(x) for x in olds]
        h_new = [pinned_copy(x) for x in news]
        h_pl = [torch.empty(p.numel(), dtype=torch.uint8, pin_memory=True) for p in payloads]
        d_in = [([torch.empty_like(x) for x in olds], [torch.empty_like(x) for x in news]) for _ in range(2)]
        rx = [torch.empty_like(p) for p in payloads]
        cs = torch.cuda.Stream()
        h2d = d2h = 0

        def copy_inputs(slot, direction):
            nonlocal h2d
            a, b = (h_old, h_new) if direction == 0 else (h_new, h_old)
            with torch.cuda.stream(cs):
                for x, y in zip(d_in[slot][0], a):
                    x.copy_(y, non_blocking=True)
                for x, y in zip(d_in[slot][1], b):
                    x.copy_(y, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cs)
            h2d += sum(y.numel() for y in a) + sum(y.numel() for y in b)
            return ev

        def e2e_steps(k):
            nonlocal d2h, h2d
            cs.wait_stream(stream)   # the first copy starts after the timer's start event
            ready = copy_inputs(0, d[0])
            for i in range(k):
                slot = i & 1
                stream.wait_event(ready)
                if i + 1 < k:   # the next step's inputs, into the other buffer (free: its step returned)
                    ready = copy_inputs(slot ^ 1, d[0] ^ 1)
                for w in range(nw):
                    rc, size, _ = dcr.encode(plan, d_in[slot][0], d_in[slot][1], payloads[w], window=w,
                                             base_version=ver[0], target_version=ver[0] + 1, counts=False,
                                             stream=sh)
                    dcr.check(rc)
                    h_pl[w][:size].copy_(payloads[w][:size], non_blocking=True)
                    rx[w][:size].copy_(h_pl[w][:size], non_blocking=True)
                    d2h += size
                    h2d += size
                    rc, res = dcr.apply(plan, st, rx[w], size, target, stream=sh)
                    dcr.check(rc)
                ver[0] += 1
                d[0] ^= 1

        e2e_steps(2)
        h2d = d2h = 0
        torch.cuda.synchronize()
        dist_barrier(ws)
        k = max(2, min(args.steps, 5))
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        e2e_steps(k)
        t1.record(stream)
        torch.cuda.synchronize()
        ems = dist_max(t0.elapsed_time(t1), ws)
        per_step_h2d, per_step_d2h = h2d // k, d2h // k
        # the host link on its own: the same input copies with nothing else
        # running, timed on the copy stream (context for the e2e figure; it
        # varies between boxes and between runs)
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(cs)
        for i in range(2):
            copy_inputs(i & 1, i & 1)
        c1.record(cs)
        torch.cuda.synchronize()
        link = 2 * sum(x.numel() for x in h_old + h_new) / (c0.elapsed_time(c1) / 1e3) / 1e9
        e2e = {"value": round(N * k * ws / (ems / 1e3) / 1e9, 3), "unit": UNIT,
               "h2d_bytes_per_step": per_step_h2d, "d2h_bytes_per_step": per_step_d2h,
               "host_link_h2d_gbs": round(link, 1)}
        del h_old, h_new, d_in

    # pipelined refit of every window through pinned host memory
    # (dcr_refit_pipelined) against the same windows in series: encode, copy
    # the stream to host and back, apply (one GPU, rank 0 of a single run)
    pipe = None
    if args.pipeline and ws == 1:
        dev_b, host_b = dcr.pipeline_sizes(plan)
        pdev = torch.empty(dev_b, dtype=torch.uint8, device=dev)
        phost = torch.empty(host_b, dtype=torch.uint8).pin_memory()
        stage = [torch.empty(p.numel(), dtype=torch.uint8).pin_memory() for p in payloads]
        rxs = [torch.empty_like(p) for p in payloads]
        last = {}

        def serial_refit():
            a, b = (olds, news) if d[0] == 0 else (news, olds)
            for w in range(nw):
                rc, size, _ = dcr.encode(plan, a, b, payloads[w], window=w, base_version=ver[0],
                                         target_version=ver[0] + 1, counts=False, stream=sh)
                dcr.check(rc)
                stage[w][:size].copy_(payloads[w][:size], non_blocking=True)
                rxs[w][:size].copy_(stage[w][:size], non_blocking=True)
                rc, _ = dcr.apply(plan, st, rxs[w], size, target, stream=sh)
                dcr.check(rc)
            ver[0] += 1
            d[0] ^= 1

        def piped_refit():
            a, b = (olds, news) if d[0] == 0 else (news, olds)
            rc, stats, _ = dcr.refit_pipelined(plan, st, a, b, target, pdev, phost, base_version=ver[0],
                                               target_version=ver[0] + 1, counts=False, stream=sh)
            dcr.check(rc)
            assert stats.committed == 1
            last["payload"] = stats.payload_bytes
            ver[0] += 1
            d[0] ^= 1

        def timed(fn, k):
            for _ in range(2):
                fn()
            torch.cuda.synchronize()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for _ in range(k):
                fn()
            a1.record(stream)
            torch.cuda.synchronize()
            return a0.elapsed_time(a1) / k

        k = max(2, min(args.steps, 5))
        ser_ms = timed(serial_refit, k)
        pip_ms = timed(piped_refit, k)
        pipe = {"windows": nw, "value": round(N / (pip_ms / 1e3) / 1e9, 3), "unit": UNIT,
                "ms_per_refit": round(pip_ms, 4), "serial_ms_per_refit": round(ser_ms, 4),
                "payload_bytes_per_refit": int(last["payload"])}
        del pdev, phost, stage, rxs

    # abort and retry: per window the hybrid stream is applied with a fault
    # injected at half its frames, then the same change set is re-encoded in
    # overwrite-only mode and applied with dcr_apply_retry (one GPU)
    retry = None
    if args.abort_retry and ws == 1:
        rpay = []
        for w in range(nw):   # overwrite-only stream buffers sized from a first encode
            buf = torch.empty(max(plan.window(w).canonical_bytes // 6, 1 << 20), dtype=torch.uint8, device=dev)
            rc, rsize, _ = dcr.encode(plan, olds, news, buf, window=w, mode=dcr.MODE_OVERWRITE_ONLY, counts=False)
            if rc == dcr.ERR_CAPACITY:
                buf = torch.empty(min(int(rsize * 1.25), caps[w]), dtype=torch.uint8, device=dev)
            rpay.append(buf)
        rlast = {}

        def abort_retry_refit():
            a, b = (olds, news) if d[0] == 0 else (news, olds)
            rbytes = 0
            for w in range(nw):
                rc, size, _ = dcr.encode(plan, a, b, payloads[w], window=w, base_version=ver[0],
                                         target_version=ver[0] + 1, counts=False, stream=sh)
                dcr.check(rc)
                nf = int(payloads[w][48:56].cpu().numpy().view("<u8")[0])
                rc, _ = dcr.apply(plan, st, payloads[w], size, target, fault=(nf // 2, 1000), stream=sh)
                assert rc == dcr.ERR_ABORTED, rc
                rc, rsize, _ = dcr.encode(plan, a, b, rpay[w], window=w, mode=dcr.MODE_OVERWRITE_ONLY,
                                          base_version=ver[0], target_version=ver[0] + 1, counts=False, stream=sh)
                dcr.check(rc)
                rc, res = dcr.apply_retry(plan, st, rpay[w], rsize, target, stream=sh)
                dcr.check(rc)
                rbytes += rsize
            assert st.version == ver[0] + 1
            rlast["bytes"] = rbytes
            ver[0] += 1
            d[0] ^= 1

        k = max(2, min(args.steps, 5))
        for _ in range(2):
            abort_retry_refit()
        torch.cuda.synchronize()
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        r0.record(stream)
        for _ in range(k):
            abort_retry_refit()
        r1.record(stream)
        torch.cuda.synchronize()
        rms = r0.elapsed_time(r1) / k
        # the retry stream alone, both ways: encoded again from old and new
        # (overwrite-only mode) or built from the XOR stream and new
        # (dcr_encode_retry, no read of old); same bytes
        a, b = (olds, news) if d[0] == 0 else (news, olds)
        xs = []
        for w in range(nw):
            rc, size, _ = dcr.encode(plan, a, b, payloads[w], window=w, counts=False, stream=sh)
            dcr.check(rc)
            xs.append(size)

        def time_retry(from_xor):
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(k):
                for w in range(nw):
                    if from_xor:
                        rc, _ = dcr.encode_retry(plan, payloads[w], xs[w], b, rpay[w], stream=sh)
                    else:
                        rc, _, _ = dcr.encode(plan, a, b, rpay[w], window=w, mode=dcr.MODE_OVERWRITE_ONLY,
                                              counts=False, stream=sh)
                    dcr.check(rc)
            t1.record(stream)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1) / k

        time_retry(True)
        ms_ow, ms_x = time_retry(False), time_retry(True)
        retry = {"ms_per_refit": round(rms, 4), "value": round(N / (rms / 1e3) / 1e9, 3), "unit": UNIT,
                 "abort": "half of each window's frames applied, one split mid-frame",
                 "retry_payload_bytes_per_refit": int(rlast["bytes"]),
                 "retry_stream_ms": {"from_old_and_new": round(ms_ow, 4), "from_xor_stream_and_new": round(ms_x, 4)}}
        del rpay

    # ownership-sharded encode: rank r encodes part r of every window on its
    # GPU, the compressed parts are gathered to rank 0 (all-gather of sizes,
    # gather of the frames), which applies the assembled stream
    shard = None
    if args.shard:
        from wl import descs_of as _descs
        import torch.distributed as dist
        if ws == 1 and not dist.is_initialized():
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            os.environ.setdefault("MASTER_PORT", "29512")
            dist.init_process_group("nccl", rank=0, world_size=1, device_id=dev)
        splan = dcr.Plan(_descs(wl), window_bytes=(args.window_mb << 20) or wl.window_bytes,
                         codec=dcr.CODEC_SNAPPY if args.codec == "snappy" else dcr.CODEC_LZ4)
        slast = {}

        def sharded_refit():
            a, b = (olds, news) if d[0] == 0 else (news, olds)
            pbytes = 0
            for w in range(nw):
                rc, sz, _ = dcr.encode_part(splan, a, b, rank, ws, window=w, counts=False, stream=sh)
                dcr.check(rc)

                def write(fo, fr, ix):
                    dcr.check(dcr.encode_part_write(splan, fo, fr, fr.numel(), ix, stream=sh))

                out = dcr.gather_stream(splan, w, rank, ws, sz, write, ver[0], ver[0] + 1, device=dev)
                if rank == 0:
                    rc, _ = dcr.apply(plan, st, out, out.numel(), target, stream=sh)
                    dcr.check(rc)
                    pbytes += out.numel()
            ver[0] += 1
            d[0] ^= 1
            slast["payload"] = pbytes

        k = max(2, min(args.steps, 5))
        for _ in range(2):
            sharded_refit()
        torch.cuda.synchronize()
        dist_barrier(ws)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(k):
            sharded_refit()
        s1.record(stream)
        torch.cuda.synchronize()
        sms = dist_max(s0.elapsed_time(s1) / k, ws)
        shard = {"parts": ws, "ms_per_refit": round(sms, 4), "value": round(N / (sms / 1e3) / 1e9, 3),
                 "unit": UNIT, "payload_bytes_per_refit": int(slast["payload"]) if rank == 0 else None,
                 "exchange": "all-gather of part sizes, gather of compressed parts to rank 0 (torch.distributed)"}
        splan.close()

    # the receiver really holds the last step's target weights
    # (with --shard only rank 0 applied the sharded refits)
    if not (shard and rank != 0):
        ref = torch.empty_like(target)
        dcr.check(dcr.dense_refit(plan, olds if d[0] == 0 else news, ref))
        assert torch.equal(ref, target), "receiver arena differs from a dense refit"
        del ref

    P = statistics.mean(sizes)
    peak, peak_kind = measured_peak()
    alg_bytes = 2 * N / nw + P  # per encode launch: read old+new of the window, write payload
    achieved = alg_bytes / (statistics.mean(enc_ms) / 1e3) / 1e9
    traffic = ncu_traffic(args, N / nw)
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": run_config(args, wl, nw, ws),
        "encode_gbs": round(N / (statistics.mean(enc_ms) * nw / 1e3) / 1e9, 3),
        "apply_gbs": round(N / (statistics.mean(app_ms) * nw / 1e3) / 1e9, 3),
        "encode_kernel_ms": round(statistics.mean(enc_ms), 4),
        "apply_kernel_ms": round(statistics.mean(app_ms), 4),
        # the rest of the library's GPU time per window: frame scan, copy and
        # spill kernels after the encode, commit check after the apply
        "other_kernels_ms": round(statistics.mean(rest_ms), 4),
        # per window, by launch group: the encoder's main kernel; its scan,
        # copy and second-pass kernels; the first apply kernel; the deferred
        # frame kernels; the commit check
        "kernel_ms_by_group": {k: round(statistics.mean(v), 4) for k, v in parts_ms.items()},
        # apply against the dense byte model (reads N + P, writes N)
        "apply_model_frac": round((2 * N / nw + P) / (statistics.mean(app_ms) / 1e3) / 1e9 / peak, 4),
        "payload_bytes": int(P), "changed_values": int(statistics.mean(changed)) if changed else None,
        "roofline": {"bound": "hbm", "kernel": "encode_kernel", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": int(alg_bytes)},
        # the library's kernels in the timed steps, as its calls report them
        "gpu_launches": int(sum(launches)),
        "clocks": clocks,
    }
    if e2e:
        line["e2e"] = e2e
    if pipe:
        line["pipelined"] = pipe
    if retry:
        line["abort_retry"] = retry
    if shard:
        line["sharded"] = shard
    if rank == 0 and not args.no_cpu_baseline:
        cb = cpu_baseline(wl, codec=args.codec)
        # payload against the oracle's on identical bytes: the GPU encodes the
        # oracle's sample too (one refit, old -> new)
        swl = cb.pop("sample_workload")
        if swl is wl:
            gpu_sample_payload = P * nw
        else:
            splan = dcr.Plan(descs_of(swl), window_bytes=swl.window_bytes,
                             codec=dcr.CODEC_SNAPPY if args.codec == "snappy" else dcr.CODEC_LZ4)
            so, sn = swl.device_arenas(torch)
            gpu_sample_payload = 0
            for w in range(splan.n_windows):
                buf = torch.empty(splan.window(w).payload_bound, dtype=torch.uint8, device=dev)
                rc, size, _ = dcr.encode(splan, so, sn, buf, window=w, counts=False)
                dcr.check(rc)
                gpu_sample_payload += size
            del so, sn, buf
            splan.close()
        line["payload_vs_oracle"] = round(gpu_sample_payload / cb.pop("payload_bytes"), 4)
        line["payload_vs_oracle_on"] = "the oracle's sample: " + cb.pop("sample_what")
        line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line))
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="moe", choices=sorted(WORKLOAD_NAMES))
    ap.add_argument("--moe-layers", type=int, default=16, help="layers of the MoE stack (profiler captures)")
    ap.add_argument("--frac", type=float, default=None,
                    help="change rate (sweep: 1 or more = fully random new buffer)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--window-mb", type=int, default=0, help="window size in MiB (0: the workload's)")
    ap.add_argument("--codec", default="lz4", choices=["lz4", "snappy"], help="block codec of the XOR masks")
    ap.add_argument("--encoder", default="auto", choices=sorted(ENCODER_VARIANTS),
                    help="encoder kernel: auto, wide (warp per chunk), deep (warp per chunk, 12 landing "
                         "stages), cta (CTA per chunk)")
    ap.add_argument("--apply", default="auto", choices=sorted(APPLY_VARIANTS),
                    help="apply kernels: auto, warp (one warp per frame), cta (one CTA per frame), "
                         "lane (one thread per ZSRC frame)")
    ap.add_argument("--overflow-kib", type=int, default=0,
                    help="encoder overflow heap in KiB (0: one eighth of the window, -1: none)")
    ap.add_argument("--abort-retry", action="store_true",
                    help="also time refits aborted at half the frames and completed by the overwrite-only retry")
    ap.add_argument("--pipeline", action="store_true",
                    help="also time dcr_refit_pipelined against the same windows in series")
    ap.add_argument("--shard", action="store_true",
                    help="also time the ownership-sharded encode: each rank encodes its part of every window, "
                         "the compressed parts are gathered to rank 0, which applies them")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
