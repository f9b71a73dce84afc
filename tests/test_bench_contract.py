"""bench.py's reference arm (the CPU oracle timed on the host cores) prints
one JSON line with the keys the benchmark contract asks for; runs on a
machine without a GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "single", "--steps", "1", "--warmup", "1"],
                         stdout=subprocess.PIPE, stderr=subprocess.PIPE, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr.decode()[-2000:]
    lines = [l for l in out.stdout.decode().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["warmup"] >= 3 and d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["config"]["workload"].startswith("single")
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def _bench():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    return bench


def test_ncu_traffic_only_for_the_profiled_configuration():
    import argparse
    bench = _bench()
    for wl in ("dense", "moe"):
        base = dict(workload=wl, frac=None, codec="lz4", window_mb=0)
        t = bench.ncu_traffic(argparse.Namespace(**base), 1 << 30)
        assert t is None or t > 0   # None once encode.cu changed since the capture
        for k, v in (("frac", 0.03), ("codec", "snappy"), ("window_mb", 64)):
            assert bench.ncu_traffic(argparse.Namespace(**dict(base, **{k: v})), 1 << 30) is None, k
    assert bench.ncu_traffic(argparse.Namespace(workload="gqa", frac=None, codec="lz4", window_mb=0),
                             1 << 30) is None


def test_default_workload_is_the_largest_single_gpu_config():
    bench = _bench()
    from synth import configs
    sizes = {w: bench.build_workload(w).canonical_bytes for w in bench.WORKLOAD_NAMES}
    assert max(sizes, key=sizes.get) == "moe"
    import argparse
    ap_default = [a for a in open(os.path.join(ROOT, "bench.py")).read().splitlines()
                  if '"--workload", default=' in a]
    assert ap_default and 'default="moe"' in ap_default[0]


def test_oracle_sample_holds_the_workloads_own_bytes():
    import numpy as np
    from synth import configs
    for wl, budget in ((configs.mini(5), 200000), (configs.mini(3), 100000), (configs.mini(4), 300000)):
        s, what = configs.sample(wl, budget)
        assert s.canonical_bytes <= max(budget, wl.tensors[0].nbytes) and what
        olds, news = wl.host_arenas()
        so, sn = s.host_arenas()
        for t, u in zip(s.tensors, wl.tensors):
            for r in t.holders(wl.tp):
                lb = t.local_bytes(wl.tp)
                assert np.array_equal(so[r][t.shard_offset[r]:t.shard_offset[r] + lb],
                                      olds[r][u.shard_offset[r]:u.shard_offset[r] + lb])
                assert np.array_equal(sn[r][t.shard_offset[r]:t.shard_offset[r] + lb],
                                      news[r][u.shard_offset[r]:u.shard_offset[r] + lb])
