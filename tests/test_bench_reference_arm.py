"""The reference arm of bench.py (the oracle timed on the host cores) prints
one JSON line with the same metric, unit and workload keys as the GPU arm,
a cpu_baseline describing the run and an e2e block with no device copies."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    sys.path.insert(0, ROOT)
    import bench
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    cfg = d["config"]
    assert cfg["workload"] == bench.WORKLOAD_TEXT["tiny"]
    for key in ("B", "T", "H", "d", "seed", "flops_per_step"):
        assert key in cfg
    assert cfg["d"] == 128 and cfg["flops_per_step"] == 4 * cfg["B"] * cfg["H"] * cfg["T"] ** 2 * 128
    assert "l2" in cfg
    # one head per worker process: the cores reported are the workers that ran
    assert cb["cores"] == min(cfg["H"], bench.host_cores())


def test_reference_arm_variant_flags_reach_the_config():
    sys.path.insert(0, ROOT)
    import bench
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "3", "--pcast", "1",
                        "--vsmooth", "0", "--reverse", "--S", "448", "--beta", "0.3"],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    cfg = json.loads(r.stdout.strip().splitlines()[-1])["config"]
    assert cfg["pcast"] == "ExpCast" and cfg["vsmooth"] is False and cfg["kv_order"] == "reverse"
    assert cfg["S"] == 448.0 and cfg["beta"] == 0.3
