"""The benchmark's reference arm (the oracle on the host cores) as the base
contract wants its JSON line: one line, the decode workload's metric and
config, a cpu_baseline that describes the run, an e2e with no host-link
bytes.  Runs here: the arm touches no GPU."""
import json
import os
import subprocess
import sys

import bench
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "LOCAL_RANK", "WORLD_SIZE")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3", "--ref-seconds", "3"],
                       env=env, capture_output=True, text=True, timeout=240, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 3, 3)
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["vs_baseline"] is None
    assert d["data"] == "synthetic" and d["scaling"] == "weak"
    cfg = d["config"]
    for k, v in bench.decode_config(W.DECODE).items():
        assert cfg[k] == v, k
    assert cfg["seeds"]["layers"] == [W.DECODE.seed]
    n = cfg["tokens_per_step_sample"]
    assert 1 <= n <= W.DECODE.T
    # the value is the sampled tokens over the timed steps' wall time
    assert abs(d["value"] - n * 1000.0 / d["ms_per_step"]) <= 1e-6 * d["value"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"] and str(n) in cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
