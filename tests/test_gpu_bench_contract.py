"""bench.py's output line: one JSON object with the keys and types its
readers depend on, for both arms, on the tiny list (a few seconds)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                         cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_our_arm_line():
    d = run_bench("--workload", "tiny", "--steps", "3", "--warmup", "3",
                  "--e2e-steps", "2", "--cpu-seconds", "1", "--no-other-configs")
    for k, t in (("metric", str), ("value", float), ("unit", str), ("n_gpus", int),
                 ("steps", int), ("warmup", int), ("ms_per_step", float),
                 ("higher_is_better", bool), ("scaling", str), ("dtype", str),
                 ("data", str), ("config", dict), ("roofline", dict),
                 ("e2e", dict), ("cpu_baseline", dict), ("clocks", dict),
                 ("gpu_launches", int)):
        assert isinstance(d[k], t), k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"]
    assert d["vs_baseline"] is None and d["config"]["workload"] == "tiny"
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] == 4
    # the link measured alone and the loop's own copies, beside the loop
    assert e["link_copy_ms"] > 0 and e["link_gbs"] > 0
    lc = e["loop_copy_ms"]
    assert 0 < lc["min"] <= lc["median"] <= lc["max"]
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0
    assert d["gpu_launches"] == 3 * d["steps"]      # cast amax, fused pass, update
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])


def test_reference_arm_line():
    d = run_bench("--impl", "reference", "--workload", "tiny", "--steps", "2",
                  "--warmup", "1")
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
