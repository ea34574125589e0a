"""bench.py's JSON line on the GPU, on two quick invocations (the tiny prefill
workload and the split-KV decode, K steps only): one line of valid JSON with
the fields the benchmark contract names, positive rates, a roofline whose
fraction is the achieved rate over the peak, an end-to-end rate with its
copy sizes, the launch count, and the clock record."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + list(args), capture_output=True,
                         text=True, cwd=ROOT, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


@pytest.mark.parametrize("workload,unit,launches", [("tiny", "TFLOP/s", 1), ("decode", "GB/s", 2)])
def test_bench_line(workload, unit, launches):
    d = _bench("--workload", workload, "--steps", "4", "--warmup", "3", "--no-cpu-baseline", "--no-workloads")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["unit"] == unit and d["n_gpus"] == 1 and d["steps"] == 4 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["gpu_launches"] == launches * 4
    r = d["roofline"]
    assert r["bound"] in ("tensor", "hbm") and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert "sm_max_mhz" in d["clocks"] and "reasons" in d["clocks"]
    assert d["config"]["workload"]


def test_bench_line_with_every_workload():
    """The default run's extra objects on short settings: every other workload
    timed in the same process with its own roofline and clocks, the decode
    entries measured against the read probe as well, the sustained block."""
    d = _bench("--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--workload-steps", "3",
               "--sustained-seconds", "0.2")
    wl = d["workloads"]
    for name in ("train", "gqa", "long", "window", "decode", "decode_paged"):
        e = wl[name]
        assert e["value"] > 0 and e["steps"] == 3 and e["roofline"]["peak"] > 0, name
        assert abs(e["frac"] - e["roofline"]["achieved"] / e["roofline"]["peak"]) < 1e-9, name
        assert "sm_max_mhz" in e["clocks"], name
    for name in ("decode", "decode_paged"):
        assert wl[name]["read_gbs"] > 0 and wl[name]["frac_of_read"] > 0
    assert wl["read_probe"]["read_gbs"] > 0
    s = d["sustained"]
    assert s["value"] > 0 and s["steps"] >= 10 and "sm_mhz" in s["clocks"]
    assert d["e2e_serial"]["value"] > 0
