"""The benchmark's one-GPU line end to end: a short run of bench.py with
every key the line promises (headline, roofline, end to end, clocks) and an
`extras` row for every other forward and backward workload it times."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_bench_line_has_every_key_and_extras_row():
    import bench
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3",
                          "--warmup", "3", "--no-cpu-baseline", "--e2e-steps", "2",
                          "--extra-steps", "2", "--extra-warmup", "1"],
                         cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "gpu_launches", "roofline", "e2e", "clocks", "extras"):
        assert key in d, key
    assert d["value"] > 0 and d["n_gpus"] == 1 and d["gpu_launches"] == 3
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9 and "traffic_source" in r
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == 3 * 8 * 32 * 8192 * 64 * 2
    assert e["d2h_bytes_per_step"] == 8 * 32 * 8192 * (64 * 2 + 4)
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    want = {("fwd", w.name) for w in bench.EXTRA_FWD} | {("bwd", w.name) for w in bench.EXTRA_BWD}
    got = {(x["pass"], x["workload"]) for x in d["extras"]}
    assert got == want
    for x in d["extras"]:
        assert x["kernel_ms"] > 0 and x["tflops"] > 0 and 0 < x["frac"] < 1.5, x
        assert "sm_mhz" in x["clocks"]
