"""bench.py's JSON line on the GPU: one short decode_32k run checked against the line's
contract (the keys, the whole-job rate, the headline roofline taken from the step's
dominant kernel, the launch count from the step graph, the end-to-end copies)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_bench_line_contract():
    steps, warmup = 4, 3
    r = subprocess.run([sys.executable, "bench.py", "--steps", str(steps), "--warmup", str(warmup),
                        "--no-extras", "--no-cpu-baseline"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "rooflines", "gpu_launches", "clocks", "e2e", "kernel_ms"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    # whole-job rate: 32 query rows per step
    assert d["value"] == pytest.approx(32 / (d["ms_per_step"] * 1e-3), rel=1e-6)
    # two launches per step (the indexer, the one-call top-k + sparse MLA)
    assert d["gpu_launches"] == 2 * steps
    # the headline roofline is the kernel with the largest warm time of the step
    roof, allk = d["roofline"], d["rooflines"]
    assert roof["kernel"] == max(allk.values(), key=lambda x: x["ms"])["kernel"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    assert roof["achieved"] == pytest.approx(roof["algorithmic_bytes"] / (roof["ms"] * 1e-3) / 1e9)
    assert 0.05 < roof["frac"] < 1.2
    km = d["kernel_ms"]
    assert roof["ms"] in (km["indexer"], km.get("topk_and_sparse_mla_one_call"))
    # the calls overlap a little, so the step is at most the sum of its two launches
    assert d["ms_per_step"] <= 1.1 * (km["indexer"] + km["topk_and_sparse_mla_one_call"])
    # end to end: pinned host copies in both directions every step
    e2e = d["e2e"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert e2e["ms_per_step"] >= d["ms_per_step"] * 0.9
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
