"""bench.py end to end on the GPU, short: one JSON line on stdout with every
key of the benchmark contract, a roofline object for the dominant kernel, the
end-to-end number through host buffers, the CPU baseline, the launch count
and the sampled clocks."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--steps", "3", "--warmup", "3", "--no-extra"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["scaling"] == "weak" and d["dtype"] == "bf16" and "workload" in d["config"]
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert 0.3 < rf["frac"] < 1.3, rf  # a plain read stream near the copy peak
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]
    ag = cb["agreement_with_gpu"]  # the oracle's rounds against the timed step's outputs
    # at least two trees are sampled; every difference from the oracle must be
    # a counted near-tie (builder) or near-boundary (draw) flip, and flips stay
    # rare
    assert ag["trees"] >= 2, ag
    assert ag["builder_mismatch"] == 0 and ag["draw_mismatch"] == 0, ag
    assert ag["builder_flips"] <= 2 and ag["draw_flips"] <= 1, ag
    assert ag["max_rel_err_exit_mass"] < 1e-5, ag
    rf_src = rf.get("duration_from", "")
    assert "second timed region" in rf_src, rf
    assert d["gpu_launches"] == 8 * 3
    assert d["clocks"]["sm_max_mhz"] > 0
