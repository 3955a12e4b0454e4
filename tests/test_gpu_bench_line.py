"""The bench line's contract on a GPU: one JSON line with the metric, the timing
fields, the roofline of the dominant kernel, per-kernel durations with the
attention's two roofline terms, the clock record, the end-to-end figure through the
binding and, where an input set fits in L2, the hot-L2 figure. Runs the small
float32 workload and the LLaDA-shaped layer (bf16 tensor-core path) for a few
hundred steps each."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _line(workload, steps=300):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", workload,
                        "--steps", str(steps), "--warmup", "5", "--no-cpu-baseline"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


@pytest.mark.parametrize("workload,dtype", [("tiny", "f32"), ("llada", "bf16")])
def test_bench_line(workload, dtype):
    d = _line(workload)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "kernels", "gpu_launches", "clocks", "e2e"):
        assert k in d, k
    assert d["steps"] == 300 and d["warmup"] >= 3 and d["n_gpus"] == 1 and d["dtype"] == dtype
    assert d["value"] > 0 and abs(d["value"] * d["ms_per_step"] / 1000.0 - 1.0) < 1e-6
    assert d["gpu_launches"] >= 2 * d["steps"]
    ka, kc = d["kernels"]["block_attn"], d["kernels"]["commit"]
    # the attention is the step less the commit
    assert ka["us"] + kc["us"] == pytest.approx(d["ms_per_step"] * 1000.0, rel=1e-6)
    rt = ka["roofline"]
    assert rt["hbm_us"] > 0 and rt["bound"] in ("hbm", "tensor")
    assert (rt["tensor_us"] is None) == (dtype == "f32")
    assert 0 < rt["frac_of_roofline"] <= 1.5
    roof = d["roofline"]
    assert roof["bound"] == "hbm" and roof["peak"] > 0
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"], rel=1e-9)
    assert d["e2e"]["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] > 0
    assert d["e2e"]["d2h_bytes_per_step"] > 0
    hot = d.get("hot_l2")
    assert hot is not None and hot["us_per_step"] > 0  # both input sets fit in half of L2
