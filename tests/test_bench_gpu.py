"""bench.py's JSON line on the GPU: the keys and the consistency of the
numbers that the measurement contract fixes (a short run of the default
workload, B=8 H=16 N=4096 d=128 causal).

Checked: one JSON line; value = counted FLOPs per step / ms_per_step; the
roofline object's fraction = achieved / peak, with achieved within the
plausible range of its bound; the end-to-end leg's copy volumes equal the
bytes of q, k, v, dO in and O, dQ, dK, dV (and LSE) out; the clock fields and the CPU
oracle baseline are present; gpu_launches counts four launches per step.
"""
import json
import os
import subprocess
import sys

import pytest

from io_aware_exact_14_gb300 import counts
from io_aware_exact_14_gb300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run_bench(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_default_bench_line_keeps_the_contract():
    steps, warmup = 5, 3
    d = _run_bench("--steps", str(steps), "--warmup", str(warmup), "--cpu-seconds", "1")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "clocks", "gpu_launches"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True and d["dtype"] == "bf16"

    w = WORKLOADS[5]
    assert d["config"]["workload"] == w.name
    B, H, N, dim = w.shape
    flops = counts.attn_flops(B, H, N, dim, True, "fwd") + counts.attn_flops(B, H, N, dim, True, "bwd")
    assert d["value"] == pytest.approx(flops / (d["ms_per_step"] * 1e-3) / 1e12, rel=2e-3)

    roof = d["roofline"]
    assert roof["bound"] in ("tensor", "hbm")
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"], abs=2e-3)
    assert 0.2 < roof["frac"] < 1.3
    if roof["traffic"] is not None:   # dram bytes per launch from the committed capture
        assert roof["traffic"] > 0

    e2e = d["e2e"]
    tensor_bytes = B * H * N * dim * 2
    assert e2e["h2d_bytes_per_step"] == 4 * tensor_bytes                  # q, k, v, dO
    assert e2e["d2h_bytes_per_step"] == 4 * tensor_bytes + B * H * N * 4  # O, dQ, dK, dV and LSE
    assert 0 < e2e["value"] <= d["value"] * 1.05

    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] > 0
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]   # a 5-step run may see no sample
    assert d["gpu_launches"] == 4 * steps
