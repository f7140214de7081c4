"""The JSON line bench.py prints: the keys a reader of the benchmark relies on,
and the arithmetic that ties them together (roofline fraction = achieved /
peak, launches = 2 per step).  Both arms are checked on the CPU: the GPU arm's
line through emit_line with fixed timings, the reference arm (the oracle on
host cores) end to end on the small workload."""

import contextlib
import io
import json
import os
import subprocess
import sys
import types

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

TOP_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
            "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches"}


def _emit(**over):
    args = types.SimpleNamespace(warmup=5, no_cpu_baseline=True, cpu_seconds=0.0)
    e2e = {"value": 1000.0, "unit": "TFLOP/s", "h2d_bytes_per_step": 10, "d2h_bytes_per_step": 5}
    clocks = {"sm_mhz": 2000.0, "sm_max_mhz": 2070.0, "reasons": []}
    kw = dict(args=args, world=1, n=20, step_ms_max=6.2, pre_ms=6.0, dec_ms=0.09, pre_ms_max=6.0, dec_ms_max=0.09,
              pre_tflops=1450.0, dec_gbs=5900.0, e2e=e2e, clocks=clocks, x=None)
    kw.update(over)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.emit_line(**kw)
    lines = [ln for ln in buf.getvalue().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


def test_gpu_arm_line_keys_and_arithmetic():
    d = _emit()
    assert TOP_KEYS <= set(d)
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] >= 3
    assert d["gpu_launches"] == 2 * 20                       # one prefill and one decode launch per step
    assert d["config"]["workload"]
    r = d["roofline"]
    assert {"bound", "achieved", "peak", "unit", "frac", "traffic"} <= set(r)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(bench.prefill_flops(bench.PREFILL_B, bench.PREFILL_S) / 6.0e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    dr = d["decode"]["roofline"]
    assert dr["bound"] == "hbm" and dr["frac"] == pytest.approx(dr["achieved"] / dr["peak"])
    assert dr["achieved"] == pytest.approx(bench.decode_bytes(bench.DECODE_B, bench.DECODE_CTX) / 0.09e-3 / 1e9)
    assert {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"} <= set(d["e2e"])
    assert d["clocks"]["sm_max_mhz"] == 2070.0


def test_gpu_arm_optional_objects():
    d = _emit(bwd={"bwd_ms": 28.0, "bwd_ms_local": 28.0, "fwd_ms": 6.0, "reps": 10})
    pf = bench.prefill_flops(bench.PREFILL_B, bench.PREFILL_S)
    assert d["backward"]["value"] == pytest.approx(2.5 * pf / 28.0e-3 / 1e12)
    assert d["backward"]["roofline"]["frac"] == pytest.approx(d["backward"]["roofline"]["achieved"] /
                                                              d["backward"]["roofline"]["peak"])


def test_reference_arm_line():
    """The oracle arm prints one line on the GPU arm's metric and unit, with its own CPU baseline."""
    env = dict(os.environ, PYTHONPATH=ROOT)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "small", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert TOP_KEYS - {"roofline"} <= set(d)                # no kernel, so no kernel roofline
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_grid_summary_reports_both_bars():
    peaks = {"bf16_tflops": 2000.0, "hbm_gbs": 8000.0, "source": "measured"}
    recs = [{"kind": "prefill", "S": S, "B": 1, "ms": 1.0, "TFLOP/s": 1000.0, "frac": 0.5, "timing": "graph"}
            for S in bench.GRID_PREFILL_S]
    recs += [{"kind": "decode", "ctx": c, "B": b, "us": 10.0, "GB/s": 4000.0, "frac": 0.5, "timing": "graph"}
             for c in bench.GRID_DECODE_CTX for b in bench.GRID_B]
    recs += [{"kind": "decode_long", "ctx": c, "B": b, "us": 30.0, "GB/s": 6000.0, "frac": 0.9, "timing": "graph"}
             for b, c in bench.GRID_LONG_DECODE]
    g = bench.grid_summary(recs, peaks)
    assert len(g["prefill_b1"]) == 4 and len(g["decode"]) == 16
    assert g["prefill_bar_mean_frac"] == pytest.approx(0.5) and g["decode_bar_mean_frac"] == pytest.approx(0.5)
    assert len(g["decode_long_ctx"]) == len(bench.GRID_LONG_DECODE)      # reported, outside the README's bar
    d = _emit(grid=g)
    assert d["grid"]["decode"]["B1_ctx8192"]["frac"] == 0.5


def test_traffic_is_null_unless_captured_on_the_current_sources():
    b, src = bench.traffic("prefill")
    assert src["current_sources"] == bench.sources_hash("prefill")
    if src["captured_on_sources"] != src["current_sources"]:
        assert b is None and src["fresh"] is False
    else:
        assert b is not None and src["fresh"] is True
