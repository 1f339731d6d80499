"""The benchmark's JSON line (no GPU): keys, types and the arithmetic of the
derived figures, built from a made-up decode record."""
import argparse
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _args(**kw):
    a = argparse.Namespace(cpu_exec=0, pool="pinned")
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _dec(T=1, K=100):
    return dict(value=200.0, elapsed=0.5, K=K, W=8, T=T, clocks={"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []},
                status=0, t_init=0.0, hits=800.0, misses=200.0, fills=150.0, cpu=50.0, P=4,
                shares={"control": 0.1, "fill": 0.5, "experts": 0.35, "merge": 0.05},
                ms_per_token={"control": 0.6, "fill": 4.0, "experts": 3.0, "merge": 0.3},
                launches={"control": 192}, ex_bytes=2.0e9, ex_ms=1000.0, ex_n=100, fill_bytes=1.0e9, fill_ms=6.0,
                fill_n=50, control_us=7.0, route_us=0.0, eager_ms=8.0, e2e=190.0, h2d=1000, d2h=2000)


PEAKS = dict(hbm_gbs=6750.0, bf16_tflops=1960.0, bf16_tflops_sustained=1700.0, source="measured")


def test_line_has_the_contract_keys():
    w = dict(bench.A3B)
    line = bench.build_line(_args(), w, 1, _dec(), 211.0, None, None, PEAKS)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert k in line, k
    assert line["unit"] == "tok/s" and line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["data"] == "synthetic" and "workload" in line["config"]
    r = line["roofline"]
    assert set(r) >= {"bound", "achieved", "peak", "unit", "frac", "traffic"}
    # achieved = fill bytes / fill time; frac = achieved / peak
    assert r["achieved"] == pytest.approx(1.0e9 / 6.0e-3 / 1e9, abs=0.05)
    assert r["frac"] == pytest.approx(r["achieved"] / 211.0, abs=1e-3)
    e = line["e2e"]
    assert set(e) == {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}
    assert line["ms_per_step"] == pytest.approx(0.5 / 100 * 1e3)
    assert line["gpu_launches"] == 100 * w["L"] * 5  # control, fill, two expert launches, merge per layer


def test_per_token_counters_divide_by_the_batch():
    w = dict(bench.A3B, T=16)
    line = bench.build_line(_args(), w, 1, _dec(T=16), 211.0, None, None, PEAKS)
    c = line["components"]
    assert c["fills_per_step"] == pytest.approx(1.5)
    assert c["fills_per_token"] == pytest.approx(1.5 / 16, abs=1e-3)
    assert c["kernel_ms_per_token"]["fill"] == pytest.approx(4.0 / 16, abs=1e-4)
    assert "batch 16" in line["metric"]


def test_metric_names():
    assert bench.metric_name(_args(), dict(bench.A3B)) == bench.METRIC
    v4 = bench.metric_name(_args(), dict(bench.V4))
    assert "V4-Flash-style MXFP4" in v4 and "batch 1" in v4
    assert "CPU expert executor" in bench.metric_name(_args(cpu_exec=8), dict(bench.A3B))
