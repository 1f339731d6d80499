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
LINK = {"whole_pool_gbs": 211.0, "chunks": 54, "chunk_gbs_min": 200.0, "chunk_gbs_median": 210.0,
        "chunk_gbs_max": 211.5, "burst_first_1p21gb_gbs": 211.3}


def test_line_has_the_contract_keys():
    w = dict(bench.A3B)
    line = bench.build_line(_args(), w, 1, _dec(), LINK, None, None, PEAKS)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert k in line, k
    assert line["unit"] == "tok/s" and line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["data"] == "synthetic" and "workload" in line["config"]
    r = line["roofline"]
    assert set(r) >= {"bound", "achieved", "peak", "unit", "frac", "traffic"}
    # achieved = fill bytes / fill time; frac = achieved / peak
    assert r["achieved"] == pytest.approx(1.0e9 / 6.0e-3 / 1e9, abs=0.05)
    # the link peak of the fill is the median 1 GiB chunk rate, not the whole-pool rate
    assert r["peak"] == 210.0 and r["frac"] == pytest.approx(r["achieved"] / 210.0, abs=1e-3)
    e = line["e2e"]
    assert set(e) == {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}
    assert line["ms_per_step"] == pytest.approx(0.5 / 100 * 1e3)
    assert line["gpu_launches"] == 100 * w["L"] * 5  # control, fill, two expert launches, merge per layer


def test_per_token_counters_divide_by_the_batch():
    w = dict(bench.A3B, T=16)
    line = bench.build_line(_args(), w, 1, _dec(T=16), LINK, None, None, PEAKS)
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


def test_timed_window_and_host_link_are_reported():
    w = dict(bench.A3B)
    line = bench.build_line(_args(), w, 1, _dec(), LINK, None, None, PEAKS)
    tw = line["timed_window"]
    assert tw["tokens"] == [8, 108] and tw["every"] == 1 and tw["hit_rate"] == pytest.approx(0.8)
    # beside the end-to-end twin, value's tokens are every second one of 2K
    tw2 = bench.build_line(_args(), w, 1, dict(_dec(), stride=2), LINK, None, None, PEAKS)["timed_window"]
    assert tw2["tokens"] == [8, 208] and tw2["every"] == 2
    assert line["host_link"]["whole_pool_gbs"] == 211.0 and line["roofline"]["peak"] == 210.0
    # the config object is the workload alone (the reference arm prints the same one)
    assert line["config"] == bench.line_config(_args(), w, 1)


def test_traffic_is_null_once_the_kernel_source_changes(monkeypatch):
    t, note = bench.ncu_traffic("decode_experts", 1.0e8)
    assert t is None or t == round(bench.NCU_TRAFFIC["decode_experts"]["ratio"] * 1.0e8)
    monkeypatch.setitem(bench.NCU_TRAFFIC, "decode_experts", dict(bench.NCU_TRAFFIC["decode_experts"], sha16="0" * 16))
    t, note = bench.ncu_traffic("decode_experts", 1.0e8)
    assert t is None and "changed" in note


def test_reference_arm_prints_the_same_config_and_integer_steps():
    """The oracle as the reference arm, on a tiny workload so it runs here."""
    w = dict(bench.A3B, L=2, E=16, k=2, d=256, f=128, S=8, K_max=16, desc="tiny decode")
    args = _args(steps=4, warmup=3, ref_budget_s=30.0)
    ref = bench.run_reference(args, w, 1)
    assert ref["impl"] == "reference" and ref["steps"] == 4 and isinstance(ref["steps"], int)
    assert ref["warmup"] == 3 and ref["config"] == bench.line_config(args, w, 1)
    assert ref["metric"] == bench.metric_name(args, w) and ref["unit"] == "tok/s" and ref["value"] > 0
    assert set(ref["e2e"]) == {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}


def test_fused_resident_phase_needs_resident_experts():
    """Fused path: the experts' HBM rate is the resident phase's bytes over its
    span, and is not reported when the window held less than one resident
    expert per launch (hit rate ~0), nor is a traffic figure."""
    bx = 9_437_184
    dec = dict(_dec(), path="fused", bx=bx,
               meters={"resident_bytes": 8 * bx * 10.0, "resident_s": 10 * 20e-6, "resident_launches": 10})
    gbs, how = bench.experts_rate(dec)
    assert gbs == pytest.approx(8 * bx / 20e-6 / 1e9) and "resident" in how
    per, tr, note = bench.experts_traffic(dict(bench.A3B), dec)
    assert per == pytest.approx(8 * bx)
    dec_none = dict(dec, meters={"resident_bytes": 0.3 * bx * 10, "resident_s": 10 * 2e-6, "resident_launches": 10})
    assert bench.experts_rate(dec_none) == (0.0, None)
    dec_zero = dict(dec, meters={"resident_bytes": 0.0, "resident_s": 0.0, "resident_launches": 0})
    per, tr, note = bench.experts_traffic(dict(bench.A3B), dec_zero)
    assert tr is None and "no resident" in note


def test_e2e_token_sets_report_their_fills():
    """The device-timed and the end-to-end contexts are timed on different
    halves of the same 2K tokens: the line shows each half's fills per token."""
    w = dict(bench.A3B)
    line = bench.build_line(_args(), w, 1, dict(_dec(), e2e_fills=(140.0, 150.0)), LINK, None, None, PEAKS)
    f = line["components"]["e2e_fills_per_token"]
    assert f == {"e2e_tokens": 1.4, "value_tokens": 1.5}
