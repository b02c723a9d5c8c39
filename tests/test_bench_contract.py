"""The bench line committed with the profiles is well formed: every key of the
bench contract, a roofline whose fraction is achieved / peak, a DRAM traffic
figure near the dominant kernel's algorithmic bytes, an end-to-end figure with
its copy sizes, the CPU baseline and the clock record.  CPU only (reads JSON)."""
import json
import os

import pytest

from conftest import ROOT

LINE = os.path.join(ROOT, "profiles", "bench_line_prefill_t4096_decode_t32.json")


@pytest.fixture(scope="module")
def line():
    with open(LINE) as f:
        return json.load(f)


def test_top_level_keys(line):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in line, k
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["scaling"] == "weak" and line["n_gpus"] >= 1
    assert line["warmup"] >= 3 and line["steps"] >= 1
    assert line["vs_baseline"] is None            # no published number for this metric and workload
    assert line["config"]["workload"] == "prefill_t4096"
    # value is tokens per second over the timed steps
    T = line["config"]["T"]
    assert line["value"] == pytest.approx(line["n_gpus"] * T / (line["ms_per_step"] * 1e-3), rel=2e-3)
    assert line["gpu_launches"] == 3 * line["steps"]


def test_roofline(line):
    r = line["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-3)
    assert 0.0 < r["frac"] < 1.5
    # the W1/W3 GEMM moves its algorithmic bytes about once (no re-reads)
    assert r["traffic"] is not None
    algorithmic = 2181038080
    assert 0.95 * algorithmic <= r["traffic"] <= 1.10 * algorithmic


def test_decode_roofline(line):
    d = line["decode_t32"]["roofline"]
    assert d["bound"] == "hbm" and d["unit"] == "GB/s"
    assert d["frac"] == pytest.approx(d["achieved"] / d["peak"], rel=1e-3)


def test_e2e_cpu_baseline_and_clocks(line):
    e = line["e2e"]
    for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert k in e, k
    T, d = line["config"]["T"], line["config"]["d"]
    assert e["h2d_bytes_per_step"] == T * d * 2 and e["d2h_bytes_per_step"] == T * d * 2
    assert e["value"] < line["value"] * 1.05    # host copies can only add time
    c = line["cpu_baseline"]
    for k in ("value", "unit", "cores", "kind", "sample"):
        assert k in c, k
    assert c["kind"] == "oracle" and c["cores"] >= 1
    k = line["clocks"]
    for key in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert key in k, key
    assert not set(k["reasons"]) & {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


def test_roofline_duration_comes_from_the_headline_run(line):
    # the W1/W3 duration is the headline's ms per call times the kernel's share of
    # the per-kernel event times, and the peak is the one for that window's length
    r = line["roofline"]
    assert r["duration_us"] == pytest.approx(line["ms_per_step"] * 1e3 * r["share"], rel=2e-3)
    assert r["achieved"] == pytest.approx(r["flops_per_launch"] / (r["duration_us"] * 1e-6) / 1e12, rel=2e-3)
    window_ms = line["ms_per_step"] * line["steps"]
    assert ("burst" if window_ms <= 250.0 else "sustained") in r["peak_kind"]
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-3)
    share = line["stages_us"]["expert_w1w3_swiglu"] / sum(line["stages_us"].values())
    assert r["share"] == pytest.approx(share, abs=2e-3)


def test_sustained_leg_and_near_ties(line):
    s = line["sustained"]
    assert s["timed_seconds"] >= 2.0
    r = s["roofline"]
    assert "sustained" in r["peak_kind"] and r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-3)
    assert s["clocks"]["samples"] >= 5
    assert not set(s["clocks"]["reasons"]) & {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    nt = line["near_ties"]
    assert nt["tokens"] == line["config"]["T"]
    assert nt["index_mismatches_outside_near_ties"] == 0
