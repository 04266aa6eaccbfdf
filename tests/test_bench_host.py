"""Host-side pieces of bench.py (no GPU): every workload's byte and op counts,
metric names and the reference arm's JSON line on a tiny sample."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("name", sorted(bench.WORKLOADS))
def test_workload_counts(name):
    w = bench.WORKLOADS[name]
    wb, sb = bench.weight_bytes(w), bench.step_bytes(w)
    assert 0 < wb < sb
    kp = w["K"] + (w["K"] & 1)
    packed = w["N"] * (w["K"] if w["kind"] == "w8a16" else kp // 2)
    assert wb >= packed
    assert bench.step_ops(w) == 2 * w["M"] * w["N"] * w["K"]
    value, unit = bench.metric_of(w, 1.0)
    assert value > 0 and unit in ("GB/s", "TOPS", "TFLOP/s")
    assert ("decode" in bench.metric_name(w)) == (w["regime"] == "decode")


def test_default_workload_bytes():
    """The default line's algorithmic bytes: weights + f16 scales + bf16 x + f32 y."""
    w = bench.WORKLOADS["w4a16_gemv_m1"]
    assert bench.step_bytes(w) == 2048 * 1024 + 2048 * 64 * 2 + 2048 * 2 + 2048 * 4


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0", "--cpu-seconds", "0.5"], capture_output=True, text=True, timeout=600,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_extra_lines_cover_the_benchmark_set():
    """The default run's extra lines: every decode-grid and prefill workload exists."""
    for name in bench.EXTRA_DECODE + bench.EXTRA_PREFILL:
        assert name in bench.WORKLOADS, name
    grid = {(w["kind"], w["M"], w["N"], w["layout"]) for n in bench.EXTRA_DECODE
            for w in [bench.WORKLOADS[n]] if n.startswith(("w4a16_decode", "w4a8_decode"))}
    for kind in ("w4a16", "w4a8"):
        for M in (1, 4, 16):
            for N in (13312, 3072):
                for lay in (0, 1):
                    assert (kind, M, N, lay) in grid, (kind, M, N, lay)
    pre = {(bench.WORKLOADS[n]["kind"], bench.WORKLOADS[n]["N"]) for n in bench.EXTRA_PREFILL}
    assert {(k, n) for k in ("w4a8", "w4a16") for n in (2048, 3072, 13312)} <= pre


def test_reference_arm_bounded_for_many_steps():
    """Many steps with a tiny budget: each step samples output channels
    instead of whole calls, so the run ends quickly and says so."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps",
                          "20000", "--warmup", "1", "--cpu-seconds", "0.5"], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["steps"] == 20000 and line["value"] > 0
    assert "output channels sampled" in line["cpu_baseline"]["sample"]


def test_cpu_model_is_named():
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()


def test_microdecoder_extra_line_has_clocks_and_oracle():
    """The default run's microdecoder line: every mode keeps its figures and
    gets the clocks sampled inside its own timed region; the oracle's frame
    rate sits beside them."""
    import datetime as dt
    t0 = dt.datetime(2026, 1, 1, 12, 0, 0).timestamp()
    sampler = bench.ClockSampler(None)
    for i in range(20):  # one sample every 50 ms; a power-cap sample inside the second region
        ts = dt.datetime.fromtimestamp(t0 + 0.05 * i).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        cap = "Active" if i == 12 else "Not Active"
        sampler.lines.append(f"{ts}, {2070 - i}, 2070, 900.00, 0x0, Not Active, Not Active, Not Active, {cap}")
    figures = {"ms_per_frame": 0.9, "frames_per_s": 1111.1, "weight_gbs": 570.0, "weight_sets": 9,
               "frac_of_hbm": 0.084, "launches_per_frame": 1}
    md = {"chain_rotating": {**figures, "t0": t0 + 0.02, "t1": t0 + 0.33},
          "chain_l2_resident": {**figures, "t0": t0 + 0.52, "t1": t0 + 0.80}}
    line = bench.microdecoder_extra(md, sampler, 0.05)
    assert line["workload"] == bench.MICRODECODER
    for k in md:
        assert "t0" not in line[k] and line[k]["weight_gbs"] == 570.0
    first, second = line["chain_rotating"]["clocks"], line["chain_l2_resident"]["clocks"]
    assert first["samples"] == 6 and first["reasons"] == [] and first["sm_max_mhz"] == 2070
    assert second["samples"] == 6 and second["reasons"] == ["sw_power_cap"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cpu_model"]
    assert bench.microdecoder_extra(md, sampler, None).get("cpu_baseline") is None
    json.dumps(line)


def test_measure_line_reports_cold_and_warm(monkeypatch):
    """measure_line's host logic with the device parts faked: the cold figure
    rotates input copies, the warm one runs every step on copy 0, and both
    come from the same workload object."""
    seen = []

    class FakeWorkload:
        launches_per_step = 1

        def __init__(self, w, copies):
            self.w, self.copies = w, copies

    def fake_time_steps(wl, steps, warmup, kernel_only=False):
        seen.append((wl.copies, kernel_only))
        us = 2.0 if wl.copies == 1 else 4.0   # warm: weights already in L2
        return steps * us / 1e3, 100.0, 100.1

    monkeypatch.setattr(bench, "Workload", FakeWorkload)
    monkeypatch.setattr(bench, "time_steps", fake_time_steps)
    sampler = bench.ClockSampler(None)
    name = "w4a16_decode_m1_n13312"
    w = bench.WORKLOADS[name]
    line = bench.measure_line(name, 128 << 20, {"hbm_gbs": 6759.9}, sampler, None)
    copies = bench.copies_for(w, 128 << 20)
    assert seen == [(copies, False), (copies, True), (1, False)]
    assert line["us_per_step"] == 4.0 and line["warm_l2_resident"]["us_per_step"] == 2.0
    assert line["warm_l2_resident"]["value"] == round(2 * line["value"], 2) or \
        abs(line["warm_l2_resident"]["value"] - 2 * line["value"]) < 0.02
    assert "cpu_baseline" not in line
