"""Host logic of the benchmark that decides whether a measurement is valid or what
it reports, run on CPU: the clock-sample summary (throttle reasons, the SM clock
under load) and the ncu traffic record, which is used only while the kernel
source is unchanged since the capture."""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(sm, reasons=("Not Active",) * 4, mx=2070):
    # index, clocks.sm, clocks.max.sm, power.draw, reasons.active, hw_slowdown,
    # hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
    return ", ".join(["0", str(sm), str(mx), "812.3", "0x0000000000000000"] + list(reasons))


def test_clock_summary_median_of_the_busy_half_and_reasons():
    c = bench.ClockSampler(0)
    c.lines = [_line(v) for v in (345, 345, 2070, 2055, 2070, 1980)] + ["garbage", ""]
    s = c.summary()
    assert s["samples"] == 6 and s["sm_max_mhz"] == 2070.0
    # the idle edges (345 MHz) fall in the lower half: median of 2055, 2070, 2070
    assert s["sm_mhz"] == 2070.0
    assert s["reasons"] == []


def test_clock_summary_reports_each_throttle_reason():
    c = bench.ClockSampler(0)
    c.lines = [_line(1500, ("Active", "Not Active", "Not Active", "Not Active")),
               _line(1490, ("Not Active", "Not Active", "Active", "Active")),
               _line(1510)]
    s = c.summary()
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]


def test_clock_summary_without_samples():
    c = bench.ClockSampler(0)
    c.lines = ["[N/A], [N/A]"]
    assert c.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_traffic_record_only_for_the_captured_source(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// kernel v1\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    digest = hashlib.sha256(src.read_bytes()).hexdigest()
    (prof / "gmm1_decode_ncu.md").write_text(
        "summary\n\n    traffic_bytes_per_launch: 123456789\n    source_sha256: %s\n" % digest)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("gmm1", "decode", str(src)) == 123456789
    assert bench.traffic_record("gmm1", "prefill", str(src)) is None  # no capture of that workload
    src.write_text("// kernel v2\n")  # the kernel changed since the counters were taken
    assert bench.traffic_record("gmm1", "decode", str(src)) is None


def test_roofline_picks_the_bound_and_flags_fractions_above_the_peak():
    import synth
    w = synth.CONFIGS["prefill"]
    ei, _ = synth.routing(w.seed, w.M, w.E, w.topK, w.routing)
    alg, active = bench.algorithmic(w, ei)
    peaks = {"hbm_gbs": 6785.9, "bf16_tflops": 1833.7, "source": "measured"}
    t = alg["gmm1"]["ops"] / (0.8 * peaks["bf16_tflops"] * 1e12)  # 80% of the tensor peak
    r = bench.roofline_of(w, {"gmm1": t * 1e3, "gmm2": t * 0.5e3}, alg, peaks)
    assert r["bound"] == "tensor" and abs(r["frac"] - 0.8) < 1e-3 and "above_peak" not in r
    r = bench.roofline_of(w, {"gmm1": t * 0.7e3, "gmm2": t * 0.5e3}, alg, peaks)
    assert r["frac"] > 1 and r["above_peak"] is True
    d = synth.CONFIGS["decode"]
    ei, _ = synth.routing(d.seed, d.M, d.E, d.topK, d.routing)
    alg, active = bench.algorithmic(d, ei)
    r = bench.roofline_of(d, {"gmm1": 1.1, "gmm2": 0.6}, alg, peaks)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"


def test_single_thread_oracle_baseline():
    import synth
    res = bench.single_thread_oracle({"tiny": synth.make_inputs("tiny")})
    assert res["tiny"]["cores"] == 1 and res["tiny"]["value"] > 0
    import oracle
    assert oracle.max_threads() > 1 or os.cpu_count() == 1  # the previous count is restored


def test_launches_per_step_follow_the_engine_choice():
    """The bench's count of our kernels per layer step (its `gpu_launches` claim) for
    every workload, written out from the engine rules it restates: the sort fused into
    the quant kernel up to 4096 routes and two launches above 8192; one GEMM engine up to
    24 rows per expert on average and from 256 on, three launches per GEMM between (the
    warp-MMA share on 16-row and on 32-row tiles, then the tcgen05 pairs); SwiGLU inside
    GMM1 above 24 rows per expert.  The ncu launch lists show the same kernels per step
    (prefill 6, skewed 10, decode 5)."""
    import synth
    expect = {
        "tiny": 0 + 1 + 2 * 1 + 1 + 1,     # 32 routes, 4 rows per expert
        "decode": 0 + 1 + 2 * 1 + 1 + 1,   # 1024 routes, 4 rows per expert
        "mid": 0 + 1 + 2 * 1 + 1 + 1,      # 4096 routes, 16 rows per expert
        "skewed": 2 + 1 + 2 * 3 + 0 + 1,   # 16384 routes, 64 rows per expert: split, fused SwiGLU
        "prefill": 2 + 1 + 2 * 1 + 0 + 1,  # 49152 routes, 768 rows per expert: pairs only
    }
    for name, n in expect.items():
        assert bench.launches_per_step(synth.CONFIGS[name]) == n, name
