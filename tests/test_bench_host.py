"""Host-side helpers of bench.py on CPU: the clock-sample summary that decides whether a
run is kept, the DRAM-traffic record keyed to the kernel source, the FLOP count of a
step and the choice of the peak a fraction is taken against."""
import hashlib
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from gemm_overlap_gemms_gb300 import synth  # noqa: E402


def _line(sm, mx, hw="Not Active", hw_th="Not Active", sw_th="Not Active", cap="Not Active"):
    # index, clocks.sm, clocks.max.sm, power.draw, reasons.active, then the four reasons
    return "0, %s, %s, 1012.5, 0x0000000000000004, %s, %s, %s, %s" % (sm, mx, hw, hw_th, sw_th, cap)


def test_clock_summary_median_max_and_reasons():
    lines = [_line(2070, 2070), _line(1995, 2070, cap="Active"), _line(2032, 2070),
             "garbage", "0, [N/A], 2070, 1, 0, Not Active, Not Active, Not Active, Not Active"]
    c = bench.parse_clocks(lines)
    assert c == {"sm_mhz": 2032.0, "sm_max_mhz": 2070.0, "samples": 3, "reasons": ["sw_power_cap"]}


def test_clock_summary_reports_every_slowdown_it_saw():
    lines = [_line(1600, 2070, hw="Active"), _line(1500, 2070, hw_th="Active"),
             _line(1700, 2070, sw_th="Active")]
    c = bench.parse_clocks(lines)
    assert c["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert c["sm_mhz"] == 1600.0


def test_clock_summary_without_samples():
    assert bench.parse_clocks([]) is None
    assert bench.parse_clocks(["a, b", "0, x, y, 1, 0, A, A, A, A"]) is None


def test_traffic_record_follows_the_kernel_source(monkeypatch):
    sha = bench.kernel_src_sha()
    assert sha == hashlib.sha256(b"".join(open(f, "rb").read() for f in bench.KERNEL_SRC)).hexdigest()[:16]
    rec = {"sha256_16": sha, "bytes": 1.0e9, "T": 8192, "source": "profiles/x.md"}
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {"rs": rec})
    t = bench.kernel_traffic("rs", 4096.0)
    assert t["bytes_per_launch"] == pytest.approx(0.5e9)      # scaled by the launches' mean T
    assert t["captured_T"] == 8192 and t["scaled_to_mean_T"] == 4096.0
    assert bench.kernel_traffic("ag_swiglu", 4096.0) is None  # no record
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {"rs": dict(rec, sha256_16="0" * 16)})
    assert bench.kernel_traffic("rs", 4096.0) is None         # stale once the source changed


def test_step_flops_are_the_algorithmic_counts():
    w = synth.WORKLOADS["swiglu"]
    ag, rs = bench.step_flops([1024, 2048], w)
    H, N, K, tp = w.hidden, w.ag_n[0], w.rs_k[0], w.tp
    assert ag == 2.0 * 3072 * H * N
    assert rs == 2.0 * 3072 * K * H * tp


def test_peak_values_measured_or_fallback(monkeypatch, tmp_path):
    assert bench._peak_value({"bf16_tflops_sustained": 1650}, "bf16_tflops_sustained") == 1650.0
    assert bench._peak_value({"hbm_gbs": {"median": 7100.5}}, "hbm_gbs") == 7100.5
    assert bench._peak_value({"bf16_tflops": 1900.0}, "bf16_tflops_sustained", "bf16_tflops") == 1900.0
    assert bench._peak_value({}, "hbm_gbs") is None
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d, src = bench.peaks()
    assert src == "fallback" and d == bench.FALLBACK
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 7000.0}')
    d, src = bench.peaks()
    assert src == "measured" and d["hbm_gbs"] == 7000.0


def test_sweep_counts_are_algorithmic():
    # AG: 2*T*H*N FLOPs; bytes = weight once + shards read + buffer written + Y written
    fl, nb = bench.op_flops_bytes("ag", 512, 4096, 4, N=3072)
    assert fl == 2.0 * 512 * 4096 * 3072
    assert nb == 2.0 * (3072 * 4096 + 2 * 512 * 4096 + 512 * 3072)
    # SwiGLU writes half the columns
    _, nb_glu = bench.op_flops_bytes("ag_swiglu", 512, 4096, 4, N=7168)
    assert nb_glu == 2.0 * (7168 * 4096 + 2 * 512 * 4096 + 512 * 3584)
    # RS: 2*T*K*H*tp FLOPs; bytes = tp weights + tp A_j + the T output rows
    fl, nb = bench.op_flops_bytes("rs", 64, 4096, 4, K=3584)
    assert fl == 2.0 * 64 * 3584 * 4096 * 4
    assert nb == 2.0 * (4 * 3584 * 4096 + 4 * 64 * 3584 + 64 * 4096)


def test_roofline_point_names_the_limiting_roof():
    # 1 GFLOP over 10 MB (100 FLOP/B) in 1 ms against 2000 TFLOP/s and 8000 GB/s:
    # the ridge is 250 FLOP/B, so HBM bounds it at 100 * 8000 GB/s = 800 TFLOP/s
    p = bench.roofline_point(1e9, 1e7, 1e-3, 2000.0, 8000.0)
    assert p["bound"] == "hbm"
    assert p["tflops"] == pytest.approx(1.0)
    assert p["hbm_gbs"] == pytest.approx(10.0)
    assert p["frac_of_roofline"] == pytest.approx(1.0 / 800.0)
    # far right of the ridge: the tensor peak bounds it
    q = bench.roofline_point(1e12, 1e8, 1e-3, 2000.0, 8000.0)
    assert q["bound"] == "tensor" and q["frac_of_roofline"] == pytest.approx(1000.0 / 2000.0)
    assert q["frac_of_peak"] == pytest.approx(0.5)


def test_default_sweep_covers_the_metric_ladder():
    names = {n: Ts for n, _, _, Ts in bench.DEFAULT_SWEEP}
    assert set(names) == {"fc1_ag_swiglu", "fc2_rs", "qkv_ag", "large_rs_k1024", "large_rs_k3584"}
    for n, Ts in names.items():
        w = synth.WORKLOADS[dict((a, b) for a, b, _, _ in bench.DEFAULT_SWEEP)[n]]
        assert all(T % w.tp == 0 and w.tp <= T <= w.max_tokens for T in Ts), n
    assert min(names["fc2_rs"]) == 4 and max(names["large_rs_k3584"]) == 16384


def test_interleaved_medians_take_turns_and_return_each_ones_median():
    """The bulk-overlap timings: one call of each timing function per round, in turn,
    so that a drift over the run (clocks under the power cap) reaches all of them alike;
    the result is each function's own median, not a pooled one."""
    calls = []

    def fake(name, values):
        it = iter(values)

        def f():
            calls.append(name)
            return next(it)
        return f

    a = fake("a", [5.0, 1.0, 3.0, 9.0, 7.0])
    b = fake("b", [10.0, 30.0, 20.0, 50.0, 40.0])
    assert bench.interleaved_medians([a, b], rounds=5) == [5.0, 30.0]
    assert calls == ["a", "b"] * 5


def test_event_regions_split_around_the_headline():
    assert bench.split_around(20) == (10, 10)
    assert bench.split_around(5) == (2, 3)
    assert bench.split_around(1) == (0, 1)


def test_median_region_ignores_one_slow_region():
    """The end-to-end figure: one region slowed by the host does not move the median,
    and every region is listed per step."""
    med, note = bench.median_region([114.6, 209.2, 114.7], 10)
    assert med == 114.7
    assert note == "median of 3 regions of 10 steps each: 11.46, 20.92, 11.47 ms per step"


def test_no_gc_keeps_the_collector_off_inside_and_restores_it():
    import gc
    assert gc.isenabled()
    with bench.no_gc():
        assert not gc.isenabled()
    assert gc.isenabled()
    gc.disable()
    try:
        with bench.no_gc():            # already off: nothing collected, nothing changed
            assert not gc.isenabled()
        assert not gc.isenabled()      # left as it was found
    finally:
        gc.enable()
