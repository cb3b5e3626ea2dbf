"""Host logic of bench.py that needs no GPU: the choice of the roofline's bf16 denominator from the
sampled clocks, and the rule that a stored DRAM-traffic figure is reported only for the kernel
sources it was captured from."""
import bench


PEAKS = dict(hbm=6794.5, bf16=1962.7, bf16_sustained=1707.1, src="measured")


def test_burst_peak_without_power_cap():
    assert bench.choose_peak(PEAKS, []) == (1962.7, "burst")
    assert bench.choose_peak(PEAKS, ["hw_slowdown"]) == (1962.7, "burst")
    assert bench.choose_peak(PEAKS, None) == (1962.7, "burst")     # no clock samples at all


def test_sustained_peak_under_power_cap():
    assert bench.choose_peak(PEAKS, ["sw_power_cap"]) == (1707.1, "sustained")
    no_sustained = dict(PEAKS, bf16_sustained=None)
    assert bench.choose_peak(no_sustained, ["sw_power_cap"]) == (1962.7, "burst")


def test_traffic_follows_the_kernel_sources(monkeypatch):
    digest = bench.gemm_source_digest()
    assert len(digest) == 16 and digest == bench.gemm_source_digest()
    monkeypatch.setattr(bench, "GEMM_TRAFFIC", {"w": (123, digest), "stale": (456, "0" * 16)})
    assert bench.gemm_traffic("w") == 123
    assert bench.gemm_traffic("stale") is None        # captured from other sources
    assert bench.gemm_traffic("absent") is None


def test_clock_summary_windows():
    c = bench.ClockSampler(0)
    row = "0, {mhz}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {cap}"
    c.samples = [(1.0, row.format(mhz=2070, cap="Not Active")), (2.0, row.format(mhz=2070, cap="Not Active")),
                 (5.0, row.format(mhz=1500, cap="Active")), (6.0, row.format(mhz=1400, cap="Active"))]
    c.window = (0.5, 2.5)
    s = c.summary()
    assert s["sm_mhz"] == 2070 and s["reasons"] == [] and s["samples"] == 2
    s2 = c.summary((4.5, 6.5))
    assert s2["sm_mhz"] == 1450 and s2["reasons"] == ["sw_power_cap"]
