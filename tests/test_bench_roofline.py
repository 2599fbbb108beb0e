"""The bench's tensor roofline (CPU): the denominator is the measured burst
rate, or the measured sustained rate when the leg's own clock record shows the
power cap; the fraction of the burst rate is reported either way."""

import pytest

import bench

PEAKS = (6789.0, 1891.3, 1716.0, "measured")


def test_burst_when_no_cap():
    clk = {"sm_mhz": 2070, "reasons": []}
    r = bench.tensor_roofline(1800.0, clk, PEAKS)
    assert r["peak"] == pytest.approx(1891.3)
    assert r["frac"] == pytest.approx(1800.0 / 1891.3)
    assert r["frac_of_burst"] == pytest.approx(r["frac"])
    assert "burst" in r["peak_source"] and r["bound"] == "tensor" and r["unit"] == "TFLOP/s"


def test_sustained_when_power_capped():
    clk = {"sm_mhz": 1425, "reasons": ["sw_power_cap"]}
    r = bench.tensor_roofline(1700.0, clk, PEAKS)
    assert r["peak"] == pytest.approx(1716.0)
    assert r["frac"] == pytest.approx(1700.0 / 1716.0)
    assert r["frac_of_burst"] == pytest.approx(1700.0 / 1891.3)
    assert "sustained" in r["peak_source"]


@pytest.mark.parametrize("clk", [None, {}, {"reasons": None}, {"reasons": ["hw_slowdown"]}])
def test_no_record_or_other_reason_keeps_burst(clk):
    r = bench.tensor_roofline(1000.0, clk, PEAKS)
    assert r["peak"] == pytest.approx(1891.3)


def test_sparse_scale():
    r = bench.tensor_roofline(2700.0, {"reasons": []}, PEAKS, scale=2.0)
    assert r["peak"] == pytest.approx(2 * 1891.3)
    assert r["peak_source"].startswith("2 x ")
    r = bench.tensor_roofline(2500.0, {"reasons": ["sw_power_cap"]}, PEAKS, scale=2.0)
    assert r["peak"] == pytest.approx(2 * 1716.0)
    assert r["frac_of_burst"] == pytest.approx(2500.0 / (2 * 1891.3))


def test_load_peaks_reads_the_measured_file():
    hbm, burst, sustained, src = bench.load_peaks()
    assert src in ("measured", "fallback")
    assert hbm > 0 and burst > 0 and 0 < sustained <= burst
