"""The roofline object of bench.py on CPU: which bf16 peak is the denominator and
which resource a kernel's roofline is.

- The burst figure is used for a kernel that ran at full clock in a short timed
  region, and the sustained one when the power cap was active or the region
  lasted seconds.
- The single-launch kernel for m <= 128 is reported against HBM when its
  compulsory bytes take longer at the HBM peak than its products at the tensor
  peak.
- Both fractions of a tensor-bound kernel are in the line.
"""
import pytest

import bench

PEAKS = {"hbm_gbs": 6785.2, "bf16_tflops": 1917.5, "bf16_tflops_sustained": 1719.8}


class _Bucket:
    def __init__(self, single):
        self.ns_single_kernel = single


class _Nsm:
    def __init__(self, single):
        self.single = single

    def muon_get_bucket_info(self, plan, b):
        return _Bucket(self.single)


class _Info:
    n_buckets = 1


@pytest.mark.parametrize("reasons, timed_s, want", [
    ([], 0.6, 1917.5),                  # full clock, sub-second region: burst
    (["sw_power_cap"], 0.6, 1719.8),    # the power cap held the clock down: sustained
    ([], 5.0, 1719.8),                  # seconds-long region: sustained
    (["sw_power_cap"], 5.0, 1719.8),
])
def test_peak_choice(reasons, timed_s, want):
    peak, name = bench.choose_bf16_peak(PEAKS, "measured", {"reasons": reasons}, timed_s)
    assert peak == want
    assert ("sustained" in name) == (want == 1719.8)


def test_peak_choice_without_a_sustained_figure():
    peaks = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
    assert bench.choose_bf16_peak(peaks, "fallback", {"reasons": ["sw_power_cap"]}, 1.0)[0] == 1900.0


def test_hbm_binds_by_time_at_each_peak():
    # the per-head launch: 5.66 GB and 1.126 TFLOP -> 0.83 ms of HBM against 0.59 ms of products
    assert bench.hbm_binds(5.66e9, 1.126e12, 6785.2, 1917.5)
    # the layer's NS: 5.2 GB moved and 4.6 TFLOP -> products dominate
    assert not bench.hbm_binds(5.2e9, 4.6e12, 6785.2, 1917.5)


def test_tensor_bound_entry():
    ns_ms, launches, flops = 2.7, 15, 4.6e12
    tf = flops / (ns_ms * 1e-3) / 1e12
    r = bench.roofline_entry(_Nsm(0), None, _Info(), False, False, ns_ms, launches, flops, 0, tf,
                             1917.5, "measured bf16 burst", PEAKS, 1719.8, 348.4e6)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == 1917.5
    assert r["frac"] == pytest.approx(tf / 1917.5)
    assert r["frac_of_burst"] == pytest.approx(tf / 1917.5)
    assert r["frac_of_sustained"] == pytest.approx(tf / 1719.8)
    assert r["algorithmic_flops_per_launch"] == pytest.approx(flops / launches)
    assert r["per_launch_ms"] == pytest.approx(ns_ms / launches)
    assert r["traffic"] == 348.4e6


def test_hbm_bound_entry():
    ns_ms, nbytes, flops = 2.27, 5.66e9, 1.126e12
    tf = flops / (ns_ms * 1e-3) / 1e12
    r = bench.roofline_entry(_Nsm(1), None, _Info(), False, True, ns_ms, 1, flops, nbytes, tf,
                             1917.5, "measured bf16 burst", PEAKS, 1719.8, None)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6785.2
    assert r["achieved"] == pytest.approx(nbytes / (ns_ms * 1e-3) / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6785.2)
    assert r["tensor_frac"] == pytest.approx(tf / 1917.5)
    assert r["algorithmic_bytes_per_launch"] == nbytes


def test_tf32_entry_counts_three_products():
    ns_ms, launches, flops = 13.2, 15, 4.6e12
    tf = flops / (ns_ms * 1e-3) / 1e12
    peak = 1917.5 * 1.1 / 2.25
    r = bench.roofline_entry(_Nsm(0), None, _Info(), True, False, ns_ms, launches, flops, 0, tf,
                             peak, "measured bf16 burst x 1.1/2.25", PEAKS, 1719.8, None)
    assert r["achieved"] == pytest.approx(3 * tf)
    assert r["frac"] == pytest.approx(3 * tf / peak)
    assert "frac_of_burst" not in r
