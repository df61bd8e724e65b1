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
    def __init__(self, single, fused=0):
        self.ns_single_kernel = single
        self.momentum_in_ns_kernel = fused


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
    # frac is on executed flops; the algorithmic count is reported beside it
    ns_ms, launches, flops, executed = 2.7, 15, 4.6e12, 4.35e12
    tf = executed / (ns_ms * 1e-3) / 1e12
    r = bench.roofline_entry(_Nsm(0), None, _Info(), False, False, ns_ms, launches, flops, executed, 0,
                             1917.5, "measured bf16 burst", PEAKS, 1719.8, 348.4e6)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == 1917.5
    assert r["achieved"] == pytest.approx(tf)
    assert r["frac"] == pytest.approx(tf / 1917.5)
    assert r["frac_of_burst"] == pytest.approx(tf / 1917.5)
    assert r["frac_of_sustained"] == pytest.approx(tf / 1719.8)
    assert r["frac_algorithmic"] == pytest.approx(flops / (ns_ms * 1e-3) / 1e12 / 1917.5)
    assert r["algorithmic_flops_per_launch"] == pytest.approx(flops / launches)
    assert r["executed_flops_per_launch"] == pytest.approx(executed / launches)
    assert r["per_launch_ms"] == pytest.approx(ns_ms / launches)
    assert r["traffic"] == 348.4e6


def test_hbm_bound_entry():
    ns_ms, nbytes, flops, executed = 2.27, 5.66e9, 1.126e12, 1.5e12
    r = bench.roofline_entry(_Nsm(1), None, _Info(), False, True, ns_ms, 1, flops, executed, nbytes,
                             1917.5, "measured bf16 burst", PEAKS, 1719.8, None)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6785.2
    assert r["achieved"] == pytest.approx(nbytes / (ns_ms * 1e-3) / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6785.2)
    assert r["tensor_frac"] == pytest.approx(executed / (ns_ms * 1e-3) / 1e12 / 1917.5)
    assert r["algorithmic_bytes_per_launch"] == nbytes


def test_tf32_entry_counts_three_products_at_half_the_bf16_rate():
    ns_ms, launches, flops, executed = 13.2, 15, 4.6e12, 4.35e12
    tf = executed / (ns_ms * 1e-3) / 1e12
    peak = bench.tf32_peak(1917.5)
    assert peak == pytest.approx(958.75)
    r = bench.roofline_entry(_Nsm(0), None, _Info(), True, False, ns_ms, launches, flops, executed, 0,
                             peak, "measured bf16 burst x 0.5", PEAKS, 1719.8, None)
    assert r["achieved"] == pytest.approx(3 * tf)
    assert r["frac"] == pytest.approx(3 * tf / peak)
    assert "frac_of_burst" not in r


def test_executed_flops_of_the_layer_and_the_small_kernel():
    # layer: executed flops sit below the algorithmic count (POLY runs upper tiles
    # only) and above the upper-triangle minimum
    layer = [(4096, 2560), (1024, 2560), (1024, 2560), (2560, 4096), (9728, 2560), (9728, 2560), (2560, 9728)]
    alg = sum(bench.ns_flops(r, c, 5)[1] for r, c in layer)
    exe = sum(bench.ns_executed_flops(r, c, 5) for r, c in layer)
    assert alg == pytest.approx(4.616e12, rel=1e-3)
    assert 0.9 * alg < exe < alg
    # a 128 x 2560 head on the small kernel: 128 x 128 tiles, 20 chunks of 128 columns
    per_it = 2 * 128 * 128 * 2560 * 2 + 2 * 128 ** 3
    assert bench.ns_executed_flops(128, 2560, 5, small=True) == 5 * per_it
    assert bench.ns_executed_flops(100, 2500, 1, small=True) == per_it


def test_both_arms_state_the_same_config():
    spec = bench.workload_spec("layer")
    a, b = bench.arm_config(spec, 1), bench.arm_config(bench.workload_spec("layer"), 1)
    assert a == b and a["matrices_per_step"] == 7 and a["elements_per_step"] == 100_925_440
    assert a["l2"].startswith("inputs 1.01 GB")
    assert bench.offload_config(1)["matrices_per_step"] == 252


def test_compulsory_bytes_of_the_small_kernel():
    # 1728 heads of 128 x 2560, fp32 W, bf16 G: weights read and written (8 B) plus
    # X0 (2 B), or, with the momentum in the kernel, G (2 B) and M read and written (8 B)
    t = [(128, 2560, 1728)]
    e = 128 * 2560 * 1728
    assert bench.ns_compulsory_bytes(t, [4], [2], False) == 10 * e
    assert bench.ns_compulsory_bytes(t, [4], [2], True) == 18 * e


def test_launches_per_step():
    class Nsm:
        def __init__(self, kinds):
            self.kinds = kinds

        def muon_get_bucket_info(self, plan, b):
            return _Bucket(*self.kinds[b])

    class Info:
        n_buckets = 3

    nsm = Nsm([(0, 0), (1, 0), (1, 1)])   # GEMM bucket; small kernel after the momentum kernel; fused
    assert bench.launches_per_step(nsm, None, Info()) == (2 + 15) + (2 + 1) + 1
    assert bench.launches_per_step(nsm, None, Info(), ns_only=True) == 15 + 1 + 1


def test_compulsory_bytes_of_the_gram_kernel():
    # the gram method reads X0 twice (the Gram, then U = R X0): 12 B per element with
    # the momentum kernel first; computing the momentum itself it writes X0 once and
    # reads it back: G 2 + M 8 + X0 4 + W 8 = 22
    t = [(128, 2560, 1728)]
    e = 128 * 2560 * 1728
    assert bench.ns_compulsory_bytes(t, [4], [2], False, "gram") == 12 * e
    assert bench.ns_compulsory_bytes(t, [4], [2], True, "gram") == 22 * e


def test_head_traffic_scales_by_matrices():
    if bench.head_traffic("gram", 336) is None:
        pytest.skip("the gram kernel's sources changed since the capture")
    # the capture: one launch over 7 layers (336 matrices), read 868.6 MB, write 385.4 MB
    assert bench.head_traffic("gram", 336) == pytest.approx(868.6e6 + 385.4e6)
    assert bench.head_traffic("gram", 1728) == pytest.approx((868.6e6 + 385.4e6) * 1728 / 336)
