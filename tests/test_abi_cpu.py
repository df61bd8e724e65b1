"""C-ABI library: it loads without a GPU, exports what include/muon.h declares, and
its host-side planner and argument checks behave as documented (no kernel runs)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def nsm():
    import newton_schulz_muon_gb300.build as b
    b.build()
    import newton_schulz_muon_gb300 as m
    return m


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "muon.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(muon_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(nsm):
    names = _declared_functions()
    assert "muon_plan" in names and "muon_step" in names and "muon_offload_step" in names
    lib = ctypes.CDLL(nsm.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_config_default(nsm):
    c = nsm.muon_config_default()
    assert (c.ns_a, c.ns_b, c.ns_c) == pytest.approx((3.4445, -4.7750, 2.0315))
    assert c.eps == pytest.approx(1e-7)
    assert c.ns_precision == nsm.MUON_NS_BF16 and c.momentum_form == nsm.MUON_MOMENTUM_EMA
    assert c.grad_dtype == nsm.MUON_DTYPE_BF16 and c.param_dtype == nsm.MUON_DTYPE_F32
    assert c.max_inflight == 1 and c.skip_nonfinite == 1 and c.offload == 0
    assert c.ns_kernel == nsm.MUON_NS_KERNEL_AUTO
    assert c.ns_momentum_fused == 0 and c.ns_method == nsm.MUON_NS_METHOD_STANDARD


QWEN3_4B_LAYER = [(4096, 2560), (1024, 2560), (1024, 2560), (2560, 4096),
                  (9728, 2560), (9728, 2560), (2560, 9728)]


def test_plan_one_qwen3_4b_layer(nsm):
    p = nsm.muon_plan(QWEN3_4B_LAYER, bucket_cap_bytes=512 << 20)
    info = nsm.muon_get_plan_info(p)
    assert info.n_tensors == 7 and info.n_matrices == 7
    assert info.n_groups == 3            # (2560,4096) q+o, (1024,2560) k+v, (2560,9728) gate+up+down
    assert info.n_buckets == 1
    b = nsm.muon_get_bucket_info(p, 0)
    assert b.n_matrices == 7 and b.n_groups == 3
    assert b.bytes == 2 * sum(r * c for r, c in QWEN3_4B_LAYER)
    assert info.workspace_bytes >= 2 * b.bytes  # X ping-pong, plus A and B


def test_plan_experts_across_layers(nsm):
    shapes = []
    for _ in range(48):
        shapes += [(768, 2048, 128), (768, 2048, 128), (2048, 768, 128)]
    p = nsm.muon_plan(shapes, bucket_cap_bytes=512 << 20)
    info = nsm.muon_get_plan_info(p)
    assert info.n_matrices == 18432 and info.n_groups == 1
    per = (512 << 20) // (768 * 2048 * 2)
    assert per == 170
    assert info.n_buckets == -(-18432 // per) == 109
    assert info.max_bucket_matrices == 170
    assert nsm.muon_get_bucket_info(p, 108).n_matrices == 18432 - 108 * 170


def test_plan_per_head_one_batch(nsm):
    shapes = [(128, 2560, 48)] * 36
    p = nsm.muon_plan(shapes, bucket_cap_bytes=0)
    info = nsm.muon_get_plan_info(p)
    assert info.n_matrices == 1728 and info.n_buckets == 1 and info.n_groups == 1


def test_small_matrix_kernel_selection(nsm):
    # every group m <= 128 in the wide form (tall ones count by their column count)
    p = nsm.muon_plan([(128, 2560, 48)] * 2 + [(2000, 48), (3, 5)], bucket_cap_bytes=0)
    assert nsm.muon_get_bucket_info(p, 0).ns_single_kernel == 1
    # one group with m = 129 sends the bucket to the grouped GEMM launches
    assert nsm.muon_get_bucket_info(nsm.muon_plan([(128, 512), (129, 512)], bucket_cap_bytes=0),
                                    0).ns_single_kernel == 0
    # per bucket: the layer's buckets of k/v (m = 1024) stay on the GEMMs
    p = nsm.muon_plan([(64, 256, 4), (1024, 2560)], bucket_cap_bytes=200_000)
    kinds = [nsm.muon_get_bucket_info(p, b).ns_single_kernel for b in range(nsm.muon_get_plan_info(p).n_buckets)]
    assert kinds[0] == 1 and kinds[-1] == 0
    # forced off, and not used for 3xTF32
    cfg = nsm.muon_config_default(ns_kernel=nsm.MUON_NS_KERNEL_GEMM)
    assert nsm.muon_get_bucket_info(nsm.muon_plan([(128, 2560, 4)], config=cfg), 0).ns_single_kernel == 0
    cfg = nsm.muon_config_default(ns_precision=nsm.MUON_NS_TF32X3)
    assert nsm.muon_get_bucket_info(nsm.muon_plan([(128, 2560, 4)], config=cfg), 0).ns_single_kernel == 0
    with pytest.raises(nsm.MuonError):
        nsm.muon_plan([(4, 4)], config=nsm.muon_config_default(ns_kernel=2))


def test_plan_full_model_offload_layout(nsm):
    shapes = QWEN3_4B_LAYER * 36
    cfg = nsm.muon_config_default(offload=1)
    p = nsm.muon_plan(shapes, bucket_cap_bytes=512 << 20, config=cfg)
    info = nsm.muon_get_plan_info(p)
    assert info.n_matrices == 252
    assert info.max_bucket_bytes <= 512 << 20
    total = sum(nsm.muon_get_bucket_info(p, i).n_matrices for i in range(info.n_buckets))
    assert total == 252
    p2 = nsm.muon_plan(shapes, bucket_cap_bytes=512 << 20)
    assert nsm.muon_get_plan_info(p).workspace_bytes > nsm.muon_get_plan_info(p2).workspace_bytes


def test_plan_cap_smaller_than_a_matrix(nsm):
    p = nsm.muon_plan([(64, 64, 5)], bucket_cap_bytes=100)
    assert nsm.muon_get_plan_info(p).n_buckets == 5


def test_plan_labels_never_share_a_bucket(nsm):
    p = nsm.muon_plan([(32, 64), (32, 64), (32, 64)], groups=[0, 1, 0], bucket_cap_bytes=0)
    info = nsm.muon_get_plan_info(p)
    assert info.n_groups == 2
    assert info.n_buckets >= 2


def test_plan_run_limit_splits_buckets(nsm):
    p = nsm.muon_plan([(16, 32)] * 100, bucket_cap_bytes=0)
    info = nsm.muon_get_plan_info(p)
    assert info.n_buckets == 2 and info.max_bucket_matrices == 64


def test_plan_rejects_bad_arguments(nsm):
    for shapes in ([(0, 5)], [(5, 0)], [(4, 4, 0)], [(4, 4, 2, 10)]):
        with pytest.raises(nsm.MuonError) as e:
            nsm.muon_plan(shapes)
        assert e.value.status == nsm.MUON_ERR_INVALID
    with pytest.raises(nsm.MuonError):
        nsm.muon_plan([(4, 4)], config=nsm.muon_config_default(grad_dtype=7))
    with pytest.raises(nsm.MuonError):
        nsm.muon_plan([(4, 4)], config=nsm.muon_config_default(max_inflight=3))
    out = ctypes.c_void_p()
    assert nsm.lib.muon_plan(None, 0, None, 0, None, ctypes.byref(out)) == nsm.MUON_ERR_INVALID


def test_step_without_workspace_is_refused(nsm):
    p = nsm.muon_plan([(8, 16)])
    with pytest.raises(nsm.MuonError) as e:
        nsm.muon_step(p, [16], [32], [48], 0.02, 0.95, True, 0.0, stream=0)
    assert e.value.status == nsm.MUON_ERR_NO_WORKSPACE
    st = nsm.lib.muon_sync(p.handle, None, None)
    assert st == nsm.MUON_ERR_NO_WORKSPACE


def test_selftest_arguments_are_checked(nsm):
    p = nsm.muon_plan([(8, 16)])
    assert nsm.lib.muon_selftest_wait_timeout(None, 1000, None) == nsm.MUON_ERR_INVALID
    for bad in (0, -5, 1_000_001):
        assert nsm.lib.muon_selftest_wait_timeout(p.handle, bad, None) == nsm.MUON_ERR_INVALID
    # no workspace bound: refused before anything is enqueued
    assert nsm.lib.muon_selftest_wait_timeout(p.handle, 1000, None) == nsm.MUON_ERR_NO_WORKSPACE


def test_status_strings(nsm):
    for code in (0, 1, -1, -2, -3, -4, -5, -6, -7):
        assert nsm.muon_status_string(code)
    assert nsm.muon_status_string(-99) == "unknown status"


def test_synth_library_loads(nsm):
    lib = ctypes.CDLL(os.path.join(ROOT, "synth", "libmuonsynth.so"))
    assert hasattr(lib, "synth_fill_normal") and hasattr(lib, "synth_philox")


def test_minimax_schedule_agrees_with_the_oracle(nsm):
    # two constructions written apart (closed-form critical points here, a dense
    # grid in the oracle) agree to the fp32 rounding of the coefficients
    import oracle
    for lower, safety in ((1e-3, 1.0), (1e-2, 1.0), (1e-3, 1.02)):
        co, err = nsm.muon_polar_express_coefficients(7, lower, safety)
        oco, oerr = oracle.polar_express_schedule(7, lower, safety)
        for k in range(7):
            assert co[k] == pytest.approx(oco[k], rel=2e-6, abs=1e-6), (lower, safety, k)
            assert err[k] == pytest.approx(oerr[k], rel=1e-5, abs=1e-12), (lower, safety, k)


def test_schedule_arguments_are_checked(nsm):
    out = (ctypes.c_float * 48)()
    for n, lo, sf in ((0, 1e-3, 1.0), (17, 1e-3, 1.0), (3, 0.0, 1.0), (3, 1.0, 1.0), (3, 1e-3, 0.9),
                      (3, 1e-3, 2.5), (3, float("nan"), 1.0)):
        assert nsm.lib.muon_polar_express_coefficients(n, lo, sf, out, None) == nsm.MUON_ERR_INVALID, (n, lo, sf)
    assert nsm.lib.muon_polar_express_coefficients(3, 1e-3, 1.0, None, None) == nsm.MUON_ERR_INVALID
    p = nsm.muon_plan([(8, 16)])
    nsm.muon_set_ns_schedule(p, [(3.0, -3.0, 1.0)] * 16)
    nsm.muon_set_ns_schedule(p, [])
    for bad in ([(1.0, 2.0, 3.0)] * 17, [(1.0, float("inf"), 0.0)], [(float("nan"), 0.0, 0.0)]):
        with pytest.raises(nsm.MuonError) as e:
            nsm.muon_set_ns_schedule(p, bad)
        assert e.value.status == nsm.MUON_ERR_INVALID
    assert nsm.lib.muon_set_ns_schedule(None, out, 1) == nsm.MUON_ERR_INVALID
    assert nsm.lib.muon_set_ns_schedule(p.handle, None, 2) == nsm.MUON_ERR_INVALID


def test_gram_method_plans_only_small_matrix_buckets(nsm):
    cfg = nsm.muon_config_default(ns_method=nsm.MUON_NS_METHOD_GRAM)
    p = nsm.muon_plan([(128, 2560, 48), (700, 96)], config=cfg)      # every matrix has m <= 128
    assert all(nsm.muon_get_bucket_info(p, b).ns_single_kernel for b in range(nsm.muon_get_plan_info(p).n_buckets))
    for bad in ([(256, 512)], [(128, 512), (4096, 2560)]):
        with pytest.raises(nsm.MuonError) as e:
            nsm.muon_plan(bad, config=cfg)
        assert e.value.status == nsm.MUON_ERR_UNSUPPORTED
    with pytest.raises(nsm.MuonError) as e:
        nsm.muon_plan([(128, 512)], config=nsm.muon_config_default(ns_method=2))
    assert e.value.status == nsm.MUON_ERR_INVALID
