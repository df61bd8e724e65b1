"""The single-launch Newton-Schulz kernel for matrices of at most 128 rows (wide
form) against the fp64 oracle, next to the grouped GEMM launches on the same
inputs.

Every case runs the same seeded workload twice, once per kernel path, and checks
each step of each path against the oracle per logical matrix (momentum within 1
ulp, weight update within 3e-2 relative Frobenius error).  The shapes reach the
kernel's edges: m < 128 (rows of the 128-row box zero-filled), n not a multiple
of the 64-column chunk, exactly one chunk, n above 4096, tall matrices (the
update transposed back), more matrices than CTAs, several groups in one launch,
one and six iterations, and each of the three products isolated by coefficients.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import (TOL_BF16, Workload, f32, nsm, oracle_constants, rel_fro, run_steps, ulp_distance,
                      widen)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    return nsm()


def _cfg(m, kernel):
    return m.muon_config_default(ns_kernel=kernel)


def _assert_path(m, wl, kernel, cap=512 << 20):
    plan = m.muon_plan(wl.plan_shapes(), bucket_cap_bytes=cap, config=_cfg(m, kernel))
    want = 1 if kernel == m.MUON_NS_KERNEL_AUTO else 0
    info = m.muon_get_plan_info(plan)
    assert all(m.muon_get_bucket_info(plan, b).ns_single_kernel == want for b in range(info.n_buckets))


KERNELS = ["AUTO", "GEMM"]


def _kernel(m, name):
    return m.MUON_NS_KERNEL_AUTO if name == "AUTO" else m.MUON_NS_KERNEL_GEMM


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("shapes", [
    [(128, 2560, 4)],                 # per-head shape
    [(100, 700), (3, 5)],             # ragged m and n, two groups
    [(128, 64), (64, 128)],           # exactly one chunk; a tall matrix
    [(96, 1000, 3), (2000, 48)],      # tall 2000 x 48 -> wide 48 x 2000
    [(128, 4100)],                    # n above 4096, ragged last chunk
    [(1, 64), (64, 1), (1, 1)],       # single rows and columns
])
def test_small_kernel_matches_oracle(m, shapes, kernel):
    wl = Workload(shapes, m_sigma=0.02, g_sigma=1e-3)
    k = _kernel(m, kernel)
    _assert_path(m, wl, k)
    ulp, rel = run_steps(m, wl, steps=2, cfg=_cfg(m, k))
    assert ulp <= 1 and rel <= TOL_BF16


def _fused_cfg(m):
    return m.muon_config_default(ns_kernel=m.MUON_NS_KERNEL_AUTO, ns_momentum_fused=1)


def _assert_momentum_fused(m, wl, want, cap=512 << 20):
    plan = m.muon_plan(wl.plan_shapes(), bucket_cap_bytes=cap, config=_fused_cfg(m))
    info = m.muon_get_plan_info(plan)
    got = [m.muon_get_bucket_info(plan, b).momentum_in_ns_kernel for b in range(info.n_buckets)]
    assert got == [want] * info.n_buckets


# The small kernel computes the momentum itself in its first pass over each matrix
# (bf16 gradients, wide matrices, n a multiple of 8): G and M staged 32 columns at
# a time, M written back, X0 into the ring stage and the workspace, the norm summed
# in the kernel.  Momentum within 1 ulp and updates within 3e-2 of the oracle.
@pytest.mark.parametrize("shapes", [
    [(128, 2560, 4)],                 # per-head shape: 20 whole chunks
    [(100, 704), (3, 8)],             # m < 128 (rows zero in the ring), n = 5.5 chunks; one 8-column row block
    [(128, 136, 2), (1, 64)],         # one chunk and one quarter; a single row
    [(64, 4104)],                     # n above 4096, a last chunk of 8 columns
    [(96, 256, 3), (32, 512, 2), (128, 128), (16, 1024, 5)],   # four groups in one launch
])
def test_fused_momentum_matches_oracle(m, shapes):
    wl = Workload(shapes, m_sigma=0.02, g_sigma=1e-3)
    _assert_path(m, wl, m.MUON_NS_KERNEL_AUTO)
    _assert_momentum_fused(m, wl, 1)
    ulp, rel = run_steps(m, wl, steps=3, cfg=_fused_cfg(m))
    assert ulp <= 1 and rel <= TOL_BF16


@pytest.mark.parametrize("opts", [dict(form="sgd"), dict(nesterov=False), dict(wd=0.1, mu=0.5),
                                  dict(ns_steps=1), dict(ns_steps=6)])
def test_fused_momentum_options(m, opts):
    wl = Workload([(128, 640, 3), (64, 1000 + 24)], m_sigma=0.02, g_sigma=1e-3)
    _assert_momentum_fused(m, wl, 1)
    ulp, rel = run_steps(m, wl, steps=2, cfg=_fused_cfg(m), **opts)
    assert ulp <= 1 and rel <= TOL_BF16


def test_fused_momentum_more_matrices_than_ctas(m):
    # 400 + 3 matrices: each CTA runs the fused first pass for several matrices in turn
    wl = Workload([(16, 208, 400), (128, 304, 3)], m_sigma=0.02, g_sigma=1e-3)
    _assert_momentum_fused(m, wl, 1, cap=0)
    ulp, rel = run_steps(m, wl, steps=2, cfg=_fused_cfg(m), cap=0)
    assert ulp <= 1 and rel <= TOL_BF16


def test_fused_momentum_nonfinite_matrix_is_skipped(m):
    import torch
    wl = Workload([(64, 128, 3), (32, 256)], m_sigma=0.02, g_sigma=1e-3)
    _assert_momentum_fused(m, wl, 1)
    W0 = [t.clone() for t in wl.dW]
    g = wl.dG[0].clone()
    g[1, 5, 7] = float("nan")
    plan = m.muon_plan(wl.plan_shapes(), config=_fused_cfg(m))
    m.allocate_workspace(plan)
    m.muon_step(plan, wl.dW, [g, wl.dG[1]], wl.dM, 0.02, 0.95, True, 0.0, 5)
    st, nf = m.muon_sync(plan)
    assert st == m.MUON_WARN_NONFINITE and nf == 1
    assert torch.equal(wl.dW[0][1], W0[0][1])
    assert not torch.equal(wl.dW[0][0], W0[0][0]) and not torch.equal(wl.dW[1], W0[1])
    assert torch.isfinite(wl.dW[0]).all() and torch.isfinite(wl.dW[1]).all()


def test_fused_and_separate_momentum_agree(m):
    # one set of bf16 gradients given twice: as bf16 with ns_momentum_fused (the
    # small kernel computes the momentum) and widened to fp32 (the momentum kernel
    # runs first, as for any fp32 gradient).  Both round the same fp32 operations, so the new momentum is
    # bit-identical; the updates differ only through the order of the norm's sums.
    import torch
    outs = []
    for fused in (True, False):
        wl = Workload([(128, 2560, 3), (64, 512)], m_sigma=0.02, g_sigma=1e-3)
        cfg = _fused_cfg(m)
        if not fused:
            cfg.grad_dtype = m.MUON_DTYPE_F32
            wl.dG = [g.float() for g in wl.dG]
        plan = m.muon_plan(wl.plan_shapes(), config=cfg)
        assert m.muon_get_bucket_info(plan, 0).momentum_in_ns_kernel == int(fused)
        m.allocate_workspace(plan)
        W0 = [w.clone() for w in wl.dW]
        m.muon_step(plan, wl.dW, wl.dG, wl.dM, 0.02, 0.95, True, 0.0, 5)
        assert m.muon_sync(plan) == (m.MUON_OK, 0)
        torch.cuda.synchronize()
        outs.append(([w - w0 for w, w0 in zip(wl.dW, W0)], [x.clone() for x in wl.dM]))
    (dw_f, m_f), (dw_s, m_s) = outs
    for a, b in zip(m_f, m_s):
        assert torch.equal(a, b)
    for a, b in zip(dw_f, dw_s):
        for j in range(a.shape[0]):
            assert rel_fro(a[j].double().cpu().numpy(), b[j].double().cpu().numpy()) <= 1e-2


@pytest.mark.parametrize("kernel", KERNELS)
def test_more_matrices_than_ctas(m, kernel):
    # 400 + 3 matrices in one launch: each CTA takes several, of two groups
    wl = Workload([(16, 200, 400), (128, 300, 3)], m_sigma=0.02, g_sigma=1e-3)
    k = _kernel(m, kernel)
    _assert_path(m, wl, k, cap=0)
    run_steps(m, wl, cfg=_cfg(m, k), cap=0)


@pytest.mark.parametrize("waves, extra", [(4, 0), (2, 5)])
def test_start_stagger_cases(m, waves, extra):
    # matrix counts that take each branch of the start stagger: every CTA with as many
    # matrices, from four per CTA (the second half of the CTAs start later), and some
    # CTAs with one matrix fewer (those start later); no result depends on it
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    wl = Workload([(128, 256, waves * sms + extra)], m_sigma=0.02, g_sigma=1e-3)
    run_steps(m, wl, cfg=_cfg(m, m.MUON_NS_KERNEL_AUTO), cap=0)
    wl = Workload([(96, 512, waves * sms + extra)], m_sigma=0.02, g_sigma=1e-3)
    run_steps(m, wl, cfg=m.muon_config_default(ns_method=m.MUON_NS_METHOD_GRAM), cap=0, method="gram")


@pytest.mark.parametrize("ns_steps", [1, 2, 6])
def test_iteration_counts(m, ns_steps):
    wl = Workload([(128, 1024, 2), (64, 333)], m_sigma=0.02, g_sigma=1e-3)
    run_steps(m, wl, ns_steps=ns_steps, cfg=_cfg(m, m.MUON_NS_KERNEL_AUTO))


@pytest.mark.parametrize("coeffs", [(1.0, 0.0, 0.0), (0.0, 1.0, 0.0), (0.0, 0.0, 1.0), (0.5, -0.25, 0.125)])
@pytest.mark.parametrize("ns_steps", [1, 2])
def test_each_product_isolated(m, coeffs, ns_steps):
    # (1,0,0): the a X term only; (0,1,0): A X (Gram and UPDATE); (0,0,1): A A X
    # (Gram, A A and UPDATE).  Two iterations also exercise the fused Gram.
    # W starts at 0 so that the small update is not lost in the rounding of W.
    wl = Workload([(128, 640), (96, 200, 2), (500, 40)], w_sigma=0.0, g_sigma=1.0, g_dtype=synth.F32)
    run_steps(m, wl, ns_steps=ns_steps, coeffs=coeffs, mu=0.0, nesterov=False,
              cfg=_cfg(m, m.MUON_NS_KERNEL_AUTO))


def test_bf16_weights_from_zero_hold_the_update_tolerance(m):
    # W0 = 0: the bf16 rounding of W_new is at most 2^-8 of the update, so the
    # bound stays within 3.5e-2 of ||dW|| (the small kernel's per-warp bf16 update)
    from gpu_util import TOL_BF16_W
    wl = Workload([(128, 512, 3), (512, 100), (64, 2560, 2)], w_sigma=0.0, w_dtype=synth.BF16, g_sigma=1e-3)
    k = m.MUON_NS_KERNEL_AUTO
    _assert_path(m, wl, k, cap=0)
    ulp, rel = run_steps(m, wl, cfg=_cfg(m, k), cap=0, bf16_max_bound=TOL_BF16_W)
    assert ulp <= 1 and rel <= TOL_BF16_W
    wl = Workload([(128, 512, 3), (512, 100)], w_sigma=0.02, w_dtype=synth.BF16, g_sigma=1e-3)
    ulp, rel = run_steps(m, wl, lr=1.0, wd=0.1, cfg=_cfg(m, k), cap=0, bf16_max_bound=TOL_BF16_W)
    assert ulp <= 1 and rel <= TOL_BF16_W


def test_bf16_weights_and_options(m):
    wl = Workload([(128, 512, 3), (512, 100)], w_dtype=synth.BF16, g_dtype=synth.F32, g_sigma=1e-3)
    run_steps(m, wl, steps=2, wd=0.1, cfg=_cfg(m, m.MUON_NS_KERNEL_AUTO))
    wl = Workload([(128, 512, 3), (512, 100)], m_sigma=0.02, g_sigma=1e-3)
    run_steps(m, wl, steps=2, form="sgd", nesterov=False, cfg=_cfg(m, m.MUON_NS_KERNEL_AUTO))


def test_offload_emit_through_small_kernel(m):
    import torch
    wl = Workload([(128, 2560, 6), (700, 100)], m_sigma=0.02, g_sigma=1e-3)
    cfg = m.muon_config_default(offload=1, max_inflight=2, timing=1)
    plan = m.muon_plan(wl.plan_shapes(), bucket_cap_bytes=1 << 20, config=cfg)
    info = m.muon_get_plan_info(plan)
    assert info.n_buckets >= 3
    assert all(m.muon_get_bucket_info(plan, b).ns_single_kernel == 1 for b in range(info.n_buckets))
    m.allocate_workspace(plan)

    def pinned(arr, code):
        if code == synth.BF16:
            return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).pin_memory()
        return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).pin_memory()

    hG = [pinned(g, wl.g_dtype) for g in wl.G]
    hM = [pinned(x, synth.F32) for x in wl.M]
    hU = [torch.empty(x.shape, dtype=torch.float32).pin_memory() for x in wl.M]
    m.muon_offload_step(plan, hG, hM, hU, 0.95, True, 5, timeout_ms=120_000)
    mu32, omu = oracle_constants(0.95, "ema")
    coeffs = tuple(f32(v) for v in oracle.DEFAULT_COEFFS)
    for i, (r, c, k) in enumerate(wl.shapes):
        for j in range(k):
            G = widen(wl.G[i][j], wl.g_dtype)
            Mo = oracle.momentum_update(wl.M[i][j], G, mu32, one_minus_mu=omu)
            assert int(ulp_distance(hM[i][j].numpy(), Mo).max()) <= 1
            V = oracle.nesterov_blend(Mo, G, mu32, True, one_minus_mu=omu)
            Uo = oracle.offload_update(oracle.newton_schulz(V, coeffs=coeffs, eps=f32(1e-7)), r, c)
            assert rel_fro(hU[i][j].numpy(), Uo) <= TOL_BF16, (i, j)


def test_both_paths_agree_closely(m):
    # both paths round A, B and X to bf16 at the same points and differ only in
    # the order of fp32 accumulation (and the mirrored Gram of the GEMM path), so
    # their updates differ by far less than the tolerance to the oracle
    import torch
    outs = []
    for kernel in (m.MUON_NS_KERNEL_AUTO, m.MUON_NS_KERNEL_GEMM):
        wl = Workload([(128, 2560, 3)], m_sigma=0.02, g_sigma=1e-3)
        W0 = wl.dW[0].clone()
        plan = m.muon_plan(wl.plan_shapes(), config=_cfg(m, kernel))
        m.allocate_workspace(plan)
        m.muon_step(plan, wl.dW, wl.dG, wl.dM, 0.02, 0.95, True, 0.0, 5)
        torch.cuda.synchronize()
        outs.append((wl.dW[0] - W0).double().cpu().numpy())
    for j in range(3):
        assert rel_fro(outs[0][j], outs[1][j]) <= 2e-2
