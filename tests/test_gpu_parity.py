"""GPU path vs the fp64 oracle, element by element, through the C ABI.

Tolerances: fp32 momentum within 1 ulp of the oracle's rounded value (teacher
forced: each step starts both sides from the GPU's previous state); per logical
matrix, the relative Frobenius error of the weight update within 3e-2 for bf16
Newton-Schulz.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import (TOL_BF16, TOL_BF16_W, Workload, f32, nsm, oracle_constants, rel_fro, run_steps,
                      to_numpy, torch_from, ulp_distance, widen)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    return nsm()


def _run(m, wl, **kw):
    return run_steps(m, wl, **kw)


def test_synth_device_fill_is_bit_identical(m):
    import torch
    for dtype, code in ((torch.float32, synth.F32), (torch.bfloat16, synth.BF16)):
        for (stream, step, start, n, sigma) in ((3, 0, 0, 100_003, 1.0), (17, 5, 12_345, 4097, 0.02),
                                                (2, 1, 1, 1, 1e-3)):
            t = torch.empty(n, dtype=dtype, device="cuda")
            synth.fill_normal_cuda(t, synth.SEED, stream, step, sigma, start=start)
            want = synth.tensor(synth.SEED, stream, step, (n,), sigma, code, start=start)
            got = to_numpy(t, code)
            assert np.array_equal(got.view(np.uint32 if code == synth.F32 else np.uint16),
                                  want.view(np.uint32 if code == synth.F32 else np.uint16))
    rng = np.random.default_rng(0)
    ctr = rng.integers(0, 2 ** 32, size=(1000, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 2 ** 32, size=(1000, 2), dtype=np.uint64).astype(np.uint32)
    got = synth.philox_cuda(ctr, key)
    for i in range(0, 1000, 97):
        want = synth.philox4x32_10([ctr[i, 0]], [ctr[i, 1]], [ctr[i, 2]], [ctr[i, 3]], key[i, 0], key[i, 1])
        assert [int(w[0]) for w in want] == got[i].tolist()


def test_single_256x512_three_steps(m):
    # fp32 weights N(0,0.02), fp32 gradients N(0,1) fresh each step, zero momentum,
    # mu 0.95 Nesterov, lr 0.02, wd 0, 5 quintic iterations.
    wl = Workload([(256, 512)], w_sigma=0.02, g_sigma=1.0, g_dtype=synth.F32)
    ulp, rel = _run(m, wl, steps=3)
    assert ulp <= 1 and rel <= TOL_BF16


@pytest.mark.parametrize("coeffs", [(1.0, 0.0, 0.0), (0.0, 1.0, 0.0), (0.0, 0.0, 1.0), (0.5, -0.25, 0.125)])
def test_one_iteration_isolates_each_gemm(m, coeffs):
    # (1,0,0): UPDATE epilogue only; (0,1,0): GRAM + UPDATE; (0,0,1): GRAM + POLY + UPDATE.
    # W starts at 0 so that the (tiny, for a monomial) update is not lost in the
    # fp32 rounding of W.
    wl = Workload([(192, 320), (320, 192), (64, 640)], w_sigma=0.0, g_sigma=1.0, g_dtype=synth.F32)
    _run(m, wl, ns_steps=1, coeffs=coeffs, mu=0.0, nesterov=False)


def test_no_iteration_is_plain_normalisation(m):
    wl = Workload([(100, 300), (300, 100)], g_sigma=1.0, g_dtype=synth.F32)
    _run(m, wl, ns_steps=0)


@pytest.mark.parametrize("shape", [(300, 200), (100, 700), (130, 130), (1, 64), (64, 1), (777, 129),
                                   (129, 1000), (5, 3)])
def test_ragged_shapes(m, shape):
    wl = Workload([shape], m_sigma=0.02, g_sigma=1e-3)
    _run(m, wl, steps=2)


def test_batched_groups_and_fused_tensors(m):
    # several tensors, counts > 1 (experts / heads), three same-shape groups, small cap -> many buckets
    wl = Workload([(96, 256, 5), (256, 96, 3), (128, 384, 4), (384, 128, 2), (64, 64, 7)],
                  m_sigma=0.02, g_sigma=1e-3)
    _run(m, wl, cap=300_000)


@pytest.mark.parametrize("opts", [dict(form="sgd"), dict(nesterov=False), dict(wd=0.1),
                                  dict(ns_steps=1), dict(ns_steps=6), dict(mu=0.5)])
def test_options(m, opts):
    wl = Workload([(200, 330), (330, 200)], m_sigma=0.02, g_sigma=1e-3)
    _run(m, wl, steps=2, **opts)


def test_bf16_weights_fp32_grads(m):
    wl = Workload([(256, 512), (512, 256)], w_dtype=synth.BF16, g_dtype=synth.F32, g_sigma=1e-3)
    _run(m, wl, steps=2)


@pytest.mark.parametrize("g_dtype", [synth.F32, synth.BF16])
def test_bf16_weights_from_zero_hold_the_update_tolerance(m, g_dtype):
    # W0 = 0: the bf16 rounding of W_new is at most 2^-8 of the update itself, so
    # the bound stays within 3.5e-2 of ||dW|| and a 10 % error in the update fails
    wl = Workload([(256, 512), (512, 256), (130, 700), (700, 130, 2)], w_sigma=0.0, w_dtype=synth.BF16,
                  g_dtype=g_dtype, g_sigma=1.0 if g_dtype == synth.F32 else 1e-3)
    ulp, rel = _run(m, wl, bf16_max_bound=TOL_BF16_W)
    assert ulp <= 1 and rel <= TOL_BF16_W


def test_bf16_weights_large_lr_with_decay_hold_the_update_tolerance(m):
    # W ~ N(0, 0.02) with lr 1 and wd 0.1: the update (about lr * ||U||) dominates
    # the bf16 rounding of W, and the decay term rides on the old bf16 W
    wl = Workload([(256, 512), (512, 256), (200, 330, 2)], w_sigma=0.02, w_dtype=synth.BF16, g_sigma=1e-3)
    ulp, rel = _run(m, wl, lr=1.0, wd=0.1, bf16_max_bound=TOL_BF16_W)
    assert ulp <= 1 and rel <= TOL_BF16_W


def _zero_one_matrix(wl, i, j):
    # G = M = 0 for matrix j of tensor i, on the host arrays and the device tensors
    wl.G[i][j] = 0
    wl.M[i][j] = 0
    wl.dG[i] = torch_from(wl.G[i], wl.g_dtype)
    wl.dM[i] = torch_from(wl.M[i], synth.F32)


@pytest.mark.parametrize("kernel,last", [("auto", 304), ("auto", 300), ("gemm", 300)])
@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_zero_matrix_in_a_bucket(m, kernel, last, wd):
    # an all-zero G and M: V = 0, so X0 = 0 / (0 + eps) = 0 and U = 0; the matrix
    # keeps its weights (wd = 0) or only decays (wd > 0), with nothing non-finite,
    # while the other matrices of the same bucket update as usual.  With n = 304 the
    # small kernel computes the momentum itself; with 300 the momentum kernel does.
    import torch
    wl = Workload([(128, 640, 3), (96, last)], m_sigma=0.02, g_sigma=1e-3)
    _zero_one_matrix(wl, 0, 1)
    W0 = wl.dW[0].clone()
    cfg = m.muon_config_default(ns_kernel=m.MUON_NS_KERNEL_AUTO if kernel == "auto" else m.MUON_NS_KERNEL_GEMM,
                                ns_momentum_fused=1)
    ulp, rel = _run(m, wl, wd=wd, cfg=cfg)
    assert ulp <= 1 and rel <= TOL_BF16
    assert torch.isfinite(wl.dW[0]).all() and torch.isfinite(wl.dM[0]).all()
    assert int((wl.dM[0][1] != 0).sum()) == 0
    if wd == 0.0:
        assert torch.equal(wl.dW[0][1], W0[1])
    assert not torch.equal(wl.dW[0][0], W0[0]) and not torch.equal(wl.dW[0][2], W0[2])


@pytest.mark.parametrize("shape,kernel,g_dtype", [((64, 128), "auto", synth.F32), ((64, 128), "auto", synth.BF16),
                                                  ((64, 128), "gemm", synth.F32), ((200, 330), "auto", synth.F32),
                                                  ((330, 200), "auto", synth.F32)])
def test_tiny_norm_where_eps_matters(m, shape, kernel, g_dtype):
    # ||V||_F ~ 1e-6, so eps = 1e-7 in X0 = V / (||V|| + eps) shrinks every singular
    # value by ~9 % and moves the update by > 10 % (checked on the oracle here):
    # the GPU must put eps where the oracle does to stay within 3e-2 (bf16
    # gradients: the small kernel computes the norm itself)
    r, c = shape
    sigma = 1e-6 / (0.0975 * np.sqrt(r * c))        # EMA + Nesterov from M = 0: V = 0.0975 G
    wl = Workload([shape], w_sigma=0.0, g_sigma=sigma, g_dtype=g_dtype)
    V = 0.0975 * widen(wl.G[0][0], g_dtype)
    assert 0.8e-6 < np.linalg.norm(V) < 1.25e-6
    U_eps, U_none = oracle.newton_schulz(V, eps=1e-7), oracle.newton_schulz(V, eps=0.0)
    assert rel_fro(U_eps, U_none) > 3 * TOL_BF16
    cfg = m.muon_config_default(ns_kernel=m.MUON_NS_KERNEL_AUTO if kernel == "auto" else m.MUON_NS_KERNEL_GEMM,
                                ns_momentum_fused=1)
    ulp, rel = _run(m, wl, cfg=cfg)
    assert ulp <= 1 and rel <= TOL_BF16


def test_per_head_interleaved_qkv_small(m):
    # 2 layers of an interleaved [Q0..Q3,K0,V0,...] projection: 2 kv groups x 6 heads x 128 rows
    wl = Workload([(128, 512, 12), (128, 512, 12)], m_sigma=0.02, g_sigma=1e-3)
    _run(m, wl, cap=0)


def test_deterministic(m):
    import torch
    outs = []
    for _ in range(2):
        wl = Workload([(384, 640, 2), (640, 384)], m_sigma=0.02, g_sigma=1e-3)
        plan = m.muon_plan(wl.plan_shapes())
        m.allocate_workspace(plan)
        m.muon_step(plan, wl.dW, wl.dG, wl.dM, 0.02, 0.95, True, 0.0, 5)
        torch.cuda.synchronize()
        outs.append([t.clone() for t in wl.dW + wl.dM])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_nonfinite_matrix_is_skipped_and_reported(m):
    import torch
    wl = Workload([(64, 128, 3)], m_sigma=0.02, g_sigma=1e-3)
    W0 = [t.clone() for t in wl.dW]
    g = wl.dG[0].clone()
    g[1, 5, 7] = float("nan")
    plan = m.muon_plan(wl.plan_shapes())
    m.allocate_workspace(plan)
    m.muon_step(plan, wl.dW, [g], wl.dM, 0.02, 0.95, True, 0.0, 5)
    st, nf = m.muon_sync(plan)
    assert st == m.MUON_WARN_NONFINITE and nf == 1
    assert torch.equal(wl.dW[0][1], W0[0][1])         # skipped
    assert not torch.equal(wl.dW[0][0], W0[0][0])     # others updated
    assert torch.isfinite(wl.dW[0]).all()
    st, nf = m.muon_sync(plan)                        # the status word was cleared
    assert st == m.MUON_OK and nf == 0


def test_argument_validation_on_device(m):
    import torch
    wl = Workload([(64, 128)])
    plan = m.muon_plan(wl.plan_shapes())
    m.allocate_workspace(plan)
    with pytest.raises(m.MuonError) as e:
        m.muon_step(plan, wl.dW, wl.dG, wl.dM[:0] + [0], 0.02, 0.95, True, 0.0)
    assert e.value.status == m.MUON_ERR_INVALID
    bad = torch.empty(64 * 128 + 1, dtype=torch.float32, device="cuda")[1:]
    with pytest.raises(m.MuonError):
        m.muon_step(plan, [bad], wl.dG, wl.dM, 0.02, 0.95, True, 0.0)
    with pytest.raises(m.MuonError):
        m.muon_step(plan, wl.dW, wl.dG, wl.dM, 0.02, 0.95, True, 0.0, ns_steps=17)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(m.MuonError) as e:
        m.muon_plan_bind_workspace(m.muon_plan(wl.plan_shapes()), small)
    assert e.value.status == m.MUON_ERR_NO_WORKSPACE


def test_device_wait_timeout_is_reported_and_the_context_stays_usable(m):
    # the failure path without a fault: a kernel's bounded wait runs out (a
    # barrier nothing arrives on, 20 ms limit), the status word records it,
    # muon_sync reports and clears it, and the next steps run and match the oracle
    import time
    import torch
    wl = Workload([(128, 640), (300, 200)], m_sigma=0.02, g_sigma=1e-3)
    plan = m.muon_plan(wl.plan_shapes())
    m.allocate_workspace(plan)
    t0 = time.perf_counter()
    m.muon_selftest_wait_timeout(plan, 20_000)
    with pytest.raises(m.MuonError) as e:
        m.muon_sync(plan)
    waited = time.perf_counter() - t0
    assert e.value.status == m.MUON_ERR_DEVICE
    assert 0.015 <= waited < 5.0
    assert m.muon_sync(plan) == (m.MUON_OK, 0)  # cleared by the read
    m.muon_step(plan, wl.dW, wl.dG, wl.dM, 0.02, 0.95, True, 0.0, 5)  # the same plan steps on
    assert m.muon_sync(plan) == (m.MUON_OK, 0)
    torch.cuda.synchronize()
    ulp, rel = run_steps(m, wl, steps=2)
    assert ulp <= 1 and rel <= TOL_BF16


# --- fp32 (3xTF32) Newton-Schulz mode: per-matrix tolerance 1e-4 --------------

@pytest.mark.parametrize("shapes", [[(256, 512)], [(300, 200), (100, 700)], [(128, 384, 3), (640, 384)],
                                    [(1, 64), (130, 130)]])
def test_tf32x3_mode(m, shapes):
    from gpu_util import TOL_TF32X3
    wl = Workload(shapes, m_sigma=0.02, g_sigma=1e-3)
    cfg = m.muon_config_default(ns_precision=m.MUON_NS_TF32X3)
    ulp, rel = _run(m, wl, cfg=cfg, tol=TOL_TF32X3, steps=2)
    assert rel <= TOL_TF32X3


@pytest.mark.parametrize("coeffs", [(1.0, 0.0, 0.0), (0.0, 1.0, 0.0), (0.0, 0.0, 1.0)])
def test_tf32x3_one_iteration_each_gemm(m, coeffs):
    from gpu_util import TOL_TF32X3
    wl = Workload([(192, 320), (320, 192)], w_sigma=0.0, g_sigma=1.0, g_dtype=synth.F32)
    cfg = m.muon_config_default(ns_precision=m.MUON_NS_TF32X3)
    _run(m, wl, cfg=cfg, ns_steps=1, coeffs=coeffs, mu=0.0, nesterov=False, tol=TOL_TF32X3)


# --- offload: pinned host gradients and momentum --------------------------------

def _pinned(arr, dtype_code):
    import torch
    if dtype_code == synth.BF16:
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32))
    return t.pin_memory()


def _offload(m, wl, cap, inflight, ns_steps=5, mu=0.95, zero_copy=0):
    import torch
    cfg = m.muon_config_default(offload=1, max_inflight=inflight, timing=1, offload_zero_copy=zero_copy)
    cfg.grad_dtype = wl.g_dtype
    plan = m.muon_plan(wl.plan_shapes(), bucket_cap_bytes=cap, config=cfg)
    m.allocate_workspace(plan)
    hG = [_pinned(g, wl.g_dtype) for g in wl.G]
    hM = [_pinned(x, synth.F32) for x in wl.M]
    hU = [torch.empty(x.shape, dtype=torch.float32).pin_memory() for x in wl.M]
    m.muon_offload_step(plan, hG, hM, hU, mu, True, ns_steps, timeout_ms=120_000)
    st = m.muon_get_stats(plan)
    return [x.numpy().copy() for x in hM], [u.numpy().copy() for u in hU], st, plan


def test_offload_matches_oracle_and_is_order_independent(m):
    shapes = [(256, 512), (300, 200, 2), (64, 640), (512, 128, 3)]
    wl = Workload(shapes, m_sigma=0.02, g_sigma=1e-3)
    M1, U1, st, plan = _offload(m, wl, cap=400_000, inflight=1)
    assert m.muon_get_plan_info(plan).n_buckets >= 3
    assert st.h2d_bytes > 0 and st.d2h_bytes > 0
    mu32, omu = oracle_constants(0.95, "ema")
    for i, (r, c, k) in enumerate(wl.shapes):
        for j in range(k):
            G = widen(wl.G[i][j], wl.g_dtype)
            Mo = oracle.momentum_update(wl.M[i][j], G, mu32, one_minus_mu=omu)
            assert int(ulp_distance(M1[i][j], Mo).max()) <= 1
            V = oracle.nesterov_blend(Mo, G, mu32, True, one_minus_mu=omu)
            Uo = oracle.offload_update(oracle.newton_schulz(V, coeffs=tuple(f32(v) for v in oracle.DEFAULT_COEFFS),
                                                            eps=f32(1e-7)), r, c)
            assert rel_fro(U1[i][j], Uo) <= TOL_BF16, (i, j)
    # two buckets in writeback while one computes gives the same bytes
    M2, U2, _, _ = _offload(m, wl, cap=400_000, inflight=2)
    for a, b in zip(M1 + U1, M2 + U2):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("shapes", [
    [(256, 512), (300, 200, 2), (64, 640), (512, 128, 3)],   # grouped GEMM buckets
    [(128, 1024, 4), (96, 700), (700, 96)],                  # small-matrix kernel buckets
])
def test_zero_copy_offload_is_bitwise_the_staged_one(m, shapes):
    # the same kernels read and write the pinned host buffers directly instead of
    # device staging slots: same bytes out, a smaller workspace, fewer launches of
    # nothing but copies
    wl = Workload(shapes, m_sigma=0.02, g_sigma=1e-3)
    M1, U1, st1, p1 = _offload(m, wl, cap=400_000, inflight=2)
    M2, U2, st2, p2 = _offload(m, wl, cap=400_000, inflight=2, zero_copy=1)
    for a, b in zip(M1 + U1, M2 + U2):
        assert np.array_equal(a, b)
    assert st2.h2d_bytes == st1.h2d_bytes and st2.d2h_bytes == st1.d2h_bytes
    assert m.muon_get_plan_info(p2).workspace_bytes < m.muon_get_plan_info(p1).workspace_bytes


def _offload_check(wl, hM_prev, hM, hU):
    """Every matrix of an offload step against the oracle, teacher forced from the
    momentum the step started from."""
    mu32, omu = oracle_constants(0.95, "ema")
    coeffs = tuple(f32(v) for v in oracle.DEFAULT_COEFFS)
    for i, (r, c, k) in enumerate(wl.shapes):
        for j in range(k):
            G = widen(wl.G[i][j], wl.g_dtype)
            Mo = oracle.momentum_update(hM_prev[i][j], G, mu32, one_minus_mu=omu)
            assert int(ulp_distance(hM[i][j], Mo).max()) <= 1, (i, j)
            V = oracle.nesterov_blend(Mo, G, mu32, True, one_minus_mu=omu)
            Uo = oracle.offload_update(oracle.newton_schulz(V, coeffs=coeffs, eps=f32(1e-7)), r, c)
            assert rel_fro(hU[i][j], Uo) <= TOL_BF16, (i, j)


def _offload_plan(m, wl, cap):
    import torch
    cfg = m.muon_config_default(offload=1, max_inflight=2)
    cfg.grad_dtype = wl.g_dtype
    plan = m.muon_plan(wl.plan_shapes(), bucket_cap_bytes=cap, config=cfg)
    m.allocate_workspace(plan)
    hG = [_pinned(g, wl.g_dtype) for g in wl.G]
    hM = [_pinned(x, synth.F32) for x in wl.M]
    hU = [torch.empty(x.shape, dtype=torch.float32).pin_memory() for x in wl.M]
    return plan, hG, hM, hU


def test_offload_timeout_then_recovers(m):
    # the failure path of the offload's bounded host wait, without a fault: a
    # kernel holds the compute stream for 300 ms (the failure-path self-test's
    # bounded wait on a barrier nothing arrives on), so the step cannot finish
    # within its 50 ms and returns MUON_ERR_TIMEOUT.  Its work completes later and
    # matches the oracle; the next step of the same plan matches it too.
    import torch
    wl = Workload([(256, 512, 3), (300, 200, 2), (128, 640, 4)], m_sigma=0.02, g_sigma=1e-3)
    plan, hG, hM, hU = _offload_plan(m, wl, cap=600_000)
    assert m.muon_get_plan_info(plan).n_buckets >= 3
    cs = torch.cuda.Stream()
    M0 = [x.numpy().copy() for x in hM]
    m.muon_selftest_wait_timeout(plan, 300_000, stream=cs)
    with pytest.raises(m.MuonError) as e:
        m.muon_offload_step(plan, hG, hM, hU, 0.95, True, 5, compute=cs, timeout_ms=50)
    assert e.value.status == m.MUON_ERR_TIMEOUT
    torch.cuda.synchronize()
    with pytest.raises(m.MuonError) as e:            # the self-test's own record
        m.muon_sync(plan, stream=cs)
    assert e.value.status == m.MUON_ERR_DEVICE
    M1 = [x.numpy().copy() for x in hM]
    _offload_check(wl, M0, M1, [u.numpy() for u in hU])
    m.muon_offload_step(plan, hG, hM, hU, 0.95, True, 5, compute=cs, timeout_ms=120_000)
    _offload_check(wl, M1, [x.numpy() for x in hM], [u.numpy() for u in hU])
    assert m.muon_sync(plan, stream=cs) == (m.MUON_OK, 0)


@pytest.mark.parametrize("nth", [0, 3, 6])
def test_offload_injected_copy_failure_then_recovers(m, nth):
    # a host-link copy that fails to enqueue (injected: the call reports it as if
    # cudaMemcpy2DAsync had failed).  Copies per bucket: an upload of G and of M
    # per run, then a writeback of M and of U' per run; the first bucket holds one
    # run (copies 0-3), the second two (4-11).  nth 0: the first upload, nothing
    # enqueued; 3: the first bucket's U' writeback, after its M writeback; 6: the
    # second bucket's second run, after the whole first bucket.  The step returns
    # MUON_ERR_CUDA, the work enqueued before the failure completes, and the next
    # step of the same plan runs to the end and matches the oracle from whatever
    # momentum the failed step left in each matrix.
    import torch
    wl = Workload([(256, 512, 3), (300, 200, 2), (128, 640, 4)], m_sigma=0.02, g_sigma=1e-3)
    plan, hG, hM, hU = _offload_plan(m, wl, cap=600_000)
    assert m.muon_get_plan_info(plan).n_buckets >= 3
    M0 = [x.numpy().copy() for x in hM]
    m.muon_inject_copy_failure(plan, nth)
    with pytest.raises(m.MuonError) as e:
        m.muon_offload_step(plan, hG, hM, hU, 0.95, True, 5)
    assert e.value.status == m.MUON_ERR_CUDA and "injected" in str(e.value)
    torch.cuda.synchronize()
    M1 = [x.numpy().copy() for x in hM]
    changed = sum(int(not np.array_equal(a, b)) for a, b in zip(M0, M1))
    assert changed == {0: 0, 3: 1, 6: 1}[nth]      # tensors whose momentum the failed step wrote back
    m.muon_offload_step(plan, hG, hM, hU, 0.95, True, 5)   # the injection was cleared
    _offload_check(wl, M1, [x.numpy() for x in hM], [u.numpy() for u in hU])


def test_offload_rejects_pageable_host_memory(m):
    import torch
    wl = Workload([(64, 128)])
    cfg = m.muon_config_default(offload=1)
    plan = m.muon_plan(wl.plan_shapes(), config=cfg)
    m.allocate_workspace(plan)
    g = torch.zeros((64, 128), dtype=torch.bfloat16)          # pageable
    mm = torch.zeros((64, 128), dtype=torch.float32).pin_memory()
    u = torch.zeros((64, 128), dtype=torch.float32).pin_memory()
    with pytest.raises(m.MuonError) as e:
        m.muon_offload_step(plan, [g], [mm], [u], 0.95, True, 5)
    assert e.value.status == m.MUON_ERR_NOT_PINNED
    plan2 = m.muon_plan(wl.plan_shapes())                      # no staging slots
    m.allocate_workspace(plan2)
    with pytest.raises(m.MuonError) as e:
        m.muon_offload_step(plan2, [g.pin_memory()], [mm], [u], 0.95, True, 5)
    assert e.value.status == m.MUON_ERR_NO_WORKSPACE


def test_resume_from_copied_state_is_bitwise_identical(m):
    import torch
    shapes = [(256, 384, 2), (384, 256)]
    run = Workload(shapes, m_sigma=0.0, g_sigma=1e-3)
    plan = m.muon_plan(run.plan_shapes())
    m.allocate_workspace(plan)
    for step in range(4):
        run.new_grads(step)
        m.muon_step(plan, run.dW, run.dG, run.dM, 0.02, 0.95, True, 0.01, 5)
        if step == 1:   # checkpoint: copy the caller-owned state out
            ckpt = [t.cpu().clone() for t in run.dW + run.dM]
    torch.cuda.synchronize()
    res = Workload(shapes, m_sigma=0.0, g_sigma=1e-3)
    n = len(shapes)
    res.dW = [t.cuda() for t in ckpt[:n]]
    res.dM = [t.cuda() for t in ckpt[n:]]
    plan2 = m.muon_plan(res.plan_shapes())                      # fresh plan and workspace
    m.allocate_workspace(plan2)
    for step in (2, 3):
        res.new_grads(step)
        m.muon_step(plan2, res.dW, res.dG, res.dM, 0.02, 0.95, True, 0.01, 5)
    torch.cuda.synchronize()
    for a, b in zip(run.dW + run.dM, res.dW + res.dM):
        assert torch.equal(a, b)


# --- metrics: per-bucket records and input norms ("Muon Optimizer + FSDP", 需要记录的指标) ---

@pytest.mark.parametrize("g_dtype,fused", [(synth.BF16, 1), (synth.BF16, 0), (synth.F32, 0)])
def test_input_norms_match_the_oracle(m, g_dtype, fused):
    # ||V||_F of every matrix, tensor order: grouped-GEMM buckets, small-matrix
    # buckets (with the momentum in the small kernel the norm is summed there;
    # otherwise by the momentum kernel), a tall matrix; a NaN matrix reports a
    # non-finite norm
    import math
    wl = Workload([(256, 512), (128, 640, 3), (700, 96), (64, 128, 2)], m_sigma=0.02, g_sigma=1e-3,
                  g_dtype=g_dtype)
    g = wl.dG[3].clone()
    g[1, 2, 3] = float("nan")
    plan = m.muon_plan(wl.plan_shapes(), bucket_cap_bytes=300_000,
                       config=m.muon_config_default(grad_dtype=g_dtype, ns_momentum_fused=fused))
    assert m.muon_get_plan_info(plan).n_buckets >= 3
    m.allocate_workspace(plan)
    m.muon_step(plan, wl.dW, wl.dG[:3] + [g], wl.dM, 0.02, 0.95, True, 0.0, 5)
    st, nf = m.muon_sync(plan)
    assert st == m.MUON_WARN_NONFINITE and nf == 1
    norms = m.muon_get_input_norms(plan)
    mu32, omu = oracle_constants(0.95, "ema")
    idx = 0
    for i, (r, c, k) in enumerate(wl.shapes):
        for j in range(k):
            if (i, j) == (3, 1):
                assert not math.isfinite(norms[idx])
            else:
                G = widen(wl.G[i][j], g_dtype)
                Mo = oracle.momentum_update(wl.M[i][j], G, mu32, one_minus_mu=omu)
                V = oracle.nesterov_blend(Mo, G, mu32, True, one_minus_mu=omu)
                assert abs(norms[idx] - np.linalg.norm(V)) <= 1e-5 * np.linalg.norm(V), (i, j)
            idx += 1


def test_bucket_stats_add_up_to_the_step(m):
    import torch
    wl = Workload([(256, 512, 2), (128, 640, 3), (300, 200)], m_sigma=0.02, g_sigma=1e-3)
    cfg = m.muon_config_default(timing=1)
    plan = m.muon_plan(wl.plan_shapes(), bucket_cap_bytes=300_000, config=cfg)
    m.allocate_workspace(plan)
    m.muon_step(plan, wl.dW, wl.dG, wl.dM, 0.02, 0.95, True, 0.0, 5)
    torch.cuda.synchronize()
    total = m.muon_get_stats(plan)
    info = m.muon_get_plan_info(plan)
    bs = [m.muon_get_bucket_stats(plan, b) for b in range(info.n_buckets)]
    assert sum(b.n_matrices for b in bs) == info.n_matrices == 6
    assert sum(b.ns_ms for b in bs) == pytest.approx(total.ns_ms, rel=1e-6)
    assert sum(b.prep_ms for b in bs) == pytest.approx(total.prep_ms, rel=1e-6, abs=1e-9)
    assert all(b.ns_ms > 0 and b.h2d_bytes == 0 and b.ns_workspace_bytes > 0 for b in bs)
    for b, want in zip(bs, (m.muon_get_bucket_info(plan, i) for i in range(info.n_buckets))):
        assert (b.m, b.n, b.bytes, b.n_groups) == (want.m, want.n, want.bytes, want.n_groups)
    # offload: per-bucket host-link bytes add up to the step's
    wl = Workload([(256, 512, 3), (300, 200, 2)], m_sigma=0.02, g_sigma=1e-3)
    _, _, st, plan = _offload(m, wl, cap=600_000, inflight=2)
    info = m.muon_get_plan_info(plan)
    bs = [m.muon_get_bucket_stats(plan, b) for b in range(info.n_buckets)]
    assert sum(b.h2d_bytes for b in bs) == st.h2d_bytes == sum(r * c * k * 6 for r, c, k in wl.shapes)
    assert sum(b.d2h_bytes for b in bs) == st.d2h_bytes
    assert all(b.h2d_ms > 0 and b.d2h_ms > 0 for b in bs)
