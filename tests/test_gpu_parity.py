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
from gpu_util import (TOL_BF16, Workload, check_step, f32, nsm, oracle_constants, rel_fro, to_numpy,
                      torch_from, ulp_distance, widen)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    return nsm()


def _run(m, wl, *, lr=0.02, mu=0.95, nesterov=True, wd=0.0, ns_steps=5, cap=512 << 20, cfg=None,
         steps=1, form="ema", coeffs=oracle.DEFAULT_COEFFS, sample=None, tol=TOL_BF16):
    import torch
    cfg = cfg or m.muon_config_default()
    cfg.grad_dtype = wl.g_dtype
    cfg.param_dtype = wl.w_dtype
    cfg.momentum_form = m.MUON_MOMENTUM_SGD if form == "sgd" else m.MUON_MOMENTUM_EMA
    cfg.ns_a, cfg.ns_b, cfg.ns_c = coeffs
    plan = m.muon_plan(wl.plan_shapes(), bucket_cap_bytes=cap, config=cfg)
    m.allocate_workspace(plan)
    worst = (0, 0.0)
    for step in range(steps):
        if step > 0:
            wl.new_grads(step)
        W_prev = [to_numpy(t, wl.w_dtype) for t in wl.dW]
        M_prev = [to_numpy(t, synth.F32) for t in wl.dM]
        m.muon_step(plan, wl.dW, wl.dG, wl.dM, lr, mu, nesterov, wd, ns_steps)
        st, nf = m.muon_sync(plan)
        assert st == m.MUON_OK and nf == 0
        torch.cuda.synchronize()
        W_new = [to_numpy(t, wl.w_dtype) for t in wl.dW]
        M_new = [to_numpy(t, synth.F32) for t in wl.dM]
        u, r = check_step(wl, W_prev, M_prev, W_new, M_new, lr=lr, mu=mu, nesterov=nesterov, wd=wd,
                          ns_steps=ns_steps, coeffs=coeffs, form=form, sample=sample, tol=tol)
        worst = (max(worst[0], u), max(worst[1], r))
    return worst


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
