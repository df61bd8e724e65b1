"""Full-size workloads through the C ABI, in the launch configuration bench.py uses,
checked against the oracle on sampled logical matrices and by properties on all.

Inputs of sampled matrices are generated on the CPU by synth and compared bit for
bit with the device-filled tensors before the step, so the oracle never sees a
value that came from the CUDA path.
"""
import numpy as np
import pytest

import synth
from gpu_util import (TOL_BF16, Workload, check_matrix, device_tensor, host_matrix, nsm, run_steps,
                      to_numpy)

pytestmark = pytest.mark.gpu

QWEN3_4B_LAYER = [(4096, 2560), (1024, 2560), (1024, 2560), (2560, 4096),
                  (9728, 2560), (9728, 2560), (2560, 9728)]
SEED = synth.SEED


@pytest.fixture(scope="module")
def m():
    return nsm()


def _same_bits(dev, host, code):
    got = to_numpy(dev, code)
    return np.array_equal(got.view(np.uint16 if code == synth.BF16 else np.uint32),
                          np.ascontiguousarray(host).view(np.uint16 if code == synth.BF16 else np.uint32))


def test_qwen3_4b_layer_full_size(m):
    # every one of the 7 matrices of the layer, at full size, two steps
    wl = Workload(QWEN3_4B_LAYER, w_sigma=0.02, m_sigma=0.02, g_sigma=1e-3)
    ulp, rel = run_steps(m, wl, steps=2)
    assert ulp <= 1 and rel <= TOL_BF16


def _sampled_step(m, tensors, shapes, plan, samples, *, w_code, g_code, w_sigma, m_sigma, g_sigma, lr=0.02,
                  mu=0.95, bf16_max_bound=None):
    """tensors: list of (W, M, G) device tensors; samples: [(tensor index, matrix index)]."""
    import torch
    pre = {}
    for (ti, j) in samples:
        r, c = shapes[ti][:2]
        W0 = host_matrix((r, c), j, w_code, SEED, synth.stream_id(ti, synth.ROLE_W), 0, w_sigma)
        M0 = host_matrix((r, c), j, synth.F32, SEED, synth.stream_id(ti, synth.ROLE_M), 0, m_sigma)
        G0 = host_matrix((r, c), j, g_code, SEED, synth.stream_id(ti, synth.ROLE_G), 0, g_sigma)
        W, M, G = tensors[ti]
        assert _same_bits(W[j], W0, w_code) and _same_bits(M[j], M0, synth.F32) and _same_bits(G[j], G0, g_code)
        pre[(ti, j)] = (W0, M0, G0)
    m.muon_step(plan, [t[0] for t in tensors], [t[2] for t in tensors], [t[1] for t in tensors],
                lr, mu, True, 0.0, 5)
    st, nf = m.muon_sync(plan)
    assert st == m.MUON_OK and nf == 0
    torch.cuda.synchronize()
    worst = 0.0
    for (ti, j), (W0, M0, G0) in pre.items():
        W, M, _ = tensors[ti]
        _, rel = check_matrix(W0, M0, G0, to_numpy(W[j], w_code), to_numpy(M[j], synth.F32),
                              w_dtype=w_code, g_dtype=g_code, lr=lr, mu=mu, bf16_max_bound=bf16_max_bound)
        worst = max(worst, rel)
    return worst


def test_per_head_qkv_36_layers_full_size(m):
    # fused interleaved [Q0..Q3,K0,V0,...] projections [6144, 2560] x 36 layers; each
    # 128-row head is one logical matrix: 1728 matrices in one batched Newton-Schulz
    import torch
    layers, heads, hd, cols = 36, 48, 128, 2560
    shapes = [(hd, cols, heads)] * layers
    plan = m.muon_plan([(hd, cols, heads, 0)] * layers, bucket_cap_bytes=0)
    assert m.muon_get_plan_info(plan).n_buckets == 1
    m.allocate_workspace(plan)
    tensors = []
    for i in range(layers):
        W = device_tensor((heads, hd, cols), synth.F32, SEED, synth.stream_id(i, synth.ROLE_W), 0, 0.02)
        M = device_tensor((heads, hd, cols), synth.F32, SEED, synth.stream_id(i, synth.ROLE_M), 0, 0.02)
        G = device_tensor((heads, hd, cols), synth.BF16, SEED, synth.stream_id(i, synth.ROLE_G), 0, 1e-3)
        tensors.append((W, M, G))
    W_before = torch.stack([t[0] for t in tensors]).clone()
    rng = np.random.default_rng(7)
    samples = [(0, 0), (0, 4), (0, 5), (0, 47), (17, 23), (35, 0), (35, 46), (35, 47)]
    samples += [(int(rng.integers(layers)), int(rng.integers(heads))) for _ in range(8)]
    worst = _sampled_step(m, tensors, shapes, plan, samples, w_code=synth.F32, g_code=synth.BF16,
                          w_sigma=0.02, m_sigma=0.02, g_sigma=1e-3)
    assert worst <= TOL_BF16
    # every head: the update is finite and its singular values sit in the quintic's band
    U = (W_before - torch.stack([t[0] for t in tensors])).reshape(layers * heads, hd, cols) / 0.02
    assert torch.isfinite(U).all()
    ev = torch.linalg.eigvalsh((U.double() @ U.double().transpose(1, 2)))
    sv = ev.clamp_min(0).sqrt()
    assert float(sv.min()) > 0.5 and float(sv.max()) < 1.35


def test_moe_experts_48_layers_full_size(m):
    # gate/up [128, 768, 2048] and down [128, 2048, 768] per layer, 48 layers: 18432
    # matrices, same-shape groups merged across layers, micro-buckets of 512 MiB.
    import torch
    layers, E = 48, 128
    shapes = []
    for _ in range(layers):
        shapes += [(768, 2048, E), (768, 2048, E), (2048, 768, E)]
    plan = m.muon_plan([(r, c, k, 0) for (r, c, k) in shapes], bucket_cap_bytes=512 << 20,
                       config=m.muon_config_default(param_dtype=m.MUON_DTYPE_BF16))
    info = m.muon_get_plan_info(plan)
    assert info.n_matrices == 18432 and info.n_buckets == 109
    m.allocate_workspace(plan)
    tensors = []
    for i, (r, c, k) in enumerate(shapes):
        W = device_tensor((k, r, c), synth.BF16, SEED, synth.stream_id(i, synth.ROLE_W), 0, 0.02)
        M = torch.zeros((k, r, c), dtype=torch.float32, device="cuda")
        G = device_tensor((k, r, c), synth.BF16, SEED, synth.stream_id(i, synth.ROLE_G), 0, 1e-3)
        tensors.append((W, M, G))
    # first and last matrix of every bucket (bucket b holds global matrices
    # [170b, 170b+170)), the last matrix, and eight more at random
    samples = []
    for b in range(109):
        for g in (170 * b, min(170 * b + 169, 18431)):
            samples.append((g // E, g % E))
    samples.append((143, 127))
    rng = np.random.default_rng(7)
    samples += [(int(rng.integers(len(shapes))), int(rng.integers(E))) for _ in range(8)]
    # lr 2: the update outweighs the bf16 rounding of W ~ N(0, 0.02) (||W|| ~ 25 against
    # ||dW|| ~ 50-80), so the weights are held to the per-matrix tolerance: the bound,
    # 3e-2 plus the half-ulp allowance of W_new, is at most 3.5e-2 of ||dW||
    worst = _sampled_step(m, tensors, shapes, plan, samples, w_code=synth.BF16, g_code=synth.BF16,
                          w_sigma=0.02, m_sigma=0.0, g_sigma=1e-3, lr=2.0, bf16_max_bound=0.035)
    assert worst <= 0.035
    for W, M, _ in tensors[::17]:
        assert torch.isfinite(W.float()).all() and torch.isfinite(M).all()


def test_moe_expert_layer_bf16_weights_from_zero(m):
    # one layer of the expert workload (384 matrices of 768 x 2048 in the wide form,
    # buckets of 170, 170 and 44) with bf16 weights starting at 0: the fused bf16
    # weight update of full 170-matrix buckets, held to 3.5e-2 of ||dW|| (the bf16
    # rounding of W_new is then at most 2^-8 of the update)
    from gpu_util import TOL_BF16_W
    import torch
    E = 128
    shapes = [(768, 2048, E), (768, 2048, E), (2048, 768, E)]
    plan = m.muon_plan([(r, c, k, 0) for (r, c, k) in shapes], bucket_cap_bytes=512 << 20,
                       config=m.muon_config_default(param_dtype=m.MUON_DTYPE_BF16))
    info = m.muon_get_plan_info(plan)
    assert info.n_buckets == 3 and info.max_bucket_matrices == 170
    m.allocate_workspace(plan)
    tensors = []
    for i, (r, c, k) in enumerate(shapes):
        W = torch.zeros((k, r, c), dtype=torch.bfloat16, device="cuda")
        M = torch.zeros((k, r, c), dtype=torch.float32, device="cuda")
        G = device_tensor((k, r, c), synth.BF16, SEED, synth.stream_id(i, synth.ROLE_G), 0, 1e-3)
        tensors.append((W, M, G))
    # first and last matrix of each bucket (global matrices [0,170), [170,340), [340,384)), and more
    samples = [(0, 0), (1, 41), (1, 42), (2, 83), (2, 84), (2, 127), (0, 77), (1, 100), (2, 5)]
    worst = _sampled_step(m, tensors, shapes, plan, samples, w_code=synth.BF16, g_code=synth.BF16,
                          w_sigma=0.0, m_sigma=0.0, g_sigma=1e-3, bf16_max_bound=TOL_BF16_W)
    assert worst <= TOL_BF16_W
    for W, M, _ in tensors:
        assert torch.isfinite(W.float()).all() and bool((W != 0).any(dim=(1, 2)).all())


def test_offload_full_qwen3_4b_36_layers(m):
    # 36 layers of Qwen3-4B shapes (3.63B Muon parameters) with momentum and gradients
    # in pinned host memory; 512 MiB buckets, one bucket in writeback while one computes
    import torch
    layers = 36
    shapes = [(r, c, 1) for _ in range(layers) for (r, c) in QWEN3_4B_LAYER]
    cfg = m.muon_config_default(offload=1, max_inflight=1, timing=1)
    plan = m.muon_plan([(r, c, 1, 0) for (r, c, _) in shapes], bucket_cap_bytes=512 << 20, config=cfg)
    m.allocate_workspace(plan)
    hG, hM, hU = [], [], []
    for i, (r, c, _) in enumerate(shapes):
        g = device_tensor((r, c), synth.BF16, SEED, synth.stream_id(i, synth.ROLE_G), 0, 1e-3)
        mm = device_tensor((r, c), synth.F32, SEED, synth.stream_id(i, synth.ROLE_M), 0, 0.02)
        hG.append(torch.empty((r, c), dtype=torch.bfloat16, pin_memory=True).copy_(g))
        hM.append(torch.empty((r, c), dtype=torch.float32, pin_memory=True).copy_(mm))
        hU.append(torch.empty((r, c), dtype=torch.float32, pin_memory=True))
        del g, mm
    samples = [1, 2, 7 * 35 + 1, 7 * 17 + 3, 7 * 35 + 6]   # k/v of layer 0, k of 35, o of 17, down of 35
    pre = {}
    for i in samples:
        r, c, _ = shapes[i]
        G0 = host_matrix((r, c), 0, synth.BF16, SEED, synth.stream_id(i, synth.ROLE_G), 0, 1e-3)
        M0 = host_matrix((r, c), 0, synth.F32, SEED, synth.stream_id(i, synth.ROLE_M), 0, 0.02)
        assert np.array_equal(hG[i].view(torch.int16).numpy().view(np.uint16), G0)
        assert np.array_equal(hM[i].numpy(), M0)
        pre[i] = (G0, M0)
    m.muon_offload_step(plan, hG, hM, hU, 0.95, True, 5, timeout_ms=600_000)
    st = m.muon_get_stats(plan)
    assert st.h2d_bytes == sum(r * c * 6 for (r, c, _) in shapes)
    assert st.d2h_bytes == sum(r * c * 8 for (r, c, _) in shapes)
    import oracle
    from gpu_util import f32, oracle_constants, rel_fro, ulp_distance, widen
    mu32, omu = oracle_constants(0.95, "ema")
    for i, (G0, M0) in pre.items():
        r, c, _ = shapes[i]
        G = widen(G0, synth.BF16)
        Mo = oracle.momentum_update(M0, G, mu32, one_minus_mu=omu)
        assert int(ulp_distance(hM[i].numpy(), Mo).max()) <= 1
        V = oracle.nesterov_blend(Mo, G, mu32, True, one_minus_mu=omu)
        Uo = oracle.offload_update(oracle.newton_schulz(V, coeffs=tuple(f32(v) for v in oracle.DEFAULT_COEFFS),
                                                        eps=f32(1e-7)), r, c)
        assert rel_fro(hU[i].numpy(), Uo) <= TOL_BF16
    for u in hU[::25]:
        assert torch.isfinite(u).all()


def test_expert_shapes_update_through_offload(m):
    # the bf16 weights of the expert workload hide the update under bf16 rounding; the
    # fp32 update U' of the offload path checks the same Newton-Schulz tightly
    import torch
    import oracle
    from gpu_util import f32, oracle_constants, rel_fro, widen
    shapes = [(768, 2048, 6), (2048, 768, 5)]
    wl = Workload(shapes, m_sigma=0.0, g_sigma=1e-3)
    cfg = m.muon_config_default(offload=1)
    plan = m.muon_plan(wl.plan_shapes(), bucket_cap_bytes=4 * 768 * 2048 * 2, config=cfg)
    m.allocate_workspace(plan)
    hG = [torch.from_numpy(np.ascontiguousarray(g).view(np.int16)).view(torch.bfloat16).pin_memory() for g in wl.G]
    hM = [torch.from_numpy(x.copy()).pin_memory() for x in wl.M]
    hU = [torch.empty(x.shape, dtype=torch.float32).pin_memory() for x in wl.M]
    m.muon_offload_step(plan, hG, hM, hU, 0.95, True, 5)
    mu32, omu = oracle_constants(0.95, "ema")
    for i, (r, c, k) in enumerate(wl.shapes):
        for j in range(k):
            G = widen(wl.G[i][j], synth.BF16)
            Mo = oracle.momentum_update(wl.M[i][j], G, mu32, one_minus_mu=omu)
            V = oracle.nesterov_blend(Mo, G, mu32, True, one_minus_mu=omu)
            Uo = oracle.offload_update(oracle.newton_schulz(V, coeffs=tuple(f32(v) for v in oracle.DEFAULT_COEFFS),
                                                            eps=f32(1e-7)), r, c)
            assert rel_fro(hU[i].numpy()[j], Uo) <= TOL_BF16
