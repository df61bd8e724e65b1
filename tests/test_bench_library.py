"""The bench's library baseline computes the same Muon step as the oracle.

bench.library_step is the step written as a loop of torch ops (batched bf16 GEMMs
with fp32 accumulation); the GPU arm times it beside the hand-written kernels. Here
it runs on the CPU, on a wide and a tall tensor of a few matrices, and each
matrix's weight update must match the fp64 oracle to the bf16 Newton-Schulz
tolerance, and its fp32 momentum to fp32 rounding (the library form rounds twice,
after the multiply and after the add, so it is not held to the kernels' 1 ulp).
"""
import numpy as np
import pytest
import torch

import bench
import oracle

RNG_SEED = 1234


@pytest.mark.parametrize("rows, cols, count", [(48, 96, 3), (96, 40, 2)])
def test_library_step_matches_the_oracle(rows, cols, count):
    rng = np.random.default_rng(RNG_SEED + rows)
    W = (0.02 * rng.standard_normal((count, rows, cols))).astype(np.float32)
    M = (0.02 * rng.standard_normal((count, rows, cols))).astype(np.float32)
    G = (1e-3 * rng.standard_normal((count, rows, cols))).astype(np.float32)
    tW, tM, tG = torch.from_numpy(W.copy()), torch.from_numpy(M.copy()), torch.from_numpy(G.copy())
    lr, mu = 0.02, 0.95
    bench.library_step(torch, [tW], [tM], [tG], [bench.NS_COEFFS] * 5, lr=lr, mu=mu, wd=0.0)
    omu = float(np.float32(1.0) - np.float32(mu))
    for j in range(count):
        Wo, Mo, _ = oracle.muon_matrix_step(W[j].astype(np.float64), M[j], G[j].astype(np.float64), lr,
                                            float(np.float32(mu)), True, 0.0, one_minus_mu=omu)
        bound = 2 * np.finfo(np.float32).eps * (np.abs(mu * M[j]) + np.abs(omu * G[j]))
        assert np.all(np.abs(tM[j].numpy().astype(np.float64) - Mo) <= bound)
        dw = tW[j].numpy().astype(np.float64) - W[j]
        dw_or = Wo - W[j]
        rel = np.linalg.norm(dw - dw_or) / np.linalg.norm(dw_or)
        assert rel <= 3e-2, rel
