"""Seeded random workloads against the fp64 oracle.

Each case draws 2-4 tensors with random rows and cols (1 to ~1700) and counts (1 to
3). So a plan mixes tall and wide matrices, ragged 256-blocks, groups of at most 128
rows beside larger ones, several buckets under a small cap, and both Newton-Schulz
kernels. Every logical matrix of two optimizer steps is checked: momentum within 1
ulp, the update within the bf16 tolerance. The draws are fixed (seeded), so a
failure reproduces.
"""
import numpy as np
import pytest

from gpu_util import TOL_BF16, Workload, nsm, run_steps

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    return nsm()


def _draw(seed):
    rng = np.random.default_rng(seed)
    shapes = []
    for _ in range(int(rng.integers(2, 5))):
        kind = rng.integers(0, 4)
        if kind == 0:      # a head-like slice: few rows, wide
            r, c = int(rng.integers(1, 129)), int(rng.integers(64, 1700))
        elif kind == 1:    # square-ish
            r = int(rng.integers(100, 1100)); c = int(r + rng.integers(-90, 90))
        else:              # anything
            r, c = int(rng.integers(1, 1700)), int(rng.integers(1, 1700))
        if rng.integers(0, 2):
            r, c = c, r
        shapes.append((max(r, 1), max(c, 1), int(rng.integers(1, 4))))
    cap = int(rng.choice([0, 1 << 20, 8 << 20, 512 << 20]))
    return shapes, cap


@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("kernel", ["AUTO", "GEMM"])
def test_random_workload_matches_oracle(m, seed, kernel):
    shapes, cap = _draw(1000 + seed)
    wl = Workload(shapes, m_sigma=0.02, g_sigma=1e-3)
    k = m.MUON_NS_KERNEL_AUTO if kernel == "AUTO" else m.MUON_NS_KERNEL_GEMM
    ulp, rel = run_steps(m, wl, steps=2, cap=cap, cfg=m.muon_config_default(ns_kernel=k))
    assert ulp <= 1 and rel <= TOL_BF16, (shapes, cap)
