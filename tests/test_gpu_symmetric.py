"""Symmetric products written from their upper tiles, against the fp64 oracle.

In bf16 the GRAM and POLY launches compute only the 256 x 256 blocks on and above
the diagonal. A diagonal block is written whole, and a block above it also writes
its transpose, so A and B' = aI + bA + cAA are whole when the next GEMM reads their
rows in place.

The shapes cover:
- ragged 256-blocks (m not a multiple of 256), down to a last block of one row;
- a tall matrix;
- groups of different sizes in one launch;
- CTA pairs and single CTAs (a bucket holding a group of at most 128 rows).

Single iterations with chosen coefficients isolate each product:
- (1, 0, 0): B' = I, so the UPDATE epilogue stands alone;
- (0, 1, 0): B' = A, copied whole by POLY's epilogue;
- (0, 0, 1): A A, both operands read from the mirrored A.
"""
import pytest

from gpu_util import TOL_BF16, Workload, nsm, run_steps
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    return nsm()


@pytest.mark.parametrize("shapes", [
    [(1600, 1800)],                 # 7 ragged 256-blocks
    [(1600, 1700), (700, 1000)],    # two sizes in one launch
    [(2000, 1540)],                 # tall: 1540 x 2000, ragged
    [(513, 1100, 2)],               # 3 blocks, the last one a single row
    [(100, 700), (700, 1000)],      # a group of <= 128 rows: single-CTA 128 x 256 tiles
    [(100, 300), (1600, 1700)],     # single-CTA tiles, 7 blocks
])
def test_symmetric_storage_matches_oracle(m, shapes):
    wl = Workload(shapes, m_sigma=0.02, g_sigma=1e-3)
    ulp, rel = run_steps(m, wl, steps=2)
    assert ulp <= 1 and rel <= TOL_BF16


@pytest.mark.parametrize("coeffs", [(1.0, 0.0, 0.0), (0.0, 1.0, 0.0), (0.0, 0.0, 1.0)])
def test_symmetric_storage_isolated_products(m, coeffs):
    # W starts at 0 so that the small update is not lost in the rounding of W
    wl = Workload([(1600, 1700), (700, 1000)], w_sigma=0.0, g_sigma=1.0, g_dtype=synth.F32)
    run_steps(m, wl, ns_steps=1, coeffs=coeffs, mu=0.0, nesterov=False)
