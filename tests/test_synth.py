"""The seeded input generator: Philox known answers, determinism, distribution, bf16 rounding."""
import os

import numpy as np
import pytest

import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def _kat_rows():
    rows = []
    with open(os.path.join(HERE, "golden", "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(t, 16) for t in line.split()])
    return rows


@pytest.mark.parametrize("row", _kat_rows())
def test_philox_known_answers(row):
    c, k, want = row[:4], row[4:6], row[6:]
    got = synth.philox4x32_10([c[0]], [c[1]], [c[2]], [c[3]], k[0], k[1])
    assert [int(g[0]) for g in got] == want


def test_counter_based_slices_agree():
    full = synth.normal_f32(synth.SEED, 5, 2, 0, 100_001)
    for start, count in [(0, 1), (1, 1), (7, 1000), (99_999, 2), (65_535, 3)]:
        assert np.array_equal(synth.normal_f32(synth.SEED, 5, 2, start, count),
                              full[start:start + count])


def test_streams_and_steps_differ():
    a = synth.normal_f32(synth.SEED, 1, 0, 0, 64)
    assert not np.array_equal(a, synth.normal_f32(synth.SEED, 2, 0, 0, 64))
    assert not np.array_equal(a, synth.normal_f32(synth.SEED, 1, 1, 0, 64))


def test_normal_moments():
    z = synth.normal_f32(synth.SEED, 9, 0, 0, 1_000_000).astype(np.float64)
    assert abs(z.mean()) < 5e-3
    assert abs(z.std() - 1.0) < 5e-3
    assert abs(np.mean(np.abs(z) > 2.0) - 0.0455) < 2e-3
    assert np.all(np.isfinite(z))


def test_log_and_cos_accuracy():
    u = np.linspace(2.0 ** -25, 1 - 2.0 ** -24, 200_001).astype(np.float32)
    assert np.max(np.abs(synth._ln32(u) - np.log(u.astype(np.float64)))) < 2e-6
    assert np.max(np.abs(synth._cos2pi32(u) - np.cos(2 * np.pi * u.astype(np.float64)))) < 1e-6


def test_bf16_round_to_nearest_even():
    f = np.array([0x3F800000, 0x3F808000, 0x3F818000, 0x3F808001, 0xBF80FFFF, 0x00000000],
                 dtype=np.uint32).view(np.float32)
    want = [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xBF81, 0x0000]
    assert synth.f32_to_bf16_bits(f).tolist() == want
    assert np.array_equal(synth.bf16_bits_to_f32(np.array(want, np.uint16)).view(np.uint32),
                          np.array(want, np.uint32) << 16)


def test_tensor_shapes_and_dtypes():
    t = synth.tensor(synth.SEED, 3, 0, (4, 5), 0.02, synth.F32)
    assert t.shape == (4, 5) and t.dtype == np.float32
    b = synth.tensor(synth.SEED, 3, 0, (4, 5), 0.02, synth.BF16)
    assert b.dtype == np.uint16
    assert np.array_equal(b, synth.f32_to_bf16_bits(t))
    assert np.allclose(synth.as_f64(b, synth.BF16), t, rtol=2 ** -8, atol=0)
