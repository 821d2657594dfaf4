"""Checks of the seeded input generator (it feeds both the oracle and the GPU)."""
import numpy as np

import synth


def test_deterministic_and_sub_ranges():
    a = synth.normal(7, (1000,))
    assert np.array_equal(a, synth.normal(7, (1000,)))
    assert np.array_equal(a[123:456], synth.normal(7, (333,), start=123))
    assert not np.array_equal(a, synth.normal(8, (1000,)))
    t = synth.student_t(9, (500,), dtype=synth.BF16)
    assert np.array_equal(t[100:], synth.student_t(9, (400,), start=100, dtype=synth.BF16))


def test_moments():
    x = synth.normal(1, (1_000_000,), mean=0.0, std=0.02).astype(np.float64)
    assert abs(x.mean()) < 1e-4 and abs(x.std() - 0.02) < 1e-4
    u = synth.uniform(2, 1_000_000)
    assert u.min() > 0 and u.max() < 1 and abs(u.mean() - 0.5) < 2e-3
    t = synth.student_t(3, (1_000_000,), df=3).astype(np.float64)
    # median of |t_3| is 0.7649; its variance is 3
    assert abs(np.median(np.abs(t)) - 0.7649) < 5e-3
    assert abs(np.var(t[np.abs(t) < 50]) - 3.0) < 0.3


def test_bf16_bits_are_rne_of_the_f32_draw():
    f = synth.normal(4, (10000,), std=3.0)
    b = synth.normal(4, (10000,), std=3.0, dtype=synth.BF16)
    u = f.view(np.uint32)
    want = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(b, want)
