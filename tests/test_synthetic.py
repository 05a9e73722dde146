"""The seeded generator: deterministic, counter-based, and its C implementation
agrees with the plain numpy statement of the same recipe."""
import numpy as np

import synthetic


def test_c_matches_numpy_recipe():
    a = synthetic.normal_f64(3, 1, 1001, 50001)
    b = synthetic.normal_f64_numpy(3, 1, 1001, 50001)
    assert np.max(np.abs(a - b)) < 1e-13
    x = synthetic.draw(0, 0, (37, 129), 0.0, 1.0, "bf16")
    y = synthetic.draw_numpy(0, 0, (37, 129), 0.0, 1.0, "bf16")
    assert np.mean(x == y) > 0.9999


def test_row_blocks_are_independent_of_request():
    full = synthetic.draw(0, 2, (64, 77), 0.5, 2.0, "f32")
    part = synthetic.draw(0, 2, (64, 77), 0.5, 2.0, "f32", row_start=13, row_count=5)
    assert np.array_equal(full[13:18], part)


def test_distribution_moments():
    z = synthetic.to_f64(synthetic.draw(0, 1, (512, 1024), 1.0, 0.1, "bf16"), "bf16")
    assert abs(z.mean() - 1.0) < 1e-3 and abs(z.std() - 0.1) < 1e-3
    s = synthetic.normal_f64(0, 4, 0, 1 << 20)
    assert abs(s.mean()) < 5e-3 and abs(s.std() - 1.0) < 5e-3
    assert abs(np.mean(s ** 3)) < 1e-2 and abs(np.mean(s ** 4) - 3.0) < 3e-2


def test_streams_and_seeds_differ():
    a = synthetic.draw(0, 0, (8, 8), 0, 1, "f32")
    assert not np.array_equal(a, synthetic.draw(0, 1, (8, 8), 0, 1, "f32"))
    assert not np.array_equal(a, synthetic.draw(1, 0, (8, 8), 0, 1, "f32"))
    assert np.array_equal(a, synthetic.draw(0, 0, (8, 8), 0, 1, "f32"))


def test_bf16_rounding_is_nearest_even():
    v = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20], np.float32)
    bits = synthetic.f32_to_bf16_bits(v)
    assert bits.tolist() == [0x3F80, 0x3F80, 0x3F82, 0x3F81]
