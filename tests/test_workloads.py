"""The seeded input generator: determinism, distribution and storage rounding."""
import numpy as np

from workloads import (WORKLOADS, bf16_bits_to_f32, f32_to_bf16_bits, gen_matrix,
                       normal_f64, splitmix_draws)


def test_splitmix_known_first_draw():
    # SplitMix64 seeded with 0: the first output of the published generator
    # (state += 0x9E3779B97F4A7C15, then the two multiply-xorshift rounds).
    assert int(splitmix_draws(0, 0, 1)[0]) == 0xE220A8397B1DCDAF


def test_normal_stats_and_determinism():
    x = normal_f64(123, 0, 1 << 18)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert np.array_equal(x[:1000], normal_f64(123, 0, 1000))
    assert not np.array_equal(x[:1000], normal_f64(123, 1, 1000))
    assert np.array_equal(normal_f64(9, 2, 7), normal_f64(9, 2, 8)[:7])


def test_bf16_bits_round_trip():
    x = (normal_f64(3, 0, 4096) * 0.02).astype(np.float32)
    b = f32_to_bf16_bits(x)
    y = bf16_bits_to_f32(b)
    assert np.all(np.abs(y - x) <= np.abs(x) * 2.0 ** -8)
    assert np.array_equal(f32_to_bf16_bits(y), b)


def test_gen_matrix_shapes():
    m = gen_matrix(2001, 0, 7, 13, 0.5, "bf16")
    assert m.data.shape == (7, 13) and m.data.dtype == np.uint16
    f = gen_matrix(2001, 0, 7, 13, 0.5, "f32")
    assert f.data.dtype == np.float32
    assert np.array_equal(f32_to_bf16_bits(f.data), m.data)


def test_workload_counts():
    assert WORKLOADS["bucket_512_small_bf16"].count == 512
    assert WORKLOADS["stack_24L_h2048_bf16"].count == 168
    w5 = WORKLOADS["stack_32L_7b_bf16_f32mom"]
    assert w5.count == 224
    params = sum(r * c * k for r, c, k in w5.shapes)
    assert abs(params - 6.98e9) / 6.98e9 < 0.01
