"""The seeded input generator: published splitmix64 outputs, bf16 rounding, distribution."""
import numpy as np

import fa_inputs as fi


def test_splitmix64_published_outputs():
    # the first three outputs of splitmix64 seeded with 0 (Steele, Lea and Flood's generator)
    got = [int(x) for x in fi.splitmix64(np.uint64(0), 0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_bf16_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -20, -2.0,
                  3.140625, 65504.0], dtype=np.float32)
    got = fi.f32_to_bf16_bits(x).tolist()
    # ties go to the even neighbour; just above a tie rounds up
    assert got == [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xC000, 0x4049, 0x4780]
    assert np.array_equal(fi.bf16_bits_to_f64(np.array(got, dtype=np.uint16))[:3], [1.0, 1.0, 1.0 + 2 ** -6])


def test_generator_is_deterministic_and_streams_differ():
    a = fi.make_qkv(1, 2, 64, 64, seed=3)
    b = fi.make_qkv(1, 2, 64, 64, seed=3)
    c = fi.make_qkv(1, 2, 64, 64, seed=4)
    assert np.array_equal(a.q_bits, b.q_bits) and np.array_equal(a.v_bits, b.v_bits)
    assert not np.array_equal(a.q_bits, a.k_bits)
    assert not np.array_equal(a.q_bits, c.q_bits)
    # a chunk boundary does not change the stream: a prefix of a longer draw is the shorter draw
    long = fi.normal_bf16_bits(5, 1, 3 * (1 << 20) + 7)
    short = fi.normal_bf16_bits(5, 1, 1001)
    assert np.array_equal(long[:1001], short)


def test_normal_moments_and_sigma():
    x = fi.bf16_bits_to_f64(fi.normal_bf16_bits(1, 1, 1 << 20))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    y = fi.bf16_bits_to_f64(fi.normal_bf16_bits(1, 1, 1 << 18, sigma=3.0))
    assert abs(y.std() - 3.0) < 0.03
    # bf16 values are exact in float64 and finite
    assert np.all(np.isfinite(x))
