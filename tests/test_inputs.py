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


def test_e4m3_codec_against_the_format():
    """Values fixed by the OCP FP8 e4m3 definition: bias 7, 3 mantissa bits, max 448, 0x7F NaN."""
    import math

    v = fi.E4M3_VALUES
    assert v[0x38] == 1.0 and v[0xB8] == -1.0 and v[0x00] == 0.0
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0 and math.isnan(v[0x7F]) and math.isnan(v[0xFF])
    assert v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9 and v[0x08] == 2.0 ** -6
    assert v[0x39] == 1.125 and v[0x40] == 2.0 and v[0x30] == 0.5
    finite = [c for c in range(256) if not math.isnan(v[c])]
    codes = np.array(finite, dtype=np.uint8)
    back = fi.f64_to_e4m3(v[codes])
    assert np.array_equal(fi.e4m3_to_f64(back), v[codes])  # every finite value round-trips (-0 -> 0 allowed)
    # ties go to the even code, saturation at 448
    assert fi.f64_to_e4m3(np.array([1.0625]))[0] == 0x38 and fi.f64_to_e4m3(np.array([1.1875]))[0] == 0x3A
    assert fi.f64_to_e4m3(np.array([500.0, -1e9]))[0] == 0x7E and fi.f64_to_e4m3(np.array([-1e9]))[0] == 0xFE
    # rounding is to the nearest value
    x = np.random.default_rng(0).standard_normal(10000) * 30
    q = fi.e4m3_to_f64(fi.f64_to_e4m3(x))
    pos = np.sort(np.unique(np.abs(v[codes])))
    nearest = pos[np.abs(np.abs(x)[:, None] - pos[None, :]).argmin(axis=1)] * np.sign(x)
    assert np.all(np.abs(q - x) <= np.abs(nearest - x) + 1e-15)
