"""The seeded input generator: determinism, distribution and recipe shape."""
import numpy as np

from attention_forward_prefill_gb300 import inputs


def test_same_seed_same_bits_and_different_seed_differs():
    a = inputs.normal_bits((3, 5, 64), 123, "bf16")
    b = inputs.normal_bits((3, 5, 64), 123, "bf16")
    c = inputs.normal_bits((3, 5, 64), 124, "bf16")
    assert a.dtype == np.uint16 and np.array_equal(a, b)
    assert not np.array_equal(a, c)


def test_stream_is_counter_based():
    whole = inputs.splitmix64(7, 0, 100)
    tail = inputs.splitmix64(7, 40, 60)
    assert np.array_equal(whole[40:], tail)


def test_splitmix64_reference_value():
    # SplitMix64 with state 0: the first output of the published generator
    # (Steele, Lea, Flood 2014) is 0xE220A8397B1DCDAF.
    assert int(inputs.splitmix64(0, 0, 1)[0]) == 0xE220A8397B1DCDAF


def test_normal_moments():
    x = inputs.normal_f64(99, 1 << 20)
    assert abs(x.mean()) < 5e-3
    assert abs(x.var() - 1.0) < 5e-3
    assert abs(np.mean(x ** 4) - 3.0) < 0.05


def test_16bit_rounding_is_nearest_even():
    # 1 + 2^-8 lies halfway between bf16 neighbours 1 and 1 + 2^-7 -> even (1.0)
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 1.0 + 2.0 ** -11])
    assert list(inputs.f64_to_bf16_bits(x)) == [0x3F80, 0x3F82, 0xC020, 0x3F80]
    assert list(inputs.f64_to_f16_bits(x)) == [0x3C04, 0x3C0C, 0xC100, 0x3C00]


def test_outlier_keys_recipe():
    B, H, N, d = 1, 2, 300, 16
    bits, rows = inputs.keys_with_outliers((B, H, N, d), 5, 6, "bf16")
    assert rows.shape == (B * H, 3)            # round(0.01 * 300) = 3
    for bh in range(B * H):
        assert len(set(rows[bh].tolist())) == 3
    x = (bits.astype(np.uint32) << 16).view(np.float32).reshape(B * H, N, d)
    big = np.abs(x[0, rows[0]]).mean()
    rest = np.abs(np.delete(x[0], rows[0], axis=0)).mean()
    assert 15 < big / rest < 25


def test_seq_lens_range_and_spread():
    lens = inputs.seq_lens(inputs.seed_for(3, 4), 4096, 4096)
    assert lens.dtype == np.int32
    assert lens.min() >= 1 and lens.max() <= 4096
    assert abs(lens.mean() - 2048.5) < 60


def test_threaded_generation_gives_the_same_bits():
    # blocks of the counter-based stream on host threads: no dependence on the
    # thread count or the block boundaries (an odd total length included)
    n = (1 << 22) * 2 + 6
    one = inputs.normal_bits((n,), 31, "bf16")
    many = inputs.normal_bits((n,), 31, "bf16", threads=6)
    assert np.array_equal(one, many)
    assert np.array_equal(inputs.normal_bits((3, 333), 5, "f16", threads=4),
                          inputs.normal_bits((3, 333), 5, "f16"))
    a, ra = inputs.keys_with_outliers((2, 3, 200, 64), 11, 12, "bf16")
    b, rb = inputs.keys_with_outliers((2, 3, 200, 64), 11, 12, "bf16", threads=5)
    assert np.array_equal(a, b) and np.array_equal(ra, rb)


def test_ranges_of_the_normal_stream_agree_with_the_whole():
    whole = inputs.normal_f64(77, 1000)
    assert np.array_equal(inputs.normal_f64_range(77, 400, 600), whole[400:])
    assert np.array_equal(inputs.normal_f64_range(77, 0, 999), whole[:999])
