"""The seeded input generator: determinism, distribution and exact bf16 bits."""
from __future__ import annotations

import numpy as np

import seeded_inputs as si

MASK64 = (1 << 64) - 1


def _splitmix_word(seed: int, tid: int, n: int) -> int:
    """Word n of stream (seed, tid), in plain Python integers (SplitMix64)."""
    def mix(z):
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        return z ^ (z >> 31)
    s0 = mix((seed * 0x9E3779B97F4A7C15 + tid) & MASK64)
    return mix((s0 + (n + 1) * 0x9E3779B97F4A7C15) & MASK64)


def test_words_match_scalar_splitmix():
    w = si.uniform_words(7, 3, 5, 4)
    assert [int(x) for x in w] == [_splitmix_word(7, 3, n) for n in range(5, 9)]


def test_deterministic_and_stream_separated():
    a = si.normal_bf16(5, si.TID_Q, 1000)
    assert np.array_equal(a, si.normal_bf16(5, si.TID_Q, 1000))
    assert not np.array_equal(a, si.normal_bf16(5, si.TID_K, 1000))
    assert not np.array_equal(a, si.normal_bf16(6, si.TID_Q, 1000))
    # counter form: any chunking gives the same values
    full = si.normal_f64(9, 1, 64)
    assert np.array_equal(full[32:], si.normal_f64(9, 1, 32, start=32))


def test_moments_are_standard_normal():
    x = si.bf16_bits_to_f32(si.normal_bf16(2, si.TID_V, 1 << 20)).astype(np.float64)
    assert abs(x.mean()) < 5e-3
    assert abs(x.std() - 1.0) < 5e-3
    assert abs((x > 1.0).mean() - 0.158655) < 2e-3


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-39, 1.0 + 2**-7], np.float32)
    got = si.f32_to_bf16_bits(vals)
    assert list(got) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x0021, 0x3F81]


def test_power_of_two_multiplier_is_exact():
    base = si.normal_bf16(4, si.TID_Q, 4096)
    x8 = si.normal_bf16(4, si.TID_Q, 4096, multiplier=8.0)
    assert np.array_equal(si.bf16_bits_to_f32(x8), si.bf16_bits_to_f32(base) * 8)


def test_sample_rows_distinct_and_required():
    r = si.sample_rows(6, 32768, 128, must_include=[0, 1, 16384, 32767])
    assert len(r) == 128 and len(set(r.tolist())) == 128
    assert {0, 1, 16384, 32767} <= set(r.tolist())
    assert np.all(np.diff(r) > 0) and r[-1] < 32768
    assert np.array_equal(r, si.sample_rows(6, 32768, 128, must_include=[0, 1, 16384, 32767]))
    small = si.sample_rows(1, 10, 50)
    assert small.tolist() == list(range(10))


def test_torch_generator_matches_host_generator():
    torch = __import__("pytest").importorskip("torch")
    n = 200_001
    host = si.normal_bf16(3, si.TID_K, n, multiplier=2.0)
    dev = si.normal_bf16_torch(3, si.TID_K, n, multiplier=2.0, device="cpu", chunk=65536)
    dev_bits = dev.view(torch.int16).numpy().view(np.uint16)
    same = host == dev_bits
    assert same.mean() > 0.9999
    # any difference is a single bf16 step
    diff = np.abs(host.astype(np.int32) - dev_bits.astype(np.int32))
    assert diff.max() <= 1


def test_e4m3_table_and_rounding():
    t = si.E4M3_MAGNITUDES
    assert t[1] == 2.0 ** -9 and t[8] == 2.0 ** -6 and t[126] == 448.0 and np.isnan(t[127])
    assert np.all(np.diff(t[:127]) > 0)
    # ties go to the even code; saturation at 448; sign bit
    mid = (t[9] + t[10]) / 2          # between codes 9 and 10 -> 10
    assert si.f64_to_e4m3_bits(np.array([mid]))[0] == 10
    mid = (t[10] + t[11]) / 2         # between 10 and 11 -> 10
    assert si.f64_to_e4m3_bits(np.array([mid]))[0] == 10
    assert list(si.f64_to_e4m3_bits(np.array([1e6, -1e6, -0.0, 2.0 ** -11]))) == [126, 254, 128, 0]
    x = np.array([1.0, -2.5, 0.0137, 300.0])
    back = si.e4m3_bits_to_f32(si.f64_to_e4m3_bits(x))
    assert list(back) == [1.0, -2.5, 0.013671875, 288.0]


def test_e4m3_matches_torch_cast_and_widens_exactly_to_bf16():
    torch = __import__("pytest").importorskip("torch")
    x = si.normal_f64(8, 1, 100_000) * 37.0
    x = np.clip(x, -448, 448)
    ours = si.f64_to_e4m3_bits(x)
    theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]
    f32 = si.e4m3_bits_to_f32(codes)
    assert np.array_equal(si.bf16_bits_to_f32(si.e4m3_bits_to_bf16_bits(codes)), f32)
