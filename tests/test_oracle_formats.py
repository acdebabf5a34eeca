"""Pins for the oracle's number formats (e4m3 codes, bf16 rounding).

The oracle's encoders are written from the format definitions; here they are
checked against closed forms (named codes, exact midpoints), against torch's own
conversions (a library routine), and exhaustively over their domains."""
import numpy as np
import pytest
import torch

import oracle


def torch_e4m3_codes(v):
    t = torch.from_numpy(np.asarray(v, dtype=np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.isnan(ours).sum() == 2          # 0x7F and 0xFF only


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
    (0x38, 1.0), (0x3C, 1.5), (0x40, 2.0), (0x7E, 448.0), (0x77, 240.0),
    (0x80, -0.0), (0xB8, -1.0), (0xFE, -448.0),
])
def test_e4m3_named_codes(code, value):
    got = oracle.e4m3_decode(np.array([code], dtype=np.uint8))[0]
    assert got == value and np.signbit(got) == np.signbit(value)
    # and the encoder inverts it
    assert oracle.e4m3_encode(np.array([value], dtype=np.float32))[0] == code


def test_e4m3_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_e4m3_midpoints_tie_to_even():
    # between adjacent positive codes c and c+1 the midpoint goes to the even code;
    # a hair above goes up, a hair below goes down (closed form, no library)
    pos = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    lo, hi = pos[:-1], pos[1:]
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)     # exact in fp32
    c = np.arange(0, 0x7E)
    even = np.where(c % 2 == 0, c, c + 1)
    assert np.array_equal(oracle.e4m3_encode(mid), even)
    assert np.array_equal(oracle.e4m3_encode(-mid), even | 0x80)
    up = np.nextafter(mid, np.float32(np.inf))
    dn = np.nextafter(mid, np.float32(0))
    assert np.array_equal(oracle.e4m3_encode(up), c + 1)
    assert np.array_equal(oracle.e4m3_encode(dn), c)


def test_e4m3_saturates():
    v = np.array([448.0, 463.9, 464.0, 470.0, 1e6, 3e38, -500.0, -1e30], dtype=np.float32)
    assert list(oracle.e4m3_encode(v)) == [0x7E] * 6 + [0xFE] * 2


def test_e4m3_signed_zero():
    v = np.array([0.0, -0.0, 1e-30, -1e-30, 2.0 ** -10, -(2.0 ** -10)], dtype=np.float32)
    # 2**-10 is the midpoint between 0 and the smallest subnormal: ties to even (zero)
    assert list(oracle.e4m3_encode(v)) == [0x00, 0x80, 0x00, 0x80, 0x00, 0x80]


def test_e4m3_encode_every_bf16_value_matches_torch():
    # every finite bf16 pattern (as fp32) in [-512, 512]
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = oracle.bf16_to_f32(bits)
    v = v[np.isfinite(v) & (np.abs(v) <= 512)]
    assert np.array_equal(oracle.e4m3_encode(v), torch_e4m3_codes(v))


def test_e4m3_encode_random_fp32_matches_torch():
    rng = np.random.default_rng(1)
    n = 1_000_000
    mant = rng.uniform(1.0, 2.0, n)
    ex = rng.integers(-14, 10, n)
    sign = rng.choice([-1.0, 1.0], n)
    v = (sign * mant * np.exp2(ex)).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(v), torch_e4m3_codes(v))


def test_bf16_decode_matches_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_bf16_round_fp32_matches_torch():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(500_000) * np.exp2(rng.integers(-130, 125, 500_000))).astype(np.float32)
    # include exact ties: bf16 value + half its ulp
    base = oracle.bf16_to_f32(rng.integers(0, 0x7F00, 20000).astype(np.uint16)).astype(np.float64)
    ulp = np.exp2(np.floor(np.log2(np.maximum(base, 2.0 ** -126))) - 7)
    ties = (base + ulp / 2).astype(np.float32)
    v = np.concatenate([v, ties, -ties, np.float32([3.4e38, -3.4e38, 1e-45, 0.0, -0.0])])
    ours = oracle.f64_to_bf16(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_round_from_fp64_is_single_rounding():
    # 1 + 2**-8 is the midpoint between bf16 1.0 and 1 + 2**-7: it goes to even (1.0);
    # a hair above (2**-40, invisible in fp32) must go up: no double rounding via fp32
    v = np.array([1 + 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -40, 1 + 3 * 2.0 ** -8], dtype=np.float64)
    got = oracle.bf16_to_f32(oracle.f64_to_bf16(v))
    assert list(got) == [1.0, 1 + 2.0 ** -7, 1 + 2.0 ** -6]
