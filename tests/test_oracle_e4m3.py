"""Pins for the oracle's FP8 E4M3FN format (used for V and for P).

The pages fix only "FP8 PV" (diffusers PR #15060, "What does this PR do?";
diffusers issue #15014, kernel contract bullets).  The oracle reads FP8 as OCP
E4M3FN with round-to-nearest-even and saturation.  These tests pin the
oracle's encoder/decoder to the format's closed-form definition and to
PyTorch's independent ``float8_e4m3fn`` cast.
"""
import numpy as np
import pytest
import torch

import oracle


def test_decode_closed_form_values():
    dec = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert dec[0x00] == 0.0 and not np.signbit(dec[0x00])
    assert dec[0x80] == 0.0 and np.signbit(dec[0x80])
    assert dec[0x01] == 2.0 ** -9            # smallest subnormal
    assert dec[0x07] == 7 * 2.0 ** -9        # largest subnormal
    assert dec[0x08] == 2.0 ** -6            # smallest normal
    assert dec[0x38] == 1.0                  # exponent field 7 = bias
    assert dec[0x39] == 1.125
    assert dec[0x7E] == 448.0                # largest finite
    assert dec[0xFE] == -448.0
    assert np.isnan(dec[0x7F]) and np.isnan(dec[0xFF])
    # 126 distinct positive finite values, strictly increasing with the code
    pos = dec[0x01:0x7F]
    assert np.all(np.diff(pos) > 0)


def test_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    dec = oracle.e4m3_decode(codes.numpy())
    finite = ~np.isnan(ref)
    assert np.array_equal(np.isnan(dec), np.isnan(ref))
    assert np.array_equal(dec[finite], ref[finite])


def test_encode_roundtrip_every_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_midpoints_round_to_even_code():
    for c in range(0x00, 0x7E):
        lo, hi = oracle.e4m3_decode(np.array([c, c + 1], dtype=np.uint8))
        mid = np.float32((lo + hi) / 2)          # exact: at most 5 significant bits
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode([mid])[0] == even, hex(c)
        assert oracle.e4m3_encode([-mid])[0] == (even | 0x80)
        above = np.nextafter(mid, np.float32(np.inf), dtype=np.float32)
        below = np.nextafter(mid, np.float32(0), dtype=np.float32)
        assert oracle.e4m3_encode([above])[0] == c + 1
        assert oracle.e4m3_encode([below])[0] == c


def test_saturation_to_448():
    big = np.array([448.0, 455.9, 464.0, 480.0, 1e6, 3.0e38, np.inf], dtype=np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)


def test_tiny_values_and_signed_zero():
    half_min_sub = np.float32(2.0 ** -10)     # tie between 0 and 2^-9: even is 0
    assert oracle.e4m3_encode([half_min_sub])[0] == 0x00
    assert oracle.e4m3_encode([-half_min_sub])[0] == 0x80
    assert oracle.e4m3_encode([np.float32(1.5 * 2.0 ** -10)])[0] == 0x01
    assert oracle.e4m3_encode([np.float32(1e-30)])[0] == 0x00
    assert oracle.e4m3_encode([np.float32(-0.0)])[0] == 0x80


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_encode_matches_torch_rne_in_range(seed):
    rng = np.random.default_rng(seed)
    # log-uniform magnitudes across subnormal and normal binades, both signs
    mag = np.exp2(rng.uniform(-12, np.log2(440.0), size=200_000))
    y = (mag * rng.choice([-1.0, 1.0], size=mag.size)).astype(np.float32)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(y), ref)


def test_encode_error_within_half_quantum():
    rng = np.random.default_rng(7)
    y = rng.uniform(-448, 448, size=100_000).astype(np.float32)
    dec = oracle.e4m3_decode(oracle.e4m3_encode(y))
    a = np.abs(y.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    quantum = np.exp2(e - 3)
    assert np.all(np.abs(dec - y) <= quantum / 2)
