"""Pins of the oracle's binary16 handling (CPU only)."""
import warnings

import numpy as np

from oracle import f16


def test_decode_matches_numpy_for_every_pattern():
    # special case that reduces to a library routine: numpy's own half decode
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = f16.bits_to_float(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zero survives
    assert np.signbit(f16.bits_to_float(np.array([0x8000])))[0]


def test_decode_known_values():
    cases = {0x3C00: 1.0, 0xC000: -2.0, 0x7BFF: 65504.0, 0x0001: 2.0 ** -24,
             0x0400: 2.0 ** -14, 0x3555: 0.333251953125, 0x2C00: 0.0625}
    for b, v in cases.items():
        assert f16.bits_to_float(np.array([b]))[0] == v
    assert np.isinf(f16.bits_to_float(np.array([0x7C00]))[0])


def test_round_is_nearest_even():
    e = 2.0 ** -11          # half an ulp of 1.0 in f16
    assert f16.round_to_f16(1.0 + e) == 1.0                 # tie -> even (1.0)
    assert f16.round_to_f16(1.0 + 3 * e) == 1.0 + 4 * e     # tie -> even (1+2^-9)
    assert f16.round_to_f16(1.0 + 1.01 * e) == 1.0 + 2 * e  # above the tie
    with warnings.catch_warnings():
        warnings.simplefilter("ignore", RuntimeWarning)
        assert np.isinf(f16.round_to_f16(65520.0))          # rounds past max
    assert f16.round_to_f16(65519.0) == 65504.0
