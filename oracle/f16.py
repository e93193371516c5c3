"""IEEE-754 binary16 for the oracle (test infrastructure only).

The TQ2 block scale ``d`` is an f16 stored as two little-endian bytes
("oxibonsai-kernels 0.2.1, tests_gemm_tq2.rs", the ``BlockTQ2_0_g128 { qs, d }``
literal of ``test_encode_gemm_tq2_matches_reference``, built with
``f16::from_f32``).  The decode below follows the binary16 definition:
1 sign bit, 5 exponent bits with bias 15, 10 fraction bits; exponent 0 is
zero / subnormal (value ``f * 2**-24``), exponent 31 is inf (f = 0) or NaN.

Rounding *to* f16 (the staging of activations, "cortiq-engine 0.8.43,
train_mm.rs", kernel ``cvt_col``: ``f16(v)``) is taken from numpy's
``astype(np.float16)``, a library primitive that rounds to nearest, ties to
even; ``tests/test_oracle_f16.py`` pins its tie behaviour.
"""
import numpy as np


def bits_to_float(bits):
    """Decode binary16 bit patterns (any integer array) to float64."""
    b = np.asarray(bits).astype(np.int64) & 0xFFFF
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    exp = (b >> 10) & 0x1F
    frac = b & 0x3FF
    sub = np.ldexp(frac.astype(np.float64), -24)                 # 0.f * 2^-14
    nrm = np.ldexp((1024 + frac).astype(np.float64), exp - 25)   # 1.f * 2^(e-15)
    mag = np.where(exp == 0, sub, nrm)
    mag = np.where(exp == 31, np.where(frac == 0, np.inf, np.nan), mag)
    return sign * mag


def round_to_f16(values):
    """Round float values to binary16 (nearest, ties to even); float64 out."""
    return np.asarray(values).astype(np.float16).astype(np.float64)


def round_to_f16_bits(values):
    """Like :func:`round_to_f16` but return the uint16 bit patterns."""
    return np.asarray(values).astype(np.float16).view(np.uint16)
