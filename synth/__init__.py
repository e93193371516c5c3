"""Seeded synthetic inputs shared by the tests, the smoke run and the bench.

This module draws random numbers and lays them out in the method's *input*
formats (``BlockTQ2_0_g128`` AoS bytes, u32 sign bitmaps, f32 arrays).  It
holds none of the method's arithmetic: no decode, no dequantization, no GEMM.

Generators
----------
* ``lcg_codes`` -- the 32-bit linear congruential generator of
  "oxibonsai-kernels 0.2.1, tests_gemm_tq2.rs" (test
  ``test_encode_gemm_tq2_matches_reference``): ``s = s*1664525 + 1013904223``
  (mod 2**32), code ``(s >> 16) % 3``.
* ``xorshift_uniform`` -- the ``rnd`` helper of
  "cortiq-engine 0.8.43, train_mm.rs" (tests module): xorshift64 seeded with
  ``seed*0x9E3779B97F4A7C15 | 1``, value ``((s>>11)/2**53*2-1)*scale``.
* For the large workloads, numpy's Philox-4x64 counter-based bit generator
  (``random_raw``, a stream that numpy keeps stable across versions) with the
  transforms written out here: uniform ``(u >> 11) * 2**-53``, normal by
  Box-Muller, ternary codes ``(u16 * 3) >> 16`` from each 16-bit quarter of a
  draw (bias below 2e-5), sign bits straight from the raw words.
"""
import numpy as np

MASK64 = (1 << 64) - 1


# --------------------------------------------------------------------------
# the pages' own generators (small sizes; pure Python)
# --------------------------------------------------------------------------
def lcg_codes_loop(count, seed=0x12345678):
    """``count`` ternary codes from the pages' LCG, in generation order (loop)."""
    s = seed & 0xFFFFFFFF
    out = np.empty(count, dtype=np.uint8)
    for i in range(count):
        s = (s * 1664525 + 1013904223) & 0xFFFFFFFF
        out[i] = (s >> 16) % 3
    return out


def lcg_codes(count, seed=0x12345678):
    """The same codes as :func:`lcg_codes_loop`, by the closed form of the
    recurrence: state ``n`` is ``a^n s0 + c (1 + a + ... + a^(n-1))`` mod 2^32
    (numpy's uint64 products and sums wrap mod 2^64, which keeps mod 2^32)."""
    count = int(count)
    if count == 0:
        return np.empty(0, dtype=np.uint8)
    a, c = np.uint64(1664525), np.uint64(1013904223)
    powers = np.empty(count + 1, dtype=np.uint64)
    powers[0] = 1
    powers[1:] = a
    powers = np.cumprod(powers)                     # a^0 .. a^count (mod 2^64)
    geo = np.cumsum(powers[:-1])                    # 1 + a + ... + a^(n-1), n = 1..count
    states = (powers[1:] * np.uint64(seed & 0xFFFFFFFF) + c * geo) & np.uint64(0xFFFFFFFF)
    return ((states >> np.uint64(16)) % np.uint64(3)).astype(np.uint8)


def xorshift_uniform(n, seed, scale):
    """``n`` float32 values in ``(-scale, scale)`` from the pages' xorshift64."""
    s = ((seed * 0x9E3779B97F4A7C15) & MASK64) | 1
    out = np.empty(n, dtype=np.float32)
    for i in range(n):
        s ^= (s << 13) & MASK64
        s ^= s >> 7
        s ^= (s << 17) & MASK64
        out[i] = np.float32((((s >> 11) / float(1 << 53)) * 2.0 - 1.0)) * np.float32(scale)
    return out


# --------------------------------------------------------------------------
# vectorised generators for the large workloads (Philox-4x64)
# --------------------------------------------------------------------------
def _raw(n, key):
    return np.random.Philox(key=key).random_raw(int(n)).astype(np.uint64)


def uniform01(n, key):
    return (_raw(n, key) >> np.uint64(11)).astype(np.float64) * (1.0 / (1 << 53))


def uniform(n, key, lo, hi):
    """float32 iid U(lo, hi)."""
    return (lo + (hi - lo) * uniform01(n, key)).astype(np.float32)


def normal(n, key):
    """float32 iid N(0, 1) by Box-Muller on Philox uniforms."""
    h = (int(n) + 1) // 2
    u = uniform01(2 * h, key)
    u1 = 1.0 - u[:h]                     # (0, 1]
    u2 = u[h:]
    rad = np.sqrt(-2.0 * np.log(u1))
    z = np.concatenate([rad * np.cos(2 * np.pi * u2), rad * np.sin(2 * np.pi * u2)])
    return z[: int(n)].astype(np.float32)


def codes3(n, key):
    """uint8 iid uniform over {0, 1, 2}."""
    q = (int(n) + 3) // 4
    r = _raw(q, key)
    parts = [(r >> np.uint64(16 * i)) & np.uint64(0xFFFF) for i in range(4)]
    u16 = np.stack(parts, axis=1).reshape(-1)[: int(n)]
    return ((u16 * np.uint64(3)) >> np.uint64(16)).astype(np.uint8)


def sign_bits(rows, r, key):
    """uint32 bitmap ``[rows][r/32]`` with iid bits (+-1 with p = 1/2)."""
    w = (r + 31) // 32
    raw = _raw((rows * w + 1) // 2, key)
    words = np.stack([raw & np.uint64(0xFFFFFFFF), raw >> np.uint64(32)], axis=1).reshape(-1)
    return words[: rows * w].astype(np.uint32).reshape(rows, w)


def f16_bits(values):
    """Round to binary16 (numpy, nearest-even); return the bit patterns."""
    return np.asarray(values, dtype=np.float32).astype(np.float16).view(np.uint16)


# --------------------------------------------------------------------------
# input format: BlockTQ2_0_g128 AoS
# --------------------------------------------------------------------------
def pack_aos(codes, d_bits):
    """Lay codes ``[N][K]`` (values 0..3) and scales ``[N][K/128]`` out as AoS bytes.

    Each block: 32 bytes, byte ``j`` = ``c[4j] | c[4j+1]<<2 | c[4j+2]<<4 |
    c[4j+3]<<6`` (the pages' packing loop), then the f16 scale little-endian.
    """
    codes = np.asarray(codes, dtype=np.uint8)
    N, K = codes.shape
    nb = K // 128
    c = codes.reshape(N * nb, 32, 4).astype(np.uint8)
    qs = c[:, :, 0] | (c[:, :, 1] << 2) | (c[:, :, 2] << 4) | (c[:, :, 3] << 6)
    d = np.asarray(d_bits, dtype=np.uint16).reshape(N * nb)
    blocks = np.empty((N * nb, 34), dtype=np.uint8)
    blocks[:, :32] = qs
    blocks[:, 32] = (d & 0xFF).astype(np.uint8)
    blocks[:, 33] = (d >> 8).astype(np.uint8)
    return blocks.tobytes()


# --------------------------------------------------------------------------
# the workloads
# --------------------------------------------------------------------------
def tiny_tq2(M_list=(1, 7, 8, 9, 100), seed=0x12345678):
    """W N=40 x K=256 from the pages' LCG and scale formula; x iid U(-0.5, 0.5).

    Scale ``d = f16(0.0625 + 0.0078125*(row + 0.5*blk))`` computed in f32, as
    in test ``test_encode_gemm_tq2_matches_reference``.
    Returns ``(aos, N, K, {M: x})``.
    """
    N, K = 40, 256
    nb = K // 128
    codes = lcg_codes(N * K, seed).reshape(N, K)
    row = np.arange(N, dtype=np.float32)[:, None]
    blk = np.arange(nb, dtype=np.float32)[None, :]
    d = np.float32(0.0625) + np.float32(0.0078125) * (row + np.float32(0.5) * blk)
    aos = pack_aos(codes, f16_bits(d))
    xs = {M: xorshift_uniform(M * K, 1, 0.5).reshape(M, K) for M in M_list}
    return aos, N, K, xs


def page_x(M, K):
    """The page's index-derived activations ``(col*0.013 - 0.4) + row*0.0007`` (f32)."""
    row = np.arange(M, dtype=np.float32)[:, None]
    col = np.arange(K, dtype=np.float32)[None, :]
    return (col * np.float32(0.013) - np.float32(0.4)) + row * np.float32(0.0007)


def random_tq2(N, K, key):
    """Codes iid U{0,1,2}, scales iid U(0.01, 0.1) rounded to f16; AoS bytes."""
    codes = codes3(N * K, key).reshape(N, K)
    d = uniform(N * (K // 128), key + 1000, 0.01, 0.1).reshape(N, K // 128)
    return pack_aos(codes, f16_bits(d))


def random_x(M, K, key):
    """Activations iid N(0, 1), float32 ``[M][K]``."""
    return normal(M * K, key).reshape(M, K)


def random_weights_f32(N, K, key):
    """Dense f32 weights ``[N][K]`` for the ternary producer: iid N(0, 1)
    times a per-row magnitude drawn log-uniformly from [1e-3, 1e3], so that
    block maxima span six decades."""
    w = normal(N * K, key).reshape(N, K)
    mag = np.exp(uniform(N, key + 1, np.log(1e-3), np.log(1e3))).astype(np.float32)
    return (w * mag[:, None]).astype(np.float32)


def blr_inputs(T, d_in, d_out, r, key):
    """One blr path: bitmaps, metric vectors and x, dy (all iid, see module doc)."""
    return dict(
        bits_u=sign_bits(d_out, r, key),
        bits_v=sign_bits(d_in, r, key + 1),
        h=uniform(d_out, key + 2, 0.5, 1.5),
        l=uniform(r, key + 3, 0.5, 1.5),
        g=uniform(d_in, key + 4, 0.5, 1.5),
        x=normal(T * d_in, key + 5).reshape(T, d_in),
        dy=normal(T * d_out, key + 6).reshape(T, d_out),
    )


# Workload parameters (name -> dict); keys below are the Philox keys.
GEMV = dict(name="tq2_gemv", M=1, N=4096, K=4096, wkey=2, xkey=4)
SKINNY = dict(name="tq2_skinny", Ms=(8, 32, 128), N=11008, K=4096, wkey=5, xkey=7)
LARGE = dict(name="tq2_large", M=4096, N=14336, K=4096, wkey=8, xkey=10)
# the two DiT shapes of the pages' Metal benchmark ("oxibonsai-kernels 0.2.1", bench over
# (M, N, K) = (1536, 27648, 3072) and (1536, 3072, 3072)), same distributions as LARGE
DIT = (dict(name="tq2_dit_wide", M=1536, N=27648, K=3072, wkey=20, xkey=21),
       dict(name="tq2_dit_square", M=1536, N=3072, K=3072, wkey=22, xkey=23))
BLR = dict(name="blr_layer", T=2048, d_in=4096, d_out=4096, r=512, key=11)
