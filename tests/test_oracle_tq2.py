"""Pins of the TQ2 oracle against the pages and plain mathematics (CPU only).

Each test is chosen so that a plausible slip in ``oracle/tq2.py`` (a wrong
bit index, a code offset other than -1, a transposed operand, a dropped
scale, a mis-read scale byte order) fails at least one of them.
"""
import numpy as np
import pytest

import synth
from oracle import tq2


def _page_pack_block(codes128, d_bits):
    """One block packed the way the page's test loop does it.

    ``for b in qs: c0..c3 = next_code(); b = c0 | c1<<2 | c2<<4 | c3<<6``,
    then the f16 scale, little-endian.
    """
    it = iter(int(c) for c in codes128)
    qs = []
    for _ in range(32):
        c0, c1, c2, c3 = next(it), next(it), next(it), next(it)
        qs.append(c0 | (c1 << 2) | (c2 << 4) | (c3 << 6))
    return bytes(qs) + bytes([d_bits & 0xFF, d_bits >> 8])


def test_parse_returns_codes_in_generation_order():
    seq = synth.lcg_codes(2 * 128 * 3)
    blocks = b"".join(_page_pack_block(seq[i * 128:(i + 1) * 128], 0x3C00) for i in range(6))
    codes, d = tq2.parse_aos(blocks, 3, 256)
    assert np.array_equal(codes.reshape(-1), seq)
    assert np.all(d == 0x3C00)


@pytest.mark.parametrize("hot", [0, 2, 3])
def test_one_hot_every_position(hot):
    # all codes 1 (weight 0) except one code at position k -> W = (hot-1)*d only at k
    d_bits, d = 0x3A00, 0.75
    for k in range(128):
        seq = np.ones(128, dtype=np.uint8)
        seq[k] = hot
        W = tq2.dequant_aos(_page_pack_block(seq, d_bits), 1, 128)
        want = np.zeros((1, 128))
        want[0, k] = (hot - 1) * d
        assert np.array_equal(W, want), k


def test_scale_bytes_little_endian_and_per_block():
    seq = np.full(256, 2, dtype=np.uint8)              # weight = +d everywhere
    aos = _page_pack_block(seq[:128], 0x3C00) + _page_pack_block(seq[128:], 0xC100)
    W = tq2.dequant_aos(aos, 1, 256)
    assert np.all(W[0, :128] == 1.0) and np.all(W[0, 128:] == -2.5)


def test_all_codes_one_gives_zero():
    N, K, M = 5, 384, 3
    codes = np.ones((N, K), dtype=np.uint8)
    d = synth.f16_bits(synth.uniform(N * 3, 1, 0.01, 0.1)).reshape(N, 3)
    W = tq2.dequant_aos(synth.pack_aos(codes, d), N, K)
    x = synth.random_x(M, K, 3)
    out = tq2.gemm(x, W)
    assert np.array_equal(out, np.zeros((M, N)))


def test_all_codes_two_closed_form():
    # out[m,n] = sum_blk d[n,blk] * sum_{k in blk} x[m,k]
    N, K, M = 7, 512, 4
    nb = K // 128
    codes = np.full((N, K), 2, dtype=np.uint8)
    d_bits = synth.f16_bits(synth.uniform(N * nb, 2, 0.01, 0.1)).reshape(N, nb)
    d = d_bits.view(np.float16).astype(np.float64)
    x = synth.random_x(M, K, 4).astype(np.float64)
    out = tq2.gemm(x, tq2.dequant_aos(synth.pack_aos(codes, d_bits), N, K))
    blocksum = x.reshape(M, nb, 128).sum(axis=2)           # [M][nb]
    want = np.array([[sum(d[n, b] * blocksum[m, b] for b in range(nb)) for n in range(N)]
                     for m in range(M)])
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)


def test_unit_vectors_recover_columns():
    # N != K so a transposed operand cannot even run; e_k picks column k of W
    N, K = 3, 256
    aos = synth.random_tq2(N, K, 20)
    codes, d_bits = tq2.parse_aos(aos, N, K)
    d = d_bits.view(np.float16).astype(np.float64)
    for k in (0, 1, 5, 127, 128, 200, 255):
        x = np.zeros((1, K))
        x[0, k] = 1.0
        out = tq2.gemm(x, tq2.dequant(codes, d_bits))
        want = (codes[:, k].astype(np.float64) - 1.0) * d[:, k // 128]
        assert np.array_equal(out[0], want)


def test_linearity():
    N, K = 9, 384
    W = tq2.dequant_aos(synth.random_tq2(N, K, 30), N, K)
    x1 = synth.random_x(3, K, 31).astype(np.float64)
    x2 = synth.random_x(3, K, 32).astype(np.float64)
    a, b = 0.75, -1.5
    np.testing.assert_allclose(tq2.gemm(a * x1 + b * x2, W),
                               a * tq2.gemm(x1, W) + b * tq2.gemm(x2, W), rtol=1e-12, atol=1e-12)


def test_dequant_f16_is_exact():
    N, K = 6, 256
    aos = synth.random_tq2(N, K, 40)
    codes, d_bits = tq2.parse_aos(aos, N, K)
    bits = tq2.dequant_f16_bits(codes, d_bits)
    back = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(back, tq2.dequant(codes, d_bits))
    assert set(np.unique(codes)) <= {0, 1, 2}


def test_page_cpu_reference_loop_on_page_data():
    # the page's own reference: dequant to f32, then a naive f32 loop
    aos, N, K, xs = synth.tiny_tq2(M_list=(1, 7, 8, 9))
    W = tq2.dequant_aos(aos, N, K)
    W32 = W.astype(np.float32)
    for M, x in list(xs.items()) + [(3, synth.page_x(3, K))]:
        ref = np.zeros((M, N), dtype=np.float32)
        for m in range(M):
            for n in range(N):
                acc = np.float32(0.0)
                for k in range(K):
                    acc = np.float32(acc + x[m, k] * W32[n, k])
                ref[m, n] = acc
        out = tq2.gemm(x, W)
        assert np.max(np.abs(out - ref)) < 1e-4
        assert np.any(np.abs(out) > 1e-6)


def test_gemm_elem_matches_full():
    N, K, M = 11, 640, 2
    aos = synth.random_tq2(N, K, 50)
    codes, d_bits = tq2.parse_aos(aos, N, K)
    x = synth.random_x(M, K, 51)
    W = tq2.dequant(codes, d_bits)
    full, fa = tq2.gemm(x, W), tq2.gemm_abs(x, W)
    for m in range(M):
        for n in range(N):
            v, a = tq2.gemm_elem(x[m], codes[n], d_bits[n])
            assert abs(v - full[m, n]) < 1e-12 and abs(a - fa[m, n]) < 1e-12


def test_rejects_bad_shapes():
    with pytest.raises(ValueError):
        tq2.parse_aos(b"\0" * 34, 1, 100)
    with pytest.raises(ValueError):
        tq2.parse_aos(b"\0" * 33, 1, 128)


def test_vectorised_lcg_equals_the_page_loop():
    for seed in (0x12345678, 0xDEADBEEF ^ 3072, 0x9E3779B1 ^ (40 << 8) ^ 256):
        assert np.array_equal(synth.lcg_codes(5000, seed), synth.lcg_codes_loop(5000, seed))


# ---- ternary producer ("rlx-mlx 0.2.13, src/lower/helpers.rs", FakeQuantize helpers, 2 bits)

def _random_codes_scales(N, K, seed):
    """Codes in {0,1,2} with at least one nonzero weight (code 0 or 2) per block,
    and positive normal f16 scales."""
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 3, size=(N, K)).astype(np.uint8)
    codes.reshape(N, K // 128, 128)[:, :, 0] = rng.choice([0, 2], size=(N, K // 128))
    d = rng.uniform(0.01, 0.1, size=(N, K // 128))
    return codes, tq2.f16.round_to_f16_bits(d).astype(np.uint16)


def test_quantize_inverts_dequant():
    # W = (c - 1) * d exactly in f32; the block maximum is d, so w / d = c - 1
    # exactly and the producer must return the same codes and scales
    codes, d_bits = _random_codes_scales(7, 512, 11)
    W = tq2.dequant(codes, d_bits).astype(np.float32)
    c2, d2 = tq2.quantize(W)
    assert np.array_equal(c2, codes)
    assert np.array_equal(d2, d_bits)
    assert tq2.pack_aos(c2, d2) == tq2.pack_aos(codes, d_bits)


def test_quantize_ties_round_half_to_even():
    w = np.zeros((1, 128), dtype=np.float32)
    w[0, 0] = 1.0                                  # block maximum: scale 1
    w[0, 1], w[0, 2] = 0.5, -0.5                   # ties -> 0 (even), not +-1
    w[0, 3], w[0, 4] = np.nextafter(np.float32(0.5), np.float32(1)), np.nextafter(np.float32(-0.5), np.float32(-1))
    w[0, 5], w[0, 6] = np.nextafter(np.float32(0.5), np.float32(0)), -1.0
    codes, d_bits = tq2.quantize(w)
    assert list(codes[0, :7]) == [2, 1, 1, 2, 0, 1, 0]
    assert int(d_bits[0, 0]) == 0x3C00             # f16 1.0


def test_quantize_zero_block_and_floor():
    # max|w| = 0: the 1e-12 floor keeps the division finite; f16(1e-12) is 0
    codes, d_bits = tq2.quantize(np.zeros((2, 256), dtype=np.float32))
    assert np.all(codes == 1) and np.all(d_bits == 0)


def test_quantize_scale_per_block_not_per_row():
    w = np.zeros((1, 256), dtype=np.float32)
    w[0, :128] = np.linspace(-2.0, 2.0, 128, dtype=np.float32)      # block 0: max 2
    w[0, 128:] = np.linspace(-0.25, 0.25, 128, dtype=np.float32)    # block 1: max 0.25
    codes, d_bits = tq2.quantize(w)
    assert int(d_bits[0, 0]) == 0x4000 and int(d_bits[0, 1]) == 0x3400   # f16 2.0, 0.25
    # each block uses its own maximum: the same relative pattern gives the same codes
    assert np.array_equal(codes[0, :128], codes[0, 128:])
    assert codes[0, 0] == 0 and codes[0, 127] == 2 and codes[0, 64] == 1


def test_quantize_error_and_sign_bounds():
    rng = np.random.default_rng(5)
    W = (rng.standard_normal((9, 640)) * rng.uniform(0.01, 10, size=(9, 1))).astype(np.float32)
    codes, d_bits = tq2.quantize(W)
    Wq = tq2.dequant(codes, d_bits)
    blocks = np.abs(W.reshape(9, 5, 128)).max(axis=2)                       # the f32 scales
    d = tq2.f16.bits_to_float(d_bits)
    bound = np.repeat(np.abs(d - blocks) + blocks / 2, 128, axis=1)          # |q(d - s)| + s/2
    assert np.all(np.abs(Wq - W) <= bound * (1 + 1e-6))
    q = codes.astype(np.int64) - 1
    assert np.all(q * np.sign(W) >= 0)                                       # never the opposite sign


def test_quantize_scale_outside_the_f16_range():
    w = np.zeros((1, 256), dtype=np.float32)
    w[0, 5] = 1e5                          # above the f16 maximum 65504: d rounds to +inf
    w[0, 128 + 9] = -3e-8                  # f16 subnormal range: d = 3e-8 rounds to 2^-25 -> 0x0000 or 0x0001
    codes, d_bits = tq2.quantize(w)
    assert int(d_bits[0, 0]) == 0x7C00
    assert codes[0, 5] == 2 and codes[0, 128 + 9] == 0
    assert int(d_bits[0, 1]) == 0x0000 or int(d_bits[0, 1]) == 0x0001
    # 3e-8 lies between 2^-25 (the midpoint of 0 and the smallest subnormal 2^-24) and 2^-24: rounds up
    assert int(d_bits[0, 1]) == 0x0001


# ---- pins of pack_aos (the inverse of the page's block layout) -------------

def test_pack_aos_bytes_equal_the_page_packing_loop():
    # several rows and blocks of LCG codes; every block must come out byte for
    # byte as the page's loop packs it ({qs, d} with qs[j] = c0|c1<<2|c2<<4|c3<<6)
    N, K = 3, 384
    codes = synth.lcg_codes(N * K, 0x2468ACE1).reshape(N, K)
    d_bits = np.array([[0x3C00, 0x2E66, 0xB800], [0x0001, 0x7BFF, 0x8000], [0x1234, 0x4321, 0xFC00]],
                      dtype=np.uint16)
    want = b"".join(_page_pack_block(codes[n, 128 * b:128 * (b + 1)], int(d_bits[n, b]))
                    for n in range(N) for b in range(K // 128))
    assert tq2.pack_aos(codes, d_bits) == want


def test_pack_aos_one_hot_byte_positions():
    # all codes 0 except code v at element e: only byte e//4 is nonzero and it
    # holds v << 2*(e%4); the scale follows as two little-endian bytes
    for v in (1, 2, 3):
        for e in (0, 1, 2, 3, 4, 37, 126, 127):
            codes = np.zeros((1, 128), dtype=np.uint8)
            codes[0, e] = v
            blk = tq2.pack_aos(codes, np.array([[0xABCD]], dtype=np.uint16))
            assert len(blk) == 34
            want = bytearray(34)
            want[e // 4] = v << (2 * (e % 4))
            want[32], want[33] = 0xCD, 0xAB
            assert blk == bytes(want), (v, e)


def test_pack_aos_literal_block():
    # codes 0,1,2,3 repeating: every qs byte is 0 | 1<<2 | 2<<4 | 3<<6 = 0xE4
    codes = np.tile(np.array([0, 1, 2, 3], dtype=np.uint8), 32).reshape(1, 128)
    assert tq2.pack_aos(codes, np.array([[0x3C00]], dtype=np.uint16)) == bytes([0xE4] * 32 + [0x00, 0x3C])
    # all codes 1 (weight 0): 0b01010101 = 0x55
    ones = np.ones((1, 128), dtype=np.uint8)
    assert tq2.pack_aos(ones, np.array([[0x0102]], dtype=np.uint16)) == bytes([0x55] * 32 + [0x02, 0x01])


def test_pack_then_parse_round_trips_including_code_3():
    rng = np.random.default_rng(7)
    N, K = 5, 512
    codes = rng.integers(0, 4, size=(N, K)).astype(np.uint8)          # code 3 included
    d_bits = rng.integers(0, 1 << 16, size=(N, K // 128)).astype(np.uint16)
    c2, d2 = tq2.parse_aos(tq2.pack_aos(codes, d_bits), N, K)
    assert np.array_equal(c2, codes) and np.array_equal(d2, d_bits)
    assert 3 in set(np.unique(codes))


# ---- pins of gemm_abs (the scale of the tensor-path bound) -----------------

def test_gemm_abs_hand_computed():
    # x = [1, -2, 0.5, -4], W rows [1, 1, -1, 0] and [-0.5, 2, 2, -1]:
    #   row 0: |1*1| + |-2*1| + |0.5*-1| + |-4*0| = 1 + 2 + 0.5 + 0 = 3.5
    #   row 1: |1*-0.5| + |-2*2| + |0.5*2| + |-4*-1| = 0.5 + 4 + 1 + 4 = 9.5
    # while the signed sums are 1 - 2 - 0.5 = -1.5 and -0.5 - 4 + 1 + 4 = 0.5
    x = np.array([[1.0, -2.0, 0.5, -4.0]])
    W = np.array([[1.0, 1.0, -1.0, 0.0], [-0.5, 2.0, 2.0, -1.0]])
    assert np.array_equal(tq2.gemm_abs(x, W), np.array([[3.5, 9.5]]))
    assert np.array_equal(tq2.gemm(x, W), np.array([[-1.5, 0.5]]))


def test_gemm_abs_bounds_the_signed_sum_with_equality_for_one_sign():
    N, K, M = 6, 256, 3
    W = tq2.dequant_aos(synth.random_tq2(N, K, 60), N, K)
    x = synth.random_x(M, K, 61).astype(np.float64)
    s, a = tq2.gemm(x, W), tq2.gemm_abs(x, W)
    assert np.all(np.abs(s) <= a * (1 + 1e-15))
    assert np.all(a > np.abs(s))                    # mixed signs: strictly larger
    # same-sign products: the absolute sum equals |signed sum|
    xp, Wp = np.abs(x), np.abs(W)
    np.testing.assert_allclose(tq2.gemm_abs(xp, Wp), tq2.gemm(xp, Wp), rtol=1e-13)
    np.testing.assert_allclose(tq2.gemm_abs(-xp, Wp), -tq2.gemm(-xp, Wp), rtol=1e-13)


def test_gemm_abs_ignores_signs_and_is_homogeneous():
    N, K, M = 4, 256, 2
    codes, d_bits = tq2.parse_aos(synth.random_tq2(N, K, 62), N, K)
    W = tq2.dequant(codes, d_bits)
    x = synth.random_x(M, K, 63).astype(np.float64)
    a = tq2.gemm_abs(x, W)
    flip = np.where(np.arange(K) % 3 == 0, -1.0, 1.0)
    np.testing.assert_allclose(tq2.gemm_abs(x * flip, W), a, rtol=1e-13)
    np.testing.assert_allclose(tq2.gemm_abs(x, -W), a, rtol=1e-13)
    np.testing.assert_allclose(tq2.gemm_abs(-3.0 * x, W), 3.0 * a, rtol=1e-13)
    # zero weights (code 1) contribute nothing: all-code-1 rows give exactly 0
    assert np.array_equal(tq2.gemm_abs(x, np.zeros((2, K))), np.zeros((M, 2)))


def test_gemm_abs_brute_force_tiny():
    # a pure-Python loop over every (m, n, k) on a 2 x 128 x 3 problem
    N, K, M = 3, 128, 2
    W = tq2.dequant_aos(synth.random_tq2(N, K, 64), N, K)
    x = synth.random_x(M, K, 65).astype(np.float64)
    got = tq2.gemm_abs(x, W)
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                p = x[m, k] * W[n, k]
                acc += p if p >= 0 else -p
            assert abs(got[m, n] - acc) <= 1e-12 * max(1.0, acc)
