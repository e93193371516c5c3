"""Ternary ``BlockTQ2_0_g128`` GEMM, written from the format definition.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "oxibonsai-kernels 0.2.1, src/gpu_backend/metal_graph/tests_gemm_tq2.rs".

* Block format (test ``test_encode_gemm_tq2_matches_reference``: the LCG code
  generator, the ``qs`` packing loop and the ``BlockTQ2_0_g128 { qs, d }``
  literal): one block covers 128 consecutive K-elements of one weight row;
  ``qs`` is 32 bytes holding 4 two-bit codes per byte, packed LSB-first in
  generation order (``c0 | c1<<2 | c2<<4 | c3<<6``); ``d`` is an f16 scale.
  A code ``c`` in {0,1,2} stands for ``c - 1`` in {-1, 0, +1}.
* AoS byte layout (reading of the struct literal and of the raw
  ``size_of_val`` bytes that are uploaded): 34 bytes per block, ``qs[0..32]``
  then ``d`` little-endian, no padding; blocks row-major, ``K/128`` per row.
* GEMM (same test, "CPU reference" comment): ``out[m,n] = sum_k x[m,k] W[n,k]``
  with ``out`` row-major ``[M][N]``.
* Code 3 never occurs in the pages' data (codes are ``% 3``); it is decoded
  arithmetically as ``3 - 1 = +2``.
"""
import numpy as np

from . import f16

BLOCK_K = 128          # K-elements per block
QS_BYTES = 32          # packed code bytes per block
BLOCK_BYTES = 34       # qs + f16 scale


def parse_aos(aos, N, K):
    """Split AoS blocks into codes ``uint8 [N][K]`` and scale bits ``uint16 [N][K/128]``.

    Code ``i`` of byte ``j`` of block ``kb`` of row ``n`` is weight
    ``W[n, 128*kb + 4*j + i]`` (4 codes per byte, least significant first).
    """
    if K % BLOCK_K:
        raise ValueError("K must be a multiple of 128")
    nb = K // BLOCK_K
    raw = np.frombuffer(bytes(aos), dtype=np.uint8)
    if raw.size != N * nb * BLOCK_BYTES:
        raise ValueError("AoS size does not match N*(K/128)*34")
    raw = raw.reshape(N * nb, BLOCK_BYTES)
    qs = raw[:, :QS_BYTES]
    d_bits = raw[:, QS_BYTES].astype(np.uint16) | (raw[:, QS_BYTES + 1].astype(np.uint16) << 8)
    codes = np.empty((N * nb, BLOCK_K), dtype=np.uint8)
    for i in range(4):                      # field i of byte j -> element 4*j + i
        codes[:, i::4] = (qs >> (2 * i)) & 3
    return codes.reshape(N, K), d_bits.reshape(N, nb)


def dequant(codes, d_bits):
    """``W[n,k] = (c - 1) * d[n, k//128]`` in float64."""
    N, K = codes.shape
    d = f16.bits_to_float(d_bits)                        # [N][nb]
    return (codes.astype(np.float64) - 1.0) * np.repeat(d, BLOCK_K, axis=1)


def dequant_f16_bits(codes, d_bits):
    """The dequantized weight as f16 bit patterns.

    ``(c - 1) * d`` with ``c - 1`` in {-1, 0, 1, 2} is exactly representable
    in f16 whenever ``2*d`` does not overflow, so this is the exact value
    (IEEE signed zero included: ``0 * d`` is ``-0`` for negative ``d``).
    """
    return f16.round_to_f16_bits(dequant(codes, d_bits))


def dequant_aos(aos, N, K):
    codes, d_bits = parse_aos(aos, N, K)
    return dequant(codes, d_bits)


def gemm(x, W):
    """``out[m,n] = sum_k x[m,k] * W[n,k]`` in float64 (library matmul as one step)."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T


def gemm_abs(x, W):
    """``sum_k |x[m,k] * W[n,k]|``: the scale of the tensor-path error bound."""
    return np.abs(np.asarray(x, dtype=np.float64)) @ np.abs(np.asarray(W, dtype=np.float64)).T


def gemm_elem(x_row, codes_row, d_row):
    """One output element from one activation row and one weight row's codes/scales.

    Used to check sampled outputs of full-size problems one by one.
    """
    w = (codes_row.astype(np.float64) - 1.0) * np.repeat(f16.bits_to_float(d_row), BLOCK_K)
    xr = np.asarray(x_row, dtype=np.float64)
    return float(np.dot(xr, w)), float(np.dot(np.abs(xr), np.abs(w)))


def pack_aos(codes, d_bits):
    """Codes ``uint8 [N][K]`` and scale bits ``uint16 [N][K/128]`` -> AoS bytes.

    The inverse of :func:`parse_aos`: code of element ``4*j + i`` of a block
    in bits ``2i, 2i+1`` of byte ``j``, then ``d`` little-endian.
    """
    codes = np.asarray(codes, dtype=np.uint8)
    N, K = codes.shape
    nb = K // BLOCK_K
    c = codes.reshape(N * nb, QS_BYTES, 4)
    qs = c[:, :, 0] | (c[:, :, 1] << 2) | (c[:, :, 2] << 4) | (c[:, :, 3] << 6)
    d = np.asarray(d_bits, dtype=np.uint16).reshape(N * nb, 1)
    out = np.concatenate([qs.astype(np.uint8), (d & 0xFF).astype(np.uint8), (d >> 8).astype(np.uint8)], axis=1)
    return out.tobytes()


def quantize(W):
    """f32 weights ``[N][K]`` -> ternary codes ``uint8 [N][K]`` and f16 scale bits ``uint16 [N][K/128]``.

    Source: "rlx-mlx 0.2.13, src/lower/helpers.rs", the FakeQuantize helpers
    (``fq_q_max``, ``fq_scale_perbatch``, ``fq_quantize_dequantize``).  For 2
    bits ``q_max = 1``; the scale is ``max|w| / q_max`` floored at ``1e-12``;
    the quantized value is ``round(w / scale)`` clamped to ``[-q_max, q_max]``
    (the page then multiplies back by the scale).  Everything runs in the
    arrays' dtype, f32.

    Readings (the page reduces per channel or per tensor and stores nothing):
      * the maximum is taken over each 128-element block of a row, the
        granularity of ``BlockTQ2_0_g128``;
      * ``round`` rounds half to even, as the page's array library does;
      * the stored code is ``q + 1`` and ``d`` is the f32 scale rounded to
        f16 (nearest, ties to even).
    """
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    if K % BLOCK_K:
        raise ValueError("K must be a multiple of 128")
    blocks = W.reshape(N, K // BLOCK_K, BLOCK_K)
    q_max = np.float32(1.0)
    scale = np.maximum(np.abs(blocks).max(axis=2, keepdims=True) / q_max, np.float32(1e-12))
    q = np.clip(np.rint(blocks / scale), -q_max, q_max)
    codes = (q + np.float32(1.0)).astype(np.uint8).reshape(N, K)
    with np.errstate(over="ignore"):                  # scales above the f16 range round to +inf
        d_bits = f16.round_to_f16_bits(scale[..., 0].astype(np.float64)).astype(np.uint16)
    return codes, d_bits
