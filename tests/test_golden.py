"""The golden fixtures (``tests/golden/``) against the oracle (CPU only).

The fixtures were written by ``tests/golden/make_golden.py`` from the oracle
and the seeded generators; recomputing them here catches any change of the
oracle's arithmetic or of the input generators.  Each file's header cites the
passage its data and formula come from.
"""
import os

import numpy as np

import synth
from oracle import blr as oblr
from oracle import tq2 as otq2

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [line.split() for line in f if line.strip() and not line.startswith("#")]


def load_matrix(name):
    return np.array([[float(v) for v in r] for r in _rows(name)], dtype=np.float64)


def test_tq2_page_tiny_outputs():
    aos, N, K, xs = synth.tiny_tq2((1, 7))
    W = otq2.dequant_aos(aos, N, K)
    for M, x in xs.items():
        want = load_matrix(f"tq2_page_tiny_M{M}.txt")
        assert want.shape == (M, N)
        assert np.array_equal(otq2.gemm(x, W), want), M


def test_tq2_quantize_bytes():
    W = synth.random_weights_f32(16, 256, 501)
    got = otq2.pack_aos(*otq2.quantize(W))
    want = bytes.fromhex("".join(r[0] for r in _rows("tq2_quantize_16x256.txt")))
    assert got == want


def test_blr_tiny_forward_backward():
    p = synth.blr_inputs(4, 128, 96, 128, 601)
    y, _, _ = oblr.forward(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], p["x"])
    dx, dh, dl, dg, _, _ = oblr.backward(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], p["x"], p["dy"])
    assert np.array_equal(y, load_matrix("blr_tiny_y.txt"))
    assert np.array_equal(dx, load_matrix("blr_tiny_dx.txt"))
    rows = _rows("blr_tiny_dh_dl_dg.txt")
    for got, want in zip((dh, dl, dg), rows):
        assert np.array_equal(got, np.array([float(v) for v in want]))
