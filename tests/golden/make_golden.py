"""Write the golden fixtures of this directory.

Calls only the oracle (``oracle/``) and the seeded input generators
(``synth``); nothing here touches the GPU path.  Run from the repository
root:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle import blr as oblr  # noqa: E402
from oracle import tq2 as otq2  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def write_matrix(name, header, rows):
    with open(os.path.join(HERE, name), "w") as f:
        for line in header:
            f.write(f"# {line}\n")
        for r in np.atleast_2d(rows):
            f.write(" ".join(f"{float(v):.17g}" for v in r) + "\n")


def tq2_page_tiny():
    aos, N, K, xs = synth.tiny_tq2((1, 7))
    W = otq2.dequant_aos(aos, N, K)
    for M, x in xs.items():
        write_matrix(f"tq2_page_tiny_M{M}.txt", [
            "out[m][n] = sum_k x[m,k] W[n,k] for the page's tiny TQ2 data, computed by the f64 oracle.",
            'Data: "oxibonsai-kernels 0.2.1, src/gpu_backend/metal_graph/tests_gemm_tq2.rs",',
            "test test_encode_gemm_tq2_matches_reference: N=40, K=256, codes from the LCG (seed",
            "0x12345678, (s>>16)%3), d = f16(0.0625 + 0.0078125*(row + 0.5*blk)), x from the",
            f"xorshift64 generator rnd(M*K, seed 1, scale 0.5).  M={M}; one line per m, N values.",
        ], otq2.gemm(x, W))


def tq2_quantize_small():
    W = synth.random_weights_f32(16, 256, 501)
    codes, d_bits = otq2.quantize(W)
    aos = otq2.pack_aos(codes, d_bits)
    with open(os.path.join(HERE, "tq2_quantize_16x256.txt"), "w") as f:
        f.write("# BlockTQ2_0_g128 bytes (hex, one 34-byte block per line) that the oracle's\n")
        f.write('# 2-bit fake-quantize ("rlx-mlx 0.2.13, src/lower/helpers.rs", FakeQuantize\n')
        f.write("# helpers, applied per 128-block) gives for synth.random_weights_f32(16, 256, 501).\n")
        for i in range(0, len(aos), 34):
            f.write(aos[i:i + 34].hex() + "\n")


def blr_tiny():
    T, d_in, d_out, r = 4, 128, 96, 128
    p = synth.blr_inputs(T, d_in, d_out, r, 601)
    y, a, c = oblr.forward(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], p["x"])
    dx, dh, dl, dg, b, dxp = oblr.backward(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], p["x"], p["dy"])
    head = ['One blr path ("cortiq-engine 0.8.43, src/gpu_wgpu/train_mm.rs", blr_forward / blr_backward),',
            f"computed by the f64 oracle on synth.blr_inputs(T={T}, d_in={d_in}, d_out={d_out}, r={r}, key=601)."]
    write_matrix("blr_tiny_y.txt", head + ["y[t][i], one line per token."], y)
    write_matrix("blr_tiny_dx.txt", head + ["dx[t][j], one line per token."], dx)
    with open(os.path.join(HERE, "blr_tiny_dh_dl_dg.txt"), "w") as f:
        for line in head + ["Three lines: dh[i], dl[k], dg[j] (the increments)."]:
            f.write(f"# {line}\n")
        for v in (dh, dl, dg):
            f.write(" ".join(f"{float(x):.17g}" for x in v) + "\n")


if __name__ == "__main__":
    tq2_page_tiny()
    tq2_quantize_small()
    blr_tiny()
