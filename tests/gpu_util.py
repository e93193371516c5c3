"""Helpers of the GPU parity tests (upload, run, compare with the oracle)."""
import numpy as np

import synth
from oracle import tq2 as otq2


def to_dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def run_gemm(bpw, w, x_np, path=None):
    import torch
    x = to_dev(x_np.astype(np.float32))
    out = torch.full((x_np.shape[0], w.N), float("nan"), dtype=torch.float32, device="cuda")
    if path is None:
        bpw.tq2_gemm(w, x, out)
    else:
        bpw.tq2_gemm_path(w, x, out, path)
    bpw.device_status()
    return out.cpu().numpy().astype(np.float64)


def oracle_gemm(aos, N, K, x):
    """Exact oracle, its |x||W| scale, and the oracle on f16-rounded x."""
    W = otq2.dequant_aos(aos, N, K)
    x64 = np.asarray(x, dtype=np.float64)
    x16 = np.asarray(x, dtype=np.float32).astype(np.float16).astype(np.float64)
    return otq2.gemm(x64, W), otq2.gemm_abs(x64, W), otq2.gemm(x16, W), otq2.gemm_abs(x16, W)


# Bounds:
#  skinny: |err| <= 1e-3 (pages, K <= 4096) and |err| <= 2^-12 * sum|x W| + 1e-7
#          (f32 accumulation over K <= 4096 terms, plus the 2^-22 split residual)
#  tensor: |err| <= 1e-2 * sum|x W| against the exact oracle (required), and
#          |err| <= 2^-11 * sum|x16 W| against the oracle on f16-rounded x
#          (only f32 accumulation differs).
def check_skinny(got, ref, absref, where=""):
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), where
    assert err.max() <= 1e-3, f"{where}: max abs err {err.max():.3e}"
    bad = err > (2.0 ** -12) * absref + 1e-7
    assert not bad.any(), f"{where}: {bad.sum()} elements above the accumulation bound"


def check_tensor(got, ref, absref, ref16, absref16, where=""):
    assert np.all(np.isfinite(got)), where
    err = np.abs(got - ref)
    bad = err > 1e-2 * absref + 1e-30
    assert not bad.any(), f"{where}: {bad.sum()} elements above 1e-2*sum|xW| (max err {err.max():.3e})"
    err16 = np.abs(got - ref16)
    bad16 = err16 > (2.0 ** -11) * absref16 + 1e-30
    assert not bad16.any(), f"{where}: {bad16.sum()} elements differ from the f16-x oracle beyond f32 accumulation"


def page_sweep_weight(N, K):
    """Weights of the page's v8/v9/v10 sweeps: LCG seed 0x9E3779B1 ^ (N<<8) ^ K,
    scale f16(0.05 + 0.003*(row%17) + 0.002*blk)."""
    nb = K // 128
    codes = synth.lcg_codes(N * K, (0x9E3779B1 ^ (N << 8) ^ K) & 0xFFFFFFFF).reshape(N, K)
    row = (np.arange(N) % 17).astype(np.float32)[:, None]
    blk = np.arange(nb, dtype=np.float32)[None, :]
    d = np.float32(0.05) + np.float32(0.003) * row + np.float32(0.002) * blk
    return synth.pack_aos(codes, synth.f16_bits(d))


def page_sweep_x(M, K):
    """Activations of the page's sweeps: sin(col*0.011 - 0.37) + row*0.0005 (f32)."""
    row = np.arange(M, dtype=np.float32)[:, None]
    col = np.arange(K, dtype=np.float32)[None, :]
    return (np.sin(col * np.float32(0.011) - np.float32(0.37)) + row * np.float32(0.0005)).astype(np.float32)
