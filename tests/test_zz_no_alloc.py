"""The allocation-free skinny GEMM (tq2_gemm_skinny_static).

Callers that must not allocate device memory during a GEMM (plugin or
custom-op interfaces that forbid allocation while enqueuing work, serving
processes that reserve all device memory up front, real-time loops) use
tq2_gemm_skinny_static, whose scratch is a fixed device array inside the
library (the fused GEMV, where it applies, needs none).  This test calls it
through the C ABI twice in a row per shape and checks each result against
the f64 oracle within the skinny kernel's bound and for bit equality with
tq2_gemm, which runs the same kernel: the fused GEMV for M <= 8 at this K,
the staged skinny kernel above that.  The file name makes pytest collect it
last.
"""
import ctypes

import numpy as np
import pytest

import synth
from gpu_util import check_skinny
from oracle import tq2 as otq2

pytestmark = pytest.mark.gpu


def _run(lib, fn_name, w, x):
    import torch
    M, K = x.shape
    xd = torch.from_numpy(x).cuda()
    out = torch.full((M, w.N), float("nan"), dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = getattr(lib.load(), fn_name)(w.handle, ctypes.c_void_p(xd.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                      M, w.N, K, stream)
    assert st == 0, lib.load().tq2_last_error()
    lib.device_status()
    return out.cpu().numpy().astype(np.float64)


def test_static_scratch_matches_oracle_and_regular_entry_point(lib):
    N, K = 3000, 4096
    aos = synth.random_tq2(N, K, 301)
    w = lib.tq2_upload(aos, N, K)
    W = otq2.dequant_aos(aos, N, K)
    for M in (1, 2, 3, 6, 9, 16):
        x = synth.random_x(M, K, 302 + M)
        ref, absref = otq2.gemm(x, W), otq2.gemm_abs(x, W)
        regular = _run(lib, "tq2_gemm", w, x)
        for call in range(2):                               # two calls in a row
            got = _run(lib, "tq2_gemm_skinny_static", w, x)
            check_skinny(got, ref, absref, f"static M={M} call {call}")
            assert np.array_equal(got, regular), M          # the same kernel as tq2_gemm


def test_static_scratch_refuses_oversized_requests(lib):
    N, K = 64, 32768                                        # M=16 needs 2 MiB of scratch
    w = lib.tq2_upload(synth.random_tq2(N, K, 310), N, K)
    import torch
    x = torch.zeros((16, K), dtype=torch.float32, device="cuda")
    out = torch.zeros((16, N), dtype=torch.float32, device="cuda")
    st = lib.load().tq2_gemm_skinny_static(w.handle, ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                           16, N, K, None)
    assert st == 2
    assert b"scratch" in lib.load().tq2_last_error()
