"""Failure detection on the GPU without a fault: a bounded device-side wait
that runs out ends as a status the host reads, and the context stays usable.

Every wait inside the library's kernels gives up after a bounded time and
records the timeout instead of hanging the GPU.  ``tq2_debug_wait_timeout``
runs that path on purpose (one thread waits on a barrier that nothing
completes, with a bound of a few milliseconds); nothing faults, traps or
hangs.
"""
import numpy as np
import pytest

import synth
from gpu_util import check_skinny, oracle_gemm, run_gemm

pytestmark = pytest.mark.gpu

TQ2_ETIMEOUT = 5


def test_bounded_wait_ends_as_a_status(lib):
    import torch
    torch.cuda.synchronize()
    lib.device_status()                                  # nothing recorded before
    lib.debug_wait_timeout(2_000_000)                    # gives up after 2 ms
    with pytest.raises(lib.TQ2Error) as info:
        lib.device_status()
    assert info.value.status == TQ2_ETIMEOUT
    lib.device_status()                                  # the record was read and cleared

    # the context still works: a small GEMM through the same library matches the oracle
    aos, N, K, xs = synth.tiny_tq2(M_list=(1, 7))
    w = lib.tq2_upload(aos, N, K)
    for M, x in xs.items():
        ref, absref, _, _ = oracle_gemm(aos, N, K, x)
        check_skinny(run_gemm(lib, w, x), ref, absref, f"after a timeout, M={M}")
    w.free()


def test_timeout_bound_is_checked(lib):
    for bad in (0, 1_000_000_001):
        with pytest.raises(lib.TQ2Error) as info:
            lib.debug_wait_timeout(bad)
        assert info.value.status == 1
