"""The C-ABI library builds, loads on a machine without a GPU and exports
every function ``include/tq2.h`` declares.  Host-side argument checks run
without touching a device (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "tq2.h")).read()
    return re.findall(r"^TQ2_API\s+[\w\s\*]+?\b(\w+)\(", src, flags=re.M)


@pytest.fixture(scope="module")
def cdll():
    from binary_packed_weight_gb300 import build
    return ctypes.CDLL(build.build())


def test_header_declares_the_boundary():
    names = set(_declared())
    for want in ("tq2_upload", "tq2_free", "tq2_gemm", "tq2_unpack", "tq2_dequant_f16", "tq2_quantize",
                 "blr_expand_bits", "blr_forward", "blr_backward"):
        assert want in names


def test_every_declared_symbol_is_exported(cdll):
    missing = [n for n in _declared() if not hasattr(cdll, n)]
    assert not missing, missing


def test_binding_covers_the_header():
    import binary_packed_weight_gb300 as bpw
    assert set(_declared()) == set(bpw._SIGS)


def test_host_side_argument_checks(cdll):
    import binary_packed_weight_gb300 as bpw
    lib = bpw.load()
    h = ctypes.c_void_p(123)
    # null pointers and bad shapes are refused before any CUDA call
    assert lib.tq2_upload(None, 4, 128, ctypes.byref(h), None) == 1
    assert h.value is None
    buf = (ctypes.c_uint8 * 34)()
    assert lib.tq2_upload(ctypes.cast(buf, ctypes.c_void_p), 1, 100, ctypes.byref(h), None) == 2
    assert lib.tq2_upload(ctypes.cast(buf, ctypes.c_void_p), 0, 128, ctypes.byref(h), None) == 2
    assert b"K % 128" in lib.tq2_last_error() or b"K %" in lib.tq2_last_error()
    assert lib.tq2_gemm(None, None, None, 1, 1, 128, None) == 1
    assert lib.tq2_free(None) == 0
    assert lib.blr_expand_bits(None, 4, 32, None, 0, None) == 1
    assert lib.tq2_status_string(5) == b"device-side wait timed out"
    assert lib.tq2_version().startswith(b"tq2-gb300")
