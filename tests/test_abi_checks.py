"""Host-side argument checks of every compute entry point, through the C ABI.

Each case here must be refused before the library makes any CUDA call: a null
pointer, a shape outside the documented limits, an unaligned operand or an
invalid gradient scale returns its status code and a message for the calling
thread.  The non-null pointers below are made-up addresses that are never
dereferenced.  So that a check that wrongly passed could never launch a
kernel on them, the cases run only on machines without a GPU.
"""
import ctypes

import pytest

TQ2_OK, TQ2_EINVAL, TQ2_ESHAPE = 0, 1, 2
A = 0x10000        # a made-up 16-byte aligned address
U = 0x10004        # a made-up address that is not 16-byte aligned


@pytest.fixture(scope="module")
def lib():
    import torch
    if torch.cuda.is_available():
        pytest.skip("made-up device addresses are only passed where no GPU exists")
    import binary_packed_weight_gb300 as bpw
    from binary_packed_weight_gb300 import build
    build.build()
    return bpw.load()


def _err(lib):
    return lib.tq2_last_error().decode()


def test_tq2_calls(lib):
    assert lib.tq2_gemm(A, A, A, 0, 16, 128, None) == TQ2_OK            # M = 0: nothing to do
    assert lib.tq2_gemm(None, A, A, 1, 16, 128, None) == TQ2_EINVAL
    assert lib.tq2_gemm(A, None, A, 1, 16, 128, None) == TQ2_EINVAL
    for M in (-1, (1 << 24) + 1):                                      # refused before the handle is read
        assert lib.tq2_gemm(A, A, A, M, 16, 128, None) == TQ2_ESHAPE, M
    assert lib.tq2_gemm_path(None, A, A, 1, 16, 128, 1, None) == TQ2_EINVAL
    assert lib.tq2_gemm_tensor_tuned(None, A, A, 32, 16, 128, 32, 1, None) == TQ2_EINVAL
    assert lib.tq2_gemm_skinny_static(None, A, A, 1, 16, 128, None) == TQ2_EINVAL
    assert lib.tq2_shape(None, None, None) == TQ2_EINVAL
    assert lib.tq2_unpack(None, A, None) == TQ2_EINVAL
    assert lib.tq2_dequant_f16(None, A, None) == TQ2_EINVAL
    hs = (ctypes.c_void_p * 1)(A)
    assert lib.tq2_gemm_grouped(None, None, None, 1, 1, 128, None) == TQ2_EINVAL
    assert lib.tq2_gemm_grouped(hs, hs, hs, 0, 1, 128, None) == TQ2_ESHAPE
    assert lib.tq2_gemm_grouped(hs, hs, hs, 65, 1, 128, None) == TQ2_ESHAPE
    assert "G <= 64" in _err(lib)
    assert lib.tq2_gemm_grouped(hs, hs, hs, 1, 9, 128, None) == TQ2_ESHAPE   # M <= 8 only
    assert lib.tq2_gemm_grouped(hs, hs, hs, 1, 2, 32768, None) == TQ2_ESHAPE  # MT*K <= 32768
    assert lib.tq2_gemm_grouped(hs, hs, hs, 1, 3, 16384, None) == TQ2_ESHAPE  # M = 3 counts as MT = 4
    assert lib.tq2_gemm_grouped(hs, hs, hs, 1, 5, 8192, None) == TQ2_ESHAPE   # M = 5 counts as MT = 8


def test_debug_wait_timeout_bound(lib):
    assert lib.tq2_debug_wait_timeout(0, None) == TQ2_EINVAL
    assert lib.tq2_debug_wait_timeout(1_000_000_001, None) == TQ2_EINVAL


def test_quantize(lib):
    assert lib.tq2_quantize(None, 1, 128, A, None) == TQ2_EINVAL
    assert lib.tq2_quantize(A, 1, 128, None, None) == TQ2_EINVAL
    for N, K in ((0, 128), (1, 0), (1, 64), (1, 200), (-1, 128)):
        assert lib.tq2_quantize(A, N, K, A, None) == TQ2_ESHAPE, (N, K)
    assert lib.tq2_quantize(A, 1 << 40, 128, A, None) == TQ2_ESHAPE


def test_expand_bits(lib):
    assert lib.blr_expand_bits(A, 0, 32, A, 0, None) == TQ2_ESHAPE
    assert lib.blr_expand_bits(A, 4, 48, A, 0, None) == TQ2_ESHAPE
    assert lib.blr_expand_bits(A, 4, 16, A, 0, None) == TQ2_ESHAPE


GOOD = (70, 64, 128, 128)          # T, d_in, d_out, r
BAD_SHAPES = [(0, 64, 128, 128), (70, 100, 128, 128), (70, 64, 96, 128), (70, 64, 128, 64),
              (70, 64, 128, 192), (70, 32, 128, 128), (1 << 22, 1024, 1024, 128)]


def _fwd(lib, T, din, dout, r, x=A, g=A, l=A, y=A):
    return lib.blr_forward(A, A, A, l, g, x, y, A, None, T, din, dout, r, None)


def _bwd(lib, T, din, dout, r, gscale=1.0, dy=A, h=A, l=A, a=A):
    return lib.blr_backward(A, A, h, l, A, A, dy, a, None, A, A, A, A, T, din, dout, r, gscale, None)


def test_blr_forward_backward(lib):
    assert lib.blr_forward(None, A, A, A, A, A, A, A, None, *GOOD, None) == TQ2_EINVAL
    for s in BAD_SHAPES:
        assert _fwd(lib, *s) == TQ2_ESHAPE, s
        assert _bwd(lib, *s) == TQ2_ESHAPE, s
    assert "r a multiple of 128" in _err(lib) or "too large" in _err(lib)
    for kw in (dict(x=U), dict(g=U), dict(l=U)):
        assert _fwd(lib, *GOOD, **kw) == TQ2_EINVAL, kw
    for kw in (dict(dy=U), dict(h=U), dict(l=U), dict(a=U)):
        assert _bwd(lib, *GOOD, **kw) == TQ2_EINVAL, kw
    for gs in (0.0, -2.0, 3.0, 0.75, float("inf"), float("nan")):
        assert _bwd(lib, *GOOD, gscale=gs) == TQ2_EINVAL, gs
        assert "power of two" in _err(lib)


def _paths(n, bad=None):
    import binary_packed_weight_gb300 as bpw
    arr = (bpw.BlrPath * max(n, 1))()
    for p in arr:
        for f, _ in bpw.BlrPath._fields_:
            setattr(p, f, A)
        p.c_save = None
    for i, (f, v) in (bad or {}).items():
        setattr(arr[i], f, v)
    return arr


def test_blr_paths(lib):
    ps = _paths(2)
    assert lib.blr_forward_paths(None, 2, A, A, *GOOD, None) == TQ2_EINVAL
    for P in (0, -1, 65):
        assert lib.blr_forward_paths(ps, P, A, A, *GOOD, None) == TQ2_EINVAL, P
        assert lib.blr_backward_paths(ps, P, A, A, A, *GOOD, 1.0, None) == TQ2_EINVAL, P
    assert "P <= 64" in _err(lib)
    for s in BAD_SHAPES:
        assert lib.blr_forward_paths(ps, 2, A, A, *s, None) == TQ2_ESHAPE, s
        assert lib.blr_backward_paths(ps, 2, A, A, A, *s, 1.0, None) == TQ2_ESHAPE, s
    assert lib.blr_forward_paths(ps, 2, U, A, *GOOD, None) == TQ2_EINVAL
    assert lib.blr_backward_paths(ps, 2, A, U, A, *GOOD, 1.0, None) == TQ2_EINVAL
    assert lib.blr_backward_paths(ps, 2, A, A, A, *GOOD, 3.0, None) == TQ2_EINVAL
    # a null or unaligned operand of a later path names that path
    assert lib.blr_forward_paths(_paths(2, {1: ("h", None)}), 2, A, A, *GOOD, None) == TQ2_EINVAL
    assert "path 1" in _err(lib)
    assert lib.blr_forward_paths(_paths(3, {2: ("g", U)}), 3, A, A, *GOOD, None) == TQ2_EINVAL
    assert "path 2" in _err(lib)
    assert lib.blr_backward_paths(_paths(2, {1: ("dl", None)}), 2, A, A, A, *GOOD, 1.0, None) == TQ2_EINVAL
    assert "path 1" in _err(lib)
    assert lib.blr_backward_paths(_paths(2, {0: ("a_save", U)}), 2, A, A, A, *GOOD, 1.0, None) == TQ2_EINVAL
    assert "path 0" in _err(lib)


def test_blr_sign_grads(lib):
    def call(T=70, din=64, dout=128, r=128, gscale=1.0, **kw):
        a = dict(bits_u=A, h=A, l=A, g=A, x=A, dy=A, a_save=A, gu=A, gv=A)
        a.update(kw)
        return lib.blr_sign_grads(a["bits_u"], a["h"], a["l"], a["g"], a["x"], a["dy"], a["a_save"], a["gu"],
                                  a["gv"], T, din, dout, r, gscale, None)
    for f in ("bits_u", "h", "l", "g", "x", "dy", "a_save", "gu", "gv"):
        assert call(**{f: None}) == TQ2_EINVAL, f
    for s in BAD_SHAPES:
        assert call(*s) == TQ2_ESHAPE, s
    for f in ("h", "l", "g", "x", "dy", "a_save"):
        assert call(**{f: U}) == TQ2_EINVAL, f
    for gs in (0.0, 3.0, float("nan")):
        assert call(gscale=gs) == TQ2_EINVAL, gs
