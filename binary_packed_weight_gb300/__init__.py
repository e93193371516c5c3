"""Python binding of the tq2-gb300 C ABI (``include/tq2.h``).

Argument marshalling only: every function forwards device pointers, sizes
and the current CUDA stream of torch to the shared library
``libtq2gb300.so`` built from ``csrc/``.  There is no fallback: if the
library is missing or fails to load, every call raises.

Tensors must live on the current CUDA device, be contiguous and have the
dtype the C ABI states (float32 for activations and outputs, uint8 / int16
bit patterns for packed data).
"""
import ctypes
import os

__all__ = [
    "load", "lib_path", "TQ2Error", "Weight", "tq2_upload", "tq2_gemm", "tq2_gemm_path", "tq2_gemm_tensor_tuned",
    "tq2_gemm_skinny_static", "tq2_gemm_grouped", "GroupedGemv", "tq2_unpack", "tq2_dequant_f16", "tq2_quantize", "blr_expand_bits", "blr_forward", "blr_backward", "blr_forward_paths", "blr_backward_paths", "blr_sign_grads",
    "device_status", "debug_wait_timeout", "PATH_AUTO", "PATH_SKINNY", "PATH_TENSOR",
]

PATH_AUTO, PATH_SKINNY, PATH_TENSOR = 0, 1, 2
_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "libtq2gb300.so")
_lib = None

_P, _I64, _I, _F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
_SIGS = {
    "tq2_status_string": (ctypes.c_char_p, [_I]),
    "tq2_last_error": (ctypes.c_char_p, []),
    "tq2_version": (ctypes.c_char_p, []),
    "tq2_device_status": (_I, [_P]),
    "tq2_debug_wait_timeout": (_I, [ctypes.c_uint64, _P]),
    "tq2_upload": (_I, [_P, _I64, _I64, ctypes.POINTER(_P), _P]),
    "tq2_free": (_I, [_P]),
    "tq2_shape": (_I, [_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
    "tq2_gemm": (_I, [_P, _P, _P, _I64, _I64, _I64, _P]),
    "tq2_gemm_path": (_I, [_P, _P, _P, _I64, _I64, _I64, _I, _P]),
    "tq2_gemm_tensor_tuned": (_I, [_P, _P, _P, _I64, _I64, _I64, _I, _I, _P]),
    "tq2_gemm_skinny_static": (_I, [_P, _P, _P, _I64, _I64, _I64, _P]),
    "tq2_gemm_grouped": (_I, [_P, _P, _P, _I, _I64, _I64, _P]),
    "tq2_unpack": (_I, [_P, _P, _P]),
    "tq2_dequant_f16": (_I, [_P, _P, _P]),
    "tq2_quantize": (_I, [_P, _I64, _I64, _P, _P]),
    "blr_expand_bits": (_I, [_P, _I64, _I64, _P, _I, _P]),
    "blr_forward": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P]),
    "blr_backward": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                          _I64, _I64, _I64, _I64, _F, _P]),
    "blr_forward_paths": (_I, [_P, _I, _P, _P, _I64, _I64, _I64, _I64, _P]),
    "blr_backward_paths": (_I, [_P, _I, _P, _P, _P, _I64, _I64, _I64, _I64, _F, _P]),
    "blr_sign_grads": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _F, _P]),
}


class BlrPath(ctypes.Structure):
    """``blr_path`` of include/tq2.h: device pointers of one path."""
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("bits_u", "bits_v", "h", "l", "g", "a_save", "c_save", "dh", "dl", "dg")]


class TQ2Error(RuntimeError):
    def __init__(self, status, where):
        msg = load().tq2_last_error().decode(errors="replace")
        name = load().tq2_status_string(status).decode()
        super().__init__(f"{where}: {name} ({status}): {msg}")
        self.status = status


def load():
    """Load the shared library (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(lib_path):
            raise RuntimeError(f"{lib_path} is missing; build it with binary_packed_weight_gb300.build.build()")
        lib = ctypes.CDLL(lib_path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
    return _lib


def _check(status, where):
    if status != 0:
        raise TQ2Error(status, where)


def _stream(stream):
    if stream is not None:
        return ctypes.c_void_p(int(stream))
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class Weight:
    """A ``BlockTQ2_0_g128`` weight resident on the GPU (owns a C handle)."""

    def __init__(self, handle, N, K):
        self._h, self.N, self.K = handle, N, K

    @property
    def handle(self):
        return self._h

    def free(self):
        if self._h:
            _check(load().tq2_free(self._h), "tq2_free")
            self._h = None

    def __del__(self):
        try:
            if self._h and _lib is not None:
                _lib.tq2_free(self._h)
        except Exception:
            pass


def tq2_upload(aos, N, K, stream=None):
    """Upload AoS block bytes (host ``bytes`` / numpy uint8) -> :class:`Weight`."""
    buf = bytes(aos) if not isinstance(aos, (bytes, bytearray)) else aos
    arr = (ctypes.c_uint8 * len(buf)).from_buffer_copy(buf)
    h = ctypes.c_void_p()
    _check(load().tq2_upload(ctypes.cast(arr, _P), N, K, ctypes.byref(h), _stream(stream)), "tq2_upload")
    return Weight(h.value, N, K)


def tq2_gemm(w, x, out, stream=None):
    M, K = x.shape
    _check(load().tq2_gemm(w.handle, _ptr(x), _ptr(out), M, w.N, K, _stream(stream)), "tq2_gemm")
    return out


def tq2_gemm_path(w, x, out, path, stream=None):
    M, K = x.shape
    _check(load().tq2_gemm_path(w.handle, _ptr(x), _ptr(out), M, w.N, K, path, _stream(stream)), "tq2_gemm_path")
    return out


def tq2_gemm_tensor_tuned(w, x, out, bn=0, splits=0, stream=None):
    """The tensor-core path with a chosen token tile (bn) and K-split count."""
    M, K = x.shape
    _check(load().tq2_gemm_tensor_tuned(w.handle, _ptr(x), _ptr(out), M, w.N, K, int(bn), int(splits),
                                        _stream(stream)), "tq2_gemm_tensor_tuned")
    return out


def tq2_gemm_skinny_static(w, x, out, stream=None):
    """Skinny GEMM (M <= 16) that allocates nothing: its scratch is a fixed
    device array inside the library (see include/tq2.h)."""
    M, K = x.shape
    _check(load().tq2_gemm_skinny_static(w.handle, _ptr(x), _ptr(out), M, w.N, K, _stream(stream)),
           "tq2_gemm_skinny_static")
    return out


def tq2_gemm_grouped(ws, xs, outs, stream=None):
    """G independent GEMVs (M <= 8, same K) in one launch: outs[g] = xs[g] @ W_g^T."""
    G = len(ws)
    M, K = xs[0].shape
    hs = (_P * G)(*[w.handle for w in ws])
    xp = (_P * G)(*[x.data_ptr() for x in xs])
    op = (_P * G)(*[o.data_ptr() for o in outs])
    _check(load().tq2_gemm_grouped(ctypes.cast(hs, _P), ctypes.cast(xp, _P), ctypes.cast(op, _P), G, M, K,
                                   _stream(stream)), "tq2_gemm_grouped")
    return outs


class GroupedGemv:
    """tq2_gemm_grouped with its arguments marshalled once: the handle and
    pointer arrays are built at construction (the tensors are kept alive), so a
    loop that calls the same group every step pays one C call per step."""

    def __init__(self, ws, xs, outs):
        self._keep = (list(ws), list(xs), list(outs))
        self.G = len(ws)
        self.M, self.K = xs[0].shape
        self._hs = (_P * self.G)(*[w.handle for w in ws])
        self._xp = (_P * self.G)(*[x.data_ptr() for x in xs])
        self._op = (_P * self.G)(*[o.data_ptr() for o in outs])
        self._args = (ctypes.cast(self._hs, _P), ctypes.cast(self._xp, _P), ctypes.cast(self._op, _P))

    def __call__(self, stream=None):
        _check(load().tq2_gemm_grouped(*self._args, self.G, self.M, self.K, _stream(stream)), "tq2_gemm_grouped")
        return self._keep[2]


def tq2_unpack(w, stream=None):
    n = w.N * (w.K // 128) * 34
    buf = (ctypes.c_uint8 * n)()
    _check(load().tq2_unpack(w.handle, ctypes.cast(buf, _P), _stream(stream)), "tq2_unpack")
    return bytes(buf)


def tq2_dequant_f16(w, out_u16, stream=None):
    _check(load().tq2_dequant_f16(w.handle, _ptr(out_u16), _stream(stream)), "tq2_dequant_f16")
    return out_u16


def tq2_quantize(w, aos_out, stream=None):
    """f32 weights ``w`` [N, K] (device) -> BlockTQ2_0_g128 blocks in ``aos_out``
    (device uint8, N*(K/128)*34 bytes)."""
    N, K = w.shape
    _check(load().tq2_quantize(_ptr(w), N, K, _ptr(aos_out), _stream(stream)), "tq2_quantize")
    return aos_out


def blr_expand_bits(bits, rows, r, plane, transpose, stream=None):
    _check(load().blr_expand_bits(_ptr(bits), rows, r, _ptr(plane), int(transpose), _stream(stream)),
           "blr_expand_bits")
    return plane


def blr_forward(bits_u, bits_v, h, l, g, x, y, a_save, c_save=None, stream=None):
    T, d_in = x.shape
    d_out, r = h.numel(), l.numel()
    _check(load().blr_forward(_ptr(bits_u), _ptr(bits_v), _ptr(h), _ptr(l), _ptr(g), _ptr(x), _ptr(y),
                              _ptr(a_save), _ptr(c_save), T, d_in, d_out, r, _stream(stream)), "blr_forward")
    return y


def blr_backward(bits_u, bits_v, h, l, g, x, dy, a_save, c_save, dx, dh, dl, dg, gscale=1.0, stream=None):
    T, d_in = x.shape
    d_out, r = h.numel(), l.numel()
    _check(load().blr_backward(_ptr(bits_u), _ptr(bits_v), _ptr(h), _ptr(l), _ptr(g), _ptr(x), _ptr(dy),
                               _ptr(a_save), _ptr(c_save), _ptr(dx), _ptr(dh), _ptr(dl), _ptr(dg),
                               T, d_in, d_out, r, float(gscale), _stream(stream)), "blr_backward")
    return dx


def _paths_array(paths):
    """List of dicts of tensors (keys as BlrPath's fields; missing ones are NULL)."""
    arr = (BlrPath * len(paths))()
    for i, p in enumerate(paths):
        for name, _ in BlrPath._fields_:
            setattr(arr[i], name, _ptr(p.get(name)))
    return arr


def blr_forward_paths(paths, x, y, stream=None):
    """y = sum over paths, combined with the pages' rounding (see include/tq2.h)."""
    T, d_in = x.shape
    d_out, r = paths[0]["h"].numel(), paths[0]["l"].numel()
    arr = _paths_array(paths)
    _check(load().blr_forward_paths(ctypes.cast(arr, _P), len(paths), _ptr(x), _ptr(y), T, d_in, d_out, r,
                                    _stream(stream)), "blr_forward_paths")
    return y


def blr_backward_paths(paths, x, dy, dx, gscale=1.0, stream=None):
    T, d_in = x.shape
    d_out, r = paths[0]["h"].numel(), paths[0]["l"].numel()
    arr = _paths_array(paths)
    _check(load().blr_backward_paths(ctypes.cast(arr, _P), len(paths), _ptr(x), _ptr(dy), _ptr(dx), T, d_in, d_out,
                                     r, float(gscale), _stream(stream)), "blr_backward_paths")
    return dx


def blr_sign_grads(bits_u, h, l, g, x, dy, a_save, gu, gv, gscale=1.0, stream=None):
    """G_U [d_out, r] and G_V [d_in, r] of one path (see include/tq2.h)."""
    T, d_in = x.shape
    d_out, r = h.numel(), l.numel()
    _check(load().blr_sign_grads(_ptr(bits_u), _ptr(h), _ptr(l), _ptr(g), _ptr(x), _ptr(dy), _ptr(a_save), _ptr(gu),
                                 _ptr(gv), T, d_in, d_out, r, float(gscale), _stream(stream)), "blr_sign_grads")
    return gu, gv


def debug_wait_timeout(limit_ns, stream=None):
    """Launch the test kernel whose bounded wait runs out after ``limit_ns``
    (see include/tq2.h); the next :func:`device_status` raises TQ2_ETIMEOUT."""
    _check(load().tq2_debug_wait_timeout(int(limit_ns), _stream(stream)), "tq2_debug_wait_timeout")


def device_status(stream=None):
    """Synchronize and raise if a kernel recorded a bounded-wait timeout."""
    _check(load().tq2_device_status(_stream(stream)), "tq2_device_status")
