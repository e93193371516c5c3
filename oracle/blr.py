"""Binary low-rank (``blr``) layer in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "cortiq-engine 0.8.43, src/gpu_wgpu/train_mm.rs".

* Module doc: one path is ``W = diag(h) S_U diag(l) S_V^T diag(g)`` with the
  signs kept as bitmaps; forward ``a = (x.g) S_V``, ``c = (a.l) S_U^T``,
  ``y += h.c``; backward ``dh = sum dy.c``, ``db = (dy.h) S_U``,
  ``dl = sum a.db``, ``dx' = (db.l) S_V^T``, ``dg = sum x.dx'``,
  ``dx += g.dx'`` (``.`` is the elementwise product, sums over tokens).
* Bitmap convention (kernels ``expand`` / ``expand_n`` / ``expand_t``): the
  bitmap is ``[rows][words]`` u32, bit ``j`` of word ``w`` is rank
  ``32*w + j``, a set bit is +1, a clear bit is -1.
* Shapes (struct ``Blr`` and ``blr_forward``): the layer is ``m x n`` (m
  outputs, n inputs), rank ``r``; ``S_U`` is ``[m][r]``, ``S_V`` is ``[n][r]``;
  ``x`` is ``[ntok][n]``, ``y`` is ``[ntok][m]``.
* The arithmetic is the f64 host reference of test ``blr_layer_matches_host``
  for one path, with ``y`` and ``dx`` written (not accumulated) and the
  metric gradients returned as the increments that ``blr_backward`` adds.
"""
import numpy as np


def expand_bits(bits, rows, r):
    """Sign bitmap ``uint32 [rows][ceil(r/32)]`` -> float64 ``[rows][r]`` of +-1."""
    w = (r + 31) // 32
    b = np.asarray(bits, dtype=np.uint32).reshape(rows, w)
    k = np.arange(r)
    bit = (b[:, k // 32] >> (k % 32).astype(np.uint32)) & np.uint32(1)
    return np.where(bit == 1, 1.0, -1.0)


def forward(bits_u, bits_v, h, l, g, x):
    """Return ``(y, a, c)`` for one path; ``x`` is ``[T][n]``."""
    x = np.asarray(x, dtype=np.float64)
    h = np.asarray(h, dtype=np.float64)
    l = np.asarray(l, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    m, n, r = h.size, g.size, l.size
    S_U = expand_bits(bits_u, m, r)
    S_V = expand_bits(bits_v, n, r)
    a = (x * g[None, :]) @ S_V            # a[t,k] = sum_j x[t,j] g[j] S_V[j,k]
    c = (a * l[None, :]) @ S_U.T          # c[t,i] = sum_k a[t,k] l[k] S_U[i,k]
    y = c * h[None, :]                    # y[t,i] = h[i] c[t,i]
    return y, a, c


def backward(bits_u, bits_v, h, l, g, x, dy):
    """Return ``(dx, dh, dl, dg, b, dxp)``; dh/dl/dg are the increments."""
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    h = np.asarray(h, dtype=np.float64)
    l = np.asarray(l, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    m, n, r = h.size, g.size, l.size
    S_U = expand_bits(bits_u, m, r)
    S_V = expand_bits(bits_v, n, r)
    _, a, c = forward(bits_u, bits_v, h, l, g, x)
    dh = np.sum(dy * c, axis=0)                    # dh[i] = sum_t dy[t,i] c[t,i]
    b = (dy * h[None, :]) @ S_U                    # b[t,k] = sum_i dy[t,i] h[i] S_U[i,k]
    dl = np.sum(a * b, axis=0)                     # dl[k] = sum_t a[t,k] b[t,k]
    dxp = (b * l[None, :]) @ S_V.T                 # dx'[t,j] = sum_k b[t,k] l[k] S_V[j,k]
    dg = np.sum(x * dxp, axis=0)                   # dg[j] = sum_t x[t,j] dx'[t,j]
    dx = dxp * g[None, :]                          # dx[t,j] = g[j] dx'[t,j]
    return dx, dh, dl, dg, b, dxp


def abs_chain(h, l, g, x, dy):
    """Magnitude scales for per-element error bounds.

    The same expressions with every factor replaced by its absolute value and
    every sign by 1; each bounds ``sum |term|`` of the matching output.
    Returns ``(ya, aa, dxa, ba, dha, dla, dga)``.
    """
    x = np.abs(np.asarray(x, dtype=np.float64))
    dy = np.abs(np.asarray(dy, dtype=np.float64))
    h = np.abs(np.asarray(h, dtype=np.float64))
    l = np.abs(np.asarray(l, dtype=np.float64))
    g = np.abs(np.asarray(g, dtype=np.float64))
    xg = (x * g[None, :]).sum(axis=1, keepdims=True)          # sum_j |x g|
    aa = np.repeat(xg, l.size, axis=1)                        # |a| <= this
    ca = np.repeat(aa[:, :1] * l.sum(), h.size, axis=1)       # |c| <= this
    ya = ca * h[None, :]
    dyh = (dy * h[None, :]).sum(axis=1, keepdims=True)
    ba = np.repeat(dyh, l.size, axis=1)
    dxpa = np.repeat(ba[:, :1] * l.sum(), g.size, axis=1)
    dxa = dxpa * g[None, :]
    dha = (dy * ca).sum(axis=0)
    dla = (aa * ba).sum(axis=0)
    dga = (x * dxpa).sum(axis=0)
    return ya, aa, dxa, ba, dha, dla, dga


def forward_paths(paths, x):
    """Several paths of one layer ("cortiq-engine 0.8.43, train_mm.rs",
    ``blr_forward`` over ``layer.paths``): ``y = sum_p h_p . c_p``.

    ``paths`` is a list of dicts with ``bits_u, bits_v, h, l, g``.  Exact in
    f64 (the sum's order does not matter here); returns ``(y, [(a_p, c_p)])``.
    """
    y = None
    saved = []
    for p in paths:
        yp, a, c = forward(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], x)
        y = yp if y is None else y + yp
        saved.append((a, c))
    return y, saved


def backward_paths(paths, x, dy):
    """Backward of :func:`forward_paths` (``blr_backward`` over the paths):
    ``dx = sum_p g_p . dx'_p``; each path's ``(dh, dl, dg)`` increments are
    those of its own single-path backward with the shared ``dy``."""
    dx = None
    grads = []
    for p in paths:
        dxp, dh, dl, dg, _, _ = backward(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], x, dy)
        dx = dxp if dx is None else dx + dxp
        grads.append((dh, dl, dg))
    return dx, grads


def sign_grads(bits_u, bits_v, h, l, g, x, dy):
    """Gradients of ``L`` with respect to one path's signs ("cortiq-engine
    0.8.43, train_mm.rs", ``blr_backward`` with sign training):
    ``G_U = diag(h) dy^T a diag(l)`` and ``G_V = diag(g) x^T b diag(l)`` with
    ``a = (x.g) S_V`` and ``b = (dy.h) S_U``.  Returns ``(G_U, G_V)``,
    ``[d_out][r]`` and ``[d_in][r]``."""
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    h = np.asarray(h, dtype=np.float64)
    l = np.asarray(l, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    _, a, _ = forward(bits_u, bits_v, h, l, g, x)
    S_U = expand_bits(bits_u, h.size, l.size)
    b = (dy * h[None, :]) @ S_U
    G_U = h[:, None] * (dy.T @ a) * l[None, :]
    G_V = g[:, None] * (x.T @ b) * l[None, :]
    return G_U, G_V
