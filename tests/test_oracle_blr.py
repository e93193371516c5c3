"""Pins of the blr oracle (CPU only): bit positions, closed forms, brute
force, finite differences and the sign-flip identity of
"cortiq-engine 0.8.43, train_mm.rs" (test ``blr_sign_flip_exact``)."""
import itertools

import numpy as np

import synth
from oracle import blr


def _bits_from_signs(S):
    rows, r = S.shape
    w = (r + 31) // 32
    b = np.zeros((rows, w), dtype=np.uint32)
    for i in range(rows):
        for k in range(r):
            if S[i, k] > 0:
                b[i, k // 32] |= np.uint32(1 << (k % 32))
    return b


def test_expand_single_bits():
    rows, r = 3, 128
    for k in (0, 31, 32, 63, 64, 95, 96, 127):
        bits = np.zeros((rows, r // 32), dtype=np.uint32)
        bits[1, k // 32] = np.uint32(1 << (k % 32))
        S = blr.expand_bits(bits, rows, r)
        want = -np.ones((rows, r))
        want[1, k] = 1.0
        assert np.array_equal(S, want), k


def test_expand_roundtrip_random():
    rows, r = 17, 96
    S = np.where(synth.uniform(rows * r, 5, -1, 1).reshape(rows, r) >= 0, 1.0, -1.0)
    assert np.array_equal(blr.expand_bits(_bits_from_signs(S), rows, r), S)


def test_all_plus_closed_form():
    T, n, m, r = 4, 6, 5, 64
    h = synth.uniform(m, 1, 0.5, 1.5).astype(np.float64)
    l = synth.uniform(r, 2, 0.5, 1.5).astype(np.float64)
    g = synth.uniform(n, 3, 0.5, 1.5).astype(np.float64)
    x = synth.random_x(T, n, 4).astype(np.float64)
    ones_u = np.full((m, r // 32), 0xFFFFFFFF, dtype=np.uint32)
    ones_v = np.full((n, r // 32), 0xFFFFFFFF, dtype=np.uint32)
    y, a, c = blr.forward(ones_u, ones_v, h, l, g, x)
    xg = (x * g).sum(axis=1)
    np.testing.assert_allclose(a, np.repeat(xg[:, None], r, axis=1), rtol=1e-13)
    np.testing.assert_allclose(y, h[None, :] * l.sum() * xg[:, None], rtol=1e-13)


def test_brute_force_forward_tiny():
    # explicit sums over every index, no matrix routine
    T, n, m, r = 2, 3, 4, 32
    rng = synth.uniform(1000, 6, -1, 1).astype(np.float64)
    SU = np.where(rng[: m * r].reshape(m, r) > 0, 1.0, -1.0)
    SV = np.where(rng[m * r: m * r + n * r].reshape(n, r) > 0, 1.0, -1.0)
    h, l, g = rng[300:300 + m], rng[400:400 + r], rng[500:500 + n]
    x = rng[600:600 + T * n].reshape(T, n)
    y, _, _ = blr.forward(_bits_from_signs(SU), _bits_from_signs(SV), h, l, g, x)
    for t, i in itertools.product(range(T), range(m)):
        v = 0.0
        for k in range(r):
            for j in range(n):
                v += h[i] * SU[i, k] * l[k] * SV[j, k] * g[j] * x[t, j]
        assert abs(v - y[t, i]) < 1e-12


def test_backward_matches_finite_differences():
    # L = sum(y * dy) is bilinear in each parameter, so central differences are exact
    T, n, m, r = 3, 5, 4, 40
    p = synth.blr_inputs(T, n, m, r, 70)
    h, l, g = (p[k].astype(np.float64) for k in ("h", "l", "g"))
    x, dy = p["x"].astype(np.float64), p["dy"].astype(np.float64)
    bu, bv = p["bits_u"], p["bits_v"]

    def L(h_, l_, g_, x_):
        return float(np.sum(blr.forward(bu, bv, h_, l_, g_, x_)[0] * dy))

    dx, dh, dl, dg, _, _ = blr.backward(bu, bv, h, l, g, x, dy)
    eps = 0.5
    for name, vec, grad in (("h", h, dh), ("l", l, dl), ("g", g, dg), ("x", x, dx)):
        flat = vec.reshape(-1)
        for i in range(flat.size):
            args = {"h": h, "l": l, "g": g, "x": x}
            up, dn = flat.copy(), flat.copy()
            up[i] += eps
            dn[i] -= eps
            args[name] = up.reshape(vec.shape)
            lu = L(**{k + "_": v for k, v in args.items()})
            args[name] = dn.reshape(vec.shape)
            ld = L(**{k + "_": v for k, v in args.items()})
            fd = (lu - ld) / (2 * eps)
            assert abs(fd - grad.reshape(-1)[i]) <= 1e-9 * (1 + abs(fd)), (name, i)


def test_sign_flip_identity():
    # L = 1/2 |y - y*|^2; flipping U[i,k] changes L by exactly
    # -2 s G_U + 2 h_i^2 l_k^2 sum_t a_tk^2, with G_U = h_i l_k sum_t dy_ti a_tk,
    # and V[j,k] by -2 s G_V + 2 g_j^2 l_k^2 (sum_t x_tj^2)(sum_i h_i^2),
    # with G_V = g_j l_k sum_t x_tj b_tk
    T, n, m, r = 6, 7, 5, 96
    p = synth.blr_inputs(T, n, m, r, 90)
    h, l, g = (p[k].astype(np.float64) for k in ("h", "l", "g"))
    x = p["x"].astype(np.float64)
    bu, bv = p["bits_u"].copy(), p["bits_v"].copy()
    y0, a, _ = blr.forward(bu, bv, h, l, g, x)
    ystar = y0 + synth.random_x(T, m, 91).astype(np.float64)
    dy = y0 - ystar
    L0 = 0.5 * np.sum((y0 - ystar) ** 2)
    _, _, _, _, b, _ = blr.backward(bu, bv, h, l, g, x, dy)
    SU = blr.expand_bits(bu, m, r)
    SV = blr.expand_bits(bv, n, r)
    for (i, k) in [(0, 0), (1, 31), (2, 32), (4, 63), (3, 64), (0, 95)]:
        GU = h[i] * l[k] * np.sum(dy[:, i] * a[:, k])
        pred = -2 * SU[i, k] * GU + 2 * h[i] ** 2 * l[k] ** 2 * np.sum(a[:, k] ** 2)
        fl = bu.copy()
        fl[i, k // 32] ^= np.uint32(1 << (k % 32))
        L1 = 0.5 * np.sum((blr.forward(fl, bv, h, l, g, x)[0] - ystar) ** 2)
        assert abs((L1 - L0) - pred) <= 1e-9 * (2 * abs(GU) + abs(pred) + 1)
    for (j, k) in [(0, 0), (6, 31), (2, 32), (5, 95)]:
        GV = g[j] * l[k] * np.sum(x[:, j] * b[:, k])
        pred = -2 * SV[j, k] * GV + 2 * g[j] ** 2 * l[k] ** 2 * np.sum(x[:, j] ** 2) * np.sum(h ** 2)
        fl = bv.copy()
        fl[j, k // 32] ^= np.uint32(1 << (k % 32))
        L1 = 0.5 * np.sum((blr.forward(bu, fl, h, l, g, x)[0] - ystar) ** 2)
        assert abs((L1 - L0) - pred) <= 1e-9 * (2 * abs(GV) + abs(pred) + 1)


def test_abs_chain_bounds_terms():
    T, n, m, r = 3, 6, 5, 64
    p = synth.blr_inputs(T, n, m, r, 95)
    ya, aa, dxa, ba, dha, dla, dga = blr.abs_chain(p["h"], p["l"], p["g"], p["x"], p["dy"])
    y, a, c = blr.forward(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], p["x"])
    dx, dh, dl, dg, b, _ = blr.backward(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], p["x"], p["dy"])
    for v, bound in ((y, ya), (a, aa), (dx, dxa), (b, ba), (dh, dha), (dl, dla), (dg, dga)):
        assert np.all(np.abs(v) <= bound * (1 + 1e-12))


# ---- several paths of one layer (blr_forward / blr_backward over layer.paths)

def _paths(P, key, T=5, d_in=64, d_out=64, r=128):
    ps = [synth.blr_inputs(T, d_in, d_out, r, key + 10 * i) for i in range(P)]
    return ps, ps[0]["x"], ps[0]["dy"]


def test_paths_single_equals_one_path():
    ps, x, dy = _paths(1, 700)
    y, saved = blr.forward_paths(ps, x)
    y1, a1, c1 = blr.forward(ps[0]["bits_u"], ps[0]["bits_v"], ps[0]["h"], ps[0]["l"], ps[0]["g"], x)
    assert np.array_equal(y, y1) and np.array_equal(saved[0][0], a1) and np.array_equal(saved[0][1], c1)
    dx, grads = blr.backward_paths(ps, x, dy)
    dx1, dh1, dl1, dg1, _, _ = blr.backward(ps[0]["bits_u"], ps[0]["bits_v"], ps[0]["h"], ps[0]["l"], ps[0]["g"], x, dy)
    assert np.array_equal(dx, dx1)
    assert all(np.array_equal(u, v) for u, v in zip(grads[0], (dh1, dl1, dg1)))


def test_paths_identical_double_and_negated_h_cancels():
    ps, x, dy = _paths(1, 710)
    p = ps[0]
    y2, _ = blr.forward_paths([p, p], x)
    y1, _, _ = blr.forward(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], x)
    assert np.array_equal(y2, 2.0 * y1)                       # exact: doubling in f64
    neg = dict(p, h=-np.asarray(p["h"]))
    y0, _ = blr.forward_paths([p, neg], x)
    assert np.array_equal(y0, np.zeros_like(y0))
    dx0, _ = blr.backward_paths([p, neg], x, dy)             # L = sum y.dy vanishes identically
    assert np.array_equal(dx0, np.zeros_like(dx0))


def test_paths_gradients_are_per_path_and_dx_sums():
    ps, x, dy = _paths(3, 720)
    dx, grads = blr.backward_paths(ps, x, dy)
    total = 0.0
    for p, (dh, dl, dg) in zip(ps, grads):
        dxp, dhp, dlp, dgp, _, _ = blr.backward(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], x, dy)
        assert np.array_equal(dh, dhp) and np.array_equal(dl, dlp) and np.array_equal(dg, dgp)
        total = total + dxp
    assert np.allclose(dx, total, rtol=0, atol=1e-12 * np.abs(total).max())
    # the layer's loss L = sum(y.dy) has dL/dx = dx: check one entry by a central difference
    x = np.asarray(x, dtype=np.float64)                      # steps exact in f64 (the layer is linear in x)
    e = np.zeros_like(x); e[2, 7] = 1e-3
    yp, _ = blr.forward_paths(ps, x + e)
    ym, _ = blr.forward_paths(ps, x - e)
    fd = (np.sum(yp * dy) - np.sum(ym * dy)) / 2e-3
    assert abs(fd - dx[2, 7]) <= 1e-9 * max(1.0, abs(fd))


# ---- sign gradients, pinned by the page's flip identity (test blr_sign_flip_exact)

def test_sign_gradients_flip_identity():
    """L = 1/2 |y - y*|^2 is quadratic in each sign, so flipping sign s of
    U[i,k] changes it by exactly -2 s G_U[i,k] + 2 h_i^2 l_k^2 sum_t a_tk^2,
    and of V[j,k] by -2 s G_V[j,k] + 2 g_j^2 l_k^2 (sum_t x_tj^2)(sum_i h_i^2).
    Each flip reruns the forward with the bit changed (this also checks the
    bit mapping)."""
    p = synth.blr_inputs(9, 64, 128, 128, 801)
    x = np.asarray(p["x"], dtype=np.float64)
    y0, a, _ = blr.forward(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], x)
    ystar = y0 + 0.7 * np.asarray(synth.normal(y0.size, 802), dtype=np.float64).reshape(y0.shape)
    dy = y0 - ystar
    L0 = 0.5 * np.sum((y0 - ystar) ** 2)
    GU, GV = blr.sign_grads(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], x, dy)
    h, l, g = (np.asarray(p[k], dtype=np.float64) for k in ("h", "l", "g"))
    SU = blr.expand_bits(p["bits_u"], h.size, l.size)
    SV = blr.expand_bits(p["bits_v"], g.size, l.size)
    for (i, k) in ((0, 0), (1, 31), (2, 32), (127, 127), (17, 63), (100, 64)):
        for side in ("U", "V"):
            bits = np.array(p["bits_u" if side == "U" else "bits_v"], dtype=np.uint32).copy()
            row = i % (h.size if side == "U" else g.size)
            bits[row, k // 32] ^= np.uint32(1 << (k % 32))
            bu, bv = (bits, p["bits_v"]) if side == "U" else (p["bits_u"], bits)
            y1, _, _ = blr.forward(bu, bv, h, l, g, x)
            dL = 0.5 * np.sum((y1 - ystar) ** 2) - L0
            if side == "U":
                s, G = SU[row, k], GU[row, k]
                quad = 2 * h[row] ** 2 * l[k] ** 2 * np.sum(a[:, k] ** 2)
            else:
                s, G = SV[row, k], GV[row, k]
                quad = 2 * g[row] ** 2 * l[k] ** 2 * np.sum(x[:, row] ** 2) * np.sum(h ** 2)
            pred = -2 * s * G + quad
            assert abs(dL - pred) <= 1e-9 * (2 * abs(G) + quad), (side, row, k, dL, pred)
