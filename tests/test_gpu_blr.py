"""GPU parity of the blr layer (bitmap expansion, forward, backward) through
the C ABI against the f64 oracle.

Bounds ("cortiq-engine 0.8.43, train_mm.rs", test blr_layer_matches_host):
relative L2 error < 3e-3 per tensor (the page's
bound) and, per element, |gpu - oracle| <= 2^-9 * (the absolute-value chain
of the same expression).  Each output passes through at most two f16
roundings (2 * 2^-11) plus f32 accumulation over at most 4096 + 512 terms.
"""
import numpy as np
import pytest

import synth
from gpu_util import to_dev
from oracle import blr as oblr

pytestmark = pytest.mark.gpu

TOL = 2.0 ** -9


def _page_inputs(T=70, d_in=384, d_out=256, r=128, pi=0):
    """The page's blr test data: rnd-based signs, h in [0.02,0.045], l in [0.5,1],
    g in [0.1,0.2], x scale 2, dy scale 1e-3."""
    def signs(rows, seed):
        return np.where(synth.xorshift_uniform(rows * r, seed, 1.0).reshape(rows, r) >= 0, 1.0, -1.0)

    def pack(S):
        rows = S.shape[0]
        b = np.zeros((rows, r // 32), dtype=np.uint32)
        for k in range(r):
            b[:, k // 32] |= np.where(S[:, k] > 0, np.uint32(1 << (k % 32)), np.uint32(0))
        return b
    su, sv = signs(d_out, 10 + pi), signs(d_in, 20 + pi)
    return dict(
        bits_u=pack(su), bits_v=pack(sv),
        h=(0.02 + np.abs(synth.xorshift_uniform(d_out, 30 + pi, 0.5)) * 0.05).astype(np.float32),
        l=(0.5 + np.abs(synth.xorshift_uniform(r, 40 + pi, 0.5))).astype(np.float32),
        g=(0.1 + np.abs(synth.xorshift_uniform(d_in, 50 + pi, 0.5)) * 0.2).astype(np.float32),
        x=synth.xorshift_uniform(T * d_in, 60, 2.0).reshape(T, d_in),
        dy=synth.xorshift_uniform(T * d_out, 61, 1e-3).reshape(T, d_out),
    )


def _run(lib, p, gscale=1.0, save_c=True):
    import torch
    T, d_in = p["x"].shape
    d_out, r = p["h"].size, p["l"].size
    d = {k: to_dev(v) for k, v in p.items()}
    d["bits_u"] = to_dev(p["bits_u"].view(np.int32))
    d["bits_v"] = to_dev(p["bits_v"].view(np.int32))
    f = dict(dtype=torch.float32, device="cuda")
    y = torch.full((T, d_out), float("nan"), **f)
    a = torch.full((T, r), float("nan"), **f)
    c = torch.full((T, d_out), float("nan"), **f) if save_c else None
    lib.blr_forward(d["bits_u"], d["bits_v"], d["h"], d["l"], d["g"], d["x"], y, a, c)
    dx = torch.full((T, d_in), float("nan"), **f)
    dh, dl, dg = torch.zeros(d_out, **f), torch.zeros(r, **f), torch.zeros(d_in, **f)
    lib.blr_backward(d["bits_u"], d["bits_v"], d["h"], d["l"], d["g"], d["x"], d["dy"], a, c, dx, dh, dl, dg,
                     gscale=gscale)
    lib.device_status()
    out = dict(y=y, a=a, dx=dx, dh=dh, dl=dl, dg=dg)
    if save_c:
        out["c"] = c
    return {k: v.cpu().numpy().astype(np.float64) for k, v in out.items()}


def _oracle(p):
    y, a, c = oblr.forward(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], p["x"])
    dx, dh, dl, dg, _, _ = oblr.backward(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], p["x"], p["dy"])
    ya, aa, dxa, _, dha, dla, dga = oblr.abs_chain(p["h"], p["l"], p["g"], p["x"], p["dy"])
    ca = ya / np.asarray(p["h"], dtype=np.float64)[None, :]
    return (dict(y=y, a=a, c=c, dx=dx, dh=dh, dl=dl, dg=dg),
            dict(y=ya, a=aa, c=ca, dx=dxa, dh=dha, dl=dla, dg=dga))


def _check(got, want, chain, where):
    for k, g in got.items():
        w, ch = want[k], chain[k]
        assert np.all(np.isfinite(g)), f"{where} {k}: not finite"
        rel = np.sqrt(np.sum((g - w) ** 2) / max(np.sum(w * w), 1e-300))
        assert rel < 3e-3, f"{where} {k}: relative L2 error {rel:.3e}"
        bad = np.abs(g - w) > TOL * ch + 1e-30
        assert not bad.any(), f"{where} {k}: {bad.sum()} elements above 2^-9 of the abs chain"


def test_expand_bits_bit_exact(lib):
    import torch
    for rows, r, key in ((256, 128, 1), (40, 96, 2), (3, 32, 3)):
        bits = synth.sign_bits(rows, r, key)
        want = oblr.expand_bits(bits, rows, r).astype(np.float16).view(np.uint16)
        db = to_dev(bits.view(np.int32))
        for tr in (0, 1):
            plane = torch.zeros((r, rows) if tr else (rows, r), dtype=torch.int16, device="cuda")
            lib.blr_expand_bits(db, rows, r, plane, tr)
            lib.device_status()
            got = plane.cpu().numpy().view(np.uint16)
            assert np.array_equal(got, want.T if tr else want), (rows, r, tr)


@pytest.mark.parametrize("gscale", [1.0, 1024.0])
@pytest.mark.parametrize("save_c", [True, False])
def test_blr_page_shape(lib, gscale, save_c):
    p = _page_inputs()
    got = _run(lib, p, gscale=gscale, save_c=save_c)
    want, chain = _oracle(p)
    _check(got, want, chain, f"page shape gs={gscale} save_c={save_c}")


@pytest.mark.parametrize("T,d_in,d_out,r", [(1, 64, 64, 128), (33, 192, 320, 256), (300, 512, 448, 384)])
def test_blr_ragged_shapes(lib, T, d_in, d_out, r):
    p = synth.blr_inputs(T, d_in, d_out, r, 200 + T)
    got = _run(lib, p, save_c=(T % 2 == 1))
    want, chain = _oracle(p)
    _check(got, want, chain, f"T={T} d_in={d_in} d_out={d_out} r={r}")


def test_blr_full_size(lib):
    cfg = synth.BLR
    p = synth.blr_inputs(cfg["T"], cfg["d_in"], cfg["d_out"], cfg["r"], cfg["key"])
    got = _run(lib, p, save_c=False)
    want, chain = _oracle(p)
    _check(got, want, chain, "T=2048 d=4096 r=512")


def test_blr_deterministic_and_accumulating(lib):
    p = synth.blr_inputs(130, 256, 192, 128, 300)
    r1 = _run(lib, p, save_c=False)
    r2 = _run(lib, p, save_c=False)
    for k in r1:
        assert np.array_equal(r1[k], r2[k]), k
    # dh/dl/dg accumulate: a second backward on the same buffers doubles them
    import torch
    T, d_in = p["x"].shape
    d_out, r = p["h"].size, p["l"].size
    d = {k: to_dev(v) for k, v in p.items() if k not in ("bits_u", "bits_v")}
    bu, bv = to_dev(p["bits_u"].view(np.int32)), to_dev(p["bits_v"].view(np.int32))
    f = dict(dtype=torch.float32, device="cuda")
    y, a = torch.empty((T, d_out), **f), torch.empty((T, r), **f)
    lib.blr_forward(bu, bv, d["h"], d["l"], d["g"], d["x"], y, a, None)
    dx = torch.empty((T, d_in), **f)
    dh, dl, dg = torch.zeros(d_out, **f), torch.zeros(r, **f), torch.zeros(d_in, **f)
    for _ in range(2):
        lib.blr_backward(bu, bv, d["h"], d["l"], d["g"], d["x"], d["dy"], a, None, dx, dh, dl, dg)
    lib.device_status()
    for k, v in (("dh", dh), ("dl", dl), ("dg", dg)):
        assert np.array_equal(v.cpu().numpy(), 2 * r1[k].astype(np.float32)), k


def test_blr_rejects_bad_arguments(lib):
    import ctypes
    import torch
    L = lib.load()
    z = torch.zeros(4096, dtype=torch.float32, device="cuda")
    pz = ctypes.c_void_p(z.data_ptr())
    # shapes: d_in not a multiple of 64, r not a multiple of 128
    assert L.blr_forward(pz, pz, pz, pz, pz, pz, pz, pz, None, 4, 96, 64, 128, None) == 2
    assert L.blr_forward(pz, pz, pz, pz, pz, pz, pz, pz, None, 4, 64, 64, 96, None) == 2
    assert L.blr_forward(None, pz, pz, pz, pz, pz, pz, pz, None, 4, 64, 64, 128, None) == 1
    # gscale must be a positive power of two
    for gs in (3.0, 0.0, -2.0):
        assert L.blr_backward(pz, pz, pz, pz, pz, pz, pz, pz, None, pz, pz, pz, pz, 4, 64, 64, 128, gs, None) == 1


# ---- several paths of one layer (blr_forward_paths / blr_backward_paths)

def _dev_path(p, T, d_out, r, d_in):
    import torch
    f = dict(dtype=torch.float32, device="cuda")
    return dict(bits_u=to_dev(p["bits_u"].view(np.int32)), bits_v=to_dev(p["bits_v"].view(np.int32)),
                h=to_dev(p["h"]), l=to_dev(p["l"]), g=to_dev(p["g"]),
                a_save=torch.full((T, r), float("nan"), **f), c_save=torch.full((T, d_out), float("nan"), **f),
                dh=torch.zeros(d_out, **f), dl=torch.zeros(r, **f), dg=torch.zeros(d_in, **f))


def _run_paths(lib, ps, gscale=1.0):
    import torch
    T, d_in = ps[0]["x"].shape
    d_out, r = ps[0]["h"].size, ps[0]["l"].size
    dps = [_dev_path(p, T, d_out, r, d_in) for p in ps]
    x, dy = to_dev(ps[0]["x"]), to_dev(ps[0]["dy"])
    y = torch.full((T, d_out), float("nan"), dtype=torch.float32, device="cuda")
    dx = torch.full((T, d_in), float("nan"), dtype=torch.float32, device="cuda")
    lib.blr_forward_paths(dps, x, y)
    lib.blr_backward_paths(dps, x, dy, dx, gscale=gscale)
    lib.device_status()
    n = lambda t: t.cpu().numpy().astype(np.float64)
    return n(y), n(dx), [(n(d["dh"]), n(d["dl"]), n(d["dg"])) for d in dps], (y, dx)


@pytest.mark.parametrize("P", [2, 3])
def test_paths_against_oracle(lib, P):
    ps = [_page_inputs(pi=i) for i in range(P)]
    y, dx, grads, _ = _run_paths(lib, ps, gscale=1024.0)
    want_y, _ = oblr.forward_paths(ps, ps[0]["x"])
    want_dx, want_grads = oblr.backward_paths(ps, ps[0]["x"], ps[0]["dy"])
    chains = [oblr.abs_chain(p["h"], p["l"], p["g"], p["x"], p["dy"]) for p in ps]
    ya, dxa = sum(c[0] for c in chains), sum(c[2] for c in chains)
    _check(dict(y=y, dx=dx), dict(y=want_y, dx=want_dx), dict(y=ya, dx=dxa), f"{P} paths")
    for i, (got, want, c) in enumerate(zip(grads, want_grads, chains)):
        _check(dict(dh=got[0], dl=got[1], dg=got[2]), dict(dh=want[0], dl=want[1], dg=want[2]),
               dict(dh=c[4], dl=c[5], dg=c[6]), f"{P} paths, path {i}")


def test_paths_combine_rounds_as_the_page(lib):
    """y = fl(fl(y0 + y1) + y2) and dx likewise, from the single-path results:
    each product and each sum rounded to f32 separately (the page's scale_acc
    passes; for two paths its one-pass scale_acc2)."""
    ps = [_page_inputs(pi=i) for i in range(3)]
    singles = [_run(lib, p) for p in ps]
    import torch
    for P in (2, 3):
        _, _, _, (y, dx) = _run_paths(lib, ps[:P])
        want_y, want_dx = np.float32(singles[0]["y"]), np.float32(singles[0]["dx"])
        for s in singles[1:P]:
            want_y = (want_y + np.float32(s["y"])).astype(np.float32)
            want_dx = (want_dx + np.float32(s["dx"])).astype(np.float32)
        assert np.array_equal(y.cpu().numpy().view(np.uint32), want_y.view(np.uint32)), P
        assert np.array_equal(dx.cpu().numpy().view(np.uint32), want_dx.view(np.uint32)), P


def test_paths_one_path_is_the_single_call(lib):
    p = _page_inputs()
    single = _run(lib, p)
    y, dx, grads, _ = _run_paths(lib, [p])
    assert np.array_equal(y, single["y"]) and np.array_equal(dx, single["dx"])
    assert np.array_equal(grads[0][0], single["dh"]) and np.array_equal(grads[0][1], single["dl"])
    assert np.array_equal(grads[0][2], single["dg"])


# ---- sign gradients (blr_sign_grads) against the oracle

SIGN_TOL = 2.0 ** -8      # a (or b) and two staged operands: three f16 roundings per product chain


@pytest.mark.parametrize("shape", [(70, 384, 256, 128), (33, 192, 320, 256), (2048, 4096, 4096, 512)],
                         ids=["page", "ragged", "C5"])
def test_sign_grads_against_oracle(lib, shape):
    import torch
    T, d_in, d_out, r = shape
    p = _page_inputs(T, d_in, d_out, r) if T == 70 else synth.blr_inputs(T, d_in, d_out, r, 900 + T)
    d = {k: to_dev(v) for k, v in p.items() if k not in ("bits_u", "bits_v")}
    bu, bv = to_dev(p["bits_u"].view(np.int32)), to_dev(p["bits_v"].view(np.int32))
    f = dict(dtype=torch.float32, device="cuda")
    y, a = torch.empty((T, d_out), **f), torch.empty((T, r), **f)
    lib.blr_forward(bu, bv, d["h"], d["l"], d["g"], d["x"], y, a)
    gu = torch.full((d_out, r), float("nan"), **f)
    gv = torch.full((d_in, r), float("nan"), **f)
    # the page's gradient scale with its 1e-3-sized dy; 1 for unit-sized dy, where
    # b.l.gs would leave the f16 range at 1024
    gs = 1024.0 if T == 70 else 1.0
    lib.blr_sign_grads(bu, d["h"], d["l"], d["g"], d["x"], d["dy"], a, gu, gv, gscale=gs)
    lib.device_status()
    GU, GV = oblr.sign_grads(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], p["x"], p["dy"])
    _, aa, _, ba, _, _, _ = oblr.abs_chain(p["h"], p["l"], p["g"], p["x"], p["dy"])
    h, l, g = (np.abs(np.asarray(p[k], dtype=np.float64)) for k in ("h", "l", "g"))
    cu = h[:, None] * (np.abs(np.asarray(p["dy"], dtype=np.float64)).T @ aa) * l[None, :]
    cv = g[:, None] * (np.abs(np.asarray(p["x"], dtype=np.float64)).T @ ba) * l[None, :]
    for name, got, want, chain in (("G_U", gu, GU, cu), ("G_V", gv, GV, cv)):
        got = got.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), name
        rel = np.sqrt(np.sum((got - want) ** 2) / max(np.sum(want * want), 1e-300))
        assert rel < 3e-3, f"{shape} {name}: relative L2 error {rel:.3e}"
        bad = np.abs(got - want) > SIGN_TOL * chain + 1e-30
        assert not bad.any(), f"{shape} {name}: {bad.sum()} elements above 2^-8 of the abs chain"
