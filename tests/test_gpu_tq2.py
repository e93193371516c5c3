"""GPU parity of the TQ2 path through the C ABI against the f64 oracle.

Upload / unpack and the f16 dequantization are bit-exact; GEMM outputs are
held to the bounds stated in ``gpu_util`` (the pages' 1e-3 for the skinny
f32-activation kernel, 1e-2 * sum|x W| for the f16-staged tensor path, plus
tighter accumulation-only bounds).
"""
import numpy as np
import pytest

import synth
from gpu_util import (check_skinny, check_tensor, oracle_gemm, page_sweep_weight, page_sweep_x, run_gemm,
                      to_dev)
from oracle import tq2 as otq2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny(lib):
    aos, N, K, xs = synth.tiny_tq2()
    return aos, N, K, xs, lib.tq2_upload(aos, N, K)


# ---------------------------------------------------------------- format ----
def test_upload_unpack_roundtrip(lib):
    for N, K, key in ((40, 256, 1), (37, 384, 2), (3, 128, 3)):
        aos = bytearray(synth.random_tq2(N, K, key))
        aos[5] = 0xFF                     # a byte of code 3s survives too
        w = lib.tq2_upload(bytes(aos), N, K)
        assert lib.tq2_unpack(w) == bytes(aos)


def test_dequant_f16_bit_exact(lib):
    import torch
    for N, K, key in ((40, 256, 4), (33, 640, 5)):
        aos = bytearray(synth.random_tq2(N, K, key))
        aos[7] = 0xFF                     # include code 3 -> +2d
        w = lib.tq2_upload(bytes(aos), N, K)
        out = torch.zeros((N, K), dtype=torch.int16, device="cuda")
        lib.tq2_dequant_f16(w, out)
        lib.device_status()
        got = out.cpu().numpy().view(np.uint16)
        codes, d_bits = otq2.parse_aos(bytes(aos), N, K)
        assert np.array_equal(got, otq2.dequant_f16_bits(codes, d_bits))


# ---------------------------------------------------------------- skinny ----
@pytest.mark.parametrize("M", [1, 7, 8, 9])
def test_tiny_skinny_matches_oracle(tiny, lib, M):
    aos, N, K, xs, w = tiny
    got = run_gemm(lib, w, xs[M])
    ref, absref, _, _ = oracle_gemm(aos, N, K, xs[M])
    check_skinny(got, ref, absref, f"tiny M={M}")
    assert np.any(np.abs(got) > 1e-6)


def test_tiny_skinny_page_activations(tiny, lib):
    aos, N, K, _, w = tiny
    for M in (1, 2, 3, 7, 8, 9, 16):
        x = synth.page_x(M, K)
        got = run_gemm(lib, w, x)
        ref, absref, _, _ = oracle_gemm(aos, N, K, x)
        check_skinny(got, ref, absref, f"page x M={M}")


@pytest.mark.parametrize("N,K", [(8, 128), (40, 256), (3072, 3072), (17, 1152), (33, 2176)])
def test_skinny_page_sweep(lib, N, K):
    aos = page_sweep_weight(N, K)
    w = lib.tq2_upload(aos, N, K)
    for M in (1, 2, 3, 7, 8, 9, 12, 16):
        x = page_sweep_x(M, K)
        got = run_gemm(lib, w, x, lib.PATH_SKINNY)
        ref, absref, _, _ = oracle_gemm(aos, N, K, x)
        check_skinny(got, ref, absref, f"sweep N={N} K={K} M={M}")


def test_gemv_tokens_full_size(lib):
    """The fused GEMV at the decode-shape weight for every token count it
    takes (M = 3 and 5..7 padded to four and eight tokens)."""
    cfg = synth.GEMV
    N, K = cfg["N"], cfg["K"]
    aos = synth.random_tq2(N, K, cfg["wkey"])
    w = lib.tq2_upload(aos, N, K)
    for M in (2, 3, 4, 5, 6, 7, 8):
        x = synth.random_x(M, K, cfg["xkey"] + M)
        got = run_gemm(lib, w, x)
        ref, absref, _, _ = oracle_gemm(aos, N, K, x)
        check_skinny(got, ref, absref, f"gemv M={M}")


def test_gemv_large_k_chunks(lib):
    # K = 16384 (M <= 2) and 8192 (M <= 4): each warp walks several 4-block chunks
    for N, K, Ms in ((300, 16384, (1, 2)), (300, 8192, (3, 4))):
        aos = synth.random_tq2(N, K, 90)
        w = lib.tq2_upload(aos, N, K)
        for M in Ms:
            x = synth.random_x(M, K, 91) * 0.5
            got = run_gemm(lib, w, x)
            ref, absref, _, _ = oracle_gemm(aos, N, K, x)
            assert np.max(np.abs(got - ref)) <= 2e-3, (M, np.max(np.abs(got - ref)))
            assert np.all(np.abs(got - ref) <= (2.0 ** -10) * absref + 1e-7), M


def test_gemv_grouped_matches_single_calls(lib):
    import torch
    K = 2048
    shapes = [(4096, 11), (40, 12), (17, 13), (1000, 14)]
    ws, auos = [], []
    for N, key in shapes:
        a = synth.random_tq2(N, K, key)
        auos.append(a)
        ws.append(lib.tq2_upload(a, N, K))
    for M in (1, 2, 3, 8):
        xs = [to_dev(synth.random_x(M, K, 50 + g)) for g in range(len(ws))]
        outs = [torch.full((M, w.N), float("nan"), device="cuda") for w in ws]
        lib.tq2_gemm_grouped(ws, xs, outs)
        lib.device_status()
        # the same group with its arguments marshalled once, called twice
        outs2 = [torch.full((M, w.N), float("nan"), device="cuda") for w in ws]
        grp = lib.GroupedGemv(ws, xs, outs2)
        for _ in range(2):
            grp()
            lib.device_status()
            for g in range(len(ws)):
                assert torch.equal(outs2[g], outs[g]), (M, g)
        for g, w in enumerate(ws):
            single = torch.empty_like(outs[g])
            lib.tq2_gemm(w, xs[g], single)
            lib.device_status()
            assert torch.equal(outs[g], single), (M, g)
            ref, absref, _, _ = oracle_gemm(auos[g], w.N, K, xs[g].cpu().numpy())
            check_skinny(outs[g].cpu().numpy().astype(np.float64), ref, absref, f"grouped M={M} g={g}")
    with pytest.raises(lib.TQ2Error):                       # M = 9 is not a grouped shape
        x9 = [torch.zeros((9, K), device="cuda") for _ in ws]
        lib.tq2_gemm_grouped(ws, x9, [torch.zeros((9, w.N), device="cuda") for w in ws])


def test_gemv_many_units_per_cta_sampled(lib):
    """N = 30000 rows at K = 4096: every CTA of the fused GEMV walks several
    units and the stage ring and scale slots wrap many times.  Sampled rows
    (all of the first and last few) against the oracle, element by element."""
    import torch
    N, K = 30000, 4096
    aos = synth.random_tq2(N, K, 92)
    w = lib.tq2_upload(aos, N, K)
    codes, d_bits = otq2.parse_aos(aos, N, K)
    rng = np.random.Generator(np.random.Philox(key=93))
    rows = sorted(set(rng.integers(0, N, 600).tolist()) | set(range(20)) | set(range(N - 20, N)))
    for M in (1, 2, 4, 8):
        x = synth.random_x(M, K, 94 + M)
        xd = to_dev(x)
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        lib.tq2_gemm(w, xd, out)
        lib.device_status()
        assert not torch.isnan(out).any().item()
        got = out.cpu().numpy().astype(np.float64)
        for m in range(M):
            for n in rows:
                ref, absref = otq2.gemm_elem(x[m], codes[n], d_bits[n])
                err = abs(got[m, n] - ref)
                assert err <= 1e-3 and err <= 2.0 ** -12 * absref + 1e-7, (m, n, got[m, n], ref)


def test_gemv_grouped_64_jobs_bit_identical(lib):
    """64 jobs of N=4096, K=4096 (the decode-shape workload) in one launch:
    each CTA walks many row groups; every output equals the single call."""
    import torch
    N, K = 4096, 4096
    ws = [lib.tq2_upload(synth.random_tq2(N, K, 100 + i), N, K) for i in range(4)]
    hs = [ws[i % 4] for i in range(64)]
    xs = [to_dev(synth.random_x(1, K, 200 + (i % 8))) for i in range(64)]
    outs = [torch.full((1, N), float("nan"), device="cuda") for _ in range(64)]
    lib.tq2_gemm_grouped(hs, xs, outs)
    lib.device_status()
    for i in range(64):
        single = torch.empty_like(outs[i])
        lib.tq2_gemm(hs[i], xs[i], single)
        lib.device_status()
        assert torch.equal(outs[i], single), i


def _sampled_gemv_check(lib, N, K, Ms, wkey, xkey, nsample=400):
    import torch
    aos = synth.random_tq2(N, K, wkey)
    w = lib.tq2_upload(aos, N, K)
    codes, d_bits = otq2.parse_aos(aos, N, K)
    rng = np.random.Generator(np.random.Philox(key=wkey + 7))
    rows = sorted(set(rng.integers(0, N, nsample).tolist()) | set(range(8)) | set(range(N - 140, N)))
    for M in Ms:
        x = synth.random_x(M, K, xkey + M)
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        lib.tq2_gemm(w, to_dev(x), out)
        lib.device_status()
        assert not torch.isnan(out).any().item()
        got = out.cpu().numpy().astype(np.float64)
        for m in range(M):
            for n in rows:
                ref, absref = otq2.gemm_elem(x[m], codes[n], d_bits[n])
                err = abs(got[m, n] - ref)
                assert err <= 1e-3 + 2e-4 * (K > 4096) and err <= 2.0 ** -12 * absref + 1e-7, (M, m, n, got[m, n], ref)


def test_gemv_row_split_ragged(lib):
    """Row-split GEMV with a ragged last unit (20000 = 156 x 128 + 32 rows)
    and a partial last stage (K = 2176: 17 blocks)."""
    _sampled_gemv_check(lib, 20000, 2176, (1, 2, 5), 110, 111)


def test_gemv_row_split_k8192(lib):
    """Row-split GEMV at K = 8192, M = 1..4 (x held in shared memory)."""
    _sampled_gemv_check(lib, 19600, 8192, (1, 2, 3, 4), 112, 113, nsample=200)


def test_gemv_grouped_distinct_x(lib):
    """A grouped call whose jobs each bring their own x: the row-split kernel
    restages x at job boundaries inside a CTA's run of units."""
    import torch
    N, K = 4096, 1024
    G = 40
    aoss = [synth.random_tq2(N, K, 120 + i) for i in range(3)]
    ws = [lib.tq2_upload(a, N, K) for a in aoss]
    Ws = [otq2.dequant_aos(a, N, K) for a in aoss]
    for M in (1, 2, 6):
        xs_np = [synth.random_x(M, K, 300 + 10 * M + g) for g in range(G)]
        hs = [ws[g % 3] for g in range(G)]
        outs = [torch.full((M, N), float("nan"), device="cuda") for _ in range(G)]
        lib.tq2_gemm_grouped(hs, [to_dev(x) for x in xs_np], outs)
        lib.device_status()
        for g in range(G):
            x64 = np.asarray(xs_np[g], dtype=np.float64)
            W = Ws[g % 3]
            check_skinny(outs[g].cpu().numpy().astype(np.float64), x64 @ W.T, np.abs(x64) @ np.abs(W).T,
                         f"M={M} job {g}")


def test_gemv_mk_limit(lib):
    """MT * K above the shared-memory limit of the fused GEMV (MT = M rounded
    up to 1, 2, 4, 8): a single call falls back to the staged skinny kernel,
    a grouped call is refused."""
    import torch
    N, K = 40, 16512                     # M = 2: M * K = 33024 > 32768
    aos = synth.random_tq2(N, K, 95)
    w = lib.tq2_upload(aos, N, K)
    for M in (1, 2, 3, 5, 8):
        x = synth.random_x(M, K, 96) * 0.5
        got = run_gemm(lib, w, x)
        ref, absref, _, _ = oracle_gemm(aos, N, K, x)
        assert np.max(np.abs(got - ref)) <= 2e-3
        assert np.all(np.abs(got - ref) <= (2.0 ** -10) * absref + 1e-7)
    x2 = torch.zeros((2, K), device="cuda")
    with pytest.raises(lib.TQ2Error):
        lib.tq2_gemm_grouped([w], [x2], [torch.zeros((2, N), device="cuda")])
    x1 = to_dev(synth.random_x(1, K, 97))
    o1 = torch.empty((1, N), device="cuda")
    lib.tq2_gemm_grouped([w], [x1], [o1])                       # M = 1 fits
    lib.device_status()
    single = torch.empty_like(o1)
    lib.tq2_gemm(w, x1, single)
    assert torch.equal(o1, single)


def test_gemv_full_size(lib):
    cfg = synth.GEMV
    N, K = cfg["N"], cfg["K"]
    aos = synth.random_tq2(N, K, cfg["wkey"])
    w = lib.tq2_upload(aos, N, K)
    x = synth.random_x(1, K, cfg["xkey"])
    got = run_gemm(lib, w, x)
    ref, absref, _, _ = oracle_gemm(aos, N, K, x)
    check_skinny(got, ref, absref, "gemv 4096x4096")


def test_skinny_m8_full_size(lib):
    cfg = synth.SKINNY
    N, K = cfg["N"], cfg["K"]
    aos = synth.random_tq2(N, K, cfg["wkey"])
    w = lib.tq2_upload(aos, N, K)
    x = synth.random_x(8, K, cfg["xkey"])
    got = run_gemm(lib, w, x)
    ref, absref, _, _ = oracle_gemm(aos, N, K, x)
    check_skinny(got, ref, absref, "skinny M=8 N=11008")


def test_skinny_deterministic(lib):
    aos = synth.random_tq2(1000, 2048, 60)
    w = lib.tq2_upload(aos, 1000, 2048)
    x = synth.random_x(5, 2048, 61)
    a = run_gemm(lib, w, x)
    b = run_gemm(lib, w, x)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- tensor ----
def test_tiny_tensor_m100(tiny, lib):
    aos, N, K, xs, w = tiny
    got = run_gemm(lib, w, xs[100])                       # M > 16 -> tensor path
    check_tensor(got, *oracle_gemm(aos, N, K, xs[100]), where="tiny M=100")


@pytest.mark.parametrize("M", [1, 7, 9, 33])
def test_tiny_tensor_forced(tiny, lib, M):
    aos, N, K, xs, w = tiny
    x = xs[M] if M in xs else synth.xorshift_uniform(M * K, 1, 0.5).reshape(M, K)
    got = run_gemm(lib, w, x, lib.PATH_TENSOR)
    check_tensor(got, *oracle_gemm(aos, N, K, x), where=f"tiny tensor M={M}")


@pytest.mark.parametrize("N,K", [(8, 128), (40, 256), (3072, 3072), (300, 640)])
def test_tensor_page_sweep(lib, N, K):
    aos = page_sweep_weight(N, K)
    w = lib.tq2_upload(aos, N, K)
    for M in (17, 32, 33, 100, 256, 257, 600):
        x = page_sweep_x(M, K)
        got = run_gemm(lib, w, x, lib.PATH_TENSOR)
        check_tensor(got, *oracle_gemm(aos, N, K, x), where=f"tensor sweep N={N} K={K} M={M}")


@pytest.mark.parametrize("M", [32, 128])
def test_tensor_skinny_config_full(lib, M):
    cfg = synth.SKINNY
    N, K = cfg["N"], cfg["K"]
    aos = synth.random_tq2(N, K, cfg["wkey"])
    w = lib.tq2_upload(aos, N, K)
    x = synth.random_x(M, K, cfg["xkey"])
    got = run_gemm(lib, w, x)
    check_tensor(got, *oracle_gemm(aos, N, K, x), where=f"N=11008 M={M}")


def test_tensor_tuned_tiles_and_splits(lib):
    """The tensor path under every token tile and K-split count the tuning
    export accepts for these shapes (ragged row tile, ragged token tile, K
    of 10 k-steps so that three splits are uneven): each within the tensor
    bound against the oracle, two splits bit-equal to one another run to run
    (the 384-token tile included: partial at M = 100, two tiles at M = 600, an
    odd number of 128-row tiles for its CTA pairs); bad tiles and split counts
    are refused."""
    import torch
    N, K = 300, 640
    aos = synth.random_tq2(N, K, 130)
    w = lib.tq2_upload(aos, N, K)
    for M, tiles in ((33, (48, 64, 128)), (100, (32, 64, 128, 256, 384)), (600, (256, 384))):
        x = synth.random_x(M, K, 131 + M)
        ref, absref, ref16, absref16 = oracle_gemm(aos, N, K, x)
        xd = to_dev(x)
        for bn in tiles:
            for splits in (1, 2, 3, 4):
                out = torch.full((M, N), float("nan"), device="cuda")
                lib.tq2_gemm_tensor_tuned(w, xd, out, bn, splits)
                lib.device_status()
                got = out.cpu().numpy().astype(np.float64)
                check_tensor(got, ref, absref, ref16, absref16, f"tuned M={M} bn={bn} splits={splits}")
                if splits <= 2:
                    again = torch.full((M, N), float("nan"), device="cuda")
                    lib.tq2_gemm_tensor_tuned(w, xd, again, bn, splits)
                    assert torch.equal(out, again), (M, bn, splits)
    x = to_dev(synth.random_x(60, K, 140))
    out = torch.zeros((60, N), device="cuda")
    for bn, splits in ((48, 1), (8, 1), (272, 1), (64, 11), (64, 17)):   # 48 < M = 60 is not a multiple of 32
        with pytest.raises(lib.TQ2Error):
            lib.tq2_gemm_tensor_tuned(w, x, out, bn, splits)


def test_tensor_stage_widths(lib):
    """Token tiles of at most 128 run pipeline stages of four, two or one
    64-k atoms: four while every K split keeps a 256-k stage, else two while
    it keeps a 128-k stage, else one.  K = 768 takes four atoms up to three
    splits, two at four to six and one at seven to twelve; ragged row and
    token tiles throughout, each within the tensor bound against the oracle,
    two splits bit-equal to one another run to run."""
    import torch
    N, K = 300, 768
    aos = synth.random_tq2(N, K, 150)
    w = lib.tq2_upload(aos, N, K)
    for M, tiles in ((33, (48, 64)), (100, (32, 128))):
        x = synth.random_x(M, K, 151 + M)
        ref, absref, ref16, absref16 = oracle_gemm(aos, N, K, x)
        xd = to_dev(x)
        for bn in tiles:
            for splits in (1, 2, 3, 4, 6, 7, 12):
                out = torch.full((M, N), float("nan"), device="cuda")
                lib.tq2_gemm_tensor_tuned(w, xd, out, bn, splits)
                lib.device_status()
                got = out.cpu().numpy().astype(np.float64)
                check_tensor(got, ref, absref, ref16, absref16, f"stages M={M} bn={bn} splits={splits}")
                if splits <= 2:
                    again = torch.full((M, N), float("nan"), device="cuda")
                    lib.tq2_gemm_tensor_tuned(w, xd, again, bn, splits)
                    assert torch.equal(out, again), (M, bn, splits)


def test_tensor_large_sampled(lib):
    """M=4096, N=14336, K=4096 in the benchmarked launch configuration; the
    oracle computes sampled outputs one by one (random elements plus two full
    rows and two full columns)."""
    _tensor_sampled(lib, synth.LARGE)


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", synth.DIT, ids=[c["name"] for c in synth.DIT])
def test_tensor_dit_shapes_sampled(lib, cfg):
    """The pages' two DiT shapes, M=1536 and K=3072 with N=27648 or 3072."""
    _tensor_sampled(lib, cfg)


def _tensor_sampled(lib, cfg):
    import torch
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    aos = synth.random_tq2(N, K, cfg["wkey"])
    w = lib.tq2_upload(aos, N, K)
    x = synth.random_x(M, K, cfg["xkey"])
    xd = to_dev(x)
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    lib.tq2_gemm(w, xd, out)
    lib.device_status()
    assert not torch.isnan(out).any().item()
    codes, d_bits = otq2.parse_aos(aos, N, K)
    rng = np.random.Generator(np.random.Philox(key=99))
    idx = [(int(m), int(n)) for m, n in zip(rng.integers(0, M, 1500), rng.integers(0, N, 1500))]
    idx += [(0, n) for n in range(0, N, 7)] + [(M - 1, n) for n in range(3, N, 11)]
    idx += [(m, 0) for m in range(0, M, 5)] + [(m, N - 1) for m in range(2, M, 9)]
    ms = torch.tensor([i[0] for i in idx], device="cuda")
    ns = torch.tensor([i[1] for i in idx], device="cuda")
    got = out[ms, ns].cpu().numpy().astype(np.float64)
    x16 = x.astype(np.float16).astype(np.float64)
    for (m, n), g in zip(idx, got):
        ref, absref = otq2.gemm_elem(x[m], codes[n], d_bits[n])
        ref16, absref16 = otq2.gemm_elem(x16[m], codes[n], d_bits[n])
        assert abs(g - ref) <= 1e-2 * absref, (m, n, g, ref)
        assert abs(g - ref16) <= 2.0 ** -11 * absref16, (m, n, g, ref16)


def test_tensor_deterministic(lib):
    aos = synth.random_tq2(700, 1024, 70)
    w = lib.tq2_upload(aos, 700, 1024)
    x = synth.random_x(300, 1024, 71)
    assert np.array_equal(run_gemm(lib, w, x), run_gemm(lib, w, x))


# ------------------------------------------------------------ edge cases ----
def test_edge_cases(lib):
    import torch
    aos = synth.random_tq2(1, 128, 80)
    w = lib.tq2_upload(aos, 1, 128)
    for M in (1, 16, 17, 40):                                   # N = 1, one block
        x = synth.random_x(M, 128, 81 + M)
        got = run_gemm(lib, w, x)
        r = oracle_gemm(aos, 1, 128, x)
        (check_skinny(got, r[0], r[1]) if M <= 16 else check_tensor(got, *r))
    # M == 0 is a no-op; shape mismatches are refused on the host
    x = torch.zeros((0, 128), device="cuda")
    out = torch.zeros((0, 1), device="cuda")
    lib.tq2_gemm(w, x, out)
    assert lib.load().tq2_gemm(w.handle, None, None, 1, 2, 128, None) != 0
    xb = torch.zeros((17, 128), device="cuda")
    with pytest.raises(lib.TQ2Error):
        lib.tq2_gemm_path(w, xb, torch.zeros((17, 1), device="cuda"), lib.PATH_SKINNY)
    # all codes 1 -> exact zeros; all codes 2 -> block sums times d
    for code in (1, 2):
        N, K = 20, 384
        codes = np.full((N, K), code, dtype=np.uint8)
        d = synth.f16_bits(synth.uniform(N * 3, 82, 0.01, 0.1)).reshape(N, 3)
        a2 = synth.pack_aos(codes, d)
        w2 = lib.tq2_upload(a2, N, K)
        for M in (1, 2, 3, 50):
            x = synth.random_x(M, K, 83)
            got = run_gemm(lib, w2, x)
            r = oracle_gemm(a2, N, K, x)
            if code == 1:
                assert np.all(got == 0.0), M    # every path, the offset-decode GEMV included
            else:
                (check_skinny(got, r[0], r[1]) if M <= 16 else check_tensor(got, *r))
    lib.device_status()


# ---- ternary producer (f32 weights -> BlockTQ2_0_g128), bit-exact against the oracle

def _quantize_gpu(lib, W):
    import torch
    N, K = W.shape
    aos = torch.zeros(N * (K // 128) * 34, dtype=torch.uint8, device="cuda")
    lib.tq2_quantize(to_dev(W), aos)
    lib.device_status()
    return aos.cpu().numpy().tobytes()


@pytest.mark.gpu
def test_quantize_matches_oracle_with_edge_blocks(lib):
    N, K = 300, 640
    W = synth.random_weights_f32(N, K, 301)
    blocks = W.reshape(N, K // 128, 128)
    blocks[3, 2, :] = 0.0                                   # all-zero block: codes 1, d = f16(1e-12) = 0
    m = np.abs(blocks[5, 1]).max()
    blocks[5, 1, 7], blocks[5, 1, 9] = 0.5 * m, -0.5 * m    # exact ties: round half to even -> 0
    blocks[6, 0, :] = -1.0                                  # every weight at the (negative) maximum
    blocks[7, 4, :] = 1e-30                                 # tiny values (f16(scale) underflows to 0)
    blocks[8, 3, 100] = 1e30                                # one huge value (f16(scale) overflows to inf)
    W = blocks.reshape(N, K)
    got = _quantize_gpu(lib, W)
    want = otq2.pack_aos(*otq2.quantize(W))
    assert got == want


@pytest.mark.gpu
def test_quantize_full_size_and_shapes(lib):
    for N, K in ((1, 128), (14336, 4096)):
        W = synth.random_weights_f32(N, K, 302 + N)
        assert _quantize_gpu(lib, W) == otq2.pack_aos(*otq2.quantize(W)), (N, K)
    import torch
    with pytest.raises(lib.TQ2Error):
        lib.tq2_quantize(torch.zeros((4, 200), device="cuda"), torch.zeros(1000, dtype=torch.uint8, device="cuda"))


@pytest.mark.gpu
def test_quantized_weights_feed_the_gemm(lib):
    """Producer -> tq2_upload -> GEMM, against the oracle on the oracle's codes.
    Weights N(0, 0.03^2), so block scales fall near the pages' U(0.01, 0.1)
    and the pages' absolute bound applies."""
    N, K = 1000, 1024
    W = (synth.random_x(N, K, 303) * np.float32(0.03)).astype(np.float32)
    aos = _quantize_gpu(lib, W)
    w = lib.tq2_upload(aos, N, K)
    for M in (1, 8, 64):
        x = synth.random_x(M, K, 304 + M)
        got = run_gemm(lib, w, x)
        ref, absref, ref16, absref16 = oracle_gemm(aos, N, K, x)
        (check_skinny(got, ref, absref, f"quantized M={M}") if M <= 16 else check_tensor(got, ref, absref, ref16, absref16, f"quantized M={M}"))


@pytest.mark.gpu
def test_quantize_quotients_next_to_one_half(lib):
    """Weights whose quotient w / s rounds to just below, exactly at, or just
    above +-0.5 in f32, for scales that are not powers of two: the producer's
    rounding decision must be the one of the correctly rounded division."""
    rows = []
    for s in (3.0, 5.0, 7.0, 0.3, 1.7e-5, 6e4):
        s = np.float32(s)
        h = np.float32(0.5) * s
        vals = [s]                                     # the block maximum
        w = h
        for _ in range(20):                            # floats walking up from s/2
            vals += [w, -w]
            w = np.nextafter(w, np.float32(np.inf))
        w = h
        for _ in range(20):                            # and down
            w = np.nextafter(w, np.float32(0))
            vals += [w, -w]
        vals = np.array(vals[:128] + [0.0] * (128 - min(len(vals), 128)), dtype=np.float32)
        rows.append(vals)
    W = np.stack(rows).astype(np.float32)
    assert _quantize_gpu(lib, W) == otq2.pack_aos(*otq2.quantize(W))


@pytest.mark.gpu
def test_tiny_page_against_golden(tiny, lib):
    """The GPU on the page's tiny data against the stored oracle outputs
    (tests/golden/tq2_page_tiny_M*.txt), within the pages' 1e-3 bound."""
    from test_golden import load_matrix
    aos, N, K, xs, w = tiny
    for M in (1, 7):
        got = run_gemm(lib, w, xs[M])
        want = load_matrix(f"tq2_page_tiny_M{M}.txt")
        assert np.abs(got - want).max() <= 1e-3, M


# ---- accuracy of the decode-shape GEMV (offset decode) on data that is not unit-scale

def _sparse_weights(N, K, key, p_nonzero, zero_rows=()):
    """Codes mostly 1 (weight 0): each code is 0 or 2 with probability p_nonzero;
    rows in zero_rows are all code 1.  Scales U(0.01, 0.1)."""
    u = synth.uniform01(N * K, key).reshape(N, K)
    c2 = synth.codes3(N * K, key + 1).reshape(N, K)
    codes = np.where(u < p_nonzero, np.where(c2 == 0, 0, 2), 1).astype(np.uint8)
    for r in zero_rows:
        codes[r] = 1
    d = synth.f16_bits(synth.uniform(N * (K // 128), key + 2, 0.01, 0.1)).reshape(N, K // 128)
    return synth.pack_aos(codes, d), codes


@pytest.mark.gpu
@pytest.mark.parametrize("p_nonzero", [0.1, 0.01])
@pytest.mark.parametrize("xscale", [1.0, 16.0, 256.0])
def test_gemv_sparse_weights_scaled_x(lib, p_nonzero, xscale):
    """M = 1, 2, 4, 8 through tq2_gemm (the fused GEMV) and tq2_gemm_grouped on
    weights with >= 90 % zero codes, rows of all code 1 mixed with dense rows,
    and x ~ N(0,1) times 1, 16 and 256: element by element within
    2^-12 * sum|x W| + 1e-7 (f32 accumulation), and exactly 0 on the all-zero
    rows.  The bound scales with the row's nonzero weights, not with x."""
    import torch
    zero_rows = (0, 5, 127, 128, 2000, 4095)
    for N, K in ((4096, 4096), (300, 8192)):
        zr = tuple(r for r in zero_rows if r < N)
        aos, codes = _sparse_weights(N, K, 700 + int(1000 * p_nonzero), p_nonzero, zr)
        w = lib.tq2_upload(aos, N, K)
        W = otq2.dequant_aos(aos, N, K)
        for M in ((1, 2, 4, 8) if K <= 4096 else (1, 2, 4)):
            x = (synth.random_x(M, K, 710 + M) * np.float32(xscale)).astype(np.float32)
            ref, absref = otq2.gemm(x, W), otq2.gemm_abs(x, W)
            got = run_gemm(lib, w, x)
            err = np.abs(got - ref)
            bad = err > 2.0 ** -12 * absref + 1e-7
            assert not bad.any(), (N, K, M, int(bad.sum()), float(err.max()))
            assert np.all(got[:, list(zr)] == 0.0), (N, K, M)
            # the same GEMV inside a grouped launch (row-split when the group fills the GPU)
            outs = [torch.full((M, N), float("nan"), device="cuda") for _ in range(40)]
            xd = to_dev(x)
            lib.tq2_gemm_grouped([w] * 40, [xd] * 40, outs)
            lib.device_status()
            for o in (outs[0], outs[39]):
                g2 = o.cpu().numpy().astype(np.float64)
                assert np.array_equal(g2, got), (N, K, M)
        w.free()
