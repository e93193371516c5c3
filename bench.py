#!/usr/bin/env python3
"""Benchmark of the packed ternary GEMM (and the rest of the hot path).

Headline workload: the TQ2 GEMV (decode shape) M=1, N=K=4096, codes iid
uniform over {0,1,2}, per-block f16 scales iid U(0.01, 0.1), x iid N(0,1).
One *step* is 64 such GEMVs, each against its own copy of the weight
(64 x 4.46 MB = 285 MB > the 129 MB L2, so every GEMV streams its weight
from HBM), issued as one tq2_gemm_grouped call (the library's call for
independent GEMVs that share K and M).  ``value`` is packed-weight GB/s over
the whole job: (N*K/4 + N*K/128*2) bytes per GEMV x GEMVs / device time.
The same 64 GEMVs issued as 64 stream-ordered tq2_gemm calls (each waits
for the one before it) are reported under ``extra`` as the latency-bound
form.

The same JSON line carries, under ``extra``, the other workloads of the hot
path measured the same way (skinny M=8/32/128 x N=11008, large M=4096 x
N=14336, and the blr layer once built), each with its roofline fraction.

``--impl reference`` times the f64 CPU oracle instead (a deliberately slow
reference on the host cores; see ``oracle/``).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

GEMV_COPIES = 64
# timed replays of each secondary workload: None keeps each workload's own
# count; --extra-reps sets one count for all (e.g. 1 for a profiler's launch list)
EXTRA_REPS = None


def reps(n):
    return n if EXTRA_REPS is None else EXTRA_REPS


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-extra", action="store_true", help="skip the secondary workloads")
    p.add_argument("--only", default="", help="comma list of extra workloads to run")
    p.add_argument("--extra-reps", type=int, default=None,
                   help="timed replays of every secondary workload (default: each workload's own count)")
    p.add_argument("--oracle-job", default="", help=argparse.SUPPRESS)
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d.get("bf16_tflops_sustained"),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def src_hash(files):
    """Hash of the kernel sources `files` (names under csrc/, in order)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "binary_packed_weight_gb300", "csrc")
    for f in files:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(key):
    """DRAM bytes per launch from the committed ncu summary, if the sources
    the kernel is compiled from have not changed since it was taken (else
    None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path)).get(key)
    if not d or not d.get("sources") or d.get("src_hash") != src_hash(d["sources"]):
        return None
    return d.get("dram_bytes")


# ---------------------------------------------------------------- clocks ----
class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons around a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.05)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        busy = sorted(sm)[len(sm) // 4:] if sm else []
        return {"sm_mhz": float(np.median(busy)) if busy else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- timing ----
def time_graph(torch, fn, steps, warmup, stream):
    """Capture fn() once into a CUDA graph; replay warmup + steps times; return
    device seconds of the timed replays (CUDA events on the launch stream)."""
    with torch.cuda.stream(stream):
        fn()                                   # first call outside capture (allocator pools)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    with torch.cuda.stream(stream):            # replays run on the current stream
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3, g


def gemv_bytes(N, K):
    return N * K // 4 + N * (K // 128) * 2


def workload_config():
    """The workload both arms measure (the fields that do not depend on the arm)."""
    N, K = synth.GEMV["N"], synth.GEMV["K"]
    return {"workload": "tq2_gemv M=1 N=4096 K=4096", "gemvs_per_step": GEMV_COPIES,
            "weights": "packed BlockTQ2_0_g128, 2 bits + f16 scale per 128",
            "l2": f"inputs larger than L2: {GEMV_COPIES} distinct weight copies "
                  f"({GEMV_COPIES * gemv_bytes(N, K) / 1e6:.0f} MB) rotated every step",
            "value": "packed-weight bytes per GEMV x GEMVs / seconds"}


def max_over_ranks(torch, dist, secs, device):
    """The job ends when its slowest rank does: every rank gets the maximum of
    the ranks' timed-region seconds (unchanged without a process group)."""
    if dist is None:
        return secs
    t = torch.tensor([secs], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_gemv, gemvs_per_rank, world, secs):
    """Whole-job packed-weight GB/s: the GEMVs of every rank over the slowest
    rank's seconds (each replica runs the same work: weak scaling)."""
    return bytes_per_gemv * gemvs_per_rank * world / secs / 1e9


# ------------------------------------------------------------- workloads ----
def capture(torch, fn, stream, warmup):
    with torch.cuda.stream(stream):
        fn()                                   # first call outside capture (allocator pools)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    with torch.cuda.stream(stream):
        for _ in range(max(3, warmup)):
            g.replay()
    torch.cuda.synchronize()
    return g


def run_gemv(torch, bpw, args, stream, dev):
    cfg = synth.GEMV
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    aos = synth.random_tq2(N, K, cfg["wkey"])
    ws = [bpw.tq2_upload(aos, N, K) for _ in range(GEMV_COPIES)]
    x = torch.from_numpy(synth.random_x(M, K, cfg["xkey"])).to(dev)
    # the 64 outputs are views of one [64][M][N] buffer, so that a caller can
    # read every result back with one copy
    obuf = torch.empty((len(ws), M, N), dtype=torch.float32, device=dev)
    outs = list(obuf.unbind(0))
    xs = [x] * len(ws)

    # one tq2_gemm_grouped launch per step, issued straight onto the stream
    # with its arguments marshalled once (GroupedGemv): consecutive launches
    # overlap under programmatic dependent launch (the next one's prologue
    # and weight prefetch start while this one finishes), which separate
    # CUDA-graph replays would not
    grouped = bpw.GroupedGemv(ws, xs, outs)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            grouped(stream=stream.cuda_stream)
    torch.cuda.synchronize()
    clocks = Clocks(dev.index if dev.index is not None else 0)
    return dict(ws=ws, x=x, xs=xs, outs=outs, obuf=obuf, step=grouped, clocks=clocks, M=M, N=N, K=K, aos=aos)


def extra_chained(torch, bpw, ctx, stream, pk):
    """The same 64 GEMVs as 64 stream-ordered tq2_gemm calls (latency-bound:
    each waits for the previous kernel; weights prefetch under PDL)."""
    ws, x, N, K, M = ctx["ws"], ctx["x"], ctx["N"], ctx["K"], ctx["M"]
    out = ctx["outs"][0]

    def step():
        for w in ws:
            bpw.tq2_gemm(w, x, out, stream=stream.cuda_stream)
    n = reps(200)
    secs, _ = time_graph(torch, step, n, 5, stream)
    t = secs / n / len(ws)
    alg = gemv_bytes(N, K) + M * K * 4 + M * N * 4
    return dict(us_per_gemv=t * 1e6, gemvs_per_step=len(ws), weight_gbs=gemv_bytes(N, K) / t / 1e9,
                alg_gbs=alg / t / 1e9, hbm_frac=alg / t / 1e9 / pk["hbm"],
                kernel="tq2_gemv_kernel<1, k-split, 1 job> (one launch per GEMV)")


def e2e_gemv(torch, bpw, ctx, stream, reps):
    """Public API with host buffers, every step: pinned x -> device, one
    tq2_gemm_grouped call over the 64 weights (arguments marshalled once,
    GroupedGemv), the 64 outputs (one [64][M][N] device buffer) -> pinned host
    in one copy.  Two steps are in flight, as a
    serving loop runs them: each of two slots has its own pinned and device
    buffers, the input and output copies run on two copy streams beside the
    other step's GEMVs (an input copy never queues behind the previous
    step's output copy), and before it reuses a slot the host waits until
    that slot's previous result has landed in pinned memory."""
    M, N, K = ctx["M"], ctx["N"], ctx["K"]
    ws = ctx["ws"]
    dev = ctx["x"].device
    h2d_stream, d2h_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    slots = []
    for k in range(2):
        xd = torch.empty((M, K), dtype=torch.float32, device=dev)
        ob = torch.empty((len(ws), M, N), dtype=torch.float32, device=dev)
        outs = list(ob.unbind(0))
        slots.append(dict(xh=torch.from_numpy(synth.random_x(M, K, synth.GEMV["xkey"] + k)).pin_memory(),
                          xd=xd, ob=ob, call=bpw.GroupedGemv(ws, [xd] * len(ws), outs),
                          oh=torch.empty(tuple(ob.shape), dtype=torch.float32).pin_memory(), done=None))

    def step(i):
        sl = slots[i % 2]
        if sl["done"] is not None:
            sl["done"].synchronize()           # the slot's previous result is on the host
        h2d, comp, done = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
        with torch.cuda.stream(h2d_stream):
            sl["xd"].copy_(sl["xh"], non_blocking=True)
            h2d.record(h2d_stream)
        stream.wait_event(h2d)
        sl["call"](stream=stream.cuda_stream)
        comp.record(stream)
        d2h_stream.wait_event(comp)
        with torch.cuda.stream(d2h_stream):
            sl["oh"].copy_(sl["ob"], non_blocking=True)
            done.record(d2h_stream)
        sl["done"] = done

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(reps):
        step(i)
    for sl in slots:
        sl["done"].synchronize()
    dt = time.perf_counter() - t0
    n = reps * len(ws)
    return dict(value=gemv_bytes(N, K) * n / dt / 1e9, unit="GB/s",
                h2d_bytes_per_step=M * K * 4, d2h_bytes_per_step=M * N * 4 * len(ws),
                pipeline="two steps in flight; input and output copies on two more streams")


def extra_skinny(torch, bpw, stream, dev, pk, Ms):
    cfg = synth.SKINNY
    N, K = cfg["N"], cfg["K"]
    aos = synth.random_tq2(N, K, cfg["wkey"])
    copies = 24                                            # 24 x 12 MB > L2
    ws = [bpw.tq2_upload(aos, N, K) for _ in range(copies)]
    res = {}
    for M in Ms:
        x = torch.from_numpy(synth.random_x(M, K, cfg["xkey"])).to(dev)
        out = torch.empty((M, N), dtype=torch.float32, device=dev)

        def step():
            for w in ws:
                bpw.tq2_gemm(w, x, out, stream=stream.cuda_stream)
        n = reps(20)
        secs, _ = time_graph(torch, step, n, 3, stream)
        t = secs / (n * copies)
        wb = gemv_bytes(N, K)
        alg = wb + M * K * 4 + M * N * 4
        flops = 2.0 * M * N * K
        tfl = flops / t / 1e12
        bound = "hbm" if M <= 32 else "tensor"
        res[f"M{M}"] = dict(us=t * 1e6, tflops=tfl, weight_gbs=wb / t / 1e9, alg_gbs=alg / t / 1e9,
                            hbm_frac=alg / t / 1e9 / pk["hbm"], tensor_frac=tfl / pk["bf16"],
                            bound=bound, path="skinny" if M <= 16 else "tensor")
    for w in ws:
        w.free()
    return res


def extra_c3_sweep(torch, bpw, stream, dev, pk):
    """Token-tile x K-split sweep of the tensor path at the batched-decode
    shapes M = 8, 32 and 128, N = 11008, K = 4096 (24 weight copies, > L2):
    microseconds per GEMM (x staging included) for every tile and split
    count, plus the library's own choice for the tensor path (bn 0, splits
    0; at M = 8 tq2_gemm itself takes the fused GEMV).  The weight-row tile
    is fixed at 128 rows, the M of a one-CTA kind::f16 MMA."""
    cfg = synth.SKINNY
    N, K = cfg["N"], cfg["K"]
    aos = synth.random_tq2(N, K, cfg["wkey"])
    copies = 24
    ws = [bpw.tq2_upload(aos, N, K) for _ in range(copies)]
    res = {}
    for M, tiles in ((8, (0, 16)), (32, (0, 32)), (128, (0, 32, 64, 128))):
        x = torch.from_numpy(synth.random_x(M, K, cfg["xkey"])).to(dev)
        out = torch.empty((M, N), dtype=torch.float32, device=dev)
        row = {}
        for bn in tiles:
            for splits in ((0,) if bn == 0 else (1, 2, 4, 8, 16)):
                def step():
                    for w in ws:
                        bpw.tq2_gemm_tensor_tuned(w, x, out, bn, splits, stream=stream.cuda_stream)
                n = reps(10)
                secs, _ = time_graph(torch, step, n, 3, stream)
                t = secs / (n * copies)
                key = "auto" if bn == 0 else f"bn{bn}_k{splits}"
                row[key] = dict(us=round(t * 1e6, 2), weight_gbs=round(gemv_bytes(N, K) / t / 1e9, 1),
                                tflops=round(2.0 * M * N * K / t / 1e12, 1))
        res[f"M{M}"] = row
    for w in ws:
        w.free()
    return res


def extra_blr(torch, bpw, stream, dev, pk):
    """blr layer forward + backward, T=2048 d_in=d_out=4096 r=512 (c recomputed)."""
    cfg = synth.BLR
    T, din, dout, r = cfg["T"], cfg["d_in"], cfg["d_out"], cfg["r"]
    p = synth.blr_inputs(T, din, dout, r, cfg["key"])
    import numpy as _np
    d = {k: torch.from_numpy(_np.ascontiguousarray(v)).to(dev) for k, v in p.items() if k not in ("bits_u", "bits_v")}
    bu = torch.from_numpy(p["bits_u"].view(_np.int32)).to(dev)
    bv = torch.from_numpy(p["bits_v"].view(_np.int32)).to(dev)
    f = dict(dtype=torch.float32, device=dev)
    y, a = torch.empty((T, dout), **f), torch.empty((T, r), **f)
    dx = torch.empty((T, din), **f)
    dh, dl, dg = torch.zeros(dout, **f), torch.zeros(r, **f), torch.zeros(din, **f)

    def fwd():
        bpw.blr_forward(bu, bv, d["h"], d["l"], d["g"], d["x"], y, a, None, stream=stream.cuda_stream)

    def bwd():
        bpw.blr_backward(bu, bv, d["h"], d["l"], d["g"], d["x"], d["dy"], a, None, dx, dh, dl, dg,
                         stream=stream.cuda_stream)

    def step():
        fwd()
        bwd()
    gu, gv = torch.empty((dout, r), **f), torch.empty((din, r), **f)

    def sgn():
        bpw.blr_sign_grads(bu, d["h"], d["l"], d["g"], d["x"], d["dy"], a, gu, gv, stream=stream.cuda_stream)
    n = reps(20)
    tf, _ = time_graph(torch, fwd, n, 3, stream)
    tb, _ = time_graph(torch, bwd, n, 3, stream)
    ts, _ = time_graph(torch, step, n, 3, stream)
    tg, _ = time_graph(torch, sgn, n, 3, stream)
    tf, tb, ts, tg = tf / n, tb / n, ts / n, tg / n
    sflops = 3 * 2.0 * T * dout * r                     # b, G_U and G_V: three GEMMs of 2*T*4096*512
    flops = 4 * 2.0 * T * din * r                       # four GEMMs of 2*T*4096*512 (c recomputed: a fifth)
    alg_bytes = 5 * T * din * 4 + 2 * dout * r // 8 + 2 * T * r * 4
    return dict(fwd_us=tf * 1e6, bwd_us=tb * 1e6, step_us=ts * 1e6, tflops=flops / ts / 1e12,
                alg_gbs=alg_bytes / ts / 1e9, hbm_frac=alg_bytes / ts / 1e9 / pk["hbm"],
                tensor_frac=flops / ts / 1e12 / pk["bf16"], algorithmic_bytes=alg_bytes, flops=flops,
                note="forward + backward of one path; dh from a recomputed c (no c_save)",
                sign_grads_us=tg * 1e6, sign_grads_tflops=sflops / tg / 1e12,
                sign_grads_tensor_frac=sflops / tg / 1e12 / pk["bf16"])


def extra_large(torch, bpw, stream, dev, pk):
    cfg = synth.LARGE
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    aos = synth.random_tq2(N, K, cfg["wkey"])
    w = bpw.tq2_upload(aos, N, K)
    x = torch.from_numpy(synth.random_x(M, K, cfg["xkey"])).to(dev)
    out = torch.empty((M, N), dtype=torch.float32, device=dev)

    def step():
        bpw.tq2_gemm(w, x, out, stream=stream.cuda_stream)
    n = reps(10)
    secs, _ = time_graph(torch, step, n, 3, stream)
    t = secs / n
    flops = 2.0 * M * N * K
    tfl = flops / t / 1e12
    w.free()
    return dict(us=t * 1e6, tflops=tfl, weight_gbs=gemv_bytes(N, K) / t / 1e9, tensor_frac=tfl / pk["bf16"],
                tensor_frac_sustained=tfl / pk["bf16_sus"] if pk.get("bf16_sus") else None,
                bound="tensor", includes="x f32->f16 staging kernel + GEMM")


def extra_dit(torch, bpw, stream, dev, pk):
    """The pages' two DiT shapes on the large-M tensor path (M=1536, K=3072)."""
    res = {}
    for cfg in synth.DIT:
        M, N, K = cfg["M"], cfg["N"], cfg["K"]
        w = bpw.tq2_upload(synth.random_tq2(N, K, cfg["wkey"]), N, K)
        x = torch.from_numpy(synth.random_x(M, K, cfg["xkey"])).to(dev)
        out = torch.empty((M, N), dtype=torch.float32, device=dev)

        def step():
            bpw.tq2_gemm(w, x, out, stream=stream.cuda_stream)
        n = reps(10)
        secs, _ = time_graph(torch, step, n, 3, stream)
        t = secs / n
        tfl = 2.0 * M * N * K / t / 1e12
        w.free()
        res[f"M{M}_N{N}_K{K}"] = dict(us=t * 1e6, tflops=tfl, tensor_frac=tfl / pk["bf16"],
                                      tensor_frac_sustained=tfl / pk["bf16_sus"] if pk.get("bf16_sus") else None,
                                      bound="tensor", includes="x f32->f16 staging kernel + GEMM")
    return res


def extra_quantize(torch, bpw, stream, dev, pk):
    """The ternary producer at the large GEMM's weight shape: f32 [N][K] in,
    BlockTQ2_0_g128 blocks out (inputs larger than L2)."""
    cfg = synth.LARGE
    N, K = cfg["N"], cfg["K"]
    W = torch.from_numpy(synth.random_weights_f32(N, K, cfg["wkey"] + 40)).to(dev)
    aos = torch.empty(N * (K // 128) * 34, dtype=torch.uint8, device=dev)

    def step():
        bpw.tq2_quantize(W, aos, stream=stream.cuda_stream)
    n = reps(20)
    secs, _ = time_graph(torch, step, n, 3, stream)
    t = secs / n
    nbytes = N * K * 4 + N * (K // 128) * 34
    return dict(us=t * 1e6, alg_gbs=nbytes / t / 1e9, hbm_frac=nbytes / t / 1e9 / pk["hbm"], bound="hbm",
                algorithmic_bytes=nbytes, workload=f"f32 W [{N}][{K}] -> BlockTQ2_0_g128")


# ------------------------------------------------------------ cpu oracle ----
def oracle_gemv_sample(budget_s=12.0):
    """The f64 oracle on the GEMV workload, repeated for about budget_s seconds."""
    from oracle import tq2 as otq2
    cfg = synth.GEMV
    N, K = cfg["N"], cfg["K"]
    aos = synth.random_tq2(N, K, cfg["wkey"])
    x = synth.random_x(1, K, cfg["xkey"])
    n = 0
    c0, t0 = os.times(), time.perf_counter()
    while True:
        W = otq2.dequant_aos(aos, N, K)
        otq2.gemm(x, W)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    c1 = os.times()
    cpu = (c1.user - c0.user) + (c1.system - c0.system)
    return dict(value=gemv_bytes(N, K) * n / dt / 1e9, unit="GB/s", cores=max(1, round(cpu / dt)),
                kind="oracle", sample=f"{n} full GEMVs M=1 N=K=4096 (AoS parse + f64 dequant + f64 GEMV) "
                                      f"in {dt:.1f} s; cpu/wall {cpu / dt:.2f}")


def oracle_samples(budget_s=3.0):
    """The f64 oracle as it stands on bounded samples of the other workloads,
    each repeated for about budget_s seconds on the host cores.  GFLOP/s of
    the sample (2 x tokens x rows x K per GEMM); a reported baseline beside
    the GPU figures, never a target."""
    from oracle import blr as oblr
    from oracle import tq2 as otq2

    def timed(fn, flops, sample):
        n, c0, t0 = 0, os.times(), time.perf_counter()
        while True:
            fn()
            n += 1
            if time.perf_counter() - t0 > budget_s:
                break
        dt = time.perf_counter() - t0
        c1 = os.times()
        cpu = (c1.user - c0.user) + (c1.system - c0.system)
        return dict(gflops=flops * n / dt / 1e9, cores=max(1, round(cpu / dt)), kind="oracle",
                    sample=f"{n} x {sample} in {dt:.1f} s; cpu/wall {cpu / dt:.2f}")

    res = {}
    # skinny M=8 and the large GEMM: weight rows and tokens sampled, K and the
    # distributions of the workload kept; each pass parses and dequantizes the
    # sampled rows and multiplies in f64
    for name, cfg, M, rows in (("tq2_skinny_M8", synth.SKINNY, 8, 1024), ("tq2_large", synth.LARGE, 512, 512)):
        K = cfg["K"]
        aos = synth.random_tq2(rows, K, cfg["wkey"])
        x = synth.random_x(M, K, cfg["xkey"])
        res[name] = timed(lambda: otq2.gemm(x, otq2.dequant_aos(aos, rows, K)), 2.0 * M * rows * K,
                          f"{M} tokens x {rows} of N={cfg['N']} rows, K={K}")
    # blr: forward + backward of one path on a token sample of C5 (4 GEMMs)
    c = synth.BLR
    T = 128
    p = synth.blr_inputs(T, c["d_in"], c["d_out"], c["r"], c["key"])

    def blr_step():
        oblr.forward(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], p["x"])
        oblr.backward(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], p["x"], p["dy"])
    # the oracle's backward recomputes the forward: 3 forward-sized GEMM pairs per step
    res["blr_fwd_bwd"] = timed(blr_step, 6 * 2.0 * T * c["r"] * (c["d_in"] + c["d_out"]) / 2,
                               f"forward + backward, T={T} of {c['T']} tokens, d_in=d_out={c['d_in']}, r={c['r']}")
    return res


def _oracle_job(name):
    """One full-size run of the f64 oracle (called in a child process whose BLAS
    thread count the parent fixes); returns (seconds, cpu seconds, flops,
    sample) of the oracle's work, input generation excluded."""
    from oracle import blr as oblr
    from oracle import tq2 as otq2

    def clock():
        c = os.times()
        return time.perf_counter(), c.user + c.system
    t0, c0 = clock()
    if name == "tq2_tiny_C1":
        aos, N, K, xs = synth.tiny_tq2(M_list=(1, 7, 8, 9, 100))
        W = otq2.dequant_aos(aos, N, K)
        for x in xs.values():
            otq2.gemm(x, W)
        flops = sum(2.0 * M * N * K for M in xs)
        sample = f"N={N} K={K}, M in 1,7,8,9,100 (AoS parse + f64 dequant + f64 GEMM)"
    elif name in ("tq2_gemv_C2", "tq2_skinny_M8_C3", "tq2_large_C4"):
        cfg, M = {"tq2_gemv_C2": (synth.GEMV, 1), "tq2_skinny_M8_C3": (synth.SKINNY, 8),
                  "tq2_large_C4": (synth.LARGE, synth.LARGE["M"])}[name]
        N, K = cfg["N"], cfg["K"]
        aos = synth.random_tq2(N, K, cfg["wkey"])
        x = synth.random_x(M, K, cfg["xkey"])
        t0, c0 = clock()                                  # input generation is not the oracle's work
        otq2.gemm(x, otq2.dequant_aos(aos, N, K))
        flops = 2.0 * M * N * K
        sample = f"full M={M} N={N} K={K} (AoS parse + f64 dequant + f64 GEMM)"
    elif name == "blr_C5":
        c = synth.BLR
        p = synth.blr_inputs(c["T"], c["d_in"], c["d_out"], c["r"], c["key"])
        t0, c0 = clock()
        oblr.forward(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], p["x"])
        oblr.backward(p["bits_u"], p["bits_v"], p["h"], p["l"], p["g"], p["x"], p["dy"])
        # forward: 2 GEMMs; the oracle's backward recomputes a and c: 4 more
        flops = 6 * 2.0 * c["T"] * c["r"] * c["d_in"]
        sample = f"full forward + backward T={c['T']} d_in=d_out={c['d_in']} r={c['r']}"
    else:
        raise ValueError(name)
    t1, c1 = clock()
    return t1 - t0, c1 - c0, flops, sample


def oracle_full_runs(timeout_s=120.0):
    """The f64 oracle as it stands on the full workloads: single-threaded on C1,
    C2 and C3 M=8, and over all host cores on C2, C3 M=8, C4 and C5.  Each run
    is a child process with the BLAS thread count fixed through the
    environment; ``cores`` is its CPU time over wall time.  Reported beside the
    GPU figures, never a target."""
    jobs = [("tq2_tiny_C1", 1), ("tq2_gemv_C2", 1), ("tq2_skinny_M8_C3", 1),
            ("tq2_gemv_C2", 0), ("tq2_skinny_M8_C3", 0), ("tq2_large_C4", 0), ("blr_C5", 0)]
    res = {}
    for name, threads in jobs:
        env = dict(os.environ)
        if threads:
            for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
                env[v] = str(threads)
        key = f"{name}_{'1thread' if threads else 'all_cores'}"
        try:
            r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-job", name], env=env,
                               capture_output=True, text=True, timeout=timeout_s)
            res[key] = json.loads(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else \
                {"error": r.stderr.strip().splitlines()[-1:] or ["rc %d" % r.returncode]}
        except Exception as e:                    # a reported baseline only: never fail the bench on it
            res[key] = {"error": f"{type(e).__name__}: {e}"}
    return res


def oracle_job_main(name):
    secs, cpu, flops, sample = _oracle_job(name)
    print(json.dumps(dict(seconds=secs, gflops=flops / secs / 1e9, cores=max(1, round(cpu / secs)),
                          cpu_over_wall=cpu / secs, kind="oracle", sample=sample, host_cores=os.cpu_count())))


METRIC = "TQ2 GEMM TFLOP/s and weight GB/s at M=1..4096, % of GB300 roofline"


def headline_line(world, steps, warmup, secs, value, gemvs, achieved, alg, pk, cb, e2e, clk, extra):
    """The one JSON line of the default arm (the contract the driver parses).
    secs: the slowest rank's timed seconds; value: whole-job GB/s; gemvs: per
    rank; achieved: algorithmic GB/s of one launch."""
    M, N, K = synth.GEMV["M"], synth.GEMV["N"], synth.GEMV["K"]
    return dict(
        metric=METRIC, value=value, unit="GB/s", n_gpus=world, steps=steps, warmup=warmup,
        ms_per_step=secs / steps * 1e3, higher_is_better=True, scaling="weak", vs_baseline=None,
        dtype="f32", data="synthetic",
        config=dict(workload_config(), launch="one tq2_gemm_grouped call per step (64 jobs, shared x), issued directly on the stream, consecutive steps overlapping under programmatic dependent launch",
                    activations="f32 (split to two f16 terms on the GPU), f32 accumulation",
                    parallelism="replicas" if world > 1 else "single GPU"),
        tflops=2.0 * M * N * K * gemvs * world / secs / 1e12,
        roofline={"bound": "hbm", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s",
                  "frac": achieved / pk["hbm"], "traffic": profiled_traffic("tq2_gemv_grouped"),
                  "kernel": "tq2_gemv_kernel<1, row-split, 64 jobs> (one launch per step)",
                  "algorithmic_bytes_per_launch": alg, "peak_source": pk["src"] + " hbm_gbs (copy)"},
        cpu_baseline=cb, e2e=e2e, gpu_launches=steps, clocks=clk, extra=extra,
    )


# ------------------------------------------------------------------ main ----
def main():
    args = parse()
    if args.oracle_job:
        oracle_job_main(args.oracle_job)
        return
    global EXTRA_REPS
    EXTRA_REPS = args.extra_reps
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        cb = oracle_gemv_sample(budget_s=max(3.0, min(60.0, 0.5 * (args.steps + args.warmup))))
        line = dict(metric=METRIC,
                    value=cb["value"], unit="GB/s", impl="reference", n_gpus=args.gpus, steps=args.steps,
                    warmup=args.warmup, higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64",
                    data="synthetic",
                    config=dict(workload_config(), launch="the f64 oracle, one GEMV at a time on the host cores",
                                l2="host memory: each GEMV parses and dequantizes its weight afresh",
                                parallelism="host cores"),
                    cpu_baseline=cb, e2e={"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                                          "d2h_bytes_per_step": 0})
        print(json.dumps(line), flush=True)
        return

    import torch
    import binary_packed_weight_gb300 as bpw
    from binary_packed_weight_gb300 import build as _b
    _b.build()
    bpw.load()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    pk = peaks()
    stream = torch.cuda.Stream(device=dev)

    ctx = run_gemv(torch, bpw, args, stream, dev)
    step, clocks = ctx["step"], ctx["clocks"]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            step(stream=stream.cuda_stream)
        e1.record(stream)
    e1.synchronize()
    clk = clocks.stop()
    secs = e0.elapsed_time(e1) / 1e3
    secs = max_over_ranks(torch, dist, secs, dev)
    if dist:
        dist.barrier()
    N, K, M = ctx["N"], ctx["K"], ctx["M"]
    gemvs = args.steps * GEMV_COPIES
    wbytes = gemv_bytes(N, K)
    value = job_gbs(wbytes, gemvs, world, secs)
    t_launch = secs / args.steps                      # one grouped launch per step
    alg = GEMV_COPIES * (wbytes + M * K * 4 + M * N * 4)
    achieved = alg / t_launch / 1e9
    e2e = e2e_gemv(torch, bpw, ctx, stream, reps=max(20, min(200, args.steps // 10)))

    extra = {}
    # the secondary workloads run in single-GPU runs only: a multi-GPU run
    # measures the replicated headline step and nothing else
    if not args.no_extra and world == 1:
        only = set(filter(None, args.only.split(",")))
        if not only or "skinny" in only:
            extra["tq2_skinny_N11008"] = extra_skinny(torch, bpw, stream, dev, pk, (8, 32, 128))
        if not only or "chained" in only:
            extra["tq2_gemv_chained_64"] = extra_chained(torch, bpw, ctx, stream, pk)
        if not only or "large" in only:
            extra["tq2_large_M4096_N14336"] = extra_large(torch, bpw, stream, dev, pk)
        if not only or "blr" in only:
            extra["blr_T2048_d4096_r512"] = extra_blr(torch, bpw, stream, dev, pk)
        if not only or "dit" in only:
            extra["tq2_dit_M1536_K3072"] = extra_dit(torch, bpw, stream, dev, pk)
        if not only or "quantize" in only:
            extra["tq2_quantize_N14336_K4096"] = extra_quantize(torch, bpw, stream, dev, pk)
        if "c3sweep" in only:                     # on request only (a tuning table)
            extra["tq2_c3_sweep_N11008"] = extra_c3_sweep(torch, bpw, stream, dev, pk)

    if rank != 0:
        return
    cb = oracle_gemv_sample(budget_s=12.0) if world == 1 else None
    if world == 1 and not args.no_extra:
        try:
            extra["oracle_cpu_samples"] = oracle_samples()
        except Exception as e:                    # a reported baseline only: never fail the bench on it
            extra["oracle_cpu_samples"] = {"error": f"{type(e).__name__}: {e}"}
        if not args.only or "oracle_full" in args.only:
            extra["oracle_cpu_full"] = oracle_full_runs()
    line = headline_line(world=world, steps=args.steps, warmup=args.warmup, secs=secs, value=value,
                         gemvs=gemvs, achieved=achieved, alg=alg, pk=pk, cb=cb, e2e=e2e, clk=clk, extra=extra)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
