"""Host logic of bench.py's multi-rank path, on CPU.

With N > 1 the bench runs one independent replica per GPU (the GEMMs shard by
weight rows with no exchange step, so there is no data-path collective).  The
only cross-rank steps are the barriers around the timed region and the
maximum of the ranks' times; the reference arm runs on rank 0 alone.  These
run here as world-size-2 gloo process groups and as subprocesses.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_worker(rank, world, port, secs, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        m = bench.max_over_ranks(torch, dist, secs[rank], torch.device("cpu"))
        v = bench.job_gbs(1e9, 10, world, m)
        dist.barrier()
        q.put((rank, m, v))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_world2_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    secs = [0.25, 0.75]
    ps = [ctx.Process(target=_rank_worker, args=(r, 2, port, secs, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank sees the slowest rank's time, and the job value counts both ranks' work
    assert [g[1] for g in got] == [0.75, 0.75]
    assert all(g[2] == pytest.approx(2 * 10 * 1e9 / 0.75 / 1e9) for g in got)


def test_single_process_keeps_its_time():
    import torch

    import bench
    assert bench.max_over_ranks(torch, None, 0.5, torch.device("cpu")) == 0.5
    assert bench.job_gbs(4.46e6, 64, 1, 1e-3) == pytest.approx(4.46e6 * 64 / 1e-3 / 1e9)


def _bench_reference(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--gpus", str(world), "--steps", "1", "--warmup", "1"],
                          capture_output=True, text=True, env=env, timeout=300)


def test_reference_arm_other_ranks_exit_without_work():
    r = _bench_reference(1, 2)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    r = _bench_reference(0, 2)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_oracle_samples_report_every_workload():
    import bench
    r = bench.oracle_samples(budget_s=0.05)
    assert set(r) == {"tq2_skinny_M8", "tq2_large", "blr_fwd_bwd"}
    for v in r.values():
        assert v["kind"] == "oracle" and v["gflops"] > 0 and v["cores"] >= 1 and v["sample"]


def test_headline_line_keeps_the_contract():
    import bench
    pk = bench.peaks()
    secs, steps, world = 1.7, 20000, 1
    gemvs = steps * bench.GEMV_COPIES
    wb = bench.gemv_bytes(4096, 4096)
    alg = bench.GEMV_COPIES * (wb + 4 * 4096 * 2)
    line = bench.headline_line(world=world, steps=steps, warmup=5, secs=secs,
                               value=bench.job_gbs(wb, gemvs, world, secs), gemvs=gemvs,
                               achieved=alg / (secs / steps) / 1e9, alg=alg, pk=pk,
                               cb={"value": 0.04, "unit": "GB/s", "cores": 8, "kind": "oracle", "sample": "s"},
                               e2e={"value": 1.0, "unit": "GB/s", "h2d_bytes_per_step": 16384,
                                    "d2h_bytes_per_step": 1048576},
                               clk={"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}, extra={})
    s = json.dumps(line)                                       # serialisable as one line
    assert "\n" not in s
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
              "gpu_launches", "clocks"):
        assert k in line, k
    assert line["metric"] == bench.METRIC and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["scaling"] == "weak" and line["vs_baseline"] is None and line["n_gpus"] == 1
    assert line["ms_per_step"] == pytest.approx(secs / steps * 1e3)
    assert line["config"]["workload"] == bench.workload_config()["workload"]
    rf = line["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] == pk["hbm"]
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"])
    assert set(line["e2e"]) == {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}
    assert line["gpu_launches"] == steps
