"""The benchmark's multi-rank host logic on CPU: two gloo ranks (127.0.0.1), each with
its own step time.  The path runs replicas only (no collective on the data path); the
timing takes the slowest rank and the job value counts every rank's pairs.  The
reference arm runs on rank 0 alone."""

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


def _rank(rank, world, port, times, out):
    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], torch.device("cpu"))
        out.put((rank, ms, bench.job_value(world, 1000, ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [3.0, 5.0]
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in res:
        assert ms == 5.0
        assert value == pytest.approx(2 * 1000 / 5e-3)


def test_single_process_needs_no_group():
    import torch

    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(4.0, torch.device("cpu")) == 4.0
    assert bench.job_value(1, 1000, 2.0) == pytest.approx(5e5)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--config", "1", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "1", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    # the same workload description as the GPU arm's line, with the view's pair count
    # taken from the oracle's own binning
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    import synthetic_scenes as ss

    sc, cam = ss.make_config(1)
    counts = oracle.bin_sort(cam, oracle.project(sc, cam), None)
    expect = {"workload": ss.CONFIG_NAMES[1], "gaussians": sc.n,
              "image": f"{cam.width}x{cam.height}", "sh_degree": sc.sh_degree,
              "tile_pairs": int(counts.counts.sum()), "sh_storage": "f32",
              "parallelism": "single", "l2": bench.l2_note(sc, "gradients", 1)}
    assert line["config"] == expect
