"""The bench's multi-process path on the CPU: world_size-2 gloo ranks (the GPU runs use
NCCL with the same calls).  The path has no exchange step -- ranks are independent
replicas -- so what is shared is the timing: every rank must end up with the slowest
rank's step time, and the whole-job value counts the units of all ranks over it."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_setup()
        assert (ws, r, local) == (world, rank, rank)
        ms = bench.max_over_ranks(dist, times[rank], "cpu")
        dist.barrier()
        out[rank] = (ms, bench.job_value(ws, 7.4e9, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    world, port = 2, _free_port()
    times = [0.025, 0.031]  # rank 1 is the slow one
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, port, times, out), nprocs=world, start_method="spawn", join=True)
        res = dict(out)
    for r in range(world):
        ms, value = res[r]
        assert ms == pytest.approx(0.031)
        assert value == pytest.approx(2 * 7.4e9 / 0.031e-3)


def test_single_process_is_identity():
    assert bench.max_over_ranks(None, 0.02, "cpu") == 0.02
    assert bench.job_value(1, 1e9, 1.0) == pytest.approx(1e12)


def _run_bench(args, rank, world):
    import subprocess
    import sys
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    return subprocess.run([sys.executable, os.path.join(root, "bench.py"), *args], capture_output=True, text=True,
                          env=env, timeout=600)


def test_reference_arm_rank0_prints_other_ranks_exit_quietly():
    import json
    r0 = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "3"], 0, 2)
    assert r0.returncode == 0, r0.stderr
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    r1 = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "3"], 1, 2)
    assert r1.returncode == 0, r1.stderr
    assert r1.stdout.strip() == ""
