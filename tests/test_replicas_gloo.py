"""Multi-rank host logic of the benchmark (replicas: every rank runs the same workload, no exchange).

Two gloo ranks on the CPU stand in for two GPUs: the step time is the slowest rank's, the job
throughput counts every rank's work over that time, and the reference arm (the CPU oracle) runs on
rank 0 only while the other ranks leave at once.
"""
import io
import multiprocessing as mp
import os
import socket
import sys
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, rank_ms, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        ms, tflops = bench.job_tflops(world, 2.0e9, rank_ms[rank], device="cpu")
        out.put((rank, ms, tflops))
    finally:
        dist.destroy_process_group()


def test_job_throughput_uses_the_slowest_rank():
    world, port = 2, _free_port()
    rank_ms = [1.0, 4.0]
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, rank_ms, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, tflops in res:
        assert ms == 4.0   # max over ranks, the same on every rank
        # 2 ranks x 2 GFLOP in 4 ms
        assert abs(tflops - 2 * 2.0e9 / 4.0e-3 / 1e12) < 1e-12


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    ms, tflops = bench.job_tflops(1, 3.0e9, 2.0, device="cpu")
    assert ms == 2.0 and abs(tflops - 1.5) < 1e-12


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"])
    assert rc == 0 and buf.getvalue() == ""
