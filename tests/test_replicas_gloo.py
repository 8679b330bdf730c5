"""The N > 1 path of bench.py on CPU (gloo, world size 2): every rank's
time goes into a max-over-ranks all-reduce and the whole-job throughput
counts the work of all ranks (replicas of the step, no data-path
collective); the reference arm prints from rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                                         world_size=world)
    torch.distributed.barrier()
    ms = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
    value = bench.whole_job_tflops(1e12, world, ms)
    out.put((rank, ms, value))
    torch.distributed.barrier()
    torch.distributed.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [3.0, 5.0]
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in res:
        assert ms == 5.0                                  # the slowest replica sets the time
        assert value == pytest.approx(2 * 1e12 / 5e-3 / 1e12)  # both ranks' work counted


def test_reference_arm_prints_from_rank_0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
