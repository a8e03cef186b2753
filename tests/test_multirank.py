"""The benchmark's multi-rank bookkeeping on the CPU: two gloo ranks (one
process each, rendezvous on 127.0.0.1) reduce their timings to the maximum
over ranks, and the whole-job figure counts every rank's bytes against the
slowest rank's time.  Under torchrun the reference arm runs on rank 0 only;
the other ranks exit 0 without output."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, queue):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took 10 + r ms for the timed steps and 100 - r ms end to end
        got = bench.max_over_ranks([10.0 + rank, 100.0 - rank], world, "cpu")
        queue.put((rank, got, bench.whole_job_gbs(1e9, world, got[0])))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        results = sorted(queue.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, got, gbs in results:
        assert got == [11.0, 100.0], (rank, got)
        # 2 ranks x 1 GB in the slowest rank's 11 ms
        assert gbs == pytest.approx(2e9 / 11e-3 / 1e9)


def test_whole_job_value_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job_gbs(5e8, 1, 1.0) == pytest.approx(500.0)
    assert bench.whole_job_gbs(5e8, 4, 1.0) == pytest.approx(2000.0)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
