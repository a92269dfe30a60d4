"""The benchmark's multi-rank logic on CPU with two gloo ranks: the step time
is the slowest rank's, the job's rate counts every rank's tokens, and the
reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(1.0 + rank * 2.5, dist)
    val = bench.whole_job_tokens_per_s(2048, world, ms)
    dist.barrier()
    q.put((rank, ms, val))
    dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, val in out:
        assert ms == pytest.approx(3.5)            # the slowest rank's time on every rank
        assert val == pytest.approx(2 * 2048 / 3.5e-3)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import argparse
    import bench
    args = argparse.Namespace(workload="decode_dispatch_combine", seed=0, warmup=0, steps=1)
    bench.run_reference(args, rank=1, world=2)
    assert capsys.readouterr().out == ""
