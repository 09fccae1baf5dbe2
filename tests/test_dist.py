"""The N > 1 plumbing of the benchmark on CPU (gloo, world size 2): ranks
join, meet at the timing barrier, agree on the slowest rank's time, turn it
into the whole job's µs per token, and only rank 0 runs the reference arm.
The path itself does not shard (replicas only): no data-path collective is
involved."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    try:
        w, r, local = bench.dist_init("gloo")
        assert (w, r, local) == (ws, rank, rank)
        bench.barrier(w)
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, w)  # rank 1 took longer
        us = bench.whole_job_us_per_token(slowest, steps=5, T=1, ws=w)

        class Args:
            config, warmup, steps, gpus = 1, 0, 1, ws
        ran = bench.run_reference(Args, w, r) if r != 0 else None  # returns at once on rank != 0
        bench.barrier(w)
        q.put((rank, slowest, us, ran))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_agree_on_the_slowest_time():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(ws))
    for rank, slowest, us, ran in res:
        assert slowest == 15.0  # the max over both ranks
        assert us == pytest.approx(15.0 / 5 * 1e3 / 2)  # 2 replicas x 1 token per step
        assert ran is None
