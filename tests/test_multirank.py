"""Two-rank (gloo, CPU) test of the benchmark's multi-process plumbing: rank
set-up from the launcher's environment, the barrier, the max-over-ranks timing
and the whole-job aggregate.  The forward shards by (sequence, head) with no
exchange, so ranks run independent replicas and no collective touches the
data path."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    r, w, local = bench.dist_init()
    try:
        bench.barrier(w)
        ms_local = 10.0 + 5.0 * r            # rank 1 is the slow one
        ms = bench.max_over_ranks(ms_local, w)
        value = bench.whole_job_value(1000, ms, w)
        q.put((r, w, ms, value))
    finally:
        import torch.distributed as dist
        dist.destroy_process_group()


@pytest.mark.skipif(not torch.distributed.is_available(), reason="torch.distributed missing")
def test_two_rank_timing_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p_ in procs:
        p_.start()
    for p_ in procs:
        p_.join(120)
        assert p_.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, w, ms, value in res:
        assert w == 2
        assert ms == pytest.approx(15.0)          # max over ranks
        assert value == pytest.approx(2 * 1000 / 15e-3)
