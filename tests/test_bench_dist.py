"""The multi-replica path of bench.py on CPU: two gloo ranks agree on the
slowest rank's timings and the whole-job bandwidth counts every replica's
bytes (the decode shards by (sequence, KV head) with no exchange, so the
ranks are independent replicas)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    ms, e2e = bench.slowest_rank(dist, [0.10 + 0.05 * rank, 0.30 - 0.1 * rank], "cpu")
    dist.barrier()
    q.put((r, w, local, ms, e2e, bench.whole_job_gbs(w, 1e9, ms)))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, w, local, ms, e2e, gbs) in enumerate(out):
        assert (r, w, local) == (rank, 2, rank)
        assert ms == pytest.approx(0.15) and e2e == pytest.approx(0.30)
        assert gbs == pytest.approx(2 * 1e9 / 0.15e-3 / 1e9)


def test_single_process_is_identity():
    assert bench.slowest_rank(None, [1.0, 2.0], "cpu") == [1.0, 2.0]
    assert bench.whole_job_gbs(1, 5e8, 1.0) == pytest.approx(500.0)
