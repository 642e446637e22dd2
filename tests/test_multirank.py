"""The benchmark's multi-rank bookkeeping on CPU (gloo, world size 2).

The decode path has no exchange step, so N GPUs run N independent replicas;
the only collectives are the timing reductions: the max of the ranks' elapsed
times and the sum of their bytes.  The reference arm prints from rank 0 only.
"""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    bench.init_dist(world, "gloo")
    t = bench.max_over_ranks(1.5 + rank, world, "cpu")
    b = bench.sum_over_ranks(1000.0 * (rank + 1), world, "cpu")
    bench.barrier(world)
    q.put((rank, t, b))
    dist.destroy_process_group()


def test_timing_reductions_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    assert [r[1] for r in res] == [2.5, 2.5]        # max over ranks
    assert [r[2] for r in res] == [3000.0, 3000.0]  # total bytes of all replicas


def test_reference_arm_prints_only_on_rank_zero(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""
