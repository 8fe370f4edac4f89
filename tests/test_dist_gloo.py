"""The multi-process side of bench.py on CPU: two ranks with the gloo backend
(127.0.0.1), as torchrun starts them on one node. Each rank runs its own
replica of the workload; the timing is the maximum over ranks and the value
counts the units of all ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    d = bench.Dist("gloo")
    try:
        d.barrier()
        local_ms = 10.0 + 5.0 * rank  # a slower rank sets the step time
        el = d.max(local_ms)
        q.put((rank, d.world, el, bench.dist_env()))
    finally:
        d.close()


def test_two_gloo_ranks_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got.sort()
    assert [g[0] for g in got] == [0, 1]
    for rank, world, el, env in got:
        assert world == 2 and el == pytest.approx(15.0)
        assert env == (2, rank, rank)


def test_single_process_needs_no_process_group(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    d = bench.Dist("gloo")
    assert d.pg is None and d.max(3.5) == 3.5
    d.barrier()
    d.close()
