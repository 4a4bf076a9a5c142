"""Multi-process host logic of bench.py on CPU (gloo, 2 ranks): environment
parsing, the barrier and the max over ranks that the timing uses.  Rows are
independent, so the benchmark's ranks are replicas with no data-path
collective; this is the only cross-rank step."""
import os
import socket

import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    got = bench.reduce_max(10.0 + rank * 2.5, dist)
    out.put((rank, got))
    dist.destroy_process_group()


def test_two_rank_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 12.5, 1: 12.5}


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max(3.25, None) == 3.25
    bench.barrier(None)
