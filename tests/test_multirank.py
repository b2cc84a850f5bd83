"""The N > 1 host logic of bench.py on CPU: two `gloo` ranks, each a replica,
agree on the max-over-ranks time and the rank/world parsing.  No GPU."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    r, w, local = bench.dist_env()
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    mx = bench.reduce_max(10.0 + rank * 5.0, w)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    out.put((r, w, local, mx))


@pytest.mark.timeout(120)
def test_two_gloo_ranks_reduce_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert res == [(0, 2, 0, 15.0), (1, 2, 1, 15.0)]


def test_single_rank_defaults(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.reduce_max(3.5, 1) == 3.5
    args = bench.parse_args([])
    assert args.gpus == 1 and args.warmup >= 3 and args.impl == "own"
