"""The bench's multi-rank plumbing on CPU: two gloo ranks (replicas only, no data-path
collective), barrier, max over ranks, and the whole-job aggregate."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    r, n, local = bench.dist_init(ws)
    bench.barrier(n)
    ms = 10.0 * (r + 1)  # rank 1 is the slower replica
    mx = bench.allmax(ms, n)
    v = bench.aggregate_tokens_per_s(2065, n, ms)
    bench.barrier(n)
    q.put((r, n, mx, v))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = sorted(q.get(timeout=100) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, n, mx, v in got:
        assert n == 2
        assert mx == 20.0  # every rank sees the slowest rank's time
        assert v == pytest.approx(2065 * 2 / 0.020)  # all tokens over the max time
