"""Multi-rank paths on CPU with two gloo ranks: the bench's replica plumbing (no data-path
collective; barrier, max over ranks, whole-job aggregate), and the expert-parallel split
of the layer (whole experts per rank, one sum all-reduce), checked on the oracle."""
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


def _ep_rank(rank, ws, port, q):
    """One rank of an expert-parallel split of the oracle layer: the router is replicated,
    the rank evaluates only the routed experts it owns (and rank 0 the shared expert), and
    one sum all-reduce of the fp64 partial outputs gives the layer."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import numpy as np
    import torch
    import torch.distributed as dist

    import gen
    import oracle
    from _support import make_experts, shared_expert
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    s = gen.LayerSpec("ep", hidden=256, inter=128, n_experts=16, top_k=4,
                      router="sigmoid_grouped", n_shared=1, n_group=4, topk_group=2, rsf=2.5,
                      bias_std=0.1, x_dtype="f32")
    seed, T = 5, 12
    wr, bias = gen.router_weights(s, seed), gen.router_bias(s, seed)
    x, _ = gen.hidden_states(s, seed, 0, T)
    x64 = x.astype(np.float64)
    ids, w, _ = oracle.route(s, oracle.router_logits(s, x64, wr), bias)
    owner = (np.arange(s.n_experts) * ws) // s.n_experts  # contiguous halves
    mine = np.nonzero(owner == rank)[0]
    ids_r = np.where(owner[ids] == rank, ids, -1).astype(np.int32)
    s_r = s if rank == 0 else s.replace(n_shared=0)
    part = oracle.layer_experts(s_r, x64, ids_r, w, make_experts(s, seed, 0, mine),
                                shared_expert(s_r, seed, 0))
    t = torch.from_numpy(part.copy())
    dist.all_reduce(t)
    full = oracle.layer_experts(s, x64, ids, w, make_experts(s, seed, 0), shared_expert(s, seed, 0))
    q.put((rank, int(np.count_nonzero(ids_r >= 0)), t.numpy(), full))
    dist.destroy_process_group()


@pytest.mark.timeout(180)
def test_expert_parallel_split_of_the_oracle_sums_to_the_layer():
    """Whole experts per rank plus one sum all-reduce reproduce the layer: the sharding a
    multi-GPU layer would use, checked on the oracle with two gloo ranks."""
    sys.path.insert(0, ROOT)
    import numpy as np

    import oracle
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_ep_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = sorted((q.get(timeout=150) for _ in ps), key=lambda g: g[0])
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, n0, sum0, full), (_, n1, sum1, _) = got
    assert n0 > 0 and n1 > 0 and n0 + n1 == 12 * 4  # both ranks own selected experts
    np.testing.assert_array_equal(sum0, sum1)      # every rank holds the same sum
    scale = np.sqrt(np.mean(full ** 2))
    np.testing.assert_allclose(sum0, full, rtol=0, atol=1e-12 * scale)
