"""Expert-parallel shares of the layer on the GPU (moe_layer_forward_experts).

The pages place whole experts on devices and never split one ("Show HN: 如何在我的低配置电脑上
运行 GLM-5.2", 实验性常驻 CUDA 后端); the per-device results are added.  Here each share
(a range of routed experts, the shared expert on one share only) runs through the C ABI on
the one GPU, and:
  - every share's partial output matches the oracle's partial layer (the token's slots of
    other experts dropped, the shared expert on or off) within the parity tolerance, taken
    on the scale of the whole layer's output (a share is a part of that output: max|err|
    <= 2e-3 RMS(layer), ||err||_F <= 1e-3 ||layer||_F);
  - the partials of disjoint shares covering all experts add up to moe_layer_forward;
  - two processes (gloo, world size 2), each computing its share on the GPU, sum their
    partials with one all-reduce and get the layer.
The partial forwards do not wait on each other, so running the two ranks on one GPU is
only a way to exercise the exchange, not a stand-in for two GPUs' timing.
"""
import os

import numpy as np
import pytest
import torch

import gen
import routed_expert_ffn_route_gb300 as moe
from _gpu_support import GpuLayer, get_layer, inputs, oracle_out, oracle_out_many
from _support import FROB_REL, MAX_REL_RMS, err_stats

pytestmark = pytest.mark.gpu

SMALL = gen.LayerSpec("ep_small", hidden=512, inter=384, n_experts=16, top_k=4,
                      router="sigmoid_grouped", n_shared=1, inter_shared=256, n_group=4,
                      topk_group=2, rsf=2.5, bias_std=0.1)


def share_forward(L, xd, b, e, sh):
    T = xd.shape[0]
    s = L.spec
    out = torch.full((T, s.hidden), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, s.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, s.top_k), dtype=torch.float32, device="cuda")
    ws = L.ws(T)
    moe.moe_layer_forward_experts(L.cfg, L.packed, xd, b, e, sh, out, ids, w, ws)
    st = moe.moe_read_status(ws)
    assert st == moe.MOE_OK, moe.moe_status_str(st)
    return out, ids, w


def oracle_share(L, x, ids, w, b, e, sh, tokens):
    """The oracle's partial layer: slots of experts outside [b, e) dropped (id -1), the
    shared expert only when sh."""
    spec = L.spec if sh else L.spec.replace(n_shared=0)
    keep = np.where((ids >= b) & (ids < e), ids, -1).astype(np.int32)
    if not (keep >= 0).any() and not sh:
        return np.zeros((len(tokens), L.spec.hidden))
    many = len(tokens) * (spec.top_k + 1) * spec.hidden * spec.inter > 4e9
    return (oracle_out_many(spec, L, x, keep, w, tokens) if many
            else oracle_out(spec, L, x, keep, w, tokens))


def share_close(got, ref, layer, what):
    """A share's error on the scale of the whole layer's output."""
    d = got.astype(np.float64) - ref
    rms = np.sqrt(np.mean(layer * layer))
    mx, fr = float(np.abs(d).max() / rms), float(np.linalg.norm(d) / np.linalg.norm(layer))
    print(f"{what}: max|err|/RMS(layer) = {mx:.2e}, |err|_F/|layer|_F = {fr:.2e}")
    assert mx <= MAX_REL_RMS and fr <= FROB_REL


def shares(E, n):
    cut = [round(i * E / n) for i in range(n + 1)]
    return [(cut[i], cut[i + 1], 1 if i == 0 else 0) for i in range(n)]


@pytest.mark.parametrize("T", [5, 37])
@pytest.mark.parametrize("n", [2, 4])
def test_shares_match_oracle_and_sum_to_layer(T, n):
    # T = 5: the fused decode front and register-MMA kernels; T = 37: the separate launches
    L = get_layer(SMALL, 7)
    x, xd, ids_o, w_o, *_ = inputs(SMALL, L, 0, T)
    full, _, _ = L.forward(xd)
    layer = oracle_out(SMALL, L, x, ids_o, w_o)
    total = torch.zeros_like(full)
    for b, e, sh in shares(SMALL.n_experts, n):
        out, ids, w = share_forward(L, xd, b, e, sh)
        assert np.array_equal(ids.cpu().numpy(), ids_o)  # the routing is always complete
        ref = oracle_share(L, x, ids_o, w_o, b, e, sh, np.arange(T))
        got = out.cpu().numpy()
        if np.abs(ref).max() == 0:
            assert np.array_equal(got, ref)
        else:
            share_close(got, ref, layer, f"T={T} share [{b},{e}) shared={sh}")
        total += out
    mx, fr = err_stats(total.cpu().numpy(), full.cpu().numpy())
    print(f"T={T}, {n} shares summed vs the layer: {mx:.2e} / {fr:.2e}")
    assert mx <= 1e-5 and fr <= 1e-6  # the same products; only fp32 additions reordered


def test_empty_share_is_the_shared_expert_or_zero():
    L = get_layer(SMALL, 7)
    x, xd, ids_o, w_o, *_ = inputs(SMALL, L, 1, 9)
    out, _, _ = share_forward(L, xd, 6, 6, 0)
    assert torch.equal(out, torch.zeros_like(out))
    out, _, _ = share_forward(L, xd, 6, 6, 1)
    ref = oracle_share(L, x, ids_o, w_o, 6, 6, 1, np.arange(9))
    share_close(out.cpu().numpy(), ref, oracle_out(SMALL, L, x, ids_o, w_o), "shared expert alone")


@pytest.mark.parametrize("T", [16, 2048])
def test_full_size_two_shares(T):
    s = gen.spec("dsv3")
    L = get_layer(s)
    x, xd, ids_o, w_o, *_ = inputs(s, L, 2, T)
    full, _, _ = L.forward(xd)
    parts = [share_forward(L, xd, b, e, sh)[0] for b, e, sh in shares(s.n_experts, 2)]
    mx, fr = err_stats((parts[0] + parts[1]).cpu().numpy(), full.cpu().numpy())
    print(f"dsv3 T={T}: two shares summed vs the layer: {mx:.2e} / {fr:.2e}")
    assert mx <= 1e-5 and fr <= 1e-6
    tok = np.arange(T) if T <= 16 else np.unique(np.linspace(0, T - 1, 8).round().astype(int))
    refs = [oracle_share(L, x, ids_o, w_o, b, e, sh, tok) for b, e, sh in shares(s.n_experts, 2)]
    layer = refs[0] + refs[1]
    for (b, e, sh), p, ref in zip(shares(s.n_experts, 2), parts, refs):
        share_close(p.cpu().numpy()[tok], ref, layer, f"dsv3 T={T} share [{b},{e}) shared={sh}")


def test_split_down_shares_sum_to_layer():
    """At T = 1 the Mixtral-shaped layer's down launch splits each work item's contraction;
    two expert shares, each with its own split launch and planes, still add up to the
    layer."""
    s = gen.LayerSpec("ep_mix_split", hidden=1024, inter=2048, n_experts=8, top_k=2,
                      router="softmax")
    L = get_layer(s, 3)
    x, xd, ids_o, w_o, *_ = inputs(s, L, 4, 1)
    full, _, _ = L.forward(xd)
    parts = [share_forward(L, xd, b, e, 0)[0] for b, e, _ in shares(s.n_experts, 2)]
    mx, fr = err_stats((parts[0] + parts[1]).cpu().numpy(), full.cpu().numpy())
    print(f"mix_split T=1: two shares summed vs the layer: {mx:.2e} / {fr:.2e}")
    assert mx <= 1e-5 and fr <= 1e-6
    layer = oracle_out(s, L, x, ids_o, w_o)
    for (b, e, _), p in zip(shares(s.n_experts, 2), parts):
        share_close(p.cpu().numpy(), oracle_share(L, x, ids_o, w_o, b, e, 0, np.arange(1)),
                    layer, f"mix_split T=1 share [{b},{e})")


def _rank(rank, world, port, T, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        L = GpuLayer(SMALL, 7)
        _, xd, *_ = inputs(SMALL, L, 3, T)
        b, e, sh = shares(SMALL.n_experts, world)[rank]
        part, _, _ = share_forward(L, xd, b, e, sh)
        buf = part.cpu()
        dist.all_reduce(buf, op=dist.ReduceOp.SUM)
        if rank == 0:
            full, _, _ = L.forward(xd)
            q.put(err_stats(buf.numpy(), full.cpu().numpy()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_all_reduce_their_shares():
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, 21, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    mx, fr = q.get(timeout=5)
    print(f"two ranks, all-reduced shares vs the layer: {mx:.2e} / {fr:.2e}")
    assert mx <= 1e-5 and fr <= 1e-6
