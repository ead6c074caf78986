"""GPU-side helpers of the parity tests: a packed seeded layer and oracle references."""
from __future__ import annotations

import numpy as np
import torch

import gen
import oracle
import routed_expert_ffn_route_gb300 as moe
from gen.device import build_packed_layer, hidden_to_device
from _support import filtered_hidden, make_experts, shared_expert

_LAYER_CACHE = {}


class GpuLayer:
    """A seeded layer packed on cuda:0 plus a workspace sized for T tokens."""

    def __init__(self, spec, seed=0, layer=0, bias=None):
        self.spec, self.seed, self.layer = spec, seed, layer
        self.cfg, self.packed = build_packed_layer(spec, seed, layer, "cuda", bias=bias)
        self.wr = gen.router_weights(spec, seed, layer)
        self.bias = bias if bias is not None else gen.router_bias(spec, seed, layer)
        self._ws = {}

    def ws(self, T):
        if T not in self._ws:
            n = moe.moe_workspace_bytes(self.cfg, T)
            self._ws = {T: torch.zeros(n, dtype=torch.uint8, device="cuda")}
        return self._ws[T]

    def forward(self, x_dev):
        T = x_dev.shape[0]
        k, H = self.spec.top_k, self.spec.hidden
        out = torch.empty((T, H), dtype=torch.float32, device="cuda")
        ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        ws = self.ws(T)
        moe.moe_layer_forward(self.cfg, self.packed, x_dev, out, ids, w, ws)
        st = moe.moe_read_status(ws)
        assert st == moe.MOE_OK, moe.moe_status_str(st)
        return out, ids, w

    def route(self, x_dev):
        T = x_dev.shape[0]
        k = self.spec.top_k
        ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        ws = self.ws(T)
        moe.moe_route_topk(self.cfg, self.packed, x_dev, ids, w, ws)
        assert moe.moe_read_status(ws) == moe.MOE_OK
        return ids, w

    def permutation(self, T):
        off = torch.empty(self.spec.n_experts + 1, dtype=torch.int32, device="cuda")
        perm = torch.empty(T * self.spec.top_k, dtype=torch.int32, device="cuda")
        moe.moe_debug_permutation(self.cfg, self.ws(T), T, off, perm)
        torch.cuda.synchronize()
        return off.cpu().numpy(), perm.cpu().numpy()


def get_layer(spec, seed=0, layer=0) -> GpuLayer:
    key = (spec, seed, layer)
    if key not in _LAYER_CACHE:
        _LAYER_CACHE.clear()  # keep one big layer resident at a time
        torch.cuda.empty_cache()
        _LAYER_CACHE[key] = GpuLayer(spec, seed, layer)
    return _LAYER_CACHE[key]


def inputs(spec, L: GpuLayer, batch, T):
    """Margin-filtered hidden states (host fp32, device tensor) and the oracle routing."""
    x, bits, ids, w, margin, redraws = filtered_hidden(spec, L.seed, batch, T, L.wr, L.bias)
    return x, hidden_to_device(spec, x, bits), ids, w, margin, redraws


def oracle_out(spec, L: GpuLayer, x, ids, w, tokens=None):
    """fp64 oracle output for the given tokens (all when None), routed by (ids, w)."""
    tok = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
    need = sorted(set(int(e) for e in ids[tok].ravel()))
    experts = make_experts(spec, L.seed, L.layer, need)
    sh = shared_expert(spec, L.seed, L.layer)
    return oracle.layer_experts(spec, x[tok].astype(np.float64), ids[tok], w[tok], experts, sh,
                                mode=1)


def make_experts_fast(spec, seed, layer, which) -> dict:
    """As _support.make_experts, with the codes drawn by the generator's device variant
    (the same counter-based stream, bit-identical to the host one; see test_gen) and copied
    to the host: the GPU tests build many large experts for the oracle."""
    from _support import make_expert  # noqa: F401 (same fields)
    out = {}
    for e in which:
        e = int(e)
        codes = {w: gen.expert_codes_torch(spec, seed, layer, e, w, "cuda").cpu().numpy()
                 for w in ("gate", "up", "down")}
        out[e] = oracle.Expert(gate=codes["gate"], up=codes["up"], down=codes["down"],
                               s_gate=gen.expert_scales(spec, seed, layer, e, "gate"),
                               s_up=gen.expert_scales(spec, seed, layer, e, "up"),
                               s_down=gen.expert_scales(spec, seed, layer, e, "down"))
    return out


def _masked(ids, keep):
    """ids with every slot whose expert is not in `keep` dropped (id -1)."""
    return np.where(np.isin(ids, list(keep)), ids, -1).astype(np.int32)


def oracle_out_many(spec, L: GpuLayer, x, ids, w, tokens, chunk=32, threads=None,
                    in_flight=24):
    """fp64 oracle output for many tokens of a large layer, in bounded host memory.

    The layer output is a sum over slots (out[t] = shared(x_t) + sum_j w[t][j] y_j), so it
    is computed as independent partial layers that the oracle evaluates, each on a chunk of
    at most `chunk` tokens: one routed expert at a time (the token's other slots dropped,
    id -1, no shared expert), plus the shared expert alone.  The partials run in a thread
    pool (the oracle releases the interpreter while it computes) and are summed in fp64;
    experts are drawn (on the device, bit-identical to the host stream) as they are
    needed, at most `in_flight` at a time."""
    import concurrent.futures as cf
    import os
    tok = np.asarray(tokens)
    x64 = x[tok].astype(np.float64)
    ids_t, w_t = ids[tok], w[tok]
    out = np.zeros((len(tok), spec.hidden), dtype=np.float64)
    threads = threads or max(1, min(16, os.cpu_count() or 1))
    routed_only = spec.replace(n_shared=0)

    def run(sp, rows, ids_m, ex, sh):
        return rows, oracle.layer_experts(sp, x64[rows], ids_m, w_t[rows], ex, sh, mode=1)

    with cf.ThreadPoolExecutor(threads) as pool:
        pending = []

        def drain(limit):
            while len(pending) > limit:
                rows, part = pending.pop(0).result()
                out[rows] += part

        if spec.n_shared:
            sh = make_experts_fast(spec, L.seed, L.layer, [spec.n_experts])[spec.n_experts]
            none = np.full_like(ids_t, -1)
            for s0 in range(0, len(tok), chunk):
                rows = np.arange(s0, min(len(tok), s0 + chunk))
                pending.append(pool.submit(run, spec, rows, none[rows], {}, sh))
        for e in sorted(set(int(v) for v in ids_t.ravel() if v >= 0)):
            ex = make_experts_fast(spec, L.seed, L.layer, [e])
            users = np.nonzero((ids_t == e).any(1))[0]
            for s0 in range(0, len(users), chunk):
                rows = users[s0:s0 + chunk]
                pending.append(pool.submit(run, routed_only, rows, _masked(ids_t[rows], {e}),
                                           ex, None))
            drain(in_flight)
        drain(0)
    return out


def prefill_sample(ids, n_experts, busiest=3, spread=32):
    """Tokens whose outputs a full-size prefill check compares: every token routed to the
    `busiest` most-loaded experts (each of their groups, so every m-tile of a group and
    both groups of an expert split in two), plus `spread` tokens evenly over the batch
    (one in every group of the shared expert)."""
    T = ids.shape[0]
    load = np.bincount(ids[ids >= 0].ravel(), minlength=n_experts)
    top = np.argsort(-load, kind="stable")[:busiest]
    users = np.nonzero(np.isin(ids, top).any(1))[0]
    even = np.unique(np.linspace(0, T - 1, spread).round().astype(int))
    return np.union1d(users, even), top, load[top]
