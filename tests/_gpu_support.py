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
