"""Seeded synthetic layers materialised on the GPU through the library's packing API.

Weight codes are drawn on the device with the same counter-based stream as
gen.expert_codes (bit-identical), then handed to moe_pack_router / moe_pack_expert.
Float tensors (router weights and bias, row scales, hidden states) are drawn on the host
and uploaded.  Nothing here computes any part of the MoE layer.
"""
from __future__ import annotations

import numpy as np

from . import inputs as G


def config_for(s: G.LayerSpec):
    import routed_expert_ffn_route_gb300 as moe
    return moe.make_config(s.hidden, s.inter, s.n_experts, s.top_k, router=s.router,
                           n_shared=s.n_shared, inter_shared=s.inter_shared, n_group=s.n_group,
                           topk_group=s.topk_group, norm_topk=s.norm_topk,
                           routed_scaling_factor=s.rsf, weight_bits=s.weight_bits,
                           act_q8_0=s.act_q8_0, expert_top_p=s.top_p)


def build_packed_layer(s: G.LayerSpec, seed: int, layer: int = 0, device="cuda", bias=None,
                       packed=None, host_codes=False):
    """Pack the seeded layer (router + all experts + shared) into a device buffer.

    bias: optional host fp32 [E] overriding the spec's N(0, bias_std) bias.
    host_codes: draw the weight codes on the host (numpy) and upload them, instead of
    drawing them on the device (same values; a few copies instead of many small device
    kernels, for small layers).
    Returns (cfg, packed uint8 tensor)."""
    import torch
    import routed_expert_ffn_route_gb300 as moe
    cfg = config_for(s)
    nbytes = moe.moe_packed_bytes(cfg)
    if nbytes == 0:
        raise ValueError(f"unsupported layer spec {s}")
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=device)
    wr = torch.from_numpy(G.router_weights(s, seed, layer)).to(device)
    b = bias if bias is not None else G.router_bias(s, seed, layer)
    bt = None if b is None else torch.from_numpy(np.ascontiguousarray(b, np.float32)).to(device)
    moe.moe_pack_router(cfg, wr, bt, packed)
    bufs = {}
    for e in range(s.n_experts + s.n_shared):
        mats = {}
        for which in ("gate", "up", "down"):
            rows, cols = G.expert_rows_cols(s, which, shared=(e >= s.n_experts))
            key = (which, rows, cols)
            if host_codes:
                mats[which] = torch.from_numpy(
                    np.ascontiguousarray(G.expert_codes(s, seed, layer, e, which))).to(device)
                continue
            if key not in bufs:
                bufs[key] = torch.empty((rows, cols), dtype=torch.int8, device=device)
            mats[which] = G.expert_codes_torch(s, seed, layer, e, which, device, out=bufs[key])
        sc = [torch.from_numpy(G.expert_scales(s, seed, layer, e, w)).to(device)
              for w in ("gate", "up", "down")]
        moe.moe_pack_expert(cfg, e, mats["gate"], mats["up"], mats["down"], *sc, packed)
    torch.cuda.current_stream().synchronize()
    return cfg, packed


def hidden_to_device(s: G.LayerSpec, x_f32: np.ndarray, bits, device="cuda"):
    """Upload hidden states in the spec's dtype (bf16 from the exact bit patterns)."""
    import torch
    if s.x_dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
            torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(x_f32, np.float32)).to(device)
