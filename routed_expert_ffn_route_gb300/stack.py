"""A stack of MoE layers through the C ABI ("colibrì 深度拆解" §4.3: a layer's merged output
feeds the next layer).

The stacking arithmetic is the library's reading (the pages leave it open): the stack
keeps an fp32 residual stream r; r_0 = x (the bf16 input), layer l runs on
bf16(RMSNorm(r_l)) and r_{l+1} = r_l + MoE_l(...).  Every step runs in the library's
kernels (`moe_layer_forward_next`, whose combine warms the next layer's router weights into
L2, then `moe_residual_rmsnorm`); this module only owns the buffers and issues the calls, so
a whole prefill or decode step can be captured in one CUDA graph.
"""
from __future__ import annotations

import torch

from . import (moe_layer_forward, moe_layer_forward_next, moe_read_status, moe_residual_rmsnorm,
               moe_workspace_bytes, MOE_OK, MoEError)


class Stack:
    """Layers (cfg, packed) applied in order to T <= t_max tokens, all on the current device."""

    def __init__(self, layers, t_max: int, eps: float = 1e-6):
        if not layers:
            raise ValueError("empty stack")
        self.layers = list(layers)
        cfg0 = self.layers[0][0]
        self.H, self.k = cfg0.hidden, cfg0.top_k
        for cfg, _ in self.layers:
            if cfg.hidden != self.H or cfg.top_k != self.k:
                raise ValueError("stacked layers must share hidden size and top_k")
        self.t_max, self.eps = t_max, eps
        dev = "cuda"
        self.ws = torch.zeros(max(moe_workspace_bytes(c, t_max) for c, _ in self.layers),
                              dtype=torch.uint8, device=dev)
        self.resid = torch.empty((t_max, self.H), dtype=torch.float32, device=dev)
        self.x = torch.empty((t_max, self.H), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((t_max, self.H), dtype=torch.float32, device=dev)
        self.ids = [torch.empty((t_max, self.k), dtype=torch.int32, device=dev) for _ in layers]
        self.w = [torch.empty((t_max, self.k), dtype=torch.float32, device=dev) for _ in layers]

    def forward(self, x0):
        """x0: bf16 [T, H] on the device.  Returns the residual stream
        after the last layer (fp32 [T, H], a view of the stack's buffer); the per-layer
        routing stays in self.ids[l][:T], self.w[l][:T]."""
        T = x0.shape[0]
        if T > self.t_max or x0.shape[1] != self.H:
            raise ValueError("x0 does not fit the stack")
        r, x, out = self.resid[:T], self.x[:T], self.out[:T]
        moe_residual_rmsnorm(r, None, x, x0=x0, eps=self.eps)
        for l, (cfg, packed) in enumerate(self.layers):
            if l + 1 < len(self.layers):  # the combine warms the next layer's router into L2
                ncfg, npacked = self.layers[l + 1]
                moe_layer_forward_next(cfg, packed, x, out, self.ids[l][:T], self.w[l][:T],
                                       self.ws, ncfg, npacked)
            else:
                moe_layer_forward(cfg, packed, x, out, self.ids[l][:T], self.w[l][:T], self.ws)
            moe_residual_rmsnorm(r, out, x, eps=self.eps)
        return r

    def status(self):
        st = moe_read_status(self.ws)
        if st != MOE_OK:
            raise MoEError(st, "stack forward")
