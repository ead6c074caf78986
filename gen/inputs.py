"""Counter-based seeded generator for synthetic MoE-layer inputs.

Every value is a pure function of (seed, tensor tag, sub-stream, element index),
so any slice of any tensor can be regenerated independently, on the host with
numpy or on the device with torch, with identical integer results.

The mixing function is Chris Wellons' "lowbias32" 32-bit integer hash
(published in his hash-prospector project):
    x ^= x >> 16; x *= 0x7feb352d; x ^= x >> 15; x *= 0x846ca68b; x ^= x >> 16
An element's 32-bit draw is  h = lowbias32(lowbias32(idx ^ key) + key)  with
key = the sub-stream key derived from (seed, tag, sub).

Weight codes (int8 containers) come from h with integer arithmetic only, so
the numpy and torch versions agree bit for bit.  Floating-point tensors
(hidden states, router weights and bias, row scales) are produced on the host
only (numpy float64 then rounded), so no device math library enters them.

Distributions follow the workloads: codes uniform over the int4 range [-8,7],
the int8 range [-127,127] or the int2 range [-2,1]; row scales U[0.005,0.02];
router weights N(0, 0.02); router bias N(0, 0.1) for the grouped router;
hidden states N(0,1) in fp32 or rounded to bf16.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = [
    "LayerSpec", "PRESETS", "spec", "TAG",
    "lowbias32_np", "draws_np", "draws_torch",
    "expert_codes", "expert_codes_torch", "expert_scales",
    "router_weights", "router_bias", "hidden_states", "bf16_round_bits",
    "expert_rows_cols", "zipf_bias", "zipf_rank",
]

M32 = 0xFFFFFFFF

# tensor tags of the sub-streams
TAG = {
    "x": 1, "router_w": 2, "router_b": 3,
    "gate": 4, "up": 5, "down": 6,
    "s_gate": 7, "s_up": 8, "s_down": 9,
    "zipf_perm": 10, "misc": 11,
}


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    """Shape and routing parameters of one MoE layer."""
    name: str
    hidden: int            # H
    inter: int             # I, routed expert intermediate size
    n_experts: int         # E routed experts
    top_k: int             # k
    router: str            # "softmax" or "sigmoid_grouped"
    n_shared: int = 0      # 0 or 1 shared expert
    inter_shared: int = 0  # shared expert intermediate size (defaults to I)
    n_group: int = 1
    topk_group: int = 1
    norm_topk: int = 1
    rsf: float = 1.0       # routed_scaling_factor
    weight_bits: int = 4   # 4, 8 or 2
    act_q8_0: int = 0      # 1: Q8_0 int8 activations (needs weight_bits == 8)
    x_dtype: str = "bf16"  # "f32" or "bf16"
    bias_std: float = 0.0  # router bias N(0, bias_std); 0 = no bias
    top_p: float = 0.0     # adaptive expert top-p (0 = off; lossy, opt-in)

    @property
    def inter_sh(self) -> int:
        return self.inter_shared or self.inter

    def replace(self, **kw) -> "LayerSpec":
        return dataclasses.replace(self, **kw)


PRESETS = {
    # tiny softmax layer: H=256, I=128, E=16, top-2, fp32 hidden states
    "tiny": LayerSpec("tiny", 256, 128, 16, 2, "softmax", x_dtype="f32"),
    # Mixtral-shaped: H=4096, I=14336, E=8, top-2
    "mixtral": LayerSpec("mixtral", 4096, 14336, 8, 2, "softmax"),
    # DeepSeek-V3-style: H=6144, I=2048, E=256 + 1 shared, sigmoid grouped top-8
    "dsv3": LayerSpec("dsv3", 6144, 2048, 256, 8, "sigmoid_grouped", n_shared=1,
                      n_group=8, topk_group=4, rsf=2.5, bias_std=0.1),
    # same shapes, int8 weights + Q8_0 activations
    "dsv3_int8": LayerSpec("dsv3_int8", 6144, 2048, 256, 8, "sigmoid_grouped", n_shared=1,
                           n_group=8, topk_group=4, rsf=2.5, bias_std=0.1,
                           weight_bits=8, act_q8_0=1),
    # same shapes, packed int2 weights
    "dsv3_int2": LayerSpec("dsv3_int2", 6144, 2048, 256, 8, "sigmoid_grouped", n_shared=1,
                           n_group=8, topk_group=4, rsf=2.5, bias_std=0.1, weight_bits=2),
}


def spec(name: str, **kw) -> LayerSpec:
    s = PRESETS[name]
    return s.replace(**kw) if kw else s


# ---------------------------------------------------------------- hashing

def lowbias32_np(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.uint32, copy=True)
    x ^= x >> np.uint32(16)
    x *= np.uint32(0x7FEB352D)
    x ^= x >> np.uint32(15)
    x *= np.uint32(0x846CA68B)
    x ^= x >> np.uint32(16)
    return x


def _lowbias32_int(x: int) -> int:
    x &= M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & M32
    x ^= x >> 16
    return x


def stream_key(seed: int, tag: int, sub: int) -> int:
    k = _lowbias32_int(seed & M32)
    k = _lowbias32_int(k ^ (tag * 0x9E3779B9 & M32))
    k = _lowbias32_int(k ^ (sub & M32))
    k = _lowbias32_int(k ^ ((sub >> 32) & M32))
    return k


def draws_np(seed: int, tag: int, sub: int, start: int, count: int) -> np.ndarray:
    """uint32 draws for element indices [start, start+count) of one sub-stream."""
    key = np.uint32(stream_key(seed, tag, sub))
    idx = (np.arange(start, start + count, dtype=np.uint64) & M32).astype(np.uint32)
    h = lowbias32_np(idx ^ key)
    h = lowbias32_np(h + key)  # uint32 wrap-around add
    return h


def _mul32_t(x, c: int):
    """(x * c) mod 2^32 for int64 tensors holding values in [0, 2^32), without overflow."""
    c_lo, c_hi = c & 0xFFFF, c >> 16
    return (x * c_lo + (((x * c_hi) & 0xFFFF) << 16)) & M32


def _lowbias32_t(x):
    x = x ^ (x >> 16)
    x = _mul32_t(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32_t(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def draws_torch(seed: int, tag: int, sub: int, start: int, count: int, device):
    """Same draws as draws_np, as an int64 torch tensor on `device`."""
    import torch
    key = stream_key(seed, tag, sub)
    idx = torch.arange(start, start + count, dtype=torch.int64, device=device) & M32
    h = _lowbias32_t(idx ^ key)
    h = _lowbias32_t((h + key) & M32)
    return h


# ---------------------------------------------------------------- weight codes

def expert_rows_cols(s: LayerSpec, which: str, shared: bool = False):
    inter = s.inter_sh if shared else s.inter
    if which in ("gate", "up"):
        return inter, s.hidden
    if which == "down":
        return s.hidden, inter
    raise ValueError(which)


def _sub(layer: int, expert: int) -> int:
    return (layer << 20) | expert


def _codes_from_draws(h, bits: int, xp):
    if bits == 4:
        return (h >> 28) - 8
    if bits == 2:
        return (h >> 30) - 2
    if bits == 8:
        return (((h >> 8) * 255) >> 24) - 127
    raise ValueError(bits)


def expert_codes(s: LayerSpec, seed: int, layer: int, expert: int, which: str) -> np.ndarray:
    """int8 container [rows, cols] of one expert matrix (expert == E means the shared expert)."""
    rows, cols = expert_rows_cols(s, which, shared=(expert >= s.n_experts))
    h = draws_np(seed, TAG[which], _sub(layer, expert), 0, rows * cols).astype(np.int64)
    q = _codes_from_draws(h, s.weight_bits, np)
    return q.astype(np.int8).reshape(rows, cols)


def expert_codes_torch(s: LayerSpec, seed: int, layer: int, expert: int, which: str, device,
                       out=None):
    """Device copy of expert_codes (int8 torch tensor [rows, cols]); writes into `out` if given."""
    import torch
    rows, cols = expert_rows_cols(s, which, shared=(expert >= s.n_experts))
    n = rows * cols
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.int8, device=device)
    flat = out.view(-1)
    chunk = 1 << 24
    for st in range(0, n, chunk):
        c = min(chunk, n - st)
        h = draws_torch(seed, TAG[which], _sub(layer, expert), st, c, device)
        flat[st:st + c] = _codes_from_draws(h, s.weight_bits, torch).to(torch.int8)
    return out


def _uniform01(h: np.ndarray) -> np.ndarray:
    """(0,1) doubles from uint32 draws: ((h >> 8) + 0.5) / 2^24."""
    return ((h >> np.uint32(8)).astype(np.float64) + 0.5) * (1.0 / 16777216.0)


def _normal(seed, tag, sub, n) -> np.ndarray:
    """n N(0,1) doubles by Box-Muller on pairs of draws (host only)."""
    m = (n + 1) // 2
    h = draws_np(seed, tag, sub, 0, 2 * m)
    u1 = _uniform01(h[0::2])
    u2 = _uniform01(h[1::2])
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * math.pi * u2)
    z[1::2] = r * np.sin(2.0 * math.pi * u2)
    return z[:n]


def expert_scales(s: LayerSpec, seed: int, layer: int, expert: int, which: str) -> np.ndarray:
    """fp32 per-row scales U[0.005, 0.02] of one expert matrix (which in gate/up/down)."""
    rows, _ = expert_rows_cols(s, which, shared=(expert >= s.n_experts))
    h = draws_np(seed, TAG["s_" + which], _sub(layer, expert), 0, rows)
    return (0.005 + 0.015 * _uniform01(h)).astype(np.float32)


def router_weights(s: LayerSpec, seed: int, layer: int = 0) -> np.ndarray:
    """fp32 router weights [E, H] ~ N(0, 0.02)."""
    z = _normal(seed, TAG["router_w"], _sub(layer, 0), s.n_experts * s.hidden)
    return (0.02 * z).astype(np.float32).reshape(s.n_experts, s.hidden)


def router_bias(s: LayerSpec, seed: int, layer: int = 0):
    """fp32 router bias [E] ~ N(0, bias_std), or None when the spec has no bias."""
    if s.bias_std == 0.0:
        return None
    z = _normal(seed, TAG["router_b"], _sub(layer, 0), s.n_experts)
    return (s.bias_std * z).astype(np.float32)


def zipf_rank(s: LayerSpec, seed: int, layer: int) -> np.ndarray:
    """The Zipf rank (1..E) of every expert of a layer: a seeded permutation."""
    h = draws_np(seed, TAG["zipf_perm"], _sub(layer, 0), 0, s.n_experts)
    rank = np.empty(s.n_experts, dtype=np.int64)
    rank[np.argsort(h, kind="stable")] = np.arange(1, s.n_experts + 1)
    return rank


def zipf_bias(s: LayerSpec, seed: int, layer: int, beta: float, zipf_s: float = 1.1) -> np.ndarray:
    """Zipf-shaped router bias: b_e = -beta * zipf_s * ln(rank_e), rank a seeded permutation 1..E."""
    rank = zipf_rank(s, seed, layer)
    return (-beta * zipf_s * np.log(rank.astype(np.float64))).astype(np.float32)


def bf16_round_bits(v32: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    b = np.ascontiguousarray(v32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def hidden_states(s: LayerSpec, seed: int, batch: int, T: int, draws=None, rows=None):
    """Hidden states [T, H] ~ N(0,1).

    Row t is drawn from its own sub-stream (batch, t, draw index), so a single
    row can be redrawn (draws[t] > 0) without touching the others.  With
    `rows` given, only those row indices are produced (in that order).
    Returns (values_fp32 [n,H], bf16_bits [n,H] uint16 or None).  For bf16 specs
    the fp32 values are exactly the bf16 numbers.
    """
    H = s.hidden
    rows = range(T) if rows is None else [int(r) for r in rows]
    out = np.empty((len(rows), H), dtype=np.float32)
    for i, t in enumerate(rows):
        d = 0 if draws is None else int(draws[t])
        sub = (batch << 40) | (d << 24) | t
        out[i] = _normal(seed, TAG["x"], sub, H).astype(np.float32)
    if s.x_dtype == "bf16":
        bits = bf16_round_bits(out)
        vals = (bits.astype(np.uint32) << 16).view(np.float32)
        return vals.reshape(out.shape), bits.reshape(out.shape)
    return out, None
