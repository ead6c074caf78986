"""Python binding of the GB300 MoE-layer library (libmoe_gb300.so, C ABI in include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.
PyTorch provides device memory and the current stream.  There is no CPU fallback: if the
compiled library is missing, importing the binding's functions raises.

Names mirror the C entry points (moe_pack_weights, moe_route_topk, moe_layer_forward, ...).
"""
from __future__ import annotations

import ctypes as C
import os
import threading

__all__ = [
    "MoEError", "LIB_PATH", "lib", "build", "moe_layer_config", "moe_weight_src", "make_config",
    "moe_version", "moe_status_str", "moe_check_config", "moe_packed_bytes",
    "moe_workspace_bytes", "moe_pack_weights", "moe_pack_router", "moe_pack_expert",
    "moe_unpack_weights", "moe_route_topk", "moe_layer_forward", "moe_read_status",
    "moe_debug_permutation", "moe_q8_0_quantize", "moe_debug_block_dots",
    "moe_debug_wait_timeout", "moe_layer_forward_experts", "moe_layer_forward_next", "EXPORTED",
    "MOE_OK", "MOE_ERR_INVALID_ARG", "MOE_ERR_UNSUPPORTED", "MOE_ERR_WORKSPACE",
    "MOE_ERR_CUDA", "MOE_ERR_TIMEOUT", "MOE_ERR_NUMERIC", "MOE_ERR_PACKED",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, -1, -2, -3
MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_NUMERIC, MOE_ERR_PACKED = -4, -5, -6, -7
MOE_ROUTER_SOFTMAX, MOE_ROUTER_SIGMOID_GROUPED = 0, 1
MOE_DT_F32, MOE_DT_BF16 = 0, 1

# every entry point include/moe.h declares
EXPORTED = [
    "moe_version", "moe_status_str", "moe_check_config", "moe_packed_bytes",
    "moe_workspace_bytes", "moe_pack_weights", "moe_pack_router", "moe_pack_expert",
    "moe_unpack_weights", "moe_route_topk", "moe_layer_forward", "moe_read_status",
    "moe_debug_permutation", "moe_q8_0_quantize", "moe_debug_block_dots",
    "moe_debug_wait_timeout", "moe_layer_forward_timed", "moe_forward_launches",
    "moe_layer_forward_static", "moe_residual_rmsnorm", "moe_quantize_rows",
    "moe_layer_forward_experts", "moe_layer_forward_next",
]

# stages bracketed by the events of moe_layer_forward_timed
STAGES = ["router", "permute", "act_encode", "gate_up", "down", "combine"]


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_status_name(status)} ({status})")


class moe_layer_config(C.Structure):
    _fields_ = [("hidden", C.c_int), ("inter", C.c_int), ("n_experts", C.c_int),
                ("top_k", C.c_int), ("n_shared", C.c_int), ("inter_shared", C.c_int),
                ("router", C.c_int), ("n_group", C.c_int), ("topk_group", C.c_int),
                ("norm_topk", C.c_int), ("routed_scaling_factor", C.c_float),
                ("weight_bits", C.c_int), ("act_q8_0", C.c_int), ("expert_top_p", C.c_float)]


class moe_weight_src(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "gate", "up", "down", "s_gate", "s_up", "s_down", "sh_gate", "sh_up", "sh_down",
        "sh_s_gate", "sh_s_up", "sh_s_down", "router_w", "router_bias")]


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the CUDA library for sm_103a in-tree (needs nvcc)."""
    from ._build import build as _b
    return _b(force=force)


def lib():
    """The loaded library; raises if it has not been built (no fallback path exists)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build it first (routed_expert_ffn_route_gb300.build()); "
                    "this package has no CPU or eager fallback")
            _lib = _bind(C.CDLL(LIB_PATH))
        return _lib


def _bind(L):
    P, I, S = C.c_void_p, C.c_int, C.c_size_t
    sig = {
        "moe_version": (I, []),
        "moe_status_str": (C.c_char_p, [I]),
        "moe_check_config": (I, [P]),
        "moe_packed_bytes": (S, [P]),
        "moe_workspace_bytes": (S, [P, I]),
        "moe_pack_weights": (I, [P, P, P, S, P]),
        "moe_pack_router": (I, [P, P, P, P, S, P]),
        "moe_pack_expert": (I, [P, I, P, P, P, P, P, P, P, S, P]),
        "moe_unpack_weights": (I, [P, P, I, P, P, P, P, P, P, P]),
        "moe_route_topk": (I, [P, P, P, I, I, P, P, P, S, P]),
        "moe_layer_forward": (I, [P, P, P, I, I, P, P, P, P, S, P]),
        "moe_read_status": (I, [P, P]),
        "moe_debug_permutation": (I, [P, P, I, P, P, P]),
        "moe_q8_0_quantize": (I, [P, I, I, I, P, P, P]),
        "moe_debug_block_dots": (I, [P, P, I, I, P, I, P, I, P, P]),
        "moe_debug_wait_timeout": (I, [P, S, I, P]),
        "moe_layer_forward_timed": (I, [P, P, P, I, I, P, P, P, P, S, P, I, P]),
        "moe_forward_launches": (I, [P, I, I]),
        "moe_layer_forward_static": (I, [P, P, P, I, I, P, P, P, P, P]),
        "moe_residual_rmsnorm": (I, [I, I, P, P, P, C.c_float, P, P]),
        "moe_quantize_rows": (I, [P, I, I, I, I, P, P, P]),
        "moe_layer_forward_experts": (I, [P, P, P, I, I, I, I, I, P, P, P, P, S, P]),
        "moe_layer_forward_next": (I, [P, P, P, I, I, P, P, P, P, S, P, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


def _status_name(s: int) -> str:
    try:
        return lib().moe_status_str(int(s)).decode()
    except Exception:  # pragma: no cover
        return "status"


def _ck(status: int, where: str):
    if status != MOE_OK:
        raise MoEError(status, where)


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _dtype(x) -> int:
    import torch
    if x.dtype == torch.float32:
        return MOE_DT_F32
    if x.dtype == torch.bfloat16:
        return MOE_DT_BF16
    raise TypeError(f"hidden states must be float32 or bfloat16, got {x.dtype}")


def make_config(hidden, inter, n_experts, top_k, router="softmax", n_shared=0, inter_shared=0,
                n_group=1, topk_group=1, norm_topk=1, routed_scaling_factor=1.0, weight_bits=4,
                act_q8_0=0, expert_top_p=0.0) -> moe_layer_config:
    r = {"softmax": MOE_ROUTER_SOFTMAX, "sigmoid_grouped": MOE_ROUTER_SIGMOID_GROUPED}.get(
        router, router)
    return moe_layer_config(hidden, inter, n_experts, top_k, n_shared, inter_shared, int(r),
                            n_group, topk_group, norm_topk, float(routed_scaling_factor),
                            weight_bits, act_q8_0, float(expert_top_p))


def moe_version() -> int:
    return lib().moe_version()


def moe_status_str(s: int) -> str:
    return lib().moe_status_str(int(s)).decode()


def moe_check_config(cfg) -> int:
    return lib().moe_check_config(C.byref(cfg))


def moe_packed_bytes(cfg) -> int:
    return lib().moe_packed_bytes(C.byref(cfg))


def moe_workspace_bytes(cfg, max_tokens: int) -> int:
    return lib().moe_workspace_bytes(C.byref(cfg), int(max_tokens))


def moe_pack_weights(cfg, src: dict, packed, stream=None):
    """src: dict with the moe_weight_src field names -> device tensors (router_bias may be None)."""
    s = moe_weight_src(**{k: (None if v is None else v.data_ptr()) for k, v in src.items()})
    _ck(lib().moe_pack_weights(C.byref(cfg), C.byref(s), _p(packed), packed.numel(),
                               _stream(stream)), "moe_pack_weights")


def moe_pack_router(cfg, router_w, router_bias, packed, stream=None):
    _ck(lib().moe_pack_router(C.byref(cfg), _p(router_w), _p(router_bias), _p(packed),
                              packed.numel(), _stream(stream)), "moe_pack_router")


def moe_pack_expert(cfg, expert, gate, up, down, s_gate, s_up, s_down, packed, stream=None):
    _ck(lib().moe_pack_expert(C.byref(cfg), int(expert), _p(gate), _p(up), _p(down), _p(s_gate),
                              _p(s_up), _p(s_down), _p(packed), packed.numel(), _stream(stream)),
        "moe_pack_expert")


def moe_unpack_weights(cfg, packed, expert, gate=None, up=None, down=None, s_gate=None,
                       s_up=None, s_down=None, stream=None):
    _ck(lib().moe_unpack_weights(C.byref(cfg), _p(packed), int(expert), _p(gate), _p(up),
                                 _p(down), _p(s_gate), _p(s_up), _p(s_down), _stream(stream)),
        "moe_unpack_weights")


def moe_route_topk(cfg, packed, x, ids, w, ws, stream=None):
    T = x.shape[0]
    _ck(lib().moe_route_topk(C.byref(cfg), _p(packed), _p(x), _dtype(x), T, _p(ids), _p(w),
                             _p(ws), ws.numel(), _stream(stream)), "moe_route_topk")


def moe_layer_forward(cfg, packed, x, out, ids, w, ws, stream=None):
    T = x.shape[0]
    _ck(lib().moe_layer_forward(C.byref(cfg), _p(packed), _p(x), _dtype(x), T, _p(out), _p(ids),
                                _p(w), _p(ws), ws.numel(), _stream(stream)), "moe_layer_forward")


def moe_layer_forward_experts(cfg, packed, x, expert_begin, expert_end, with_shared, out, ids,
                              w, ws, stream=None):
    """Expert-parallel share: out = [shared] + the routed experts in [begin, end) only."""
    T = x.shape[0]
    _ck(lib().moe_layer_forward_experts(C.byref(cfg), _p(packed), _p(x), _dtype(x), T,
                                        int(expert_begin), int(expert_end), int(with_shared),
                                        _p(out), _p(ids), _p(w), _p(ws), ws.numel(),
                                        _stream(stream)), "moe_layer_forward_experts")


def moe_layer_forward_next(cfg, packed, x, out, ids, w, ws, next_cfg, next_packed, stream=None):
    """moe_layer_forward that also warms the next stacked layer's router weights into L2."""
    T = x.shape[0]
    _ck(lib().moe_layer_forward_next(C.byref(cfg), _p(packed), _p(x), _dtype(x), T, _p(out),
                                     _p(ids), _p(w), _p(ws), ws.numel(), C.byref(next_cfg),
                                     _p(next_packed), _stream(stream)), "moe_layer_forward_next")


def moe_layer_forward_timed(cfg, packed, x, out, ids, w, ws, events, stream=None):
    """events: 7 torch.cuda.Event(enable_timing=True); see STAGES for what they bracket."""
    T = x.shape[0]
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event lazily, on its first record
            e.record()
    arr = (C.c_void_p * len(events))(*[C.c_void_p(e.cuda_event) for e in events])
    _ck(lib().moe_layer_forward_timed(C.byref(cfg), _p(packed), _p(x), _dtype(x), T, _p(out),
                                      _p(ids), _p(w), _p(ws), ws.numel(), arr, len(events),
                                      _stream(stream)), "moe_layer_forward_timed")


def moe_layer_forward_static(cfg, packed, x, out, ids, w, status=None, stream=None):
    """Allocation-free forward: scratch lives in the library's own 32 MiB device array."""
    T = x.shape[0]
    _ck(lib().moe_layer_forward_static(C.byref(cfg), _p(packed), _p(x), _dtype(x), T, _p(out),
                                       _p(ids), _p(w), _p(status), _stream(stream)),
        "moe_layer_forward_static")


def moe_forward_launches(cfg, T, dtype=None) -> int:
    """Kernel launches of one forward of T tokens (dtype: MOE_DT_BF16 by default)."""
    d = MOE_DT_BF16 if dtype is None else int(dtype)
    return lib().moe_forward_launches(C.byref(cfg), d, int(T))


def moe_read_status(ws, stream=None) -> int:
    return lib().moe_read_status(_p(ws), _stream(stream))


def moe_debug_permutation(cfg, ws, T, offsets, perm, stream=None):
    _ck(lib().moe_debug_permutation(C.byref(cfg), _p(ws), int(T), _p(offsets), _p(perm),
                                    _stream(stream)), "moe_debug_permutation")


def moe_q8_0_quantize(x, q, d, stream=None):
    T, n = x.shape
    _ck(lib().moe_q8_0_quantize(_p(x), _dtype(x), T, n, _p(q), _p(d), _stream(stream)),
        "moe_q8_0_quantize")


def moe_debug_block_dots(cfg, packed, expert, which, rows, qa, dots, stream=None):
    _ck(lib().moe_debug_block_dots(C.byref(cfg), _p(packed), int(expert), int(which), _p(rows),
                                   rows.numel(), _p(qa), qa.shape[0], _p(dots), _stream(stream)),
        "moe_debug_block_dots")


def moe_debug_wait_timeout(ws, iterations, stream=None):
    _ck(lib().moe_debug_wait_timeout(_p(ws), ws.numel(), int(iterations), _stream(stream)),
        "moe_debug_wait_timeout")


def moe_residual_rmsnorm(resid, add, x_next, x0=None, eps=1e-6, stream=None):
    """Stack step: resid = x0 (bf16 [T,H]) if given, else resid += add (fp32 [T,H], in place;
    add may be None); then x_next (bf16 [T,H]) = RMSNorm(resid) rounded to bf16."""
    T, H = resid.shape
    _ck(lib().moe_residual_rmsnorm(T, H, _p(resid), None if add is None else _p(add),
                                   None if x0 is None else _p(x0), float(eps), _p(x_next),
                                   _stream(stream)), "moe_residual_rmsnorm")


def moe_quantize_rows(w, bits, q, scale, stream=None):
    """Per-row quantiser: w fp32/bf16 [rows, cols] -> q int8 [rows, cols], scale fp32 [rows]."""
    rows, cols = w.shape
    _ck(lib().moe_quantize_rows(_p(w), _dtype(w), rows, cols, int(bits), _p(q), _p(scale),
                                _stream(stream)), "moe_quantize_rows")
