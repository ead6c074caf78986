"""ctypes wrapper of the plain C fp64 oracle of one MoE layer forward.

TEST INFRASTRUCTURE ONLY: the test-suite, the smoke check and the benchmark's
CPU-baseline leg may use it; the product path (the CUDA library and its Python
binding) never imports it.  The oracle shares no code with the CUDA path.

Parity pins: every function here is pinned by `tests/test_oracle_*.py` against
properties the pages and mathematics fix (brute force, closed forms, library
routines, bit identities); see the test files for which pin covers what.
"""
from __future__ import annotations

import ctypes as C
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libmoe_oracle.so")
_SRC = os.path.join(_HERE, "moe_oracle.c")
_HDR = os.path.join(_HERE, "moe_oracle.h")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall"]


def build(force: bool = False, src: str = _SRC, out: str = _SO) -> str:
    """Compile the oracle into a shared library (gcc/cc), if stale."""
    stale = force or not os.path.exists(out) or any(
        os.path.getmtime(p) > os.path.getmtime(out) for p in (src, _HDR))
    if stale:
        cc = os.environ.get("CC", "cc")
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call([cc, *CFLAGS, "-I", _HERE, src, "-o", tmp, "-lm"])
        os.replace(tmp, out)
    return out


class _Cfg(C.Structure):
    _fields_ = [("hidden", C.c_int), ("inter", C.c_int), ("n_experts", C.c_int),
                ("top_k", C.c_int), ("n_shared", C.c_int), ("inter_shared", C.c_int),
                ("router", C.c_int), ("n_group", C.c_int), ("topk_group", C.c_int),
                ("norm_topk", C.c_int), ("rsf", C.c_double), ("act_q8_0", C.c_int),
                ("top_p", C.c_double)]


class _Expert(C.Structure):
    _fields_ = [("gate", C.c_void_p), ("up", C.c_void_p), ("down", C.c_void_p),
                ("s_gate", C.c_void_p), ("s_up", C.c_void_p), ("s_down", C.c_void_p),
                ("inter", C.c_int)]


def load(path: str = None):
    global _lib
    with _lock:
        if path is not None:
            return _bind(C.CDLL(path))
        if _lib is None:
            # MOE_ORACLE_SO lets the mutation test load a deliberately broken build
            alt = os.environ.get("MOE_ORACLE_SO")
            _lib = _bind(C.CDLL(alt if alt else build()))
        return _lib


def _bind(lib):
    P = C.c_void_p
    lib.orc_silu.restype = C.c_double
    lib.orc_silu.argtypes = [C.c_double]
    lib.orc_router_logits.argtypes = [P, P, C.c_int, P, P]
    lib.orc_route.argtypes = [P, P, P, C.c_int, P, P, P]
    lib.orc_permutation.argtypes = [C.c_int, C.c_int, C.c_int, P, P, P]
    lib.orc_expert_forward.argtypes = [P, P, P, C.c_int, P]
    lib.orc_layer_forward.argtypes = [P, P, C.c_int, P, P, P, P, C.c_int, P, P, P]
    lib.orc_layer_experts.argtypes = [P, P, C.c_int, P, P, P, P, C.c_int, P]
    lib.orc_q8_0_encode.argtypes = [P, C.c_int, P, P]
    lib.orc_block_dot.restype = C.c_int32
    lib.orc_block_dot.argtypes = [P, P]
    for f in ("orc_pack_int4", "orc_unpack_int4", "orc_pack_int2", "orc_unpack_int2"):
        getattr(lib, f).argtypes = [P, C.c_size_t, P]
    lib.orc_residual_rmsnorm.argtypes = [C.c_int, C.c_int, P, P, C.c_double, P]
    lib.orc_quantize_rows.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P]
    return lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.c_void_p)


def config(spec) -> _Cfg:
    """Oracle config from a gen.LayerSpec."""
    return _Cfg(spec.hidden, spec.inter, spec.n_experts, spec.top_k, spec.n_shared,
                spec.inter_sh, 0 if spec.router == "softmax" else 1, spec.n_group,
                spec.topk_group, spec.norm_topk, float(spec.rsf), spec.act_q8_0,
                float(spec.top_p))


@dataclasses.dataclass
class Expert:
    """One expert's int8 containers and fp32 row scales (numpy)."""
    gate: np.ndarray
    up: np.ndarray
    down: np.ndarray
    s_gate: np.ndarray
    s_up: np.ndarray
    s_down: np.ndarray

    def c(self) -> _Expert:
        for a, dt in ((self.gate, np.int8), (self.up, np.int8), (self.down, np.int8),
                      (self.s_gate, np.float32), (self.s_up, np.float32),
                      (self.s_down, np.float32)):
            assert a.dtype == dt and a.flags["C_CONTIGUOUS"]
        return _Expert(self.gate.ctypes.data, self.up.ctypes.data, self.down.ctypes.data,
                       self.s_gate.ctypes.data, self.s_up.ctypes.data, self.s_down.ctypes.data,
                       self.gate.shape[0])


def silu(z: float) -> float:
    return load().orc_silu(float(z))


def router_logits(spec, x64: np.ndarray, wr: np.ndarray) -> np.ndarray:
    x64 = np.ascontiguousarray(x64, dtype=np.float64)
    wr = np.ascontiguousarray(wr, dtype=np.float32)
    T = x64.shape[0]
    out = np.empty((T, spec.n_experts), dtype=np.float64)
    cfg = config(spec)
    load().orc_router_logits(C.byref(cfg), _p(x64), T, _p(wr), _p(out))
    return out


def route(spec, logits: np.ndarray, bias=None):
    """-> ids [T,k] int32, w [T,k] float64, margin [T] float64"""
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    T = logits.shape[0]
    ids = np.empty((T, spec.top_k), dtype=np.int32)
    w = np.empty((T, spec.top_k), dtype=np.float64)
    margin = np.empty(T, dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    cfg = config(spec)
    r = load().orc_route(C.byref(cfg), _p(logits), None if b is None else _p(b), T, _p(ids),
                         _p(w), _p(margin))
    if r:
        raise ValueError(f"orc_route: unsupported config ({r})")
    return ids, w, margin


def permutation(ids: np.ndarray, n_experts: int):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    off = np.empty(n_experts + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    load().orc_permutation(T, k, n_experts, _p(ids), _p(off), _p(perm))
    return off, perm


def expert_forward(spec, ex: Expert, x64: np.ndarray) -> np.ndarray:
    x64 = np.ascontiguousarray(x64, dtype=np.float64)
    n = x64.shape[0]
    y = np.empty((n, spec.hidden), dtype=np.float64)
    cfg = config(spec)
    ce = ex.c()
    load().orc_expert_forward(C.byref(cfg), C.byref(ce), _p(x64), n, _p(y))
    return y


def _expert_array(spec, experts: dict):
    arr = (_Expert * spec.n_experts)()
    keep = []
    for e, ex in experts.items():
        arr[e] = ex.c()
        keep.append(ex)
    return arr, keep


def layer_experts(spec, x64, ids, w, experts: dict, shared=None, mode: int = 1) -> np.ndarray:
    """Expert part + combine, given routing.  experts: {expert index: Expert}."""
    x64 = np.ascontiguousarray(x64, dtype=np.float64)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float64)
    T = x64.shape[0]
    out = np.empty((T, spec.hidden), dtype=np.float64)
    arr, _keep = _expert_array(spec, experts)
    sh = shared.c() if shared is not None else None
    cfg = config(spec)
    r = load().orc_layer_experts(C.byref(cfg), _p(x64), T, _p(ids), _p(w), arr,
                                 None if sh is None else C.byref(sh), mode, _p(out))
    if r:
        raise ValueError(f"orc_layer_experts failed ({r})")
    return out


def layer_forward(spec, x64, wr, bias, experts: dict, shared=None, mode: int = 1):
    """-> ids, w, out (router + experts + combine)."""
    x64 = np.ascontiguousarray(x64, dtype=np.float64)
    wr = np.ascontiguousarray(wr, dtype=np.float32)
    T = x64.shape[0]
    ids = np.empty((T, spec.top_k), dtype=np.int32)
    w = np.empty((T, spec.top_k), dtype=np.float64)
    out = np.empty((T, spec.hidden), dtype=np.float64)
    arr, _keep = _expert_array(spec, experts)
    sh = shared.c() if shared is not None else None
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    cfg = config(spec)
    r = load().orc_layer_forward(C.byref(cfg), _p(x64), T, _p(wr),
                                 None if b is None else _p(b), arr,
                                 None if sh is None else C.byref(sh), mode, _p(ids), _p(w),
                                 _p(out))
    if r:
        raise ValueError(f"orc_layer_forward failed ({r})")
    return ids, w, out


def q8_0_encode(v: np.ndarray):
    v = np.ascontiguousarray(v, dtype=np.float32).ravel()
    assert v.size % 32 == 0
    q = np.empty(v.size, dtype=np.int8)
    d = np.empty(v.size // 32, dtype=np.float32)
    load().orc_q8_0_encode(_p(v), v.size, _p(q), _p(d))
    return q, d


def block_dot(a: np.ndarray, b: np.ndarray) -> int:
    a = np.ascontiguousarray(a, dtype=np.int8)
    b = np.ascontiguousarray(b, dtype=np.int8)
    assert a.size == 32 and b.size == 32
    return int(load().orc_block_dot(_p(a), _p(b)))


def _packer(name, per_byte):
    def f(q):
        q = np.ascontiguousarray(q, dtype=np.int8).ravel()
        out = np.empty(q.size // per_byte, dtype=np.uint8)
        getattr(load(), name)(_p(q), q.size, _p(out))
        return out
    return f


def _unpacker(name):
    def f(p, n):
        p = np.ascontiguousarray(p, dtype=np.uint8).ravel()
        q = np.empty(n, dtype=np.int8)
        getattr(load(), name)(_p(p), n, _p(q))
        return q
    return f


pack_int4 = _packer("orc_pack_int4", 2)
pack_int2 = _packer("orc_pack_int2", 4)
unpack_int4 = _unpacker("orc_unpack_int4")
unpack_int2 = _unpacker("orc_unpack_int2")


def residual_rmsnorm(r: np.ndarray, add=None, eps: float = 1e-6):
    """Stack step: r += add (in place on a copy), x = bf16(RMSNorm(r)).  -> (r, x) fp64."""
    r = np.array(r, dtype=np.float64, order="C", copy=True)
    T, H = r.shape
    a = None if add is None else np.ascontiguousarray(add, dtype=np.float64)
    xn = np.empty_like(r)
    load().orc_residual_rmsnorm(T, H, _p(r), None if a is None else _p(a), float(eps), _p(xn))
    return r, xn


def quantize_rows(w: np.ndarray, bits: int):
    """Per-row quantiser: fp32 [rows, cols] -> (codes int8 [rows, cols], scales fp32 [rows])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    q = np.empty((rows, cols), dtype=np.int8)
    s = np.empty(rows, dtype=np.float32)
    if load().orc_quantize_rows(_p(w), rows, cols, int(bits), _p(q), _p(s)):
        raise ValueError(f"unsupported bits {bits}")
    return q, s
