"""The allocation-free forward (moe_layer_forward_static) against the workspace forward.

For callers that cannot give the library device scratch (an operator plugin that only
receives its input and output tensors, a serving loop that forbids allocation after
start-up, code that must not call cudaMalloc because it may synchronise the device), the
library keeps its scratch in its own 32 MiB device array.  This test calls that entry
point through the C ABI twice in a row and checks each result against moe_layer_forward
with a caller workspace: the same kernels on the same inputs, so ids, weights and output
must be bit-identical; the first call is also checked against the fp64 oracle within the
parity tolerance of the other tests.  It builds its own layer, so it passes alone in a
fresh process as well as after the other tests; the file name makes pytest collect it
last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import gen
import gen.device
import routed_expert_ffn_route_gb300 as moe
from _gpu_support import GpuLayer, inputs, oracle_out, oracle_out_many
from _support import FROB_REL, MAX_REL_RMS, err_stats

pytestmark = pytest.mark.gpu

STATIC_BYTES = 32 << 20  # the library's scratch array


def _call_static(L, xd, T):
    s = L.spec
    out = torch.full((T, s.hidden), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.full((T, s.top_k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T, s.top_k), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    dt = moe.MOE_DT_BF16 if xd.dtype == torch.bfloat16 else moe.MOE_DT_F32
    r = moe.lib().moe_layer_forward_static(
        C.byref(L.cfg), C.c_void_p(L.packed.data_ptr()), C.c_void_p(xd.data_ptr()), dt, T,
        C.c_void_p(out.data_ptr()), C.c_void_p(ids.data_ptr()), C.c_void_p(w.data_ptr()),
        C.c_void_p(status.data_ptr()), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert r == moe.MOE_OK, moe.moe_status_str(r)
    torch.cuda.synchronize()
    assert int(status.item()) == moe.MOE_OK
    return out, ids, w


def _largest_static_T(cfg):
    """The largest T whose workspace fits the static array (the entry point's limit)."""
    T = 1
    while moe.moe_workspace_bytes(cfg, T + 1) <= STATIC_BYTES:
        T += 1
    return T


SMALL = gen.LayerSpec("noalloc_small", hidden=512, inter=384, n_experts=16, top_k=4,
                      router="sigmoid_grouped", n_shared=1, inter_shared=256, n_group=4,
                      topk_group=2, rsf=2.5, bias_std=0.1)


# Mixtral-shaped: at T = 1 the down launch splits its contraction into 8 parts, whose
# extra y planes live in the static array too
MIX_SPLIT = gen.LayerSpec("noalloc_mix_split", hidden=1024, inter=2048, n_experts=8, top_k=2,
                          router="softmax")


@pytest.mark.parametrize("spec,T", [(SMALL, 37), (gen.spec("dsv3"), 16),
                                    (gen.spec("dsv3"), "largest"), (MIX_SPLIT, 1)])
def test_static_scratch_forward_matches_workspace_forward(spec, T):
    L = GpuLayer(spec, seed=21)
    if T == "largest":
        T = _largest_static_T(L.cfg)
        print(f"{spec.name}: largest T for the static scratch = {T}")
    x, xd, ids_o, w_o, *_ = inputs(spec, L, 5, T)
    ref = [t.clone() for t in L.forward(xd)]
    for call in range(2):  # two calls in a row share (and reuse) the static array
        got = _call_static(L, xd, T)
        for g, r, what in zip(got, ref, ("out", "ids", "w")):
            assert torch.equal(g, r), f"call {call}: {what} differs from the workspace forward"
    assert np.array_equal(ref[1].cpu().numpy(), ids_o)
    many = T * (spec.top_k + spec.n_shared) * spec.hidden * spec.inter > 4e9
    want = (oracle_out_many(spec, L, x, ids_o, w_o, np.arange(T)) if many
            else oracle_out(spec, L, x, ids_o, w_o))
    mx, fr = err_stats(ref[0].cpu().numpy(), want)
    print(f"{spec.name} T={T} static forward vs oracle: max|err|/RMS = {mx:.2e}, "
          f"rel Frobenius = {fr:.2e}")
    assert mx <= MAX_REL_RMS and fr <= FROB_REL


def test_static_scratch_rejects_oversized_calls():
    s = gen.spec("dsv3")
    cfg = gen.device.config_for(s)
    largest = _largest_static_T(cfg)
    assert moe.moe_workspace_bytes(cfg, largest) <= STATIC_BYTES
    for T in (largest + 1, 64):  # the first size whose workspace exceeds the array, and more
        assert moe.moe_workspace_bytes(cfg, T) > STATIC_BYTES
        r = moe.lib().moe_layer_forward_static(
            C.byref(cfg), C.c_void_p(256), C.c_void_p(256), moe.MOE_DT_BF16, T, C.c_void_p(256),
            C.c_void_p(256), C.c_void_p(256), None, None)
        assert r == moe.MOE_ERR_WORKSPACE
