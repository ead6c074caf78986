"""The allocation-free forward (moe_layer_forward_static) against the workspace forward.

For callers that cannot give the library device scratch (an operator plugin that only
receives its input and output tensors, a serving loop that forbids allocation after
start-up, code that must not call cudaMalloc because it may synchronise the device), the
library keeps its scratch in its own 32 MiB device array.  This test calls that entry
point through the C ABI twice in a row and checks each result against moe_layer_forward
with a caller workspace, within the parity tolerance of the other tests.  It builds its
own layer, so it passes alone in a fresh process as well as after the other tests; the
file name makes pytest collect it last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import gen
import gen.device
import routed_expert_ffn_route_gb300 as moe
from _gpu_support import GpuLayer, inputs
from _support import FROB_REL, MAX_REL_RMS, err_stats

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("spec,T", [
    (gen.LayerSpec("noalloc_small", hidden=512, inter=384, n_experts=16, top_k=4,
                   router="sigmoid_grouped", n_shared=1, inter_shared=256, n_group=4,
                   topk_group=2, rsf=2.5, bias_std=0.1), 37),
    (gen.spec("dsv3"), 16),
])
def test_static_scratch_forward_matches_workspace_forward(spec, T):
    L = GpuLayer(spec, seed=21)
    _, xd, *_ = inputs(spec, L, 5, T)
    ref_out, ref_ids, ref_w = L.forward(xd)
    ref_out, ref_ids, ref_w = ref_out.cpu().numpy(), ref_ids.cpu().numpy(), ref_w.cpu().numpy()
    for _ in range(2):  # two calls in a row share (and reuse) the static array
        out, ids, w = _call_static(L, xd, T)
        assert np.array_equal(ids.cpu().numpy(), ref_ids)
        for got, ref in ((out.cpu().numpy(), ref_out), (w.cpu().numpy(), ref_w)):
            mx, fr = err_stats(got, ref)
            assert mx <= MAX_REL_RMS and fr <= FROB_REL, (mx, fr)


def test_static_scratch_rejects_oversized_calls():
    s = gen.spec("dsv3")
    cfg = gen.device.config_for(s)
    T = 64  # its workspace is far above the 32 MiB array
    assert moe.moe_workspace_bytes(cfg, T) > (32 << 20)
    r = moe.lib().moe_layer_forward_static(
        C.byref(cfg), C.c_void_p(256), C.c_void_p(256), moe.MOE_DT_BF16, T, C.c_void_p(256),
        C.c_void_p(256), C.c_void_p(256), None, None)
    assert r == moe.MOE_ERR_WORKSPACE
