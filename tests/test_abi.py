"""The C-ABI library: builds, loads, exports every declared symbol, validates on the host.

No GPU is needed: these calls return before any CUDA work."""
import ctypes as C
import os
import re

import pytest

import gen
import routed_expert_ffn_route_gb300 as moe
from gen.device import config_for

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    moe.build()
    return moe.lib()


def declared_symbols():
    txt = open(os.path.join(ROOT, "include", "moe.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", txt)))


def test_library_exports_every_declared_symbol(L):
    syms = declared_symbols()
    assert len(syms) >= 15
    for s in syms:
        assert hasattr(L, s), f"{s} declared in include/moe.h but not exported"
    assert sorted(moe.EXPORTED) == syms


def test_status_strings(L):
    for code, name in [(0, "MOE_OK"), (-1, "MOE_ERR_INVALID_ARG"), (-2, "MOE_ERR_UNSUPPORTED"),
                       (-3, "MOE_ERR_WORKSPACE"), (-5, "MOE_ERR_TIMEOUT"), (-7, "MOE_ERR_PACKED")]:
        assert moe.moe_status_str(code) == name
    assert moe.moe_version() >= 10000


@pytest.mark.parametrize("name", sorted(gen.PRESETS))
def test_presets_are_supported(name, L):
    cfg = config_for(gen.spec(name))
    assert moe.moe_check_config(cfg) == moe.MOE_OK
    assert moe.moe_packed_bytes(cfg) > 0
    assert moe.moe_workspace_bytes(cfg, 4096) > 0


def test_packed_bytes_match_the_per_expert_sizes(L):
    s = gen.spec("dsv3")
    nb = moe.moe_packed_bytes(config_for(s))
    per_expert = (2 * 2048 * 6144 + 6144 * 2048) // 2 + (2 * 2048 + 6144) * 4  # 18.92 MB
    # fp32 router matrix and bias, plus its three bf16 pieces in 128-row tensor-core tiles
    router = 256 * 6144 * 4 + 256 * 4 + 3 * 2 * (6144 // 64) * 128 * 64 * 2
    assert per_expert == 18915328
    assert 257 * per_expert + router <= nb <= 257 * (per_expert + 8192) + router + 8192
    s8 = gen.spec("dsv3_int8")
    s2 = gen.spec("dsv3_int2")
    assert moe.moe_packed_bytes(config_for(s8)) > 1.9 * nb
    assert moe.moe_packed_bytes(config_for(s2)) < 0.55 * nb


@pytest.mark.parametrize("field,value", [
    ("hidden", 100), ("inter", 96), ("top_k", 0), ("top_k", 17), ("n_experts", 257),
    ("weight_bits", 3), ("n_shared", 2), ("router", 5), ("norm_topk", 2)])
def test_unsupported_configs_rejected(field, value, L):
    cfg = config_for(gen.spec("tiny"))
    setattr(cfg, field, value)
    assert moe.moe_check_config(cfg) == moe.MOE_ERR_UNSUPPORTED
    assert moe.moe_packed_bytes(cfg) == 0
    assert moe.moe_workspace_bytes(cfg, 8) == 0


def test_grouped_router_constraints(L):
    cfg = config_for(gen.spec("dsv3"))
    for kw in [dict(n_group=7), dict(n_group=0), dict(topk_group=9), dict(topk_group=0),
               dict(n_group=64)]:
        c2 = config_for(gen.spec("dsv3"))
        for k, v in kw.items():
            setattr(c2, k, v)
        assert moe.moe_check_config(c2) == moe.MOE_ERR_UNSUPPORTED, kw
    c3 = config_for(gen.spec("dsv3"))
    c3.top_k = 8
    c3.topk_group = 1
    c3.n_group = 64 // 2  # 8 experts per group, one group kept: fewer candidates than k? 8 == k
    assert moe.moe_check_config(c3) == moe.MOE_OK
    c3.top_k = 9
    assert moe.moe_check_config(c3) == moe.MOE_ERR_UNSUPPORTED
    assert moe.moe_check_config(cfg) == moe.MOE_OK


def test_q8_requires_int8_weights(L):
    cfg = config_for(gen.spec("dsv3_int8"))
    assert moe.moe_check_config(cfg) == moe.MOE_OK
    cfg.weight_bits = 4
    assert moe.moe_check_config(cfg) == moe.MOE_ERR_UNSUPPORTED


def test_null_and_bad_arguments_rejected_before_any_launch(L):
    cfg = config_for(gen.spec("tiny"))
    P = C.c_void_p
    assert L.moe_check_config(None) == moe.MOE_ERR_INVALID_ARG
    # T == 0 is a no-op
    assert L.moe_layer_forward(C.byref(cfg), None, None, 0, 0, None, None, None, None, 0, None) == 0
    # NULL pointers with T > 0
    assert L.moe_layer_forward(C.byref(cfg), None, None, 0, 8, None, None, None, None, 0,
                               None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_route_topk(C.byref(cfg), None, None, 1, 8, None, None, None, 0,
                            None) == moe.MOE_ERR_INVALID_ARG
    # negative T, bad dtype
    assert L.moe_layer_forward(C.byref(cfg), P(256), P(256), 0, -1, P(256), P(256), P(256),
                               P(256), 1 << 30, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_route_topk(C.byref(cfg), P(256), P(256), 7, 4, P(256), P(256), P(256), 1 << 30,
                            None) == moe.MOE_ERR_INVALID_ARG
    # misaligned packed / workspace pointers
    assert L.moe_layer_forward(C.byref(cfg), P(258), P(256), 0, 4, P(256), P(256), P(256),
                               P(256), 1 << 30, None) == moe.MOE_ERR_INVALID_ARG
    # workspace too small
    assert L.moe_layer_forward(C.byref(cfg), P(256), P(256), 0, 4, P(256), P(256), P(256),
                               P(256), 64, None) in (moe.MOE_ERR_WORKSPACE, moe.MOE_ERR_UNSUPPORTED)
    # packing: bad expert index, small buffer
    assert L.moe_pack_expert(C.byref(cfg), 99, P(256), P(256), P(256), P(256), P(256), P(256),
                             P(256), 1 << 40, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_pack_router(C.byref(cfg), P(256), None, P(256), 16, None) == moe.MOE_ERR_WORKSPACE
    assert L.moe_q8_0_quantize(P(256), 0, 2, 33, P(256), P(256), None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_debug_wait_timeout(None, 0, 5, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_debug_block_dots(C.byref(cfg), P(256), 0, 0, P(256), 1, P(256), 1, P(256),
                                  None) == moe.MOE_ERR_UNSUPPORTED  # needs int8 weights


def test_workspace_grows_with_tokens(L):
    cfg = config_for(gen.spec("dsv3"))
    a, b = moe.moe_workspace_bytes(cfg, 16), moe.moe_workspace_bytes(cfg, 2048)
    assert 0 < a < b
    assert b >= 2048 * 9 * 6144 * 4  # the fp32 expert outputs of every (token, slot)


# a Mixtral-shaped small layer: few experts, a long down contraction (the decode down
# launch splits its work items' contractions and needs room for the extra y planes)
MIX_SPLIT = gen.LayerSpec("mix_split", hidden=1024, inter=2048, n_experts=8, top_k=2,
                          router="softmax")


@pytest.mark.parametrize("spec", [gen.spec("dsv3"), gen.spec("tiny"), gen.spec("dsv3_int8"),
                                  gen.spec("dsv3_int2"), gen.spec("mixtral"), MIX_SPLIT,
                                  MIX_SPLIT.replace(n_shared=1, inter_shared=1024)],
                         ids=["dsv3", "tiny", "dsv3_int8", "dsv3_int2", "mixtral", "mix_split",
                              "mix_split_shared"])
def test_workspace_never_shrinks_as_tokens_grow(spec, L):
    """A workspace sized for T tokens serves every call of T' <= T tokens, so the size is
    monotone in T (the split down launch's extra y planes are largest at small T)."""
    cfg = config_for(spec)
    sizes = [moe.moe_workspace_bytes(cfg, T) for T in list(range(1, 41)) + [64, 512, 4096]]
    assert all(0 < a <= b for a, b in zip(sizes, sizes[1:])), sizes


def test_forward_launch_counts(L):
    """Decode-sized batches run as one front launch (router, selection, permutation,
    token rows) plus gate/up, down and combine; other batches take the separate launches."""
    dsv3 = config_for(gen.spec("dsv3"))
    f32, bf16 = moe.MOE_DT_F32, moe.MOE_DT_BF16
    assert moe.moe_forward_launches(dsv3, 0) == 0
    assert moe.moe_forward_launches(dsv3, 1) == 4
    assert moe.moe_forward_launches(dsv3, 16, bf16) == 4
    assert moe.moe_forward_launches(dsv3, 8, f32) == 4      # two fp16 pieces per token
    assert moe.moe_forward_launches(dsv3, 16, f32) == 7     # 32 rows: activation tiles
    assert moe.moe_forward_launches(dsv3, 17, bf16) == 7
    assert moe.moe_forward_launches(dsv3, 2048, bf16) == 7
    # a hidden size whose T = 16 router slice does not fit the GEMV: separate launches
    wide = config_for(gen.spec("tiny").replace(hidden=12416))
    assert moe.moe_forward_launches(wide, 16, bf16) == 7
    q8 = config_for(gen.spec("dsv3_int8"))
    assert moe.moe_forward_launches(q8, 4, bf16) == 7      # Q8_0 encode, no tiles
    assert L.moe_forward_launches(C.byref(dsv3), 7, 1) == moe.MOE_ERR_INVALID_ARG


def test_top_p_validation(L):
    cfg = config_for(gen.spec("dsv3"))
    for p, ok in ((0.0, True), (0.7, True), (1.0, True), (-0.1, False), (float("nan"), False),
                  (float("inf"), False)):
        cfg.expert_top_p = p
        assert (moe.moe_check_config(cfg) == moe.MOE_OK) == ok, p


def test_expert_share_arguments_rejected_before_any_launch(L):
    cfg = config_for(gen.spec("dsv3"))
    P = C.c_void_p
    call = lambda b, e, sh, T=4: L.moe_layer_forward_experts(
        C.byref(cfg), P(256), P(256), moe.MOE_DT_BF16, T, b, e, sh, P(256), P(256), P(256),
        P(256), 1 << 40, None)
    for b, e, sh in [(-1, 4, 0), (5, 4, 0), (0, 257, 1), (0, 256, 2), (0, 256, -1)]:
        assert call(b, e, sh) == moe.MOE_ERR_INVALID_ARG, (b, e, sh)
    # an empty share is valid (its output is the shared expert, or zero); T == 0 is a no-op
    assert call(3, 3, 0, T=0) == moe.MOE_OK
    assert call(0, 256, 1, T=0) == moe.MOE_OK


def test_next_layer_forward_arguments_rejected_before_any_launch(L):
    cfg = config_for(gen.spec("dsv3"))
    bad = config_for(gen.spec("dsv3"))
    bad.hidden = 100  # not a multiple of 128
    P = C.c_void_p
    call = lambda ncfg, npk, T=4: L.moe_layer_forward_next(
        C.byref(cfg), P(256), P(256), moe.MOE_DT_BF16, T, P(256), P(256), P(256), P(256),
        1 << 40, ncfg, npk, None)
    assert call(None, P(256)) == moe.MOE_ERR_INVALID_ARG
    assert call(C.byref(cfg), None) == moe.MOE_ERR_INVALID_ARG
    assert call(C.byref(cfg), P(258)) == moe.MOE_ERR_INVALID_ARG
    assert call(C.byref(bad), P(256)) == moe.MOE_ERR_UNSUPPORTED
