"""GPU parity: the CUDA path, called through the C ABI, against the fp64 CPU oracle.

Bit-exact: expert ids (slot order included), the permutation, packing round trips,
Q8_0 codes and int32 block dots.  Floating point (layer output, routed weights):
max|err| <= 2e-3 * RMS(oracle) and ||err||_F <= 1e-3 * ||oracle||_F.
Inputs are seeded and margin-filtered (every routing decision has a score gap of at
least 1e-4); the number of redraws is printed.
"""
import numpy as np
import pytest
import torch

import gen
import gen.device
import oracle
import routed_expert_ffn_route_gb300 as moe
from _gpu_support import GpuLayer, get_layer, inputs, oracle_out, oracle_out_many, prefill_sample
from _support import FROB_REL, MAX_REL_RMS, err_stats

pytestmark = pytest.mark.gpu


def small(name="grouped", **kw):
    """Several m-tiles, a ragged token tail and both routers at small sizes."""
    if name == "grouped":
        base = dict(name="small_grouped", hidden=512, inter=384, n_experts=16, top_k=4,
                    router="sigmoid_grouped", n_shared=1, inter_shared=256, n_group=4,
                    topk_group=2, rsf=2.5, bias_std=0.1)
    else:
        base = dict(name="small_softmax", hidden=384, inter=256, n_experts=8, top_k=2,
                    router="softmax")
    base.update(kw)
    return gen.LayerSpec(**base)


def assert_close(got, ref, what):
    mx, fr = err_stats(got, ref)
    print(f"{what}: max|err|/RMS = {mx:.2e}, rel Frobenius = {fr:.2e}")
    assert mx <= MAX_REL_RMS and fr <= FROB_REL, (what, mx, fr)


def check_layer(spec, T, batch=0, sample=None, seed=0):
    """The layer forward against the oracle: ids, weights and the permutation on every
    token; the output on every token (sample None), on `sample` tokens spread over the
    batch (an int), or (sample "prefill") on every token of the three most-loaded experts
    plus 32 spread tokens."""
    L = get_layer(spec, seed)
    x, xd, ids_o, w_o, margin, redraws = inputs(spec, L, batch, T)
    out, ids, w = L.forward(xd)
    torch.cuda.synchronize()
    ids_g, w_g, out_g = ids.cpu().numpy(), w.cpu().numpy(), out.cpu().numpy()
    print(f"{spec.name} T={T}: {redraws} near-tie redraws")
    assert np.array_equal(ids_g, ids_o), "expert ids differ from the oracle"
    assert_close(w_g, w_o, f"{spec.name} T={T} weights")
    off_o, perm_o = oracle.permutation(ids_o, spec.n_experts)
    off_g, perm_g = L.permutation(T)
    assert np.array_equal(off_g, off_o) and np.array_equal(perm_g, perm_o)
    if sample == "prefill":
        tok, top, load = prefill_sample(ids_o, spec.n_experts)
        print(f"{spec.name} T={T}: output compared on {len(tok)} tokens (experts {top.tolist()} "
              f"with {load.tolist()} tokens, and 32 spread)")
    else:
        tok = None if sample is None else np.unique(
            np.linspace(0, T - 1, sample).round().astype(int))
    n = T if tok is None else len(tok)
    if n * (spec.top_k + spec.n_shared) * spec.hidden * spec.inter > 4e9:
        ref = oracle_out_many(spec, L, x, ids_o, w_o, np.arange(T) if tok is None else tok)
    else:
        ref = oracle_out(spec, L, x, ids_o, w_o, tok)
    got = out_g if tok is None else out_g[tok]
    assert_close(got, ref, f"{spec.name} T={T} output")
    return out, ids, w, xd, L


# ------------------------------------------------------------------ packing

@pytest.mark.parametrize("bits", [4, 8, 2])
def test_pack_unpack_bit_identity(bits):
    s = small("grouped", weight_bits=bits)
    L = GpuLayer(s, seed=3)
    for e in (0, 7, s.n_experts):
        rows = {w: gen.expert_rows_cols(s, w, shared=(e == s.n_experts)) for w in ("gate", "up", "down")}
        outs = {w: torch.empty(rows[w], dtype=torch.int8, device="cuda") for w in rows}
        sc = {w: torch.empty(rows[w][0], dtype=torch.float32, device="cuda") for w in rows}
        moe.moe_unpack_weights(L.cfg, L.packed, e, outs["gate"], outs["up"], outs["down"],
                               sc["gate"], sc["up"], sc["down"])
        torch.cuda.synchronize()
        for w in rows:
            assert np.array_equal(outs[w].cpu().numpy(), gen.expert_codes(s, 3, 0, e, w))
            assert np.array_equal(sc[w].cpu().numpy(), gen.expert_scales(s, 3, 0, e, w))


@pytest.mark.parametrize("bits", [4, 8, 2])
def test_pack_weights_matches_incremental_packing(bits):
    # moe_pack_weights takes every expert's containers stacked ([E][I][H] ...) in one call;
    # the blob must be byte-identical to the one moe_pack_router + moe_pack_expert write
    s = small("grouped", weight_bits=bits)
    seed = 13
    cfg = gen.device.config_for(s)
    n = moe.moe_packed_bytes(cfg)
    inc = torch.zeros(n, dtype=torch.uint8, device="cuda")
    gen.device.build_packed_layer(s, seed, 0, "cuda", packed=inc, host_codes=True)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    stack = lambda which: dev(np.stack([gen.expert_codes(s, seed, 0, e, which)
                                        for e in range(s.n_experts)]))
    sstack = lambda which: dev(np.stack([gen.expert_scales(s, seed, 0, e, which)
                                         for e in range(s.n_experts)]))
    E = s.n_experts
    src = {"gate": stack("gate"), "up": stack("up"), "down": stack("down"),
           "s_gate": sstack("gate"), "s_up": sstack("up"), "s_down": sstack("down"),
           "sh_gate": dev(gen.expert_codes(s, seed, 0, E, "gate")),
           "sh_up": dev(gen.expert_codes(s, seed, 0, E, "up")),
           "sh_down": dev(gen.expert_codes(s, seed, 0, E, "down")),
           "sh_s_gate": dev(gen.expert_scales(s, seed, 0, E, "gate")),
           "sh_s_up": dev(gen.expert_scales(s, seed, 0, E, "up")),
           "sh_s_down": dev(gen.expert_scales(s, seed, 0, E, "down")),
           "router_w": dev(gen.router_weights(s, seed, 0)),
           "router_bias": dev(gen.router_bias(s, seed, 0).astype(np.float32))}
    one = torch.zeros(n, dtype=torch.uint8, device="cuda")
    moe.moe_pack_weights(cfg, src, one)
    torch.cuda.synchronize()
    assert torch.equal(one, inc)
    # and the packed layer computes the oracle's layer
    L = GpuLayer.__new__(GpuLayer)
    L.spec, L.seed, L.layer, L.cfg, L.packed = s, seed, 0, cfg, one
    L.wr, L.bias, L._ws = gen.router_weights(s, seed, 0), gen.router_bias(s, seed, 0), {}
    x, xd, ids_o, w_o, *_ = inputs(s, L, 0, 9)
    out, ids, w = L.forward(xd)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert_close(out.cpu().numpy(), oracle_out(s, L, x, ids_o, w_o), f"packed in one call, {bits}-bit")


def test_pack_unpack_full_size_expert():
    s = gen.spec("dsv3")
    L = get_layer(s)
    for e in (5, 256):
        g = torch.empty((2048, 6144), dtype=torch.int8, device="cuda")
        d = torch.empty((6144, 2048), dtype=torch.int8, device="cuda")
        moe.moe_unpack_weights(L.cfg, L.packed, e, g, None, d)
        ref_g = gen.expert_codes_torch(s, 0, 0, e, "gate", "cuda")
        ref_d = gen.expert_codes_torch(s, 0, 0, e, "down", "cuda")
        assert torch.equal(g, ref_g) and torch.equal(d, ref_d)


# ------------------------------------------------------------------ router

@pytest.mark.parametrize("name,T", [("tiny", 8), ("tiny", 1), ("mixtral", 1), ("mixtral", 512),
                                    ("dsv3", 1), ("dsv3", 16), ("dsv3", 2048)])
def test_router_parity(name, T):
    s = gen.spec(name)
    L = get_layer(s)
    x, xd, ids_o, w_o, margin, redraws = inputs(s, L, 1, T)
    ids, w = L.route(xd)
    torch.cuda.synchronize()
    print(f"{name} T={T}: {redraws} near-tie redraws")
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert_close(w.cpu().numpy(), w_o, f"router {name} T={T} weights")
    if s.router == "sigmoid_grouped":
        assert np.allclose(w.cpu().numpy().sum(1), s.rsf, rtol=1e-5)


@pytest.mark.parametrize("kw", [dict(n_experts=1, top_k=1), dict(top_k=8),
                                dict(norm_topk=0)])
def test_router_softmax_special_cases(kw):
    s = small("softmax", **kw)
    check_layer(s, 5, seed=4)


@pytest.mark.parametrize("kw", [dict(n_group=1, topk_group=1), dict(topk_group=4),
                                dict(rsf=1.0, bias_std=0.0), dict(top_k=8, topk_group=2)])
def test_router_grouped_special_cases(kw):
    s = small("grouped", **kw)
    check_layer(s, 6, seed=5)


# ------------------------------------------------------------------ whole layer

def test_layer_tiny_full():
    check_layer(gen.spec("tiny"), 8)


@pytest.mark.parametrize("T", [1, 2, 7, 33, 37, 64])
def test_layer_small_grouped_ragged(T):
    check_layer(small("grouped"), T, seed=1)


@pytest.mark.parametrize("x_dtype,T", [("bf16", 300), ("f32", 150)])
def test_layer_small_large_groups(x_dtype, T):
    # four experts, two per token: groups of more than 64 activation rows take the
    # tensor-core kernel's widest tile (128 rows), experts with more than 128 rows split
    # into two groups, and the shared expert's tokens fill several 128-row groups; every
    # element is compared
    s = small("softmax", n_experts=4, top_k=2, n_shared=1, inter_shared=256, x_dtype=x_dtype)
    L = get_layer(s, 11)
    x, xd, ids_o, *_ = inputs(s, L, 0, T)
    rows = np.bincount(ids_o.ravel(), minlength=4) * (2 if x_dtype == "f32" else 1)
    print(f"activation rows per expert: {rows.tolist()}")
    assert rows.max() > 128
    check_layer(s, T, seed=11)


@pytest.mark.parametrize("bits", [8, 2])
def test_layer_small_other_bit_widths(bits):
    check_layer(small("grouped", weight_bits=bits), 19, seed=2)


@pytest.mark.parametrize("T", [3, 40])
def test_layer_small_q8_0(T):
    check_layer(small("grouped", weight_bits=8, act_q8_0=1), T, seed=6)


def test_layer_small_softmax_fp32():
    check_layer(small("softmax", x_dtype="f32"), 21, seed=7)


@pytest.mark.parametrize("T", [5, 16])
def test_layer_small_grouped_fp32(T):
    # T = 5: the decode front with two fp16 pieces per token; T = 16: 32 activation rows,
    # so gate/up takes the tile path while down stays on the register-MMA kernel
    check_layer(small("grouped", x_dtype="f32"), T, seed=8)


@pytest.mark.parametrize("name,T,p", [("grouped", 7, 0.6), ("grouped", 37, 0.6),
                                      ("softmax", 9, 0.55), ("grouped_q8", 9, 0.5)])
def test_layer_small_topp(name, T, p):
    # adaptive expert top-p: dropped slots (id -1, weight 0) leave the permutation and the
    # combine; T = 7 runs the fused decode front, T = 37 the separate launches
    if name == "grouped_q8":
        s = small("grouped", weight_bits=8, act_q8_0=1, top_p=p)
    else:
        s = small(name, top_p=p)
    _, ids, _, _, _ = check_layer(s, T, seed=10)
    assert (ids.cpu().numpy() < 0).any()


@pytest.mark.parametrize("T,sample", [(1, None), (16, 3), (2048, 2)])
def test_layer_dsv3_topp(T, sample):
    out, ids, w, xd, L = check_layer(gen.spec("dsv3").replace(top_p=0.7), T, sample=sample)
    kept = (ids.cpu().numpy() >= 0).sum(1)
    print(f"dsv3 top-p 0.7 T={T}: experts kept per token {kept.mean():.2f} of 8")
    assert kept.min() >= 1


def test_layer_decode_rows_without_gemv_router():
    # a hidden size whose router slices do not fit the GEMV at T = 16: the tiled router,
    # selection, permute and token-row launches feed the register-MMA kernels
    check_layer(small("softmax", hidden=12416, inter=256), 16, seed=9)


# An odd down m-tile count (H = 384: 3 m-tiles of 128 outputs; I is a multiple of 128, so
# gate/up always has an even count): the tensor-core kernels take two m-tiles per work
# item, so each group's last down item holds one.
ODD_MT = gen.LayerSpec("odd_mtiles", hidden=384, inter=256, n_experts=8, top_k=2,
                       router="softmax", n_shared=1, inter_shared=384)


@pytest.mark.parametrize("T", [40, 300])
def test_layer_odd_mtile_counts(T):
    check_layer(ODD_MT, T)


# A Mixtral-shaped small layer: few experts with a long down contraction, so the decode
# down launch has few work items and splits each item's contraction (8 parts; 4 with the
# shared expert, whose contraction has fewer code runs), the combine adding the parts' y
# planes.
MIX_SPLIT = gen.LayerSpec("mix_split", hidden=1024, inter=2048, n_experts=8, top_k=2,
                          router="softmax")


@pytest.mark.parametrize("T", [1, 2, 5, 16])
@pytest.mark.parametrize("shared", [0, 1])
def test_layer_split_down_contraction(T, shared):
    s = MIX_SPLIT.replace(n_shared=shared, inter_shared=1024 if shared else 0)
    out, ids, w, xd, L = check_layer(s, T)  # every output element against the oracle
    again, _, _ = L.forward(xd)
    assert torch.equal(out, again)  # the planes are added in a fixed order


@pytest.mark.parametrize("top_p", [0.0, 0.6])
def test_permutation_past_one_chunk_per_cta(top_p):
    """Past two 32-token chunks per SM, each permutation CTA scatters a run of chunks: the
    offsets and perm stay bit-identical to the oracle's stable order (with top-p, the
    dropped slots form perm's -1 tail)."""
    s = gen.spec("tiny").replace(top_p=top_p)
    T = 12000
    L = get_layer(s, 5)
    x, xd, ids_o, w_o, *_ = inputs(s, L, 0, T)
    out, ids, w = L.forward(xd)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    off_o, perm_o = oracle.permutation(ids_o, s.n_experts)
    off_g, perm_g = L.permutation(T)
    print(f"tiny T={T} top_p={top_p}: {int((ids_o < 0).sum())} slots dropped")
    assert np.array_equal(off_g, off_o) and np.array_equal(perm_g, perm_o)


def test_layer_deterministic_and_T0_noop():
    s = small("grouped")
    L = get_layer(s, 1)
    _, xd, *_ = inputs(s, L, 3, 29)
    a = [t.clone() for t in L.forward(xd)]
    b = L.forward(xd)
    for p, q in zip(a, b):
        assert torch.equal(p, q)
    empty = torch.empty((0, s.hidden), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((0, s.hidden), dtype=torch.float32, device="cuda")
    ids = torch.empty((0, s.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((0, s.top_k), dtype=torch.float32, device="cuda")
    moe.moe_layer_forward(L.cfg, L.packed, empty, out, ids, w, L.ws(1))


# full-size layers (the benchmark's shapes): every token up to T = 64; at prefill sizes
# every token of the three most-loaded experts (their groups cover every m-tile of the
# tensor-core kernel, and an expert with more than 128 tokens forms two groups) plus 32
# spread tokens (one in every group of the shared expert).  DSV3 at T = 256 gives an
# expert 8 tokens on average: groups of at most 64 rows, two m-tiles per work item.
@pytest.mark.parametrize("name,T,sample", [("mixtral", 1, None), ("dsv3", 1, None),
                                           ("dsv3", 16, None), ("dsv3", 256, "prefill"),
                                           ("dsv3", 2048, "prefill"),
                                           ("dsv3_int2", 1, None), ("dsv3_int8", 4, None),
                                           ("dsv3_int8", 64, None), ("mixtral", 512, "prefill")])
def test_layer_full_size(name, T, sample):
    check_layer(gen.spec(name), T, sample=sample)


# ------------------------------------------------------------------ integer paths

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_q8_0_codes_bit_exact(dtype):
    s = gen.spec("dsv3", x_dtype=dtype)
    x, bits = gen.hidden_states(s, 9, 0, 12)
    xd = gen.device.hidden_to_device(s, x, bits)
    q = torch.empty((12, s.hidden), dtype=torch.int8, device="cuda")
    d = torch.empty((12, s.hidden // 32), dtype=torch.float32, device="cuda")
    moe.moe_q8_0_quantize(xd, q, d)
    torch.cuda.synchronize()
    qo, do = oracle.q8_0_encode(x.astype(np.float32))
    assert np.array_equal(q.cpu().numpy().ravel(), qo)
    assert np.array_equal(d.cpu().numpy().ravel().view(np.uint32), do.view(np.uint32))


def test_block_dots_bit_exact():
    s = gen.spec("dsv3_int8")
    L = get_layer(s)
    x, bits = gen.hidden_states(s, 10, 0, 3)
    qx, dx = oracle.q8_0_encode(x.astype(np.float32))
    qx = qx.reshape(3, s.hidden)
    rng = np.random.default_rng(0)
    for e, which in [(3, 0), (3, 1), (200, 2), (256, 0)]:
        name = ("gate", "up", "down")[which]
        codes = gen.expert_codes(s, 0, 0, e, name)
        K = codes.shape[1]
        rows = rng.choice(codes.shape[0], 5, replace=False).astype(np.int32)
        qa = qx if which < 2 else rng.integers(-127, 128, (3, K)).astype(np.int8)
        dots = torch.empty((5, 3, K // 32), dtype=torch.int32, device="cuda")
        moe.moe_debug_block_dots(L.cfg, L.packed, e, which, torch.from_numpy(rows).cuda(),
                                 torch.from_numpy(np.ascontiguousarray(qa)).cuda(), dots)
        torch.cuda.synchronize()
        got = dots.cpu().numpy()
        for ri, r in enumerate(rows):
            for t in range(3):
                for b in range(K // 32):
                    ref = oracle.block_dot(codes[r, b * 32:(b + 1) * 32], qa[t, b * 32:(b + 1) * 32])
                    assert got[ri, t, b] == ref


# ------------------------------------------------------------------ device status

def test_packed_header_mismatch_is_reported():
    s = small("grouped")
    L = get_layer(s, 1)
    _, xd, *_ = inputs(s, L, 4, 4)
    bad = gen.device.config_for(s)
    bad.weight_bits = 8  # different layout than the blob holds
    ws = torch.zeros(moe.moe_workspace_bytes(bad, 4), dtype=torch.uint8, device="cuda")
    ids = torch.empty((4, s.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((4, s.top_k), dtype=torch.float32, device="cuda")
    big = torch.zeros(moe.moe_packed_bytes(bad), dtype=torch.uint8, device="cuda")
    big[: L.packed.numel()].copy_(L.packed)
    moe.moe_route_topk(bad, big, xd, ids, w, ws)
    assert moe.moe_read_status(ws) == moe.MOE_ERR_PACKED
    assert moe.moe_read_status(ws) == moe.MOE_OK  # read clears


def test_bounded_wait_gives_up_with_timeout_status():
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    moe.moe_debug_wait_timeout(ws, 1000)
    assert moe.moe_read_status(ws) == moe.MOE_ERR_TIMEOUT
    # the context is still usable afterwards
    t = torch.ones(16, device="cuda")
    assert float(t.sum()) == 16.0
