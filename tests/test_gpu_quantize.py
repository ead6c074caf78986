"""The per-row weight quantiser ("colibrì 深度拆解" §5.1 quantize_row) on the GPU against the
oracle: codes and scales bit for bit (both sides decide in fp32, as the page does), fp32 and
bf16 inputs, rows with exact halves, zero rows and a ragged column count; then the codes
feed moe_pack_expert and come back unchanged through moe_unpack_weights."""
import numpy as np
import pytest
import torch

import gen
import oracle
import routed_expert_ffn_route_gb300 as moe

pytestmark = pytest.mark.gpu


def seeded_rows(rows, cols, seed):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((rows, cols)) * rng.uniform(1e-3, 10.0, (rows, 1))).astype(np.float32)
    w[0] = 0.0                                           # a zero row
    w[1, : cols // 2] = 0.5 * np.arange(cols // 2) - 3.0  # exact halves when s is a power of 2
    w[1, cols // 2:] = 0.0
    w[1, 0] = 7.0 * 0.5                                  # amax 3.5 -> s = 0.5 at int4
    return w


@pytest.mark.parametrize("bits", [8, 4, 2])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", [64, 300, 6144])
def test_quantize_rows_bit_exact(bits, dtype, cols):
    w = seeded_rows(37, cols, bits * 1000 + cols)
    if dtype == "bf16":
        bits16 = gen.bf16_round_bits(w)
        w = (bits16.astype(np.uint32) << 16).view(np.float32)  # the exact bf16 values
        w_dev = torch.from_numpy(bits16.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        w_dev = torch.from_numpy(w).cuda()
    q = torch.empty(w.shape, dtype=torch.int8, device="cuda")
    s = torch.empty(w.shape[0], dtype=torch.float32, device="cuda")
    moe.moe_quantize_rows(w_dev, bits, q, s)
    q_o, s_o = oracle.quantize_rows(w, bits)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_o.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q_o)


def test_quantized_expert_packs_and_unpacks():
    """Float weights -> GPU quantiser -> pack -> unpack gives the quantiser's codes back."""
    s = gen.spec("tiny").replace(n_shared=0)
    cfg = moe.make_config(s.hidden, s.inter, s.n_experts, s.top_k, router=s.router,
                          weight_bits=4)
    packed = torch.empty(moe.moe_packed_bytes(cfg), dtype=torch.uint8, device="cuda")
    rng = np.random.default_rng(5)
    mats = {"gate": (s.inter, s.hidden), "up": (s.inter, s.hidden), "down": (s.hidden, s.inter)}
    q, sc = {}, {}
    for name, shape in mats.items():
        w = torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).cuda()
        q[name] = torch.empty(shape, dtype=torch.int8, device="cuda")
        sc[name] = torch.empty(shape[0], dtype=torch.float32, device="cuda")
        moe.moe_quantize_rows(w, 4, q[name], sc[name])
    moe.moe_pack_router(cfg, torch.zeros((s.n_experts, s.hidden), device="cuda"), None, packed)
    for e in range(s.n_experts):
        moe.moe_pack_expert(cfg, e, q["gate"], q["up"], q["down"], sc["gate"], sc["up"],
                            sc["down"], packed)
    back = {n: torch.empty_like(q[n]) for n in mats}
    moe.moe_unpack_weights(cfg, packed, 3, back["gate"], back["up"], back["down"])
    torch.cuda.synchronize()
    for n in mats:
        assert torch.equal(back[n], q[n])
