"""Pins of the CPU oracle against what the pages and mathematics fix (no GPU).

Each test names the property it pins.  None of them re-types the oracle's own
formula: they use brute force, closed forms, library routines (numpy / scipy /
sympy), hand-worked examples of the pages' rules, exact invariants, or
structured inputs whose answer is known in advance.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special as sps
import sympy

import gen
import oracle
from _support import make_expert, make_experts, shared_expert

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    for ln in open(os.path.join(GOLD, name)):
        ln = ln.strip()
        if ln and not ln.startswith("#"):
            out.append(ln.split())
    return out


# ------------------------------------------------------------------ packing

def test_int4_pack_golden_nibble_order():
    """[DEEP §5.1] first element in the high nibble (hand-worked examples of the rule)."""
    for a, b, hx in _rows("int4_pack.txt"):
        p = oracle.pack_int4(np.array([int(a), int(b)], np.int8))
        assert p[0] == int(hx, 16), (a, b, hx, p)


def test_int2_pack_golden():
    for a, b, c, d, hx in _rows("int2_pack.txt"):
        p = oracle.pack_int2(np.array([int(a), int(b), int(c), int(d)], np.int8))
        assert p[0] == int(hx, 16)


def test_int4_pack_unpack_bit_identity_all_codes_all_positions():
    """[README 量化内核] packing is bit-identical to the int8 container: every code pair."""
    codes = np.arange(-8, 8, dtype=np.int8)
    q = np.array(list(itertools.product(codes, codes)), dtype=np.int8).ravel()
    assert np.array_equal(oracle.unpack_int4(oracle.pack_int4(q), q.size), q)
    # every byte value decodes to an in-range pair and re-encodes to itself
    allb = np.arange(256, dtype=np.uint8)
    qq = oracle.unpack_int4(allb, 512)
    assert qq.min() == -8 and qq.max() == 7
    assert np.array_equal(oracle.pack_int4(qq), allb)


def test_int2_pack_unpack_bit_identity_all_codes_all_positions():
    codes = np.arange(-2, 2, dtype=np.int8)
    q = np.array(list(itertools.product(codes, repeat=4)), dtype=np.int8).ravel()
    assert np.array_equal(oracle.unpack_int2(oracle.pack_int2(q), q.size), q)
    allb = np.arange(256, dtype=np.uint8)
    assert np.array_equal(oracle.pack_int2(oracle.unpack_int2(allb, 1024)), allb)


# ------------------------------------------------------------------ SwiGLU pieces

def test_silu_closed_form():
    """silu(z) = z * sigmoid(z), evaluated with exact sympy arithmetic (30 digits)."""
    Z = sympy.Symbol("z")
    f = Z / (1 + sympy.exp(-Z))
    for z in [0, 1, -1, 2, -2, 0.5, -3.25, 7, -7, 12.5, -20]:
        ref = float(sympy.N(f.subs(Z, sympy.nsimplify(z)), 30))
        assert oracle.silu(z) == pytest.approx(ref, rel=1e-15, abs=1e-300)
    assert oracle.silu(0.0) == 0.0
    # limits: silu(z) -> z for large z, -> 0 for very negative z
    assert oracle.silu(50.0) == 50.0
    assert abs(oracle.silu(-800.0)) == 0.0
    # scipy's logistic routine
    zz = np.linspace(-30, 30, 61)
    assert np.allclose([oracle.silu(z) for z in zz], zz * sps.expit(zz), rtol=1e-15, atol=1e-300)


def _tiny_spec(**kw):
    base = dict(name="t", hidden=64, inter=32, n_experts=8, top_k=2, router="softmax",
                x_dtype="f32")
    base.update(kw)
    return gen.LayerSpec(**base)


def _onehot_expert(H, I, gate_col, up_col, down_col, gq, uq, dq, sg, su, sd):
    """gate row i = gq[i] at column gate_col[i]; up row i = uq[i] at up_col[i];
    down row o = dq[o] at column down_col[o]; everything else 0."""
    g = np.zeros((I, H), np.int8)
    u = np.zeros((I, H), np.int8)
    d = np.zeros((H, I), np.int8)
    for i in range(I):
        g[i, gate_col[i]] = gq[i]
        u[i, up_col[i]] = uq[i]
    for o in range(H):
        if down_col[o] >= 0:
            d[o, down_col[o]] = dq[o]
    return oracle.Expert(g, u, d, np.asarray(sg, np.float32), np.asarray(su, np.float32),
                         np.asarray(sd, np.float32))


def test_expert_onehot_closed_form():
    """Structured weights whose output is known element by element:
    y[o] = s_d[o] dq[o] * silu(s_g[i] gq[i] x[a_i]) * s_u[i] uq[i] x[b_i], i = down_col[o].
    Asymmetric index maps catch transposed operands, swapped gate/up and index slips."""
    H, I = 8, 4
    gate_col = [3, 0, 6, 5]
    up_col = [1, 7, 2, 4]
    down_col = [2, -1, 0, 3, -1, 1, 2, 0]
    gq = [1, -2, 3, 7]
    uq = [2, 1, -8, 5]
    dq = [1, 0, -3, 4, 0, 6, -1, 2]
    sg = [0.5, 0.25, 1.0, 0.125]
    su = [1.0, 0.5, 0.25, 2.0]
    sd = [2.0, 1.0, 0.5, 0.25, 1.0, 1.0, 4.0, 0.75]
    ex = _onehot_expert(H, I, gate_col, up_col, down_col, gq, uq, dq, sg, su, sd)
    x = np.array([[1.0, -2.0, 0.5, 3.0, -1.5, 2.5, -0.75, 1.25]])
    s = _tiny_spec(hidden=H, inter=I)
    y = oracle.expert_forward(s, ex, x)[0]
    Z = sympy.Symbol("z")
    silu = sympy.Lambda(Z, Z / (1 + sympy.exp(-Z)))
    for o in range(H):
        i = down_col[o]
        if i < 0 or dq[o] == 0:
            assert y[o] == 0.0
            continue
        gv = sympy.nsimplify(sg[i] * gq[i] * x[0, gate_col[i]])
        uv = sympy.nsimplify(su[i] * uq[i] * x[0, up_col[i]])
        ref = sympy.nsimplify(sd[o] * dq[o]) * silu(gv) * uv
        assert y[o] == pytest.approx(float(sympy.N(ref, 30)), rel=1e-14)


def _numpy_swiglu(ex, x):
    """SwiGLU expert from library primitives (numpy matmul, scipy expit)."""
    Wg = ex.s_gate.astype(np.float64)[:, None] * ex.gate.astype(np.float64)
    Wu = ex.s_up.astype(np.float64)[:, None] * ex.up.astype(np.float64)
    Wd = ex.s_down.astype(np.float64)[:, None] * ex.down.astype(np.float64)
    g = x @ Wg.T
    u = x @ Wu.T
    h = g * sps.expit(g) * u
    return h @ Wd.T


@pytest.mark.parametrize("bits", [4, 8, 2])
def test_expert_vs_library_matmul(bits):
    s = _tiny_spec(weight_bits=bits)
    ex = make_expert(s, 3, 0, 5)
    x = np.random.default_rng(0).standard_normal((5, s.hidden))
    y = oracle.expert_forward(s, ex, x)
    ref = _numpy_swiglu(ex, x)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_zero_expert_and_power_of_two_scaling_exact():
    s = _tiny_spec()
    ex = make_expert(s, 1, 0, 2)
    x = np.random.default_rng(1).standard_normal((3, s.hidden))
    y = oracle.expert_forward(s, ex, x)
    z = oracle.Expert(np.zeros_like(ex.gate), ex.up, ex.down, ex.s_gate, ex.s_up, ex.s_down)
    assert np.all(oracle.expert_forward(s, z, x) == 0.0)          # silu(0) * u = 0
    z = oracle.Expert(ex.gate, np.zeros_like(ex.up), ex.down, ex.s_gate, ex.s_up, ex.s_down)
    assert np.all(oracle.expert_forward(s, z, x) == 0.0)
    d2 = oracle.Expert(ex.gate, ex.up, ex.down, ex.s_gate, ex.s_up, ex.s_down * 2)
    assert np.array_equal(oracle.expert_forward(s, d2, x), 2 * y)  # exact in fp64
    u2 = oracle.Expert(ex.gate, ex.up, ex.down, ex.s_gate, ex.s_up * 4, ex.s_down)
    assert np.array_equal(oracle.expert_forward(s, u2, x), 4 * y)


def test_router_logits_vs_library_matmul():
    s = _tiny_spec(hidden=96, n_experts=12)
    rng = np.random.default_rng(2)
    x = rng.standard_normal((7, s.hidden))
    wr = rng.standard_normal((s.n_experts, s.hidden)).astype(np.float32)
    lg = oracle.router_logits(s, x, wr)
    assert np.allclose(lg, x @ wr.astype(np.float64).T, rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ routing

def _rank_topk(score, cand, k):
    """top-k by (score desc, index asc) via numpy lexsort."""
    cand = np.asarray(cand)
    order = np.lexsort((cand, -score[cand]))
    return cand[order[:k]]


def test_softmax_route_vs_scipy_softmax():
    s = _tiny_spec(n_experts=16, top_k=4)
    lg = np.random.default_rng(3).standard_normal((50, 16)) * 3
    ids, w, margin = oracle.route(s, lg)
    p = sps.softmax(lg, axis=1)
    for t in range(50):
        ref = _rank_topk(p[t], np.arange(16), 4)
        assert list(ids[t]) == list(ref)
        assert np.allclose(w[t], p[t, ref] / p[t, ref].sum(), rtol=1e-13)
        srt = np.sort(p[t])[::-1]
        assert margin[t] == pytest.approx(np.min(srt[:4] - srt[1:5]), rel=1e-9, abs=1e-15)


def test_softmax_ties_go_to_lower_index():
    s = _tiny_spec(n_experts=6, top_k=3)
    lg = np.array([[0.0, 1.0, 1.0, 0.5, 1.0, 0.0]])
    ids, w, margin = oracle.route(s, lg)
    assert list(ids[0]) == [1, 2, 4]
    assert margin[0] == 0.0
    assert np.allclose(w[0], 1 / 3)


def test_softmax_k_equals_E_is_dense_softmax_mixture():
    s = _tiny_spec(n_experts=8, top_k=8)
    lg = np.random.default_rng(4).standard_normal((6, 8))
    ids, w, _ = oracle.route(s, lg)
    p = sps.softmax(lg, axis=1)
    for t in range(6):
        assert np.allclose(w[t], p[t, ids[t]], rtol=1e-13)
        assert sorted(ids[t]) == list(range(8))


def test_norm_topk_off_keeps_raw_probabilities():
    s = _tiny_spec(n_experts=8, top_k=2, norm_topk=0)
    lg = np.random.default_rng(5).standard_normal((4, 8))
    ids, w, _ = oracle.route(s, lg)
    p = sps.softmax(lg, axis=1)
    for t in range(4):
        assert np.allclose(w[t], p[t, ids[t]], rtol=1e-13)


def _grouped_brute(lg_row, bias, E, G, tg, k, rsf):
    """Brute force of the grouped router: best group subset by exhaustive search over all
    C(G, tg) subsets (maximum total group score, where a group's score is the best
    pair sum over all pairs), then experts ranked by counting how many candidates beat each."""
    s = 1.0 / (1.0 + np.exp(-lg_row))
    c = s + bias
    gs = E // G
    gscore = []
    for g in range(G):
        m = c[g * gs:(g + 1) * gs]
        if gs == 1:
            gscore.append(m[0])
        else:
            gscore.append(max(m[i] + m[j] for i in range(gs) for j in range(i + 1, gs)))
    best = max(itertools.combinations(range(G), tg), key=lambda sub: sum(gscore[g] for g in sub))
    cand = [e for e in range(E) if e // gs in best]
    beats = {e: sum(1 for f in cand if c[f] > c[e] or (c[f] == c[e] and f < e)) for e in cand}
    sel = sorted([e for e in cand if beats[e] < k], key=lambda e: beats[e])
    w = s[sel] / s[sel].sum() * rsf
    return sel, w


def test_grouped_route_vs_brute_force():
    s = _tiny_spec(n_experts=32, top_k=4, router="sigmoid_grouped", n_group=8, topk_group=3,
                   rsf=2.5)
    rng = np.random.default_rng(6)
    lg = rng.standard_normal((40, 32)) * 2
    bias = (rng.standard_normal(32) * 0.3).astype(np.float32)
    ids, w, _ = oracle.route(s, lg, bias)
    for t in range(40):
        sel, wr = _grouped_brute(lg[t], bias.astype(np.float64), 32, 8, 3, 4, 2.5)
        assert list(ids[t]) == sel
        assert np.allclose(w[t], wr, rtol=1e-13)


def test_grouped_weights_sum_to_rsf_and_use_uncorrected_scores():
    s = gen.spec("dsv3")
    rng = np.random.default_rng(7)
    lg = rng.standard_normal((64, 256)) * 1.5
    bias = (rng.standard_normal(256) * 0.1).astype(np.float32)
    ids, w, _ = oracle.route(s, lg, bias)
    assert np.all(np.abs(w.sum(1) - 2.5) <= 1e-12)
    sig = sps.expit(lg)
    for t in range(64):
        assert np.allclose(w[t] / 2.5, sig[t, ids[t]] / sig[t, ids[t]].sum(), rtol=1e-13)
        # at most topk_group groups touched; ids distinct
        assert len(set(ids[t] // 32)) <= 4 and len(set(ids[t])) == 8


def test_grouped_single_group_is_plain_sigmoid_topk():
    s = _tiny_spec(n_experts=16, top_k=5, router="sigmoid_grouped", n_group=1, topk_group=1)
    rng = np.random.default_rng(8)
    lg = rng.standard_normal((20, 16))
    bias = (rng.standard_normal(16) * 0.2).astype(np.float32)
    ids, w, _ = oracle.route(s, lg, bias)
    c = sps.expit(lg) + bias.astype(np.float64)
    for t in range(20):
        assert list(ids[t]) == list(_rank_topk(c[t], np.arange(16), 5))


def test_grouped_zero_bias_rsf1_matches_softmax_free_sigmoid_weights():
    s = _tiny_spec(n_experts=16, top_k=3, router="sigmoid_grouped", n_group=4, topk_group=4)
    lg = np.random.default_rng(9).standard_normal((10, 16))
    ids, w, _ = oracle.route(s, lg, None)
    sig = sps.expit(lg)
    for t in range(10):
        # all groups kept -> plain top-k of sigmoid (monotone in the logit)
        assert list(ids[t]) == list(_rank_topk(lg[t], np.arange(16), 3))
        assert np.allclose(w[t], sig[t, ids[t]] / sig[t, ids[t]].sum(), rtol=1e-13)


def test_permutation_vs_stable_argsort():
    rng = np.random.default_rng(10)
    T, k, E = 37, 4, 11
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    off, perm = oracle.permutation(ids, E)
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(ids.ravel(), minlength=E))]))
    assert np.array_equal(perm, np.argsort(ids.ravel(), kind="stable"))


# ------------------------------------------------------------------ the whole layer

def _tiny_layer(router="softmax", **kw):
    if router == "softmax":
        s = _tiny_spec(n_experts=8, top_k=2, **kw)
    else:
        s = _tiny_spec(n_experts=16, top_k=4, router="sigmoid_grouped", n_group=4, topk_group=2,
                       rsf=2.5, n_shared=1, bias_std=0.1, **kw)
    seed = 11
    wr = gen.router_weights(s, seed)
    bias = gen.router_bias(s, seed)
    experts = make_experts(s, seed, 0)
    sh = shared_expert(s, seed, 0)
    x, _ = gen.hidden_states(s, seed, 0, 9)
    return s, x.astype(np.float64), wr, bias, experts, sh


@pytest.mark.parametrize("router", ["softmax", "sigmoid_grouped"])
def test_layer_brute_force_dense_then_mask(router):
    """Every expert evaluated densely on every token, then masked to the routed top-k."""
    s, x, wr, bias, experts, sh = _tiny_layer(router)
    ids, w, out = oracle.layer_forward(s, x, wr, bias, experts, sh, mode=1)
    dense = np.stack([_numpy_swiglu(experts[e], x) for e in range(s.n_experts)])  # [E,T,H]
    mask = np.zeros((x.shape[0], s.n_experts))
    lg = x @ wr.astype(np.float64).T
    if router == "softmax":
        p = sps.softmax(lg, axis=1)
        for t in range(x.shape[0]):
            top = _rank_topk(p[t], np.arange(s.n_experts), s.top_k)
            mask[t, top] = p[t, top] / p[t, top].sum()
    else:
        for t in range(x.shape[0]):
            sel, wt = _grouped_brute(lg[t], bias.astype(np.float64), s.n_experts, s.n_group,
                                     s.topk_group, s.top_k, s.rsf)
            mask[t, sel] = wt
    ref = np.einsum("te,eth->th", mask, dense)
    if sh is not None:
        ref += _numpy_swiglu(sh, x)
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-11 * np.abs(ref).max())
    assert np.allclose(w.sum(1), s.rsf, atol=1e-12)


@pytest.mark.parametrize("router", ["softmax", "sigmoid_grouped"])
def test_union_equals_per_token_exactly(router):
    s, x, wr, bias, experts, sh = _tiny_layer(router)
    i0, w0, o0 = oracle.layer_forward(s, x, wr, bias, experts, sh, mode=0)
    i1, w1, o1 = oracle.layer_forward(s, x, wr, bias, experts, sh, mode=1)
    assert np.array_equal(i0, i1) and np.array_equal(w0, w1)
    assert np.array_equal(o0, o1)


def test_single_expert_layer_is_plain_swiglu():
    """E=1, k=1 softmax: w = 1 and out = the expert's SwiGLU FFN."""
    s = _tiny_spec(n_experts=1, top_k=1)
    ex = make_expert(s, 12, 0, 0)
    x = np.random.default_rng(13).standard_normal((4, s.hidden))
    wr = np.ones((1, s.hidden), np.float32)
    ids, w, out = oracle.layer_forward(s, x, wr, None, {0: ex}, None)
    assert np.all(ids == 0) and np.all(w == 1.0)
    assert np.array_equal(out, oracle.expert_forward(s, ex, x))


def test_doubling_one_experts_down_scale_doubles_exactly_its_term():
    s, x, wr, bias, experts, sh = _tiny_layer("softmax")
    ids, w, out = oracle.layer_forward(s, x, wr, bias, experts, sh)
    e = int(ids[0, 0])
    ex = experts[e]
    ex2 = dict(experts)
    ex2[e] = oracle.Expert(ex.gate, ex.up, ex.down, ex.s_gate, ex.s_up, ex.s_down * 2)
    _, _, out2 = oracle.layer_forward(s, x, wr, bias, ex2, sh)
    term = np.zeros_like(out)
    for t in range(x.shape[0]):
        for j in range(s.top_k):
            if ids[t, j] == e:
                term[t] += w[t, j] * oracle.expert_forward(s, ex, x[t:t + 1])[0]
    assert np.allclose(out2 - out, term, rtol=1e-12, atol=1e-12 * np.abs(out).max())


def test_all_zero_expert_contributes_exactly_zero():
    s, x, wr, bias, experts, sh = _tiny_layer("softmax")
    ids, w, out = oracle.layer_forward(s, x, wr, bias, experts, sh)
    e = int(ids[0, 0])
    ex2 = dict(experts)
    z = experts[e]
    ex2[e] = oracle.Expert(np.zeros_like(z.gate), z.up, z.down, z.s_gate, z.s_up, z.s_down)
    _, _, out2 = oracle.layer_forward(s, x, wr, bias, ex2, sh)
    rows = [t for t in range(x.shape[0]) if e not in ids[t]]
    assert np.array_equal(out2[rows], out[rows])
    # tokens that did route to e lose exactly that term (order of the remaining sum intact
    # only for k = 2 when e sits in the last slot; check the value instead)
    for t in range(x.shape[0]):
        if e in ids[t]:
            j = list(ids[t]).index(e)
            other = [jj for jj in range(s.top_k) if jj != j]
            ref = sum(w[t, jj] * oracle.expert_forward(s, experts[int(ids[t, jj])], x[t:t + 1])[0]
                      for jj in other)
            assert np.allclose(out2[t], ref, rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------------ Q8_0 mode

def test_q8_0_hand_worked_block():
    """amax = 127 gives d = 1, so q = round-half-away(v): worked by hand."""
    v = np.zeros(32, np.float32)
    v[:8] = [127.0, 0.5, -0.5, 1.5, -2.5, 63.49, -126.6, 0.49]
    q, d = oracle.q8_0_encode(v)
    assert d[0] == 1.0
    assert list(q[:8]) == [127, 1, -1, 2, -3, 63, -127, 0]
    assert np.all(q[8:] == 0)


def test_q8_0_zero_block_and_scaling():
    q, d = oracle.q8_0_encode(np.zeros(64, np.float32))
    assert np.all(q == 0) and np.all(d == 0)
    v = np.arange(32, dtype=np.float32) - 16          # amax 16
    q, d = oracle.q8_0_encode(v)
    assert d[0] == np.float32(16) / np.float32(127)
    assert q[0] == -127 and q[-1] == round(15 * 127 / 16)


def test_q8_0_reencode_of_decoded_is_identity():
    rng = np.random.default_rng(14)
    v = (rng.standard_normal(32 * 500) * rng.uniform(0.01, 100, 32 * 500)).astype(np.float32)
    q, d = oracle.q8_0_encode(v)
    dec = (q.reshape(-1, 32).astype(np.float32) * d[:, None]).astype(np.float32).ravel()
    q2, d2 = oracle.q8_0_encode(dec)
    assert np.array_equal(q2, q)


def test_block_dot_vs_numpy_int64():
    rng = np.random.default_rng(15)
    for _ in range(200):
        a = rng.integers(-127, 128, 32).astype(np.int8)
        b = rng.integers(-128, 128, 32).astype(np.int8)
        assert oracle.block_dot(a, b) == int(a.astype(np.int64) @ b.astype(np.int64))
    a = np.full(32, -128, np.int8)
    assert oracle.block_dot(a, a) == 32 * 128 * 128


def test_q8_expert_vs_library_on_decoded_activations():
    """Q8_0 expert == SwiGLU on the Q8_0-decoded activations (library matmul), with h
    rounded to fp32 and re-encoded before the down projection."""
    s = _tiny_spec(hidden=128, inter=64, weight_bits=8, act_q8_0=1)
    ex = make_expert(s, 16, 0, 1)
    x = np.random.default_rng(17).standard_normal((3, s.hidden)).astype(np.float32)
    y = oracle.expert_forward(s, ex, x.astype(np.float64))
    qx, dx = oracle.q8_0_encode(x)
    xd = qx.reshape(3, -1, 32).astype(np.float64) * dx.reshape(3, -1, 1).astype(np.float64)
    xd = xd.reshape(3, -1)
    Wg = ex.s_gate.astype(np.float64)[:, None] * ex.gate
    Wu = ex.s_up.astype(np.float64)[:, None] * ex.up
    Wd = ex.s_down.astype(np.float64)[:, None] * ex.down
    g, u = xd @ Wg.T, xd @ Wu.T
    h = (g * sps.expit(g) * u).astype(np.float32)
    qh, dh = oracle.q8_0_encode(h)
    hd = (qh.reshape(3, -1, 32).astype(np.float64) * dh.reshape(3, -1, 1)).reshape(3, -1)
    ref = hd @ Wd.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_q8_layer_union_equals_per_token():
    s = _tiny_spec(hidden=128, inter=64, weight_bits=8, act_q8_0=1)
    seed = 18
    wr = gen.router_weights(s, seed)
    experts = make_experts(s, seed, 0)
    x, _ = gen.hidden_states(s, seed, 0, 6)
    a = oracle.layer_forward(s, x.astype(np.float64), wr, None, experts, None, mode=0)
    b = oracle.layer_forward(s, x.astype(np.float64), wr, None, experts, None, mode=1)
    assert all(np.array_equal(p, q) for p, q in zip(a, b))


# ---------------------------------------------------------------- stack harness (residual + RMSNorm)

def _bf16_exact(v):
    """True where v (fp64) is exactly a bf16 number."""
    f = v.astype(np.float32)
    return (f.astype(np.float64) == v) & ((f.view(np.uint32) & 0xFFFF) == 0)


def test_residual_rmsnorm_properties():
    """RMSNorm output has unit RMS (up to the bf16 rounding of its elements), is exactly
    invariant to scaling its input by a power of two (eps = 0), is bf16-representable, and
    the residual update is the exact fp64 sum."""
    rng = np.random.default_rng(7)
    r0 = rng.standard_normal((5, 256)) * rng.uniform(0.1, 30.0, size=(5, 1))
    add = rng.standard_normal((5, 256))
    r1, x1 = oracle.residual_rmsnorm(r0, add, eps=0.0)
    assert np.array_equal(r1, r0 + add)
    rms = np.sqrt(np.mean(x1 * x1, axis=1))
    assert np.all(np.abs(rms - 1.0) < 2.0 ** -8)
    assert np.all(_bf16_exact(x1))
    _, x2 = oracle.residual_rmsnorm(r1 * 8.0, None, eps=0.0)
    assert np.array_equal(x1, x2)
    # each element is the nearest bf16 of its exact normalised value: within half an ulp
    exact = r1 / np.sqrt(np.mean(r1 * r1, axis=1, keepdims=True))
    ulp = 2.0 ** (np.floor(np.log2(np.abs(exact))) - 7)
    assert np.all(np.abs(x1 - exact) <= 0.5 * ulp + 1e-300)


def test_residual_rmsnorm_eps_and_first_layer():
    """eps enters as mean(r^2) + eps (a constant row normalises to r/sqrt(r^2+eps)); with
    no addend r is unchanged."""
    r = np.full((1, 64), 0.01)
    r1, x = oracle.residual_rmsnorm(r, None, eps=1e-4)
    assert np.array_equal(r1, r)
    want = 0.01 / np.sqrt(1e-4 + 1e-4)
    assert np.all(np.abs(x - want) <= 2.0 ** -9 * abs(want))


# ---------------------------------------------------------------- quantiser ([DEEP] §5.1)

def test_quantize_hand_worked():
    """Rows whose scale is a power of two, so every ratio is exact: s = amax / qmax, codes
    round half away from zero ("colibrì 深度拆解" §5.1 quantize_row, roundf)."""
    # int4: amax 3.5 -> s = 0.5; ratios 7, -3.5, 0.5, 0, -7, 1.5 -> 7, -4, 1, 0, -7, 2
    q, s = oracle.quantize_rows(np.array([[3.5, -1.75, 0.25, 0.0, -3.5, 0.75]], np.float32), 4)
    assert s[0] == 0.5 and q.tolist() == [[7, -4, 1, 0, -7, 2]]
    # int8: amax 127 -> s = 1; -63.5 -> -64, 0.5 -> 1, -0.5 -> -1
    q, s = oracle.quantize_rows(np.array([[127.0, -63.5, 0.5, -0.5, 2.0, -127.0]], np.float32), 8)
    assert s[0] == 1.0 and q.tolist() == [[127, -64, 1, -1, 2, -127]]
    # int2: amax 1 -> s = 1; 0.5 -> 1, -0.5 -> -1, -1 -> -1, 0.25 -> 0
    q, s = oracle.quantize_rows(np.array([[1.0, 0.5, -0.5, -1.0, 0.25, 0.0]], np.float32), 2)
    assert s[0] == 1.0 and q.tolist() == [[1, 1, -1, -1, 0, 0]]
    # a zero row: s = 0, codes 0
    q, s = oracle.quantize_rows(np.zeros((1, 8), np.float32), 4)
    assert s[0] == 0.0 and not q.any()


@pytest.mark.parametrize("bits", [8, 4, 2])
def test_quantize_properties(bits):
    """Random rows: the largest magnitude maps to +-qmax, every code reconstructs its weight
    to within half a step, codes stay in range, and scaling a row by 2 scales s by 2 with the
    same codes (exact in fp32)."""
    rng = np.random.default_rng(bits)
    w = (rng.standard_normal((16, 96)) * rng.uniform(0.01, 5.0, (16, 1))).astype(np.float32)
    q, s = oracle.quantize_rows(w, bits)
    qmax = (1 << (bits - 1)) - 1
    assert q.min() >= -(qmax + 1) and q.max() <= qmax
    amax_col = np.argmax(np.abs(w), axis=1)
    assert np.array_equal(np.abs(q[np.arange(16), amax_col]), np.full(16, qmax))
    err = np.abs(w.astype(np.float64) - q.astype(np.float64) * s[:, None].astype(np.float64))
    assert np.all(err <= 0.5 * s[:, None] * (1 + 1e-6))
    q2, s2 = oracle.quantize_rows(w * 2, bits)
    assert np.array_equal(q2, q) and np.array_equal(s2, 2 * s)


# ------------------------------------------------------------------ adaptive expert top-p
# Reading of "Show HN" 实用调节项 (--topp, an explicit lossy override): after the top-k
# selection, in slot order keep the shortest prefix whose share of the selected weight
# sources reaches p (at least one expert); dropped slots: id -1, weight 0; kept weights
# normalised over the kept experts.

def test_topp_off_values_change_nothing():
    s = _tiny_spec(n_experts=16, top_k=4)
    lg = np.random.default_rng(21).standard_normal((30, 16)) * 2
    ref = oracle.route(s, lg)
    for p in (0.0, 1.0, 1.5):
        got = oracle.route(s.replace(top_p=p), lg)
        for a, b in zip(ref, got):
            assert np.array_equal(a, b)


def test_topp_hand_worked_softmax():
    """p = (0.5, 0.3, 0.15, 0.05), k = 3: shares of the selected mass 0.95 are
    0.526, 0.316, 0.158; at top_p 0.7 the share before slot 2 is 0.842 >= 0.7, so two
    experts stay, weighted 0.5 / 0.8 and 0.3 / 0.8."""
    s = _tiny_spec(n_experts=4, top_k=3, top_p=0.7)
    lg = np.log(np.array([[0.5, 0.3, 0.15, 0.05]]))
    ids, w, margin = oracle.route(s, lg)
    assert list(ids[0]) == [0, 1, -1]
    assert w[0] == pytest.approx([0.625, 0.375, 0.0], rel=1e-13, abs=0)
    # the closest decision: the share before the dropped slot (0.8 / 0.95) against 0.7
    assert margin[0] == pytest.approx(min(0.8 / 0.95 - 0.7, 0.7 - 0.5 / 0.95, 0.15 - 0.05),
                                      rel=1e-9)
    ids, w, _ = oracle.route(s.replace(top_p=0.5), lg)  # 0.526 > 0.5 already: one expert
    assert list(ids[0]) == [0, -1, -1] and w[0] == pytest.approx([1.0, 0.0, 0.0])


def test_topp_tiny_p_keeps_one_expert_with_the_whole_weight():
    s = _tiny_spec(n_experts=16, top_k=4, router="sigmoid_grouped", n_group=4, topk_group=2,
                   rsf=2.5, top_p=1e-9)
    lg = np.random.default_rng(22).standard_normal((20, 16))
    ids0, _, _ = oracle.route(s.replace(top_p=0.0), lg)
    ids, w, _ = oracle.route(s, lg)
    assert np.array_equal(ids[:, 0], ids0[:, 0])
    assert np.all(ids[:, 1:] == -1) and np.all(w[:, 1:] == 0.0)
    assert np.allclose(w[:, 0], 2.5, rtol=1e-14)


@pytest.mark.parametrize("router", ["softmax", "sigmoid_grouped"])
def test_topp_invariants(router):
    """Kept prefix: share before its last slot < p <= share of the whole prefix (or all
    k kept); kept weights sum to rsf; the kept ids are the top-k ids' prefix."""
    if router == "softmax":
        s = _tiny_spec(n_experts=16, top_k=6, top_p=0.6)
    else:
        s = _tiny_spec(n_experts=32, top_k=6, router="sigmoid_grouped", n_group=4,
                       topk_group=2, rsf=2.5, top_p=0.6)
    lg = np.random.default_rng(23).standard_normal((40, s.n_experts)) * 1.5
    ids0, w0, _ = oracle.route(s.replace(top_p=0.0), lg)
    ids, w, _ = oracle.route(s, lg)
    for t in range(40):
        m = int(np.sum(ids[t] >= 0))
        assert m >= 1 and np.all(ids[t, m:] == -1) and np.all(w[t, m:] == 0.0)
        assert np.array_equal(ids[t, :m], ids0[t, :m])
        share = w0[t] / w0[t].sum()  # w0 is proportional to the weight sources
        assert share[:m - 1].sum() < 0.6 and (m == s.top_k or share[:m].sum() >= 0.6)
        assert w[t, :m].sum() == pytest.approx(s.rsf, rel=1e-13)
        assert np.allclose(w[t, :m] / w[t, :m].sum(), w0[t, :m] / w0[t, :m].sum(), rtol=1e-13)


def test_topp_layer_union_equals_per_token_and_drops_experts():
    s, x, wr, bias, experts, sh = _tiny_layer("sigmoid_grouped", top_p=0.5)
    i0, w0, o0 = oracle.layer_forward(s, x, wr, bias, experts, sh, mode=0)
    i1, w1, o1 = oracle.layer_forward(s, x, wr, bias, experts, sh, mode=1)
    assert np.array_equal(i0, i1) and np.array_equal(w0, w1) and np.array_equal(o0, o1)
    assert np.any(i1 < 0)
    off, perm = oracle.permutation(i1, s.n_experts)
    n = int(np.sum(i1 >= 0))
    assert off[-1] == n and np.all(perm[n:] == -1)
    flat = i1.ravel()
    assert sorted(perm[:n].tolist()) == sorted(np.flatnonzero(flat >= 0).tolist())
    # the layer equals the plain definition: shared + sum over kept slots of w * expert
    ref = oracle.expert_forward(s, sh, x)
    for t in range(x.shape[0]):
        for j in range(s.top_k):
            if i1[t, j] >= 0:
                ref[t] += w1[t, j] * oracle.expert_forward(s, experts[i1[t, j]], x[t:t + 1])[0]
    assert np.allclose(o1, ref, rtol=1e-12, atol=1e-12)
