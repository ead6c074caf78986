"""Shared helpers of the test-suite: seeded layers for the oracle, near-tie filter."""
from __future__ import annotations

import numpy as np

import gen
import oracle


def make_expert(s: gen.LayerSpec, seed: int, layer: int, e: int) -> oracle.Expert:
    """Expert e of layer `layer` (e == E is the shared expert) from the seeded generator."""
    return oracle.Expert(
        gate=gen.expert_codes(s, seed, layer, e, "gate"),
        up=gen.expert_codes(s, seed, layer, e, "up"),
        down=gen.expert_codes(s, seed, layer, e, "down"),
        s_gate=gen.expert_scales(s, seed, layer, e, "gate"),
        s_up=gen.expert_scales(s, seed, layer, e, "up"),
        s_down=gen.expert_scales(s, seed, layer, e, "down"),
    )


def make_experts(s, seed, layer, which=None) -> dict:
    which = range(s.n_experts) if which is None else which
    return {int(e): make_expert(s, seed, layer, int(e)) for e in which}


def shared_expert(s, seed, layer):
    return make_expert(s, seed, layer, s.n_experts) if s.n_shared else None


def filtered_hidden(s, seed, batch, T, wr, bias, min_margin=1e-4, max_rounds=50):
    """Hidden states whose routing decisions all have a score margin >= min_margin.

    Tokens whose oracle margin is below the threshold are redrawn from the next
    draw index of their own row stream.  Returns (x_f32, x_bits, ids, w, margin,
    n_redraws)."""
    draws = np.zeros(T, dtype=np.int64)
    x, bits = gen.hidden_states(s, seed, batch, T, draws)
    logits = oracle.router_logits(s, x.astype(np.float64), wr)
    ids, w, margin = oracle.route(s, logits, bias)
    redraws = 0
    for _ in range(max_rounds):
        bad = np.nonzero(margin < min_margin)[0]
        if bad.size == 0:
            break
        redraws += bad.size
        draws[bad] += 1
        xb, bb = gen.hidden_states(s, seed, batch, T, draws, rows=bad)
        x[bad] = xb
        if bits is not None:
            bits[bad] = bb
        lg = oracle.router_logits(s, x[bad].astype(np.float64), wr)
        i2, w2, m2 = oracle.route(s, lg, bias)
        ids[bad], w[bad], margin[bad] = i2, w2, m2
    else:
        raise RuntimeError("near-tie filter did not converge")
    return x, bits, ids, w, margin, redraws


def err_stats(got: np.ndarray, ref: np.ndarray):
    """(max|err| / RMS(ref), ||err||_F / ||ref||_F)"""
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    d = got - ref
    rms = np.sqrt(np.mean(ref * ref))
    return float(np.max(np.abs(d)) / rms), float(np.linalg.norm(d) / np.linalg.norm(ref))


# the floating-point parity bar: max|err| <= 2e-3 * RMS(out), relative Frobenius <= 1e-3
MAX_REL_RMS = 2e-3
FROB_REL = 1e-3
