"""Writes zipf_beta.txt: the router-bias scale beta of the Zipf-skewed stack of
DeepSeek-V3-shaped layers.

Reading (the pages are silent): b_e = -beta * 1.1 * ln(rank_e) with rank a seeded
permutation of the experts, beta chosen so that the least-squares slope of
log(selection frequency) against log(rank), over ranks 8..128, is -1.1 (a token takes an
expert at most once, so the top ranks saturate and are left out of the fit).  Frequencies
come from the CPU oracle's router (fp64) on 1024 seeded tokens of layer 0; beta is found
by bisection.  Calls only oracle/ and gen/.

    python tests/golden/fit_zipf_beta.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import gen  # noqa: E402
import oracle  # noqa: E402

TOKENS, SEED, LAYER, TARGET, RANKS = 1024, 0, 0, -1.1, (8, 128)


def slope(spec, logits, rank, beta):
    ids, _, _ = oracle.route(spec, logits, gen.zipf_bias(spec, SEED, LAYER, beta))
    freq = np.bincount(ids.ravel().astype(np.int64), minlength=spec.n_experts) / logits.shape[0]
    by_rank = np.empty(spec.n_experts)
    by_rank[rank - 1] = freq
    lo, hi = RANKS
    r = np.arange(lo, hi + 1)
    f = by_rank[lo - 1:hi]
    keep = f > 0
    return np.polyfit(np.log(r[keep]), np.log(f[keep]), 1)[0], by_rank


def main():
    spec = gen.spec("dsv3")
    x, _ = gen.hidden_states(spec, SEED, 900, TOKENS)
    logits = oracle.router_logits(spec, x.astype(np.float64), gen.router_weights(spec, SEED, LAYER))
    rank = gen.zipf_rank(spec, SEED, LAYER)
    lo, hi = 0.0, 1.0
    while slope(spec, logits, rank, hi)[0] > TARGET:
        hi *= 2
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if slope(spec, logits, rank, mid)[0] > TARGET:
            lo = mid
        else:
            hi = mid
    beta = 0.5 * (lo + hi)
    s, by_rank = slope(spec, logits, rank, beta)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "zipf_beta.txt")
    with open(path, "w") as f:
        f.write("# Zipf(1.1) router-bias scale of the stacked DeepSeek-V3-shaped layers, fitted by\n"
                "# tests/golden/fit_zipf_beta.py (CPU oracle router, 1024 seeded tokens of layer 0)\n")
        f.write(f"beta {beta:.9g}\n")
        f.write(f"slope {s:.6f}  (log frequency vs log rank, ranks {RANKS[0]}..{RANKS[1]})\n")
        f.write("frequency_by_rank_1_to_16 " + " ".join(f"{v:.4f}" for v in by_rank[:16]) + "\n")
        f.write(f"experts_never_selected {int(np.sum(by_rank == 0))}\n")
    print(open(path).read())


if __name__ == "__main__":
    main()
