"""Planted mistakes in the oracle must each fail at least one pin.

Each case edits one line of a copy of the oracle's C source (a dropped term, a
wrong sign, a slipped index, a transposed operand, a wrong tie rule ...),
compiles it to a temporary library and runs the pin suite against it in a
subprocess.  The suite has to go red for every mutant.  The real oracle source
is never modified.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

MUTANTS = {
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "gate_up_swapped": ("h[i] = orc_silu(g[i]) * u[i];", "h[i] = orc_silu(u[i]) * g[i];"),
    "row_scale_index": ("wrow[cc] = (double)s[r] * (double)q[(size_t)r * cols + cc];",
                        "wrow[cc] = (double)s[cc % rows] * (double)q[(size_t)r * cols + cc];"),
    "weight_transposed": ("wrow[cc] = (double)s[r] * (double)q[(size_t)r * cols + cc];",
                          "wrow[cc] = (double)s[r] * (double)q[((size_t)cc * rows + r) % ((size_t)rows * cols)];"),
    "no_renorm": ("if (c->norm_topk) v = v / wsum;", "if (c->norm_topk) v = v;"),
    "weights_from_corrected": ("      wsrc[e] = s;\n", "      wsrc[e] = s + (bias ? (double)bias[e] : 0.0);\n"),
    "group_score_top1": ("gscore[g] = sel_score[msorted[0]] + (gs > 1 ? sel_score[msorted[1]] : 0.0);",
                         "gscore[g] = sel_score[msorted[0]];"),
    "ties_to_higher": ("if (best < 0 || score[cand[i]] > score[cand[best]]) best = i;",
                       "if (best < 0 || score[cand[i]] >= score[cand[best]]) best = i;"),
    "perm_slot_major": ("    for (int t = 0; t < T; t++)\n      for (int j = 0; j < k; j++)\n        if (ids[t * k + j] == e)",
                        "    for (int j = 0; j < k; j++)\n      for (int t = 0; t < T; t++)\n        if (ids[t * k + j] == e)"),
    "shared_dropped": ("if (c->n_shared) orc_expert_forward(c, shared, x, T, out);",
                       "if (0) orc_expert_forward(c, shared, x, T, out);"),
    "combine_weight_dropped": ("out[(size_t)t * H + h] += w[t * k + j] * yslot",
                               "out[(size_t)t * H + h] += yslot"),
    "q8_round_half_even": ("float rr = roundf(r);", "float rr = rintf(r);"),
    "q8_scale_128": ("volatile float db = amax / 127.0f;", "volatile float db = amax / 128.0f;"),
    "int4_no_sign_ext": ("q[i] = sext(p[i / 2] >> 4, 4);", "q[i] = (int8_t)(p[i / 2] >> 4);"),
    "int4_nibble_order": ("out[i / 2] = (uint8_t)(((q[i] & 0xF) << 4) | (q[i + 1] & 0xF));",
                          "out[i / 2] = (uint8_t)(((q[i + 1] & 0xF) << 4) | (q[i] & 0xF));"),
    "logit_index": ("acc += x[(size_t)t * H + h] * (double)wr[(size_t)e * H + h];",
                    "acc += x[(size_t)t * H + h] * (double)wr[((size_t)h * E + e) % ((size_t)E * H)];"),
    "sigmoid_sign": ("double s = 1.0 / (1.0 + exp(-l[e]));", "double s = 1.0 / (1.0 + exp(l[e]));"),
    "block_dot_offset": ("acc += (int32_t)a[i] * (int32_t)b[i];", "acc += (int32_t)a[i] * (int32_t)b[31 - i];"),
    "rmsnorm_sum_not_mean": ("const double inv = 1.0 / sqrt(ss / H + eps);",
                             "const double inv = 1.0 / sqrt(ss + eps);"),
    "rmsnorm_residual_dropped": ("if (add)\n      for (int h = 0; h < H; h++) rt[h] += add[(size_t)t * H + h];",
                                 "if (0)\n      for (int h = 0; h < H; h++) rt[h] += add[(size_t)t * H + h];"),
    "quant_round_half_even": ("const float rr = roundf(ratio);", "const float rr = rintf(ratio);"),
    "quant_scale_qmax_plus_1": ("volatile float sc = amax / (float)qmax;",
                                "volatile float sc = amax / (float)(qmax + 1);"),
    "quant_truncate": ("const float rr = roundf(ratio);", "const float rr = truncf(ratio);"),
    "rmsnorm_not_rounded": ("xn[(size_t)t * H + h] = round_bf16(rt[h] * inv);",
                            "xn[(size_t)t * H + h] = rt[h] * inv;"),
    "topp_not_renormalised": ("    for (int j = 0; j < m; j++) wsum += wsrc[sorted[j]];\n",
                              "    for (int j = 0; j < k; j++) wsum += wsrc[sorted[j]];\n"),
    "topp_keeps_the_crossing_slot_too": ("      if (before >= c->top_p) break;",
                                         "      if (before > c->top_p + 0.2) break;"),
    "group_score_uncorrected": (
        "gscore[g] = sel_score[msorted[0]] + (gs > 1 ? sel_score[msorted[1]] : 0.0);",
        "gscore[g] = wsrc[msorted[0]] + (gs > 1 ? wsrc[msorted[1]] : 0.0);"),
    "groups_kept_minus_one": (
        "for (int j = 0; j < c->topk_group; j++) if (gsorted[j] == g) kept = 1;",
        "for (int j = 0; j < c->topk_group - 1; j++) if (gsorted[j] == g) kept = 1;"),
    "groups_strided": ("int g = e / gs, kept = 0;", "int g = e % G, kept = 0;"),
    "bias_subtracted": ("sel_score[e] = s + (bias ? (double)bias[e] : 0.0);",
                        "sel_score[e] = s - (bias ? (double)bias[e] : 0.0);"),
    "rsf_dropped": ("w[j] = v * c->rsf;", "w[j] = v;"),
    "softmax_not_normalised": ("p[e] = p[e] / sum;", "p[e] = p[e];"),
    "silu_is_sigmoid": ("return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    "swiglu_up_dropped": (
        "for (size_t i = 0; i < (size_t)n * I; i++) h[i] = orc_silu(g[i]) * u[i];",
        "for (size_t i = 0; i < (size_t)n * I; i++) h[i] = orc_silu(g[i]);"),
    "row_scale_dropped": ("wrow[cc] = (double)s[r] * (double)q[(size_t)r * cols + cc];",
                          "wrow[cc] = (double)q[(size_t)r * cols + cc];"),
    "q8_block_scale_dropped": ("acc += (double)dx[(size_t)i * nb + b] *", "acc += 1.0 *"),
    "q8_row_scale_dropped": ("y[(size_t)i * rows + r] = (double)s[r] * acc;",
                             "y[(size_t)i * rows + r] = acc;"),
    "union_token_mod": ("int t = perm[offsets[e] + i] / k;", "int t = perm[offsets[e] + i] % k;"),
    "union_output_row": ("memcpy(yslot + (size_t)perm[offsets[e] + i] * H, ye + (size_t)i * H,",
                         "memcpy(yslot + (size_t)(offsets[e] + i) * H, ye + (size_t)i * H,"),
    "offsets_not_scanned": ("for (int e = 0; e < E; e++) offsets[e + 1] += offsets[e];", ""),
    "int4_low_nibble_twice": ("q[i] = sext(p[i / 2] >> 4, 4);", "q[i] = sext(p[i / 2] & 0xF, 4);"),
    "int4_low_no_sign_ext": ("q[i + 1] = sext(p[i / 2] & 0xF, 4);",
                             "q[i + 1] = (int8_t)(p[i / 2] & 0xF);"),
    "int2_field_order": ("q[i] = sext((p[i / 4] >> (6 - 2 * (int)(i % 4))) & 3, 2);",
                         "q[i] = sext((p[i / 4] >> (2 * (int)(i % 4))) & 3, 2);"),
    "bf16_truncates": ("double q = nearbyint(ldexp(m, 8));", "double q = trunc(ldexp(m, 8));"),
    "per_token_shared_dropped": (
        "if (c->n_shared) orc_expert_forward(c, shared, x + (size_t)t * H, 1, o);",
        "if (0) orc_expert_forward(c, shared, x + (size_t)t * H, 1, o);"),
}


def _run_mutant(name, work):
    """Compile the mutant into `work` and run the pin suite on it; True if the suite failed."""
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    work.mkdir()
    msrc = work / "moe_oracle.c"
    msrc.write_text(src.replace(old, new))
    so = str(work / "libmut.so")
    oracle.build(force=True, src=str(msrc), out=so)
    env = dict(os.environ, MOE_ORACLE_SO=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode != 0, r.stdout[-2000:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    """Every mutant's outcome, the pin-suite runs spread over the host's cores."""
    base = tmp_path_factory.mktemp("mutants")
    names = sorted(MUTANTS)
    workers = max(1, min(8, (os.cpu_count() or 2) - 1))
    with ThreadPoolExecutor(workers) as ex:
        res = list(ex.map(lambda n: _run_mutant(n, base / n), names))
    return dict(zip(names, res))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, outcomes):
    caught, tail = outcomes[name]
    assert caught, f"mutant {name} survived the pins:\n{tail}"
