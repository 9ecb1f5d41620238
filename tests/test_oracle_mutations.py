"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake into a copy of oracle/sv_oracle.c (a dropped term, a wrong
sign, index or comparison, a transposed operand), compiles the copy on the CPU, and checks
that at least one pin from test_oracle_pins.py or test_oracle_near_ties.py fails against it.  The real oracle is never
modified.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle_near_ties as nt
import test_oracle_pins as pins

SRC = open(os.path.join(os.path.dirname(oracle.__file__), "sv_oracle.c")).read()

MUTATIONS = [
    ("residual clamp dropped", "r[v] = t > 0.0 ? t : 0.0;\n                        W += r[v];",
     "r[v] = t;\n                        W += r[v];",
     [lambda o: pins.test_numpy_operator_example(o),
      lambda o: pins.test_lossless_monte_carlo(o, 4, 1, 1.0, 0, 1.0, None, None)]),
    ("accept comparison inverted", "accept = u < thr;", "accept = u > thr;",
     [lambda o: pins.test_accept_probability_examples(o, pins.GOLD["accept_probability"][0])]),
    ("ratio transposed", "double ratio = px / qx;", "double ratio = qx / px;",
     [lambda o: pins.test_accept_probability_examples(o, pins.GOLD["accept_probability"][0])]),
    ("uniform slots swapped", "double u = in->uniforms[(r0 + i) * 2 + 0];",
     "double u = in->uniforms[(r0 + i) * 2 + 1];",
     [lambda o: pins.test_numpy_operator_example(o)]),
    ("frequency penalty dropped", "double pen = pres * (c > 0 ? 1.0 : 0.0) + freq * (double)c;",
     "double pen = pres * (c > 0 ? 1.0 : 0.0);", [lambda o: pins.test_softmax_against_numpy(o)]),
    ("penalty counts the row's own draft",
     [("for (int32_t e = 0; e < nh + i; e++) {",
       "int32_t i1 = i < in->num_drafts[b] ? i + 1 : i;\n    for (int32_t e = 0; e < nh + i1; e++) {"),
      ("for (int32_t t = 0; t < i; t++) c += (d[t] == v);", "for (int32_t t = 0; t < i1; t++) c += (d[t] == v);")],
     None, [lambda o: pins.test_softmax_against_numpy(o)]),
    ("repeat counts capped at one", "for (int32_t t = 0; t < i; t++) c += (d[t] == v);",
     "for (int32_t t = 0; t < i; t++) c |= (d[t] == v);", [lambda o: pins.test_softmax_against_numpy(o)]),
    ("presence penalty sign flipped", "z[v] -= pen;", "z[v] += pen;",
     [lambda o: pins.test_softmax_against_numpy(o)]),
    ("temperature ignored", "p[v] = z[v] / T;", "p[v] = z[v];",
     [lambda o: pins.test_softmax_against_numpy(o)]),
    ("top-k off by one", "tau = zs[K - 1];", "tau = zs[K];",
     [lambda o: pins.test_filters_brute_force(o, 0), lambda o: pins.test_filters_edge_cases(o)]),
    ("top-p counts the level's own mass", "if (!cut && above / ZK < P) {",
     "if (!cut && (above + lm) / ZK < P) {",
     [lambda o, s=s: pins.test_filters_brute_force(o, s) for s in range(8)]),
    ("top-p normalised over the unfiltered row", "ZK += (p[v] >= tau) ? exp(p[v] - m) : 0.0;",
     "ZK += exp(p[v] - m);", [lambda o: pins.test_filters_edge_cases(o)]),
    ("draft row index shifted", "double qx = (double)in->draft_probs[(d0 + i) * (int64_t)V + x];",
     "double qx = (double)in->draft_probs[(d0 + (i + 1) % k) * (int64_t)V + x];",
     [lambda o: pins.test_lossless_monte_carlo(o, 8, 3, 0.7, 5, 0.8, 0.4, 0.3),
      lambda o: pins.test_accept_length_closed_form(o)]),
    ("target row always row 0", "int64_t row = row_start(in, b) + i;", "int64_t row = row_start(in, b);",
     [lambda o: pins.test_greedy_is_argmax_prefix_match(o)]),
    ("greedy tie to highest id", "if (z[v] > z[best]) best = v;", "if (z[v] >= z[best]) best = v;",
     [lambda o: pins.test_greedy_ties_go_to_lowest_id(o)]),
    ("inverse CDF not strict", "if (c > target) {", "if (c >= target) {",
     [lambda o: pins.test_inverse_cdf_never_picks_zero_weight(o)]),
    ("extra token from the wrong row", "token = inverse_cdf(p, V, in->uniforms[(r0 + k) * 2 + 1], amb.mass, &cn);",
     "token = inverse_cdf(r, V, in->uniforms[(r0 + k) * 2 + 1], amb.mass, &cn);",
     [lambda o: pins.test_expected_tokens_closed_form(o),
      lambda o: pins.test_lossless_monte_carlo(o, 4, 1, 1.0, 0, 1.0, None, None)]),
    ("one-hot: accepts on a mismatch", "const int stop = (i == k || drafts[i] != t);",
     "const int stop = (i == k || drafts[i] == t);",
     [lambda o: pins.test_onehot_joint_law(o, 5, 2, 1.0, 0, 1.0, None, None)]),
    ("one-hot: samples with the accept slot", "t = inverse_cdf(p, V, in->uniforms[(r0 + i) * 2 + 1], amb.mass, &cn);",
     "t = inverse_cdf(p, V, in->uniforms[(r0 + i) * 2 + 0], amb.mass, &cn);",
     [lambda o: pins.test_onehot_reduces_to_pinned_paths(o)]),
    ("one-hot: emits the draft at the stopping row", "token = t;", "token = i < k ? drafts[i] : t;",
     [lambda o: pins.test_onehot_joint_law(o, 5, 2, 1.0, 0, 1.0, None, None),
      lambda o: pins.test_onehot_matches_when_every_sample_matches(o)]),
    ("one-hot: scan ignores the last draft", "const int stop = (i == k || drafts[i] != t);",
     "const int stop = (i == k || (i + 1 < k && drafts[i] != t));",
     [lambda o: pins.test_onehot_matches_when_every_sample_matches(o),
      lambda o: pins.test_onehot_joint_law(o, 5, 2, 1.0, 0, 1.0, None, None)]),
    ("history: its counts dropped", "int32_t c = prior_count(in, b, v);\n        for", "int32_t c = 0;\n        for",
     [lambda o: pins.test_history_softmax_against_numpy(o)]),
    ("history: drafts not added to its counts", "for (int32_t t = 0; t < i; t++) c += (d[t] == v);",
     "if (e >= nh) for (int32_t t = 0; t < i; t++) c += (d[t] == v);",
     [lambda o, s=s: pins.test_history_is_earlier_drafts(o, s) for s in range(4)]),
    ("history: drafted tokens penalised twice", "int seen = prior_count(in, b, v) > 0;", "int seen = 0;",
     [lambda o, s=s: pins.test_history_is_earlier_drafts(o, s) for s in range(4)]),
    ("history: ignored on row 0", "for (int32_t e = 0; e < nh + i; e++) {",
     "for (int32_t e = (i == 0 ? nh : 0); e < nh + i; e++) {",
     [lambda o: pins.test_history_softmax_against_numpy(o), lambda o: pins.test_history_greedy_against_numpy(o)]),
    ("rollback keeps one row too many", "int64_t t = L - (k + 1) + 1 + a;", "int64_t t = L - (k + 1) + 2 + a;",
     [lambda o: pins.test_rollback_closed_form(o)]),
    # the near-tie classifier: a band too wide hides GPU mistakes, one too narrow fails correct
    # fp32 results; the flags must land where the GPU can part from the oracle
    ("near-tie band 100x wide", "#define NEAR_TOL 1e-5", "#define NEAR_TOL 1e-3",
     [lambda o: nt.test_accept_band(o, 1e-4, False), lambda o: nt.test_cdf_band(o, 1e-4, False, 2)]),
    ("near-tie band 100x narrow", "#define NEAR_TOL 1e-5", "#define NEAR_TOL 1e-7",
     [lambda o: nt.test_accept_band(o, 1e-6, True)]),
    ("residual-mass band 1000x wide", "#define NEAR_W 1e-6", "#define NEAR_W 1e-3",
     [lambda o: nt.test_small_residual_band(o, 1e-4, False)]),
    ("residual-mass band 10x narrow", "#define NEAR_W 1e-6", "#define NEAR_W 1e-7",
     [lambda o: nt.test_small_residual_band(o, 5e-7, True)]),
    ("accept band ignores the kept set's ambiguity", "fabs(u - thr) < NEAR_TOL + amb.mass * thr",
     "fabs(u - thr) < NEAR_TOL", [lambda o: nt.test_top_p_band_flags_accept_tests(o, 1e-6, True)]),
    ("greedy gap not relative", "return fabs(a - b) <= NEAR_TOL * s;", "return fabs(a - b) <= NEAR_TOL;",
     [lambda o: nt.test_greedy_gap_band(o, 1e-6, True)]),
    ("extra-token near-tie not located", "if (cn) mark_near(&d, k, 1);", ";",
     [lambda o: nt.test_cdf_band(o, 1e-6, True, 2)]),
    ("greedy compare near-tie not located", "if (nt && i < k) mark_near(&d, i, 0);\n                if (nt && stop)",
     "if (nt && stop)", [lambda o: nt.test_greedy_gap_flags_the_compare(o)]),
]


class _Swap:
    """Points the oracle module at a mutant library for the duration of a with-block."""

    def __init__(self, path):
        self.lib = oracle.load(path)

    def __enter__(self):
        self.saved = oracle._lib
        oracle._lib = self.lib
        return oracle

    def __exit__(self, *exc):
        oracle._lib = self.saved


@pytest.mark.parametrize("name,old,new,checks", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, oracle_lib, name, old, new, checks):
    edits = old if isinstance(old, list) else [(old, new)]
    text = SRC
    for a, b in edits:
        assert text.count(a) == 1, f"mutation anchor not unique/found: {name}"
        text = text.replace(a, b)
    src = tmp_path / "mutant.c"
    src.write_text(text)
    so = tmp_path / "mutant.so"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o",
                           str(so), str(src), "-lm"])
    caught = False
    with _Swap(str(so)) as o:
        for chk in checks:
            try:
                chk(o)
            except AssertionError:
                caught = True
                break
    assert caught, f"no pin caught the planted mistake: {name}"
