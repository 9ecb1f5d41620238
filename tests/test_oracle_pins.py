"""Pins for the float64 oracle: checks against what the source pages and the mathematics fix.

Each test names the pin it implements: closed forms, the pages' worked examples
(tests/golden/worked_examples.json), brute force on tiny vocabularies, special cases that
reduce to a library routine, and a Monte Carlo distribution (losslessness) test.  None of
them re-derives a value through the oracle's own code path.
"""
import json
import os

import numpy as np
import pytest
from scipy import stats

import sv_workloads as W

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def _rng(seed):
    return np.random.Generator(np.random.Philox(key=np.array([seed, 99], dtype=np.uint64)))


def _sample(q_rows, u):
    """Vectorised inverse-CDF draw of one token per trial from q_rows [trials, V]."""
    c = np.cumsum(q_rows.astype(np.float64), axis=-1)
    t = (u * c[..., -1])[..., None]
    return np.minimum((c <= t).sum(axis=-1), q_rows.shape[-1] - 1).astype(np.int32)


def _softmax(z):
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def _chisq_p(obs, prob):
    n = obs.sum()
    exp = prob * n
    assert np.all(obs[prob == 0] == 0), "a zero-probability token was produced"
    m = prob > 0
    if m.sum() < 2:
        return 1.0
    return stats.chisquare(obs[m], exp[m] * obs[m].sum() / exp[m].sum()).pvalue


# ------------------------------------------------------------------------------------------
# P3: worked examples printed on the pages
# ------------------------------------------------------------------------------------------

def _one(p, q, draft, u0, u1, k=1, extra_row=None):
    """Single request, k=1: row 0 has target p and draft q; row 1 (extra) is `extra_row`."""
    V = len(p)
    lg = np.log(np.asarray(p, np.float64)).astype(np.float32)
    lg = np.where(np.isfinite(lg), lg, -1e30).astype(np.float32)
    rows = np.stack([lg, lg if extra_row is None else extra_row]).astype(np.float32)
    uni = np.array([[[u0, u1], [0.5, 0.5]]], np.float32)
    return W.from_rows(V, rows, np.asarray(q, np.float32)[None], np.array([[draft]]), uni)


@pytest.mark.parametrize("case", GOLD["accept_probability"])
def test_accept_probability_examples(oracle_lib, case):
    # two-token rows: token 0 carries the printed probabilities
    p = [case["p"], 1 - case["p"]]
    q = [case["q"], 1 - case["q"]]
    a = case["accept_prob"]
    for u in [0.0, a - 2e-3, a + 2e-3, 0.999]:
        if u < 0 or u >= 1:
            continue
        r = oracle_lib.verify(_one(p, q, 0, u, 0.5))
        assert r["accept_len"][0] == (1 if u < a else 0), (case, u)
        assert r["pq"][0, 0] == pytest.approx(case["p"], abs=1e-7)


def test_numpy_operator_example(oracle_lib):
    ex = GOLD["numpy_operator_example"]
    for c in ex["cases"]:
        a = c["accept_prob"]
        for u0 in np.linspace(0, 0.999, 23):
            for u1 in [0.0, 0.3, 0.77, 0.9999]:
                r = oracle_lib.verify(_one(ex["p"], ex["q"], c["draft"], u0, u1))
                acc = bool(r["accept_len"][0] == 1)
                assert acc == (u0 < a - 1e-6 or (a >= 1.0)), (c, u0)
                if not acc:
                    res = np.asarray(c["residual"])
                    # the residual is one-hot: every u1 must land on its support
                    assert r["out_tokens"][0, 0] == int(np.argmax(res))
                    rr, Wt = oracle_lib.residual(_one(ex["p"], ex["q"], c["draft"], u0, u1), 0, 0)
                    np.testing.assert_allclose(rr, res, atol=1e-7)


def test_expected_tokens_closed_form(oracle_lib):
    """Key Topic 4: E[tokens/step] = (1 - a^(g+1)) / (1 - a) for a per-row accept rate a.

    Rows with p = [a, 1-a] and a one-hot draft q = [1, 0] accept with probability exactly a,
    so the Monte Carlo mean of accept_len + 1 must match the formula."""
    for c in GOLD["expected_tokens_per_step"]["cases"]:
        g, a = c["gamma"], c["alpha"]
        assert (1 - a ** (g + 1)) / (1 - a) == pytest.approx(c["formula"], abs=1e-5)
        n = 200_000
        lg = np.log(np.array([a, 1 - a])).astype(np.float32)
        rows = np.tile(lg, (g + 1, 1))
        q = np.tile(np.array([1.0, 0.0], np.float32), (g, 1))
        uni = _rng(int(a * 100)).random((n, g + 1, 2), dtype=np.float32)
        w = W.from_rows(2, rows, q, np.zeros((n, g), np.int32), uni)
        r = oracle_lib.verify(w, threads=4)
        tokens = r["accept_len"].astype(np.float64) + 1
        se = tokens.std() / np.sqrt(n)
        assert abs(tokens.mean() - c["formula"]) < 4 * se + 1e-3
        if c["printed_is_garbled"]:
            assert abs(c["printed"] - c["formula"]) > 0.1
        else:
            assert abs(c["printed"] - c["formula"]) < 0.01


# ------------------------------------------------------------------------------------------
# P1: losslessness -- the output distribution equals the target's (Monte Carlo, chi-square)
# ------------------------------------------------------------------------------------------

def _brute_filter(z, T, K, P):
    """Top-k then top-p straight from their definitions, O(V^2) (tiny V only)."""
    zs = z / T
    V = len(zs)
    keep = np.ones(V, bool)
    if 0 < K < V:
        keep = np.array([(zs > zs[v]).sum() < K for v in range(V)])
    e = np.where(keep, np.exp(zs - zs.max()), 0.0)
    pi = e / e.sum()
    if P < 1:
        keep2 = np.array([keep[v] and pi[keep & (zs > zs[v])].sum() < P for v in range(V)])
    else:
        keep2 = keep
    e2 = np.where(keep2, np.exp(zs - zs.max()), 0.0)
    return e2 / e2.sum()


@pytest.mark.parametrize("V,k,T,K,P,pres,freq", [
    (4, 1, 1.0, 0, 1.0, None, None),
    (8, 3, 0.7, 5, 0.8, 0.4, 0.3),
    (6, 2, 1.3, 0, 0.9, 1.0, 0.0),
])
def test_lossless_monte_carlo(oracle_lib, V, k, T, K, P, pres, freq):
    """P1 (Adding Speculative Decoding, Acceptance bars item 1): with drafts drawn from q, the
    first output token is distributed as the filtered target p_0; and given that draft 0
    was accepted, the second output is distributed as p_1 computed with d_0 counted by the
    penalties."""
    n = 1_000_000
    g = _rng(V * 10 + k)
    logits = (g.standard_normal((k + 1, V)) * 1.5).astype(np.float32)
    dl = logits[:k] + (g.standard_normal((k, V)) * 1.0).astype(np.float32)
    q = np.stack([_softmax(dl[i].astype(np.float64)) for i in range(k)]).astype(np.float32)
    drafts = np.stack([_sample(np.broadcast_to(q[i], (n, V)), g.random(n)) for i in range(k)], axis=1)
    uni = g.random((n, k + 1, 2), dtype=np.float32)
    w = W.from_rows(V, logits, q, drafts, uni, temperature=T, top_k=K, top_p=P,
                    presence=pres, frequency=freq)
    r = oracle_lib.verify(w, threads=8)
    assert (r["error"] == 0).all()
    p0 = _brute_filter(logits[0].astype(np.float64), T, K, P)
    obs0 = np.bincount(r["out_tokens"][:, 0], minlength=V)
    assert _chisq_p(obs0, p0) > 1e-3
    # second position, conditioned on the first draft accepted (out[0] = d_0)
    sel = r["accept_len"] >= 1
    for x in range(V):
        m = sel & (r["out_tokens"][:, 0] == x)
        if m.sum() < 2000:
            continue
        z1 = logits[1].astype(np.float64).copy()
        if pres or freq:
            z1[x] -= (pres or 0.0) + (freq or 0.0)
        p1 = _brute_filter(z1, T, K, P)
        obs1 = np.bincount(r["out_tokens"][m, 1], minlength=V)
        assert _chisq_p(obs1, p1) > 1e-4, (x, obs1, p1 * m.sum())


def test_dropping_residual_clamp_is_detected():
    """Sanity of the Monte Carlo pin itself: resampling from p instead of max(0, p-q)/W after
    a rejection (a plausible mistake) is biased, and the chi-square test rejects it."""
    V, n = 4, 400_000
    g = _rng(5)
    p = _softmax(g.standard_normal(V) * 1.5)
    q = _softmax(g.standard_normal(V) * 1.5)
    d = _sample(np.broadcast_to(q, (n, V)), g.random(n))
    u = g.random(n)
    acc = u < np.minimum(1, p[d] / q[d])
    wrong = np.where(acc, d, _sample(np.broadcast_to(p, (n, V)), g.random(n)))
    assert _chisq_p(np.bincount(wrong, minlength=V), p) < 1e-6


# ------------------------------------------------------------------------------------------
# P2: accept-length closed form
# ------------------------------------------------------------------------------------------

def test_accept_length_closed_form(oracle_lib):
    """E[accept_len] = sum_j prod_{i<j} beta_i with beta_i = sum_v min(p_i, q_i), the accept
    probability of row i (rows independent of the drafts: no penalties)."""
    V, k, n = 7, 4, 400_000
    g = _rng(77)
    logits = (g.standard_normal((k + 1, V)) * 1.2).astype(np.float32)
    q = np.stack([_softmax(g.standard_normal(V)) for _ in range(k)]).astype(np.float32)
    drafts = np.stack([_sample(np.broadcast_to(q[i], (n, V)), g.random(n)) for i in range(k)], axis=1)
    w = W.from_rows(V, logits, q, drafts, g.random((n, k + 1, 2), dtype=np.float32), temperature=0.9)
    r = oracle_lib.verify(w, threads=8)
    beta = [np.minimum(_softmax(logits[i].astype(np.float64) / 0.9), q[i].astype(np.float64)).sum()
            for i in range(k)]
    expect = sum(np.prod(beta[:j]) for j in range(1, k + 1))
    a = r["accept_len"].astype(np.float64)
    assert abs(a.mean() - expect) < 4 * a.std() / np.sqrt(n)


# ------------------------------------------------------------------------------------------
# P4: greedy is the one-hot special case; greedy is an argmax prefix match
# ------------------------------------------------------------------------------------------

def test_greedy_is_argmax_prefix_match(oracle_lib):
    """Adding Speculative Decoding, table 'The existing base': accept while d_j == argmax_j;
    the extra token is the argmax at the first mismatch (numpy argmax as the reference)."""
    g = _rng(11)
    B, k, V = 200, 5, 50
    logits = (g.standard_normal((B, k + 1, V))).astype(np.float32)
    am = logits.argmax(-1)
    drafts = np.where(g.random((B, k)) < 0.7, am[:, :k], g.integers(0, V, (B, k))).astype(np.int32)
    w = W.from_rows(V, logits, np.full((B, k, V), 1.0 / V, np.float32), drafts,
                    g.random((B, k + 1, 2), dtype=np.float32), greedy=1)
    r = oracle_lib.verify(w)
    for b in range(B):
        a = 0
        while a < k and drafts[b, a] == am[b, a]:
            a += 1
        assert r["accept_len"][b] == a
        assert list(r["out_tokens"][b, :a + 1]) == list(drafts[b, :a]) + [am[b, a]]
        assert (r["out_tokens"][b, a + 1:] == -1).all()


def test_greedy_equals_sampled_with_one_hot_target(oracle_lib):
    """P4: with p one-hot at the argmax (top-k = 1, no ties), the sampled algorithm returns
    exactly the greedy result for any q with q(d) > 0 and any uniforms (Adding Speculative
    Decoding, Verification and sampling item 2: greedy is the degenerate case)."""
    g = _rng(12)
    B, k, V = 300, 4, 40
    logits = g.standard_normal((B, k + 1, V)).astype(np.float32)
    am = logits.argmax(-1)
    drafts = np.where(g.random((B, k)) < 0.6, am[:, :k], g.integers(0, V, (B, k))).astype(np.int32)
    q = np.stack([[_softmax(g.standard_normal(V)) for _ in range(k)] for _ in range(B)]).astype(np.float32)
    uni = g.random((B, k + 1, 2), dtype=np.float32)
    pres = g.uniform(0, 1, B).astype(np.float32)
    wg = W.from_rows(V, logits, q, drafts, uni, greedy=1, presence=pres, frequency=0.2)
    ws = W.from_rows(V, logits, q, drafts, uni, greedy=0, top_k=1, temperature=0.8, presence=pres,
                     frequency=0.2)
    rg, rs = oracle_lib.verify(wg), oracle_lib.verify(ws)
    np.testing.assert_array_equal(rg["accept_len"], rs["accept_len"])
    np.testing.assert_array_equal(rg["out_tokens"], rs["out_tokens"])


# ------------------------------------------------------------------------------------------
# P5: invariants
# ------------------------------------------------------------------------------------------

def test_invariants_random_batches(oracle_lib):
    for seed in range(6):
        w = W.random_batch(seed, B=40, k_max=6, V=97, dtype="bf16" if seed % 2 else "f32",
                           varlen=bool(seed % 3 == 0), tie_step=0.25 if seed % 2 else 0.0)
        r = oracle_lib.verify(w)
        assert (r["error"] == 0).all()
        for b in range(w.B):
            k, a = int(w.num_drafts[b]), int(r["accept_len"][b])
            assert 0 <= a <= k
            row = r["out_tokens"][b]
            assert (row[:a + 1] >= 0).all() and (row[a + 1:] == -1).all()
            d0 = w.draft_start(b)
            assert list(row[:a]) == list(w.draft_tokens[d0:d0 + a])
            # the produced token is in the support of the distribution it was drawn from
            p = oracle_lib.row_probs(w, b, a)
            if w.greedy[b] or a == k:
                assert p[row[a]] > 0
            else:
                res, Wt = oracle_lib.residual(w, b, a)
                if Wt > 0:
                    assert res[row[a]] > 0
                    assert abs(res.sum() - 1.0) < 1e-12
                else:
                    assert p[row[a]] > 0


def test_q_equal_p_accepts_everything(oracle_lib):
    V, k, B = 8, 5, 2000
    g = _rng(21)
    logits = np.zeros((k + 1, V), np.float32)          # p uniform: exactly 1/8 in fp32 and fp64
    q = np.full((k, V), 1.0 / V, np.float32)
    drafts = g.integers(0, V, (B, k)).astype(np.int32)
    r = oracle_lib.verify(W.from_rows(V, logits, q, drafts, g.random((B, k + 1, 2), dtype=np.float32)))
    assert (r["accept_len"] == k).all()


def test_disjoint_supports_reject_at_row_zero(oracle_lib):
    V, k, B = 6, 3, 500
    g = _rng(22)
    logits = np.tile(np.array([5.0, 4.0, -30, -30, -30, -30], np.float32), (k + 1, 1))
    q = np.tile(np.array([0, 0, 0.25, 0.25, 0.25, 0.25], np.float32), (k, 1))
    drafts = g.integers(2, V, (B, k)).astype(np.int32)
    r = oracle_lib.verify(W.from_rows(V, logits, q, drafts, g.random((B, k + 1, 2), dtype=np.float32),
                                      top_k=2))
    assert (r["accept_len"] == 0).all()
    assert set(np.unique(r["out_tokens"][:, 0])) <= {0, 1}


def test_zero_drafts_is_a_plain_sample(oracle_lib):
    """k_b = 0: the request is one extra-token draw from row 0 (accept_len 0)."""
    w = W.random_batch(3, B=30, k_max=4, V=33, varlen=True)
    w.num_drafts[:] = 0
    w.row_offsets = np.arange(w.B + 1, dtype=np.int32)
    w.target_logits = np.ascontiguousarray(w.target_logits[: w.B])
    w.uniforms = np.ascontiguousarray(w.uniforms[: w.B])
    w.draft_tokens = w.draft_tokens[:0]
    w.draft_probs = w.draft_probs[:0]
    r = oracle_lib.verify(w)
    assert (r["accept_len"] == 0).all() and (r["out_tokens"][:, 0] >= 0).all()


def test_device_data_errors(oracle_lib):
    w = W.random_batch(4, B=8, k_max=3, V=20, greedy_frac=0.0)
    w.draft_tokens[1] = 20            # request 0: token out of range
    w.temperature[1] = 0.0            # request 1: T <= 0 on a sampled request
    w.top_p[2] = 1.5                  # request 2: top_p outside (0, 1]
    w.uniforms[3 * 4 + 1, 0] = 1.0    # request 3: uniform outside [0, 1)
    w.num_drafts[4] = 4               # request 4: more drafts than k_max
    r = oracle_lib.verify(w)
    assert list(r["error"][:5]) == [2, 3, 4, 5, 1]
    assert (r["accept_len"][:5] == -1).all() and (r["out_tokens"][:5] == -1).all()
    assert (r["error"][5:] == 0).all()


# ------------------------------------------------------------------------------------------
# P6 / P7: filtering by brute force, softmax against numpy
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(8))
def test_filters_brute_force(oracle_lib, seed):
    """P6: top-k then top-p from their definitions (O(V^2) counting), with forced ties."""
    g = _rng(100 + seed)
    V = int(g.integers(3, 40))
    B = 25
    step = [0.0, 0.5, 0.25, 1.0][seed % 4]
    z = g.standard_normal((B, 1, V)) * 2
    if step:
        z = np.round(z / step) * step
    z = z.astype(np.float32)
    K = g.integers(0, V + 2, B).astype(np.int32)
    P = np.where(g.random(B) < 0.7, g.uniform(0.01, 1.0, B), 1.0).astype(np.float32)
    T = g.uniform(0.2, 2.0, B).astype(np.float32)
    w = W.from_rows(V, z, np.zeros((B, 0, V), np.float32), np.zeros((B, 0), np.int32),
                    g.random((B, 1, 2), dtype=np.float32), temperature=T, top_k=K, top_p=P)
    for b in range(B):
        ref = _brute_filter(z[b, 0].astype(np.float64), float(T[b]), int(K[b]), float(P[b]))
        got = oracle_lib.row_probs(w, b, 0)
        np.testing.assert_allclose(got, ref, atol=1e-12)
        assert got.max() == got[np.argmax(z[b, 0])] > 0       # the argmax is always kept


def test_filters_edge_cases(oracle_lib):
    V = 10
    z = np.array([[3, 1, 3, 0, -1, 3, 2, 2, -5, 0]], np.float32)[None]
    mk = lambda K, P: W.from_rows(V, z, np.zeros((1, 0, V), np.float32), np.zeros((1, 0), np.int32),
                                  np.full((1, 1, 2), 0.5, np.float32), top_k=K, top_p=P)
    p = oracle_lib.row_probs(mk(1, 1.0), 0, 0)          # top-1 with a 3-way tie keeps all three
    assert set(np.nonzero(p)[0]) == {0, 2, 5}
    p = oracle_lib.row_probs(mk(4, 1.0), 0, 0)          # 4th largest is a 2-way tie at 2.0
    assert set(np.nonzero(p)[0]) == {0, 2, 5, 6, 7}
    p = oracle_lib.row_probs(mk(0, 1e-6), 0, 0)         # tiny top-p keeps the whole top level
    assert set(np.nonzero(p)[0]) == {0, 2, 5}
    p = oracle_lib.row_probs(mk(V, 1.0), 0, 0)          # top-k >= V: disabled
    assert (p > 0).all()
    # top-p acts on the top-k-renormalised mass: on a near-flat row with top-3, the third
    # token sits above 0.5 of the top-3 mass but below 0.5 of the whole row's mass
    zf = np.linspace(2.0, 1.1, V).astype(np.float32)[None, None]
    wf = W.from_rows(V, zf, np.zeros((1, 0, V), np.float32), np.zeros((1, 0), np.int32),
                     np.full((1, 1, 2), 0.5, np.float32), top_k=3, top_p=0.5)
    p = oracle_lib.row_probs(wf, 0, 0)
    assert set(np.nonzero(p)[0]) == {0, 1}
    np.testing.assert_allclose(p, _brute_filter(zf[0, 0].astype(np.float64), 1.0, 3, 0.5), atol=1e-12)


def test_softmax_against_numpy(oracle_lib):
    """P7: with no filtering, a sampled row is numpy's float64 softmax(z/T), z including the
    presence/frequency penalties of the drafts before the row (FreeToken PR #836, Design)."""
    # V = 6 makes repeated drafts common, so counts above one matter
    for w in [W.random_batch(9, B=20, k_max=5, V=301, dtype="bf16", greedy_frac=0.0),
              W.random_batch(10, B=30, k_max=8, V=6, dtype="f32", greedy_frac=0.0, draft_sigma=0.1)]:
        w.top_k[:] = 0
        w.top_p[:] = 1.0
        lg = w.logits_f32().astype(np.float64)
        for b in range(w.B):
            r0, d0 = w.row_start(b), w.draft_start(b)
            for i in range(int(w.num_drafts[b]) + 1):
                z = lg[r0 + i].copy()
                c = np.bincount(w.draft_tokens[d0:d0 + i], minlength=w.V).astype(np.float64)
                z -= w.presence[b] * (c > 0) + w.frequency[b] * c
                ref = _softmax(z / float(w.temperature[b]))
                np.testing.assert_allclose(oracle_lib.row_probs(w, b, i), ref, rtol=1e-12, atol=1e-15)


# ------------------------------------------------------------------------------------------
# P8: rollback
# ------------------------------------------------------------------------------------------

def test_rollback_closed_form(oracle_lib):
    cs = GOLD["rollback"]["cases"]
    L = np.array([c["current_len"] for c in cs])
    k = np.array([c["k"] for c in cs])
    a = np.array([c["accepted"] for c in cs])
    out, nerr = oracle_lib.rollback(L, a, k)
    assert nerr == 0
    assert list(out) == [c["committed"] for c in cs]
    out, nerr = oracle_lib.rollback([10, 10, 2], [5, -1, 0], [4, 4, 4])   # forward, negative, < 0
    assert nerr == 3 and (out == -1).all()


def test_draft_rollback_is_the_same_update(oracle_lib):
    """The draft cache appended k drafts and keeps the accepted ones: L - k + a, which is the
    target's L - (k+1) + 1 + a written differently, so one rollback serves both caches."""
    cs = GOLD["rollback_draft"]["cases"]
    L = np.array([c["current_len"] for c in cs])
    k = np.array([c["k"] for c in cs])
    a = np.array([c["accepted"] for c in cs])
    out, nerr = oracle_lib.rollback(L, a, k)
    assert nerr == 0
    assert list(out) == [c["committed"] for c in cs]


def test_greedy_ties_go_to_lowest_id(oracle_lib):
    """Exact ties (as bf16 rows have) resolve to the lowest token id, as numpy's argmax does."""
    g = _rng(13)
    B, k, V = 200, 3, 30
    logits = np.round(g.standard_normal((B, k + 1, V)) * 2).astype(np.float32)   # many exact ties
    am = logits.argmax(-1)
    drafts = np.where(g.random((B, k)) < 0.8, am[:, :k], g.integers(0, V, (B, k))).astype(np.int32)
    w = W.from_rows(V, logits, np.full((B, k, V), 1.0 / V, np.float32), drafts,
                    g.random((B, k + 1, 2), dtype=np.float32), greedy=1)
    r = oracle_lib.verify(w)
    for b in range(B):
        a = int(r["accept_len"][b])
        assert r["out_tokens"][b, a] == am[b, a]


def test_inverse_cdf_never_picks_zero_weight(oracle_lib):
    """u = 0 with leading zero-weight tokens: the draw is the first token of positive weight
    (the running sum must strictly exceed u*W)."""
    V = 8
    z = np.array([-50, -50, 1.0, 2.0, -50, 0.5, -50, -50], np.float32)
    w = W.from_rows(V, np.tile(z, (2, 1)), np.full((1, V), 1.0 / V, np.float32), np.array([[0]]),
                    np.array([[[0.99, 0.0], [0.0, 0.0]]], np.float32), top_k=3)
    r = oracle_lib.verify(w)
    assert r["accept_len"][0] == 0 and r["out_tokens"][0, 0] == 2
    w.draft_tokens[0] = 3
    w.uniforms[0, 0] = 0.0                   # accepted; the extra token is drawn with u = 0
    r = oracle_lib.verify(w)
    assert r["accept_len"][0] == 1 and list(r["out_tokens"][0]) == [3, 2]


def test_masked_tokens_have_no_mass(oracle_lib):
    """Logits of -inf (a constrained-decoding mask): weight exp(-inf) = 0 under every filter, so
    a draft on a masked token has p = 0 and is rejected, the residual max(0, p - q) puts no mass
    on masked tokens, and a top-k whose k-th largest value is -inf keeps the whole row.  Pinned
    against the filters' brute-force definitions and the residual's inverse CDF written out."""
    V = 8
    z = np.array([1.0, -np.inf, 2.0, -np.inf, 0.5, -np.inf, -np.inf, 3.0], np.float32)
    q = np.array([0.05, 0.3, 0.1, 0.2, 0.05, 0.1, 0.1, 0.1], np.float32)
    T = 0.7
    grid = (np.arange(64, dtype=np.float32) + np.float32(0.37)) / np.float32(64)
    checked = 0
    for K, P in [(0, 1.0), (2, 1.0), (6, 1.0), (0, 0.8), (6, 0.9)]:
        # (temperature and top_p reach the oracle as fp32 values)
        p = _brute_filter(z.astype(np.float64), float(np.float32(T)), K, float(np.float32(P)))
        assert p[~np.isfinite(z)].sum() == 0
        for x in (0, 2, 7):
            w = W.from_rows(V, np.tile(z, (2, 1)), q[None], np.array([[x]]),
                            np.array([[[0.999, 0.5], [0.5, 0.5]]], np.float32), temperature=T, top_k=K, top_p=P)
            r = oracle_lib.verify(w)
            assert abs(r["pq"][0, 0] - p[x]) < 1e-12, (K, P, x)
        res = np.maximum(p - q.astype(np.float64), 0.0)
        c = np.cumsum(res)
        for u in grid:
            t = np.float64(u) * c[-1]
            if np.min(np.abs(c - t)) < 1e-9:
                continue                          # a near-tie of the draw: either token is right
            w = W.from_rows(V, np.tile(z, (2, 1)), q[None], np.array([[1]]),
                            np.array([[[0.0, u], [0.5, 0.5]]], np.float32), temperature=T, top_k=K, top_p=P)
            r = oracle_lib.verify(w)
            assert r["accept_len"][0] == 0 and r["pq"][0, 0] == 0.0
            want = int(np.argmax(c > t))
            assert r["out_tokens"][0, 0] == want and np.isfinite(z[want]), (K, P, float(u))
            checked += 1
    assert checked > 250
    # greedy: the argmax among the finite logits
    for x, a, last in ((7, 1, 7), (2, 0, 7), (3, 0, 7)):
        w = W.from_rows(V, np.tile(z, (2, 1)), q[None], np.array([[x]]),
                        np.array([[[0.5, 0.5], [0.5, 0.5]]], np.float32), greedy=1)
        r = oracle_lib.verify(w)
        assert r["accept_len"][0] == a and r["out_tokens"][0, a] == last


# ------------------------------------------------------------------------------------------
# P9: the one-hot-draft scheme (FreeToken PR #836, Design: drafts are argmax proposals, so
# every verify row is sampled as decode would sample it and the matching prefix is kept)
# ------------------------------------------------------------------------------------------

def _joint_closed_form(logits, drafts, T, K, P, pres, freq):
    """Exact law of (accept_len a, final token t) for fixed drafts d_0..d_{k-1} when the
    drafts are one-hot: a = j with t != d_j (j < k), or a = k with any t, with probability
    prod_{i<j} p_i(d_i) * p_j(t).  p_i is the filtered target of row i with the drafts
    before it counted by the penalties, built from the filter definitions."""
    k, V = drafts.shape[0], logits.shape[1]
    ps = []
    for i in range(k + 1):
        z = logits[i].astype(np.float64).copy()
        c = np.bincount(drafts[:i], minlength=V).astype(np.float64)
        z -= (pres or 0.0) * (c > 0) + (freq or 0.0) * c
        ps.append(_brute_filter(z, T, K, P))
    law = np.zeros((k + 1, V))
    lead = 1.0
    for j in range(k + 1):
        law[j] = lead * ps[j]
        if j < k:
            law[j, drafts[j]] = 0.0
            lead *= ps[j][drafts[j]]
    return law, ps


@pytest.mark.parametrize("V,k,T,K,P,pres,freq", [
    (5, 2, 1.0, 0, 1.0, None, None),
    (7, 3, 0.8, 5, 0.9, 0.5, 0.3),
    (6, 2, 1.4, 0, 0.85, 1.0, 0.0),
])
def test_onehot_joint_law(oracle_lib, V, k, T, K, P, pres, freq):
    """P9a: sampling every row and keeping the matching prefix reproduces the target's
    sequential law exactly: the joint frequencies of (a, t) match the closed form, and no
    zero-probability outcome (the draft itself at the stopping row) ever appears.  The
    accept-test scheme given the same one-hot q must follow the same law (the two are equal
    in distribution and differ only in how they use the uniforms)."""
    n = 400_000
    g = _rng(1000 + V * 10 + k)
    logits = (g.standard_normal((k + 1, V)) * 1.2).astype(np.float32)
    drafts = logits[:k].argmax(-1).astype(np.int32)            # argmax proposals
    drafts[-1] = (drafts[-1] + 1) % V                          # and one that is not
    law, _ = _joint_closed_form(logits, drafts, T, K, P, pres, freq)
    q = np.zeros((k, V), np.float32)
    q[np.arange(k), drafts] = 1.0
    uni = g.random((n, k + 1, 2), dtype=np.float32)
    w = W.from_rows(V, logits, q, np.broadcast_to(drafts, (n, k)), uni, temperature=T, top_k=K, top_p=P,
                    presence=pres, frequency=freq)
    for onehot in (True, False):
        r = oracle_lib.verify(w, threads=8, onehot=onehot)
        assert (r["error"] == 0).all()
        a = r["accept_len"]
        t = r["out_tokens"][np.arange(n), a]
        obs = np.bincount(a * V + t, minlength=(k + 1) * V).astype(np.float64)
        assert _chisq_p(obs, law.reshape(-1)) > 1e-4, (onehot, obs.reshape(k + 1, V), law * n)
        assert (r["out_tokens"][:, :k][np.arange(k)[None, :] < a[:, None]] ==
                np.broadcast_to(drafts, (n, k))[np.arange(k)[None, :] < a[:, None]]).all()


def test_onehot_top_k_one_is_greedy(oracle_lib):
    """P9b: with p one-hot at the argmax (top-k = 1, no ties) every row's sample is its argmax,
    so the scheme returns the greedy result exactly, whatever the uniforms."""
    g = _rng(31)
    B, k, V = 300, 4, 40
    logits = g.standard_normal((B, k + 1, V)).astype(np.float32)
    am = logits.argmax(-1)
    drafts = np.where(g.random((B, k)) < 0.6, am[:, :k], g.integers(0, V, (B, k))).astype(np.int32)
    q = np.full((B, k, V), np.nan, np.float32)
    uni = g.random((B, k + 1, 2), dtype=np.float32)
    wg = W.from_rows(V, logits, q, drafts, uni, greedy=1, presence=0.3, frequency=0.2)
    ws = W.from_rows(V, logits, q, drafts, uni, greedy=0, top_k=1, temperature=0.7, presence=0.3,
                     frequency=0.2)
    rg = oracle_lib.verify(wg)
    rs = oracle_lib.verify(ws, onehot=True)
    np.testing.assert_array_equal(rs["accept_len"], rg["accept_len"])
    np.testing.assert_array_equal(rs["out_tokens"], rg["out_tokens"])


def test_onehot_reduces_to_pinned_paths(oracle_lib):
    """P9c: greedy requests are the same in both schemes; a request with no drafts is the
    extra-token draw of row 0 with slot 1 in both; and the scheme reads neither q nor slot 0
    (q all NaN and slot 0 out of range change nothing)."""
    w = W.random_batch(17, B=60, k_max=5, V=41, varlen=True, greedy_frac=0.4)
    ro = oracle_lib.verify(w, onehot=True)
    rr = oracle_lib.verify(w)
    gr = w.greedy.astype(bool)
    np.testing.assert_array_equal(ro["accept_len"][gr], rr["accept_len"][gr])
    np.testing.assert_array_equal(ro["out_tokens"][gr], rr["out_tokens"][gr])
    zero = w.num_drafts == 0
    assert zero.any()
    np.testing.assert_array_equal(ro["out_tokens"][zero], rr["out_tokens"][zero])
    w.draft_probs[:] = np.nan
    w.uniforms[:, 0] = 7.0
    r2 = oracle_lib.verify(w, onehot=True)
    assert (r2["error"] == 0).all()
    np.testing.assert_array_equal(r2["accept_len"], ro["accept_len"])
    np.testing.assert_array_equal(r2["out_tokens"], ro["out_tokens"])
    # out_pq: p(d_i) as the accept-test scheme reports it, q(d_i) = 1
    samp = ~np.isnan(rr["pq"][:, 0])
    np.testing.assert_array_equal(ro["pq"][samp, 0], rr["pq"][samp, 0])
    assert (ro["pq"][samp, 1] == 1.0).all()
    # slot 1 out of range is still an error
    w.uniforms[w.row_start(int(np.argmin(gr))), 1] = 1.0
    r3 = oracle_lib.verify(w, onehot=True)
    assert r3["error"][int(np.argmin(gr))] == 5


def test_onehot_matches_when_every_sample_matches(oracle_lib):
    """P9d: drafts set to the samples the rows produce (found one row at a time through the
    zero-draft reduction) are all accepted, and the output is row k's sample."""
    g = _rng(33)
    V, k = 23, 4
    logits = (g.standard_normal((k + 1, V)) * 1.5).astype(np.float32)
    u = g.random((1, k + 1, 2), dtype=np.float32)
    drafts = np.zeros((1, k), np.int32)
    for i in range(k):
        # with no penalties row i does not depend on the drafts: its sample is a zero-draft draw
        wi = W.from_rows(V, logits[i:i + 1], np.zeros((0, V), np.float32), np.zeros((1, 0), np.int32),
                         u[:, i:i + 1], temperature=0.9, top_p=0.95)
        drafts[0, i] = oracle_lib.verify(wi)["out_tokens"][0, 0]
    w = W.from_rows(V, logits, np.zeros((k, V), np.float32), drafts, u, temperature=0.9, top_p=0.95)
    r = oracle_lib.verify(w, onehot=True)
    assert r["accept_len"][0] == k
    assert list(r["out_tokens"][0, :k]) == list(drafts[0])
    wk = W.from_rows(V, logits[k:], np.zeros((0, V), np.float32), np.zeros((1, 0), np.int32), u[:, k:],
                     temperature=0.9, top_p=0.95)
    assert r["out_tokens"][0, k] == oracle_lib.verify(wk)["out_tokens"][0, 0]
    # change draft 2: the scan stops there and emits row 2's sample
    drafts[0, 2] = (drafts[0, 2] + 1) % V
    w2 = W.from_rows(V, logits, np.zeros((k, V), np.float32), drafts, u, temperature=0.9, top_p=0.95)
    r2 = oracle_lib.verify(w2, onehot=True)
    assert r2["accept_len"][0] == 2 and r2["out_tokens"][0, 2] == (drafts[0, 2] - 1) % V


# ------------------------------------------------------------------------------------------
# P10: prior history in the penalties (FreeToken PR #836, Design: what the request generated
# before a row counts as generated; the history extends that to the tokens before the drafts)
# ------------------------------------------------------------------------------------------

def _history_request(V, logits, drafts, uni, hist, pres, freq, T=0.9, K=0, P=1.0, greedy=0):
    """One request (uniform layout) with an explicit history {token: count}."""
    k = drafts.shape[0]
    w = W.from_rows(V, logits[None], np.zeros((1, k, V), np.float32), drafts[None], uni[None], temperature=T,
                    top_k=K, top_p=P, presence=pres, frequency=freq, greedy=greedy)
    toks = np.array(sorted(hist), np.int32)
    w.prior_offsets = np.array([0, toks.size], np.int32)
    w.prior_tokens = toks
    w.prior_counts = np.array([hist[t] for t in toks.tolist()], np.int32)
    return w


@pytest.mark.parametrize("seed", range(4))
def test_history_is_earlier_drafts(oracle_lib, seed):
    """P10a: the first j drafts of a request, moved into its history as counts, leave every
    later row unchanged: row i of the original equals row i - j of the request that starts at
    draft j (same logits, drafts and uniforms), for sampled and greedy requests, and so do the
    verify results.  Drafts repeat (V is small), so counts above one and tokens present both
    in the history and among the remaining drafts occur."""
    g = _rng(500 + seed)
    V, k = 9, 6
    logits = (g.standard_normal((k + 1, V)) * 1.3).astype(np.float32)
    drafts = g.integers(0, V, k).astype(np.int32)
    uni = g.random((k + 1, 2), dtype=np.float32)
    pres, freq = float(g.uniform(0.1, 1.2)), float(g.uniform(0.1, 0.9))
    for greedy in (0, 1):
        full = _history_request(V, logits, drafts, uni, {}, pres, freq, greedy=greedy, K=[0, 5][seed % 2],
                                P=[1.0, 0.85][seed // 2])
        for j in range(1, k + 1):
            hist = {}
            for t in drafts[:j].tolist():
                hist[t] = hist.get(t, 0) + 1
            cut = _history_request(V, logits[j:], drafts[j:], uni[j:], hist, pres, freq, greedy=greedy,
                                   K=[0, 5][seed % 2], P=[1.0, 0.85][seed // 2])
            for i in range(j, k + 1):
                np.testing.assert_array_equal(oracle_lib.row_probs(cut, 0, i - j), oracle_lib.row_probs(full, 0, i))


def test_history_softmax_against_numpy(oracle_lib):
    """P10b: with no filter, row i is numpy's float64 softmax((z - presence [c > 0] -
    frequency c) / T) with c = history count + count among the drafts before the row; row 0
    carries the history alone."""
    w = W.random_batch(61, B=24, k_max=5, V=40, dtype="f32", greedy_frac=0.0, draft_sigma=0.2)
    W.with_history(w, 61, 12)
    w.top_k[:] = 0
    w.top_p[:] = 1.0
    w.presence[:] = np.linspace(0.0, 1.5, w.B).astype(np.float32)
    w.frequency[:] = np.linspace(0.9, 0.0, w.B).astype(np.float32)
    lg = w.logits_f32().astype(np.float64)
    assert (np.diff(w.prior_offsets) > 0).sum() >= 10
    for b in range(w.B):
        r0, d0 = w.row_start(b), w.draft_start(b)
        h = np.zeros(w.V)
        lo, hi = w.prior_offsets[b], w.prior_offsets[b + 1]
        h[w.prior_tokens[lo:hi]] = w.prior_counts[lo:hi]
        for i in range(int(w.num_drafts[b]) + 1):
            c = h + np.bincount(w.draft_tokens[d0:d0 + i], minlength=w.V)
            z = lg[r0 + i] - (w.presence[b] * (c > 0) + w.frequency[b] * c)
            np.testing.assert_allclose(oracle_lib.row_probs(w, b, i), _softmax(z / float(w.temperature[b])),
                                       rtol=1e-12, atol=1e-15)


def test_history_greedy_against_numpy(oracle_lib):
    """P10c: a greedy request with a history accepts while the draft is numpy's argmax of the
    penalised row, the history counted on every row including row 0."""
    w = W.random_batch(62, B=40, k_max=4, V=30, dtype="f32", greedy_frac=1.0)
    lg = w.logits_f32().astype(np.float64)
    for b in range(w.B):          # drafts mostly the unpenalised argmax, so the history matters
        r0, d0 = w.row_start(b), w.draft_start(b)
        for i in range(int(w.num_drafts[b])):
            w.draft_tokens[d0 + i] = int(np.argmax(lg[r0 + i]))
    W.with_history(w, 62, 8, top_share=1.0)
    w.presence[:] = 0.8
    w.frequency[:] = 0.3
    r = oracle_lib.verify(w)
    for b in range(w.B):
        r0, d0 = w.row_start(b), w.draft_start(b)
        h = np.zeros(w.V)
        lo, hi = w.prior_offsets[b], w.prior_offsets[b + 1]
        h[w.prior_tokens[lo:hi]] = w.prior_counts[lo:hi]
        a = 0
        k = int(w.num_drafts[b])
        while True:
            c = h + np.bincount(w.draft_tokens[d0:d0 + a], minlength=w.V)
            am = int(np.argmax(lg[r0 + a] - (0.8 * (c > 0) + 0.3 * c)))
            if a == k or w.draft_tokens[d0 + a] != am:
                break
            a += 1
        assert r["accept_len"][b] == a and r["out_tokens"][b, a] == am, b


def test_history_errors(oracle_lib):
    """A malformed history (ids not ascending, a repeat, an id outside [0, V), a count below
    one, offsets that decrease) is a device-data error (code 8) of that request only."""
    w = W.random_batch(63, B=8, k_max=3, V=50, greedy_frac=0.0)
    W.with_history(w, 63, 6)
    w.prior_offsets = np.array([0, 3, 6, 9, 12, 15, 18, 21, 24], np.int32)
    w.prior_tokens = np.tile(np.array([3, 9, 20], np.int32), 8)
    w.prior_counts = np.ones(24, np.int32)
    w.prior_tokens[0:3] = [9, 3, 20]       # request 0: not ascending
    w.prior_tokens[3:6] = [3, 3, 20]       # request 1: a repeat
    w.prior_tokens[6:9] = [3, 9, 50]       # request 2: out of range
    w.prior_counts[10] = 0                 # request 3: count below one
    r = oracle_lib.verify(w)
    assert list(r["error"]) == [8, 8, 8, 8, 0, 0, 0, 0]
    w.prior_offsets[6] = 14                # request 5 ends before it starts
    r = oracle_lib.verify(w)
    assert r["error"][5] == 8 and r["error"][4] == 0
