"""Comparison of the CUDA path's outputs with the float64 oracle on the same inputs.

Rules (tolerances fixed by the method's numerics, see the design notes):
  - out_tokens and accept_len are bit-exact, except that a request may part from the oracle at
    a decision the oracle flags as a near-tie (a float64 value within 1e-5 of an accept, CDF,
    top-p or argmax boundary, or a residual mass below 1e-6).  The comparison walks the
    request's path: the first decision where the GPU and the oracle differ must be a flagged
    one -- the keep decision of the row where the two accept lengths first differ, or, with
    equal accept lengths, the final token's draw.  What follows a flagged divergence is
    excused.  Such excused mismatches are counted and must stay below 1e-4 of all decisions
    on the full-size workloads;
  - the flagged near-ties themselves are counted by kind and reported.  Accept-test near-ties
    (|u - min(1, p/q)| < 1e-5, which uniform u hits with probability about 2e-5) must stay
    below 1e-4 of the decisions of a full-size workload; how often a draw lies within 1e-5 of
    a CDF boundary is a property of the distribution drawn from (every token of probability
    below 2e-5 does), so that share is reported, not bounded;
  - p(x_i) agrees to 1e-5 absolute and q(x_i) (an input value) exactly, for every draft of a
    sampled request whose p(x_i) is not itself on a near-tie of the row's kept set;
  - a request the oracle rejects as invalid has accept_len -1 and all tokens -1.
"""
import numpy as np

P_TOL = 1e-5
NEAR_TIE_SHARE = 1e-4
NEAR_KINDS = ("near_accept", "near_cdf", "near_filter", "near_argmax", "near_w")


def first_divergence(gpu, ora, b):
    """Where request b's GPU result first parts from the oracle's: None when they agree,
    ("keep", i) when the accept lengths differ (row i = the smaller one decided differently
    whether to keep its draft), ("final", a) when only the final token differs."""
    ag, ao = int(gpu["accept_len"][b]), int(ora["accept_len"][b])
    tg, to = gpu["out_tokens"][b], ora["out_tokens"][b]
    if ag == ao and np.array_equal(tg, to):
        return None
    if ag != ao:
        return ("keep", min(ag, ao))
    assert np.array_equal(tg[:ao], to[:ao]), (b, "accepted drafts differ", tg.tolist(), to.tolist())
    return ("final", ao)


def flagged(ora, b, where):
    """Whether the oracle flagged the decision `where` (see first_divergence) of request b."""
    kind, i = where
    if kind == "final":
        return bool(ora["near_final"][b])
    return bool((int(ora["near_rows"][b]) >> i) & 1) if i < 64 else False


def compare(w, gpu, ora, requests=None, check_share=False, pq_on_path=False):
    """Asserts parity; returns a summary dict (requests compared, near-ties by kind, ...).
    pq_on_path: compare p(x_i), q(x_i) only for the drafts both sides read (i <= the smaller
    accept length) -- the lazy scheme reads no row after a request's stopping row."""
    reqs = [int(b) for b in (range(w.B) if requests is None else requests)]
    n_cmp = n_near_req = n_excused = 0
    mism, excused = [], []
    for b in reqs:
        if ora["error"][b]:
            assert gpu["accept_len"][b] == -1, (b, "invalid request must give accept_len -1")
            assert (gpu["out_tokens"][b] == -1).all(), (b, "invalid request must give -1 tokens")
            continue
        n_cmp += 1
        n_near_req += 1 if ora["near_ties"][b] > 0 else 0
        where = first_divergence(gpu, ora, b)
        if where is None:
            continue
        if flagged(ora, b, where):
            n_excused += 1
            excused.append((b,) + where)
        else:
            mism.append((b, where, int(gpu["accept_len"][b]), int(ora["accept_len"][b]),
                         gpu["out_tokens"][b].tolist(), ora["out_tokens"][b].tolist()))
    assert not mism, f"{len(mism)} requests part from the oracle at an unflagged decision, first: {mism[:5]}"
    # per-draft probabilities
    n_pq = 0
    if "pq" in gpu and w.total_drafts:
        for b in reqs:
            if ora["error"][b] or w.greedy[b]:
                continue
            d0 = w.draft_start(b)
            n_i = int(w.num_drafts[b])
            if pq_on_path:
                n_i = min(n_i, 1 + min(int(gpu["accept_len"][b]), int(ora["accept_len"][b])))
            for i in range(n_i):
                d = d0 + i
                if ora["pq_near"][d]:
                    continue
                n_pq += 1
                gp, gq = gpu["pq"][d]
                op, oq = ora["pq"][d]
                assert abs(gp - op) <= P_TOL, (b, i, float(gp), float(op))
                assert gq == np.float32(oq), (b, i, float(gq), float(oq))
    ok = [b for b in reqs if not ora["error"][b]]
    dec = int(ora["decisions"][ok].sum()) if ok else 0
    kinds = {k: int(ora[k][ok].sum()) if ok else 0 for k in NEAR_KINDS}
    near = sum(kinds.values())
    if check_share and dec:
        assert n_excused / dec < NEAR_TIE_SHARE, f"excused near-tie mismatches {n_excused}/{dec}"
        assert kinds["near_accept"] / dec < NEAR_TIE_SHARE, f"accept-test near-ties {kinds['near_accept']}/{dec}"
    return dict(requests=n_cmp, decisions=dec, near_ties=near, near_share=near / dec if dec else 0.0,
                near_by_kind=kinds, near_tie_requests=n_near_req, excused_mismatches=n_excused,
                excused=excused[:10], pq_checked=n_pq)


def check_invariants(w, gpu):
    """Properties that hold at any size, without the oracle."""
    for b in range(w.B):
        a = int(gpu["accept_len"][b])
        k = int(w.num_drafts[b])
        row = gpu["out_tokens"][b]
        assert 0 <= a <= k, (b, a, k)
        assert (row[: a + 1] >= 0).all() and (row[: a + 1] < w.V).all(), (b, row)
        assert (row[a + 1:] == -1).all(), (b, row)
        d0 = w.draft_start(b)
        assert np.array_equal(row[:a], w.draft_tokens[d0: d0 + a]), b
