"""Comparison of the CUDA path's outputs with the float64 oracle on the same inputs.

Rules (tolerances fixed by the method's numerics, see the design notes):
  - out_tokens and accept_len are bit-exact for every request whose oracle path holds no
    near-tie decision (a float64 value within 1e-5 of an accept, CDF, top-p or argmax
    boundary, or a residual mass below 1e-6);
  - a request whose path holds a near-tie may differ; such excused mismatches are counted and
    must stay below 1e-4 of all decisions (checked on large batches); the number of flagged
    near-tie decisions is reported alongside, whether or not the results differ;
  - p(x_i) agrees to 1e-5 absolute and q(x_i) (an input value) exactly, for every draft of a
    sampled request whose row's kept set is not itself on a near-tie;
  - a request the oracle rejects as invalid has accept_len -1 and all tokens -1.
"""
import numpy as np

P_TOL = 1e-5
NEAR_TIE_SHARE = 1e-4


def compare(w, gpu, ora, requests=None, check_share=False):
    """Asserts parity; returns a summary dict (requests compared, near-tie requests, ...)."""
    reqs = range(w.B) if requests is None else requests
    n_cmp = n_near_req = n_excused = 0
    mism = []
    for b in reqs:
        b = int(b)
        if ora["error"][b]:
            assert gpu["accept_len"][b] == -1, (b, "invalid request must give accept_len -1")
            assert (gpu["out_tokens"][b] == -1).all(), (b, "invalid request must give -1 tokens")
            continue
        n_cmp += 1
        same = (gpu["accept_len"][b] == ora["accept_len"][b]
                and np.array_equal(gpu["out_tokens"][b], ora["out_tokens"][b]))
        if ora["near_ties"][b] > 0:
            n_near_req += 1
            n_excused += 0 if same else 1
            continue
        if not same:
            mism.append((b, int(gpu["accept_len"][b]), int(ora["accept_len"][b]),
                         gpu["out_tokens"][b].tolist(), ora["out_tokens"][b].tolist()))
    assert not mism, f"{len(mism)} requests differ outside near-ties, first: {mism[:5]}"
    # per-draft probabilities
    n_pq = 0
    if "pq" in gpu and w.total_drafts:
        for b in reqs:
            b = int(b)
            if ora["error"][b] or w.greedy[b]:
                continue
            d0 = w.draft_start(b)
            for i in range(int(w.num_drafts[b])):
                d = d0 + i
                if ora["pq_near"][d]:
                    continue
                n_pq += 1
                gp, gq = gpu["pq"][d]
                op, oq = ora["pq"][d]
                assert abs(gp - op) <= P_TOL, (b, i, float(gp), float(op))
                assert gq == np.float32(oq), (b, i, float(gq), float(oq))
    dec = int(ora["decisions"][list(map(int, reqs))].sum()) if len(reqs) else 0
    near = int(ora["near_ties"][list(map(int, reqs))].sum()) if len(reqs) else 0
    if check_share and dec:
        assert n_excused / dec < NEAR_TIE_SHARE, f"excused near-tie mismatches {n_excused}/{dec}"
    return dict(requests=n_cmp, near_tie_requests=n_near_req, excused_mismatches=n_excused, decisions=dec,
                near_ties=near, pq_checked=n_pq)


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
