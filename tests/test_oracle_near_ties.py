"""Pins for the oracle's near-tie classifier.

A GPU result may part from the oracle only at a decision the oracle flags as a near-tie: a
float64 value within 1e-5 of a boundary (the accept test u < min(1, p/q), a CDF boundary of a
draw, the top-p mass at a value level, the top-2 gap of a penalised greedy row) or a residual
mass W below 1e-6.  Each test below builds one decision at a known distance from its
boundary -- 1e-6 (must be flagged) and 1e-4 (must not) -- from values computed here from the
definitions, and checks the flag, its kind and where on the request's path it is recorded
(the keep decision of row i, or the final token).  A band that is too wide hides GPU mistakes;
one that is too narrow fails correct fp32 results.
"""
import numpy as np
import pytest

import sv_workloads as W

F32 = np.float32


def _f32(x):
    return float(F32(x))


def _run(oracle_lib, w, onehot=False):
    r = oracle_lib.verify(w, onehot=onehot)
    return {k: (v[0] if k not in ("pq", "pq_near") else v) for k, v in r.items()}


def _kinds(r):
    return {k: int(r[k]) for k in ("near_accept", "near_cdf", "near_filter", "near_argmax", "near_w") if r[k]}


def _softmax64(z32):
    z = np.asarray(z32, np.float64)
    e = np.exp(z - z.max())
    return e / e.sum()


# ------------------------------------------------------------------------------------------
# accept test: |u - min(1, p/q)| < 1e-5
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("off,near", [(1e-6, True), (-1e-6, True), (1e-4, False), (-1e-4, False)])
def test_accept_band(oracle_lib, off, near):
    # two equal logits: p = [1/2, 1/2] exactly; q(x=0) = 0.8 (as fp32)
    q = np.array([[0.8, 0.2]], F32)
    thr = 0.5 / float(q[0, 0])
    u0 = _f32(thr + off)
    rows = np.zeros((2, 2), F32)
    w = W.from_rows(2, rows, q, np.array([[0]]), np.array([[[u0, 0.3], [0.5, 0.3]]], F32))
    r = _run(oracle_lib, w)
    assert r["accept_len"] == (1 if u0 < thr else 0)
    assert r["near_accept"] == int(near) and _kinds(r) == ({"near_accept": 1} if near else {})
    assert int(r["near_rows"]) == (1 if near else 0) and r["near_final"] == 0


def test_accept_band_locates_the_row(oracle_lib):
    """Only row 2 of 4 drafts sits on the accept boundary: bit 2 of the row mask."""
    q = np.tile(np.array([0.8, 0.2], F32), (4, 1))
    thr = 0.5 / float(q[0, 0])
    uni = np.array([[[0.1, 0.3], [0.2, 0.3], [_f32(thr - 1e-6), 0.3], [0.9, 0.3], [0.5, 0.3]]], F32)
    w = W.from_rows(2, np.zeros((5, 2), F32), q, np.zeros((1, 4), np.int32), uni)
    r = _run(oracle_lib, w)
    assert r["accept_len"] == 3 and int(r["near_rows"]) == 1 << 2 and r["near_final"] == 0


# ------------------------------------------------------------------------------------------
# CDF boundary of a draw: |cumsum_v / W - u| < 1e-5 at the chosen token
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("off,near,tok", [(1e-6, True, 2), (-1e-6, True, 1), (1e-4, False, 2),
                                          (-1e-4, False, 1)])
def test_cdf_band(oracle_lib, off, near, tok):
    # four equal logits, no drafts: the extra token is drawn from p = 1/4 each, whose CDF has
    # boundaries at 1/4, 1/2, 3/4
    u1 = _f32(0.5 + off)
    w = W.from_rows(4, np.zeros((1, 4), F32), np.zeros((0, 4), F32), np.zeros((1, 0), np.int32),
                    np.array([[[0.5, u1]]], F32))
    r = _run(oracle_lib, w)
    assert r["out_tokens"][0] == tok
    assert _kinds(r) == ({"near_cdf": 1} if near else {})
    assert r["near_final"] == int(near) and int(r["near_rows"]) == 0


def test_cdf_band_of_a_residual_draw(oracle_lib):
    """The residual draw at a rejection is the stopping row's final decision."""
    # p = [1/2, 1/2]; q = [1, 0] with draft 0: ratio 1/2; the residual is one-hot at token 1,
    # so no u is near its CDF; then a residual [1/4 .. ] spread by a 4-token row
    rows = np.zeros((2, 4), F32)
    q = np.array([[0.5, 0.5, 0.0, 0.0]], F32)           # residual = [0, 0, 1/4, 1/4] / (1/2)
    for u1, near, tok in [(_f32(0.5 + 1e-6), True, 3), (_f32(0.5 + 1e-4), False, 3), (_f32(0.5 - 1e-6), True, 2)]:
        w = W.from_rows(4, rows, q, np.array([[0]]), np.array([[[0.9, u1], [0.5, 0.5]]], F32))
        r = _run(oracle_lib, w)
        assert r["accept_len"] == 0 and r["out_tokens"][0] == tok
        assert r["near_final"] == int(near) and int(r["near_rows"]) == 0 and _kinds(r) == (
            {"near_cdf": 1} if near else {})


# ------------------------------------------------------------------------------------------
# greedy: the top-2 values of a penalised row within 1e-5 (relative)
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("rel,near", [(1e-6, True), (1e-4, False)])
def test_greedy_gap_band(oracle_lib, rel, near):
    # draft 2 is row 0's argmax and is accepted; row 1 is penalised (presence 0.5 on token 2)
    # and its top two values differ by rel x 30 (the band is relative to the larger value)
    row1 = np.array([30.0, 30.0 - 30.0 * rel, 1.0], F32)
    rows = np.stack([np.array([0.0, 0.0, 5.0], F32), row1])
    w = W.from_rows(3, rows, np.full((1, 3), 1 / 3, F32), np.array([[2]]), np.full((1, 2, 2), 0.5, F32),
                    presence=0.5, frequency=0.0, greedy=1)
    r = _run(oracle_lib, w)
    assert r["accept_len"] == 1 and r["out_tokens"][1] == 0
    assert _kinds(r) == ({"near_argmax": 1} if near else {})
    # the stopping row's argmax is the final token
    assert r["near_final"] == int(near) and int(r["near_rows"]) == 0


def test_greedy_gap_flags_the_compare(oracle_lib):
    """A near-tied argmax at a row that keeps its draft flags that row's compare."""
    rows = np.array([[0.0, 0.0, 5.0], [3.0, 3.0 - 3e-6, 1.0], [0.0, 4.0, 0.0]], F32)
    w = W.from_rows(3, rows, np.full((2, 3), 1 / 3, F32), np.array([[2, 0]]), np.full((1, 3, 2), 0.5, F32),
                    presence=0.5, frequency=0.0, greedy=1)
    r = _run(oracle_lib, w)
    assert r["accept_len"] == 2 and int(r["near_rows"]) == 1 << 1 and r["near_final"] == 0


# ------------------------------------------------------------------------------------------
# top-p: the mass strictly above a value level within 1e-5 of top_p
# ------------------------------------------------------------------------------------------

Z4 = np.log(np.array([0.5, 0.25, 0.125, 0.125])).astype(F32)
ABOVE = float(_softmax64(Z4)[:2].sum())   # mass above the level {2, 3}


@pytest.mark.parametrize("off,near", [(1e-6, True), (-1e-6, True), (1e-4, False), (-1e-4, False)])
def test_top_p_band_flags_draws(oracle_lib, off, near):
    P = _f32(ABOVE + off)
    w = W.from_rows(4, Z4[None], np.zeros((0, 4), F32), np.zeros((1, 0), np.int32),
                    np.array([[[0.5, 0.1]]], F32), top_p=P)
    r = _run(oracle_lib, w)
    assert r["out_tokens"][0] == 0
    # flipping the level {2, 3} (a quarter of the mass) moves every CDF value
    assert _kinds(r) == ({"near_filter": 1} if near else {})
    assert r["near_final"] == int(near)


@pytest.mark.parametrize("off,near", [(1e-6, True), (1e-4, False)])
def test_top_p_band_flags_accept_tests(oracle_lib, off, near):
    P = _f32(ABOVE + off)
    q = np.array([[0.8, 0.1, 0.05, 0.05]], F32)
    p = _softmax64(Z4)
    # draft 2 lies in the ambiguous level itself; draft 0 does not, but its p(x)/q(x) moves by
    # up to a quarter when the level flips, and u sits 1e-3 from it
    for x, u0 in [(2, 0.99), (0, _f32(min(1.0, p[0] / 0.8) + 1e-3))]:
        w = W.from_rows(4, np.stack([Z4, Z4]), q, np.array([[x]]), np.array([[[u0, 0.1], [0.5, 0.1]]], F32),
                        top_p=P)
        r = _run(oracle_lib, w)
        assert int(r["near_rows"]) & 1 == int(near), (x, r)
        assert r["near_filter"] >= int(near)
        assert r["pq_near"][0] == int(near)


# ------------------------------------------------------------------------------------------
# residual mass W < 1e-6
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("W_,near", [(5e-7, True), (1e-4, False)])
def test_small_residual_band(oracle_lib, W_, near):
    # draft 0 has p = W, q = 2W: ratio 1/2, rejected by u = 0.75 far from the boundary; the
    # residual is W at token 2 (and rounding crumbs elsewhere)
    p = np.array([W_, 0.5, 0.5 - W_])
    q = np.array([[2 * W_, 0.5, 0.5 - 2 * W_]], F32)
    z = np.log(p).astype(F32)
    w = W.from_rows(3, np.stack([z, z]), q, np.array([[0]]), np.array([[[0.75, 0.5], [0.5, 0.5]]], F32))
    r = _run(oracle_lib, w)
    assert r["accept_len"] == 0 and r["out_tokens"][0] == 2
    assert _kinds(r) == ({"near_w": 1} if near else {})
    assert r["near_final"] == int(near) and int(r["near_rows"]) == 0


# ------------------------------------------------------------------------------------------
# one-hot scheme: a near-tied sample flags the compare of its row, and at the stopping row the
# final token
# ------------------------------------------------------------------------------------------

def test_onehot_sample_band(oracle_lib):
    rows = np.zeros((3, 4), F32)
    # row 0 samples token 2 at u = 1/2 + 1e-6 (near) and keeps draft 2; row 1 samples token 1
    # far from a boundary and rejects draft 3
    uni = np.array([[[0.0, _f32(0.5 + 1e-6)], [0.0, 0.3], [0.0, 0.9]]], F32)
    w = W.from_rows(4, rows, np.zeros((2, 4), F32), np.array([[2, 3]]), uni)
    r = _run(oracle_lib, w, onehot=True)
    assert r["accept_len"] == 1 and r["out_tokens"][1] == 1
    assert int(r["near_rows"]) == 1 and r["near_final"] == 0 and _kinds(r) == {"near_cdf": 1}
    uni[0, 1, 1] = _f32(0.25 + 1e-6)
    r = _run(oracle_lib, W.from_rows(4, rows, np.zeros((2, 4), F32), np.array([[2, 3]]), uni), onehot=True)
    assert r["accept_len"] == 1 and r["out_tokens"][1] == 1
    assert int(r["near_rows"]) == 1 | 2 and r["near_final"] == 1


# ------------------------------------------------------------------------------------------
# the parity rule built on the flags (tests/sv_parity.py), on planted GPU results
# ------------------------------------------------------------------------------------------

def test_parity_excuses_only_a_flagged_first_divergence(oracle_lib):
    import sv_parity
    q = np.tile(np.array([0.8, 0.2], F32), (3, 1))
    thr = 0.5 / float(q[0, 0])
    # request 0: row 1's accept test is near (flagged); request 1: nothing is near
    uni = np.array([[[0.1, 0.3], [_f32(thr - 1e-6), 0.3], [0.2, 0.3], [0.5, 0.3]],
                    [[0.1, 0.3], [0.2, 0.3], [0.9, 0.3], [0.5, 0.3]]], F32)
    w = W.from_rows(2, np.zeros((4, 2), F32), q, np.zeros((2, 3), np.int32), uni)
    o = oracle_lib.verify(w)
    assert list(o["accept_len"]) == [3, 2]

    def gpu(acc, toks):
        return {"accept_len": np.array(acc, np.int32), "out_tokens": np.array(toks, np.int32)}

    same = gpu(o["accept_len"], o["out_tokens"])
    assert sv_parity.compare(w, same, o)["excused_mismatches"] == 0
    # request 0 rejecting at the flagged row 1: excused, whatever it draws
    g = gpu([1, 2], [[0, 1, -1, -1], o["out_tokens"][1]])
    assert sv_parity.compare(w, g, o)["excused_mismatches"] == 1
    # request 0 rejecting at row 0 (before the flagged row): a failure
    with pytest.raises(AssertionError):
        sv_parity.compare(w, gpu([0, 2], [[1, -1, -1, -1], o["out_tokens"][1]]), o)
    # request 1 with a different residual token: its final draw is not flagged
    t1 = o["out_tokens"][1].copy()
    t1[2] = 1 - t1[2]
    with pytest.raises(AssertionError):
        sv_parity.compare(w, gpu(o["accept_len"], [o["out_tokens"][0], t1]), o)
