"""spec_verify_lazy (no row after a request's first rejection is read) against the float64
oracle, element by element, through the C ABI.  Its results are spec_verify's: the same
oracle and the same parity rules apply, on the same batches and on the full-size workloads.
"""
import numpy as np
import pytest

import sv_workloads as W
from sv_parity import check_invariants, compare

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_12_gb300 as sv
    sv.lib()
    return sv


def run_lazy(w, want_pq=True):
    from speculative_decoding_verification_12_gb300.batch import DeviceBatch
    db = DeviceBatch.from_host(w, "cuda", want_pq=want_pq)
    db.run(lazy=True)
    return db.results(), db


def lazy_compare(oracle_lib, w, check_share=False):
    g, db = run_lazy(w)
    o = oracle_lib.verify(w, threads=16)
    return compare(w, g, o, check_share=check_share, pq_on_path=True), g, o, db


CASES = [
    # seed, B, k_max, V, dtype, varlen, tie_step, greedy_frac
    (60, 16, 4, 1000, "f32", False, 0.0, 0.3),
    (61, 24, 6, 4096, "bf16", True, 0.0, 0.3),
    (62, 20, 8, 3000, "bf16", False, 0.5, 0.2),    # forced ties
    (63, 8, 5, 1, "f32", False, 0.0, 0.5),         # V = 1
    (64, 32, 8, 20000, "bf16", True, 0.0, 0.3),
    (65, 16, 7, 65536, "f32", False, 0.125, 0.25),
    (66, 6, 64, 304, "f32", True, 0.0, 0.3),       # k_max = 64
    (67, 300, 8, 4096, "bf16", True, 0.0, 0.3),    # many rows, few CTAs per row
]


@pytest.mark.parametrize("case", CASES, ids=[f"seed{c[0]}_V{c[3]}_{c[4]}" for c in CASES])
def test_lazy_random_batches(sv, oracle_lib, case):
    seed, B, k, V, dt, varlen, tie, gf = case
    w = W.random_batch(seed, B=B, k_max=k, V=V, dtype=dt, varlen=varlen, tie_step=tie, greedy_frac=gf)
    lazy_compare(oracle_lib, w)


def test_lazy_high_acceptance(sv, oracle_lib):
    """Drafts that are the rows' argmax: most requests keep draft 0, so the second phase reads
    most rows, and long accepted prefixes end in extra-token draws."""
    w = W.random_batch(68, B=40, k_max=6, V=8192, dtype="bf16", greedy_frac=0.5)
    lg = w.logits_f32()
    for b in range(w.B):
        r0, d0 = w.row_start(b), w.draft_start(b)
        for i in range(int(w.num_drafts[b])):
            w.draft_tokens[d0 + i] = int(np.argmax(lg[r0 + i]))
    s, g, o, _ = lazy_compare(oracle_lib, w)
    assert (g["accept_len"] >= 1).sum() > w.B // 2


def test_lazy_filters_and_residual_passes(sv, oracle_lib):
    """Every kept-set path: list rows, whole-row kept sets (no filter, large top-k, top-p only,
    which take the residual kernel at a rejection) and candidate overflow."""
    w = W.random_batch(69, B=30, k_max=4, V=9000, dtype="bf16", greedy_frac=0.0, varlen=True)
    w.top_k[:] = np.array([0, 40, 3000, 0, 1, 600] * 5, np.int32)
    w.top_p[:] = np.array([1.0, 0.9, 0.7, 0.5, 1.0, 1.0] * 5, np.float32)
    lazy_compare(oracle_lib, w)


def test_lazy_zero_drafts_padding_and_errors(sv, oracle_lib):
    w = W.random_batch(70, B=30, k_max=5, V=2000, dtype="bf16", greedy_frac=0.3)
    w.num_drafts[::3] = 0
    w.num_drafts[1::3] = 2
    w.draft_tokens[w.draft_start(4) + 1] = 2000      # bad token behind draft 0
    w.temperature[7] = -1.0
    w.num_drafts[10] = 9                              # beyond k_max
    s, g, o, db = lazy_compare(oracle_lib, w)
    assert (g["accept_len"][[4, 10]] == -1).all()
    assert sv.sv_read_device_error(db.workspace)[0] != 0


def test_lazy_empty_requests_in_ragged_layout(sv, oracle_lib):
    """Requests that own no rows in row_offsets get -1 and a layout error, the others verify."""
    w = W.random_batch(71, B=12, k_max=4, V=3000, dtype="bf16", varlen=True, greedy_frac=0.3)
    ro = w.row_offsets.copy()
    # request 5 owns no rows: its rows go to the front of request 6
    ro[6] = ro[5]
    w.row_offsets = ro
    w.num_drafts[6] = min(w.k_max, int(ro[7] - ro[6]) - 1)
    # request 6's draft rows now start one slot early, on the last draft slot of the requests
    # before it: those leave that slot unused
    for b in range(5):
        w.num_drafts[b] = min(int(w.num_drafts[b]), max(0, int(ro[6]) - 6 - (int(ro[b]) - b)))
    s, g, o, db = lazy_compare(oracle_lib, w)
    assert g["accept_len"][5] == -1 and (g["out_tokens"][5] == -1).all() and o["error"][5] == 1
    assert sv.sv_read_device_error(db.workspace)[0] == 1


def test_lazy_matches_one_pass_call(sv):
    """The same batch through both entry points gives the same outputs."""
    from speculative_decoding_verification_12_gb300.batch import DeviceBatch
    w = W.random_batch(72, B=64, k_max=5, V=12000, dtype="bf16", varlen=True, greedy_frac=0.3)
    w.top_k[::4] = 0
    w.top_p[::4] = 1.0
    db = DeviceBatch.from_host(w, "cuda", want_pq=True)
    db.run()
    ref = db.results()
    db.run(lazy=True)
    got = db.results()
    np.testing.assert_array_equal(got["accept_len"], ref["accept_len"])
    np.testing.assert_array_equal(got["out_tokens"], ref["out_tokens"])
    # (p, q) agree wherever the lazy call read the row; past a row-0 rejection they are NaN
    for b in range(w.B):
        d0, k, a = w.draft_start(b), int(w.num_drafts[b]), int(ref["accept_len"][b])
        for i in range(k):
            if a == 0 and i > 0:
                assert np.isnan(got["pq"][d0 + i]).all() or w.greedy[b] or a < 0, (b, i)
            else:
                np.testing.assert_array_equal(got["pq"][d0 + i], ref["pq"][d0 + i])


@pytest.mark.parametrize("name", ["peaks", "zipf", "ragged", "stream"])
def test_lazy_full_workloads(sv, oracle_lib, name):
    w = W.make(name)
    g, _ = run_lazy(w, want_pq=False)
    check_invariants(w, g)
    o = oracle_lib.verify(w, threads=16)
    s = compare(w, g, o, check_share=True)
    print("lazy", name, s)
    assert s["requests"] == w.B
