"""spec_verify_onehot (drafts proposed as one-hot argmax tokens: every row sampled, the matching
prefix kept) against the float64 oracle's one-hot scheme, element by element, through the C ABI.
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


def run_onehot(w, want_pq=True):
    from speculative_decoding_verification_12_gb300.batch import DeviceBatch
    db = DeviceBatch.from_host(w, "cuda", want_pq=want_pq)
    db.run(onehot=True)
    return db.results(), db


def argmax_drafts(w, share, seed):
    """Replace a share of the drafts with their row's argmax (argmax proposals that agree with
    the target), so that long accepted prefixes occur."""
    g = np.random.default_rng(seed)
    lg = w.logits_f32()
    for b in range(w.B):
        r0, d0 = w.row_start(b), w.draft_start(b)
        for i in range(int(w.num_drafts[b])):
            if g.random() < share:
                w.draft_tokens[d0 + i] = int(np.argmax(lg[r0 + i]))
    return w


def full_compare(oracle_lib, w, check_share=False):
    g, db = run_onehot(w)
    o = oracle_lib.verify(w, threads=8, onehot=True)
    return compare(w, g, o, check_share=check_share), g, o


CASES = [
    # seed, B, k_max, V, dtype, varlen, tie_step, greedy_frac
    (40, 16, 4, 1000, "f32", False, 0.0, 0.3),
    (41, 24, 6, 4099, "bf16", True, 0.0, 0.3),     # odd V: unaligned rows, the one-kernel path
    (42, 20, 8, 3000, "bf16", False, 0.5, 0.2),    # forced ties at top-k / top-p boundaries
    (43, 8, 5, 1, "f32", False, 0.0, 0.5),         # V = 1: every sample is token 0
    (44, 32, 8, 20001, "bf16", True, 0.0, 0.3),
    (45, 16, 7, 65536, "f32", False, 0.125, 0.25),
    (46, 6, 64, 300, "f32", True, 0.0, 0.3),       # k_max = 64
]


@pytest.mark.parametrize("case", CASES, ids=[f"seed{c[0]}_V{c[3]}_{c[4]}" for c in CASES])
def test_onehot_random_batches(sv, oracle_lib, case):
    seed, B, k, V, dt, varlen, tie, gf = case
    w = W.random_batch(seed, B=B, k_max=k, V=V, dtype=dt, varlen=varlen, tie_step=tie, greedy_frac=gf)
    argmax_drafts(w, 0.8, seed)
    s, g, o = full_compare(oracle_lib, w)
    if V > 1:
        assert (o["accept_len"] > 0).any()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_onehot_per_row_selection(sv, oracle_lib, dtype):
    """One-hot drafts in a batch of more rows than the select kernel holds at once (per-row
    selection; no residual job can arise, so every worker but the first leaves at once)."""
    w = W.random_batch(47, B=700, k_max=3, V=2048, dtype=dtype, varlen=True, greedy_frac=0.3)
    assert w.total_rows > 1368
    argmax_drafts(w, 0.8, 47)
    s, g, o = full_compare(oracle_lib, w)
    assert (o["accept_len"] > 0).any()


def test_onehot_filters_and_fallbacks(sv, oracle_lib):
    """Every kept-set path draws on every row: candidate lists (top-k), radix select (large
    top-k, top-p only), no filter (segment sums), and an all-equal row that overflows the
    candidate buffer."""
    w = W.random_batch(47, B=30, k_max=4, V=9000, dtype="bf16", greedy_frac=0.0, penalties=True)
    w.top_k[:] = np.array([40, 3000, 0, 0, 1, 600] * 5, np.int32)
    w.top_p[:] = np.array([1.0, 0.7, 0.9, 1.0, 1.0, 0.95] * 5, np.float32)
    flat = W.f32_to_bf16_bits(np.full(w.V, 0.5, np.float32))
    w.target_logits[w.row_start(29):w.row_start(29) + 5] = flat
    argmax_drafts(w, 0.7, 47)
    full_compare(oracle_lib, w)


def test_onehot_reads_no_q_and_no_accept_slot(sv, oracle_lib):
    """The entry point takes no draft_probs; slot 0 of the uniforms is neither read nor checked
    (out-of-range values there change nothing), while slot 1 still is."""
    w = W.random_batch(48, B=20, k_max=5, V=5000, dtype="bf16", greedy_frac=0.3)
    argmax_drafts(w, 0.8, 48)
    g0, _ = run_onehot(w)
    w.uniforms[:, 0] = 3.0
    g1, db = run_onehot(w)
    np.testing.assert_array_equal(g1["accept_len"], g0["accept_len"])
    np.testing.assert_array_equal(g1["out_tokens"], g0["out_tokens"])
    code, bad = sv.sv_read_device_error(db.workspace)
    assert code == 0
    b = int(np.argmin(w.greedy))
    w.uniforms[w.row_start(b), 1] = 1.0
    g2, db = run_onehot(w)
    code, bad = sv.sv_read_device_error(db.workspace)
    assert code == 5 and bad == b
    assert g2["accept_len"][b] == -1 and (g2["out_tokens"][b] == -1).all()


def test_onehot_greedy_requests_match_accept_test_entry(sv):
    """Greedy requests give the same result through both entry points (both take the argmax
    prefix), and a sampled request with top-k = 1 (one-hot p) gives the greedy result."""
    from speculative_decoding_verification_12_gb300.batch import DeviceBatch
    w = W.random_batch(49, B=40, k_max=5, V=8000, dtype="bf16", greedy_frac=1.0)
    argmax_drafts(w, 0.7, 49)
    db = DeviceBatch.from_host(w, "cuda")
    db.run()
    ref = db.results()
    db.run(onehot=True)
    got = db.results()
    np.testing.assert_array_equal(got["accept_len"], ref["accept_len"])
    np.testing.assert_array_equal(got["out_tokens"], ref["out_tokens"])
    w.greedy[:] = 0
    w.top_k[:] = 1
    w.top_p[:] = 1.0
    db1 = DeviceBatch.from_host(w, "cuda")
    db1.run(onehot=True)
    top1 = db1.results()
    # top-k = 1 keeps every token tied for the maximum; bf16 rows of 8000 random values may
    # hold such ties, which the greedy rule breaks by lowest id -- compare untied rows only
    lg = w.logits_f32()
    for b in range(w.B):
        r0 = w.row_start(b)
        rows = lg[r0:r0 + int(w.num_drafts[b]) + 1]
        if all((r == r.max()).sum() == 1 for r in rows):
            assert top1["accept_len"][b] == ref["accept_len"][b]
            assert np.array_equal(top1["out_tokens"][b], ref["out_tokens"][b])


def test_onehot_zipf_b256_k4_v128256_full(sv, oracle_lib):
    """The 256-request bf16 workload over V = 128256 with argmax drafts, every request
    compared."""
    w = W.make("zipf")
    argmax_drafts(w, 0.75, 50)
    g, _ = run_onehot(w)
    check_invariants(w, g)
    o = oracle_lib.verify(w, threads=16, onehot=True)
    s = compare(w, g, o, check_share=True)
    print("onehot zipf", s)
    assert s["requests"] == w.B
