"""Penalties with a prior history (params.prior_*): the CUDA path against the float64 oracle,
element by element, through the C ABI -- both entry points, every kept-set path, long
histories and malformed ones.
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


def run(w, onehot=False):
    from speculative_decoding_verification_12_gb300.batch import DeviceBatch
    db = DeviceBatch.from_host(w, "cuda", want_pq=True)
    db.run(onehot=onehot)
    return db.results(), db


def full_compare(oracle_lib, w, onehot=False):
    g, db = run(w, onehot)
    o = oracle_lib.verify(w, threads=8, onehot=onehot)
    return compare(w, g, o), g, o, db


CASES = [
    # seed, B, k_max, V, dtype, varlen, tie_step, greedy_frac, history length
    (70, 16, 4, 1000, "f32", False, 0.0, 0.3, 40),
    (71, 24, 6, 4099, "bf16", True, 0.0, 0.3, 200),     # odd V: the one-kernel path
    (72, 20, 8, 3000, "bf16", False, 0.5, 0.3, 100),    # ties
    (73, 32, 8, 20001, "bf16", True, 0.0, 0.3, 2000),   # histories longer than a segment's worth
    (74, 16, 7, 65536, "f32", False, 0.125, 0.25, 500),
    (75, 6, 64, 300, "f32", True, 0.0, 0.3, 300),       # k_max = 64, history covering the row
    (76, 12, 3, 7, "bf16", True, 0.25, 0.3, 7),         # V = 7
]


@pytest.mark.parametrize("case", CASES, ids=[f"seed{c[0]}_V{c[3]}_{c[4]}_H{c[8]}" for c in CASES])
def test_history_random_batches(sv, oracle_lib, case):
    seed, B, k, V, dt, varlen, tie, gf, H = case
    w = W.random_batch(seed, B=B, k_max=k, V=V, dtype=dt, varlen=varlen, tie_step=tie, greedy_frac=gf)
    w.presence[::2] = np.maximum(w.presence[::2], 0.4)      # most requests penalised
    W.with_history(w, seed, H)
    s, g, o, _ = full_compare(oracle_lib, w)
    assert s["requests"] >= B - 1


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_history_per_row_selection(sv, oracle_lib, dtype):
    """Prior histories in a batch of more rows than the select kernel holds at once (1711 rows
    against 9 per SM on 152 SMs): the history instance of the stream kernel in the per-row
    scheme, rows streamed in the built order."""
    w = W.random_batch(79, B=700, k_max=3, V=2048, dtype=dtype, varlen=True, greedy_frac=0.3)
    assert w.total_rows > 1368
    w.presence[::2] = np.maximum(w.presence[::2], 0.4)
    W.with_history(w, 79, 300)
    s, g, o, _ = full_compare(oracle_lib, w)
    assert s["requests"] >= w.B - 2


def test_history_filters_and_onehot(sv, oracle_lib):
    """Candidate lists, radix select, no filter and greedy rows with a history; then the same
    batch through the one-hot entry point."""
    w = W.random_batch(77, B=30, k_max=4, V=9000, dtype="bf16", greedy_frac=0.2)
    w.top_k[:] = np.array([40, 3000, 0, 0, 1, 600] * 5, np.int32)
    w.top_p[:] = np.array([1.0, 0.7, 0.9, 1.0, 1.0, 0.95] * 5, np.float32)
    w.presence[:] = 0.7
    w.frequency[:] = 0.35
    W.with_history(w, 77, 400, top_share=0.8)
    full_compare(oracle_lib, w)
    lg = w.logits_f32()
    for b in range(w.B):        # argmax proposals for the one-hot scheme
        r0, d0 = w.row_start(b), w.draft_start(b)
        for i in range(int(w.num_drafts[b])):
            w.draft_tokens[d0 + i] = int(np.argmax(lg[r0 + i]))
    full_compare(oracle_lib, w, onehot=True)


def test_history_without_penalties_changes_nothing(sv):
    """With presence = frequency = 0 the history is checked but changes no result."""
    w = W.random_batch(78, B=24, k_max=5, V=5000, dtype="bf16", greedy_frac=0.3)
    w.presence[:] = 0.0
    w.frequency[:] = 0.0
    g0, _ = run(w)
    W.with_history(w, 78, 300)
    g1, db = run(w)
    np.testing.assert_array_equal(g1["accept_len"], g0["accept_len"])
    np.testing.assert_array_equal(g1["out_tokens"], g0["out_tokens"])
    assert sv.sv_read_device_error(db.workspace)[0] == 0


def test_history_errors(sv, oracle_lib):
    """A malformed history fails its own request only (code 8, outputs -1); an offset past
    prior_len is caught before any entry is read."""
    w = W.random_batch(79, B=8, k_max=3, V=50, greedy_frac=0.0)
    w.presence[:] = 0.5
    w.prior_offsets = np.array([0, 3, 6, 9, 12, 15, 18, 21, 24], np.int32)
    w.prior_tokens = np.tile(np.array([3, 9, 20], np.int32), 8)
    w.prior_counts = np.ones(24, np.int32)
    w.prior_tokens[0:3] = [9, 3, 20]       # request 0: not ascending
    w.prior_tokens[3:6] = [3, 3, 20]       # request 1: a repeat
    w.prior_tokens[6:9] = [3, 9, 50]       # request 2: out of range
    w.prior_counts[10] = 0                 # request 3: count below one
    s, g, o, db = full_compare(oracle_lib, w)
    assert list(o["error"]) == [8, 8, 8, 8, 0, 0, 0, 0]
    assert (g["accept_len"][:4] == -1).all() and (g["accept_len"][4:] >= 0).all()
    assert sv.sv_read_device_error(db.workspace) == (8, 0)
    w.prior_offsets[8] = 30                # request 7 ends past the 24 entries
    s, g, o, db = full_compare(oracle_lib, w)
    assert o["error"][7] == 8 and g["accept_len"][7] == -1 and g["accept_len"][6] >= 0


def test_history_zipf_b256_k4_v128256_full(sv, oracle_lib):
    """The 256-request bf16 workload over V = 128256 with presence/frequency penalties and
    histories of up to 1000 tokens (most segments then hold a history token), every request
    compared."""
    w = W.make("zipf")
    g0 = np.random.default_rng(80)
    w.presence = g0.uniform(0.2, 1.0, w.B).astype(np.float32)
    w.frequency = g0.uniform(0.0, 0.5, w.B).astype(np.float32)
    W.with_history(w, 80, 1000)
    g, _ = run(w)
    check_invariants(w, g)
    o = oracle_lib.verify(w, threads=16)
    s = compare(w, g, o, check_share=True)
    print("history zipf", s)
    assert s["requests"] == w.B
