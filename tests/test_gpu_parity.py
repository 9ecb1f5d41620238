"""CUDA path vs the float64 oracle, element by element, through the C ABI.

Every request of every batch is compared, the workloads at their measured sizes included.
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
    sv.lib()    # fails loudly when the library was not built
    return sv


def run_gpu(w, want_pq=True):
    from speculative_decoding_verification_12_gb300.batch import DeviceBatch
    db = DeviceBatch.from_host(w, "cuda", want_pq=want_pq)
    db.run()
    return db.results(), db


def full_compare(oracle_lib, w, check_share=False):
    g, db = run_gpu(w)
    o = oracle_lib.verify(w, threads=8)
    check_invariants_valid(w, g, o)
    return compare(w, g, o, check_share=check_share), g, o, db


def check_invariants_valid(w, g, o):
    ok = np.nonzero(o["error"] == 0)[0]
    sub = w
    for b in ok:
        a = int(g["accept_len"][b])
        assert 0 <= a <= int(w.num_drafts[b])


# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "tiny_greedy"])
def test_tiny_case(sv, oracle_lib, name):
    w = W.make(name)
    s, g, o, _ = full_compare(oracle_lib, w)
    assert s["requests"] == 1


RANDOM_CASES = [
    # seed, B, k_max, V, dtype, varlen, tie_step, greedy_frac
    (0, 16, 4, 1000, "f32", False, 0.0, 0.3),
    (1, 24, 6, 4099, "bf16", True, 0.0, 0.3),     # odd V: unaligned rows, ragged tail segment
    (2, 20, 8, 3000, "bf16", False, 0.5, 0.2),    # forced ties at top-k / top-p boundaries
    (3, 12, 3, 255, "f32", True, 0.0, 0.5),       # less than one segment
    (4, 8, 5, 1, "f32", False, 0.0, 0.5),         # V = 1
    (5, 10, 2, 7, "bf16", True, 0.25, 0.3),
    (6, 32, 8, 20001, "bf16", True, 0.0, 0.3),
    (7, 16, 7, 65536, "f32", False, 0.125, 0.25),
    (8, 40, 1, 513, "bf16", False, 0.0, 0.0),
    (9, 6, 64, 300, "f32", True, 0.0, 0.3),      # k_max = 64
]


@pytest.mark.parametrize("case", RANDOM_CASES, ids=[f"seed{c[0]}_V{c[3]}_{c[4]}" for c in RANDOM_CASES])
def test_random_batches(sv, oracle_lib, case):
    seed, B, k, V, dt, varlen, tie, gf = case
    w = W.random_batch(seed, B=B, k_max=k, V=V, dtype=dt, varlen=varlen, tie_step=tie, greedy_frac=gf)
    full_compare(oracle_lib, w)


def test_large_top_k_and_top_p_only_paths(sv, oracle_lib):
    """top-k above the candidate cap and top-p without top-k take the radix-select path."""
    w = W.random_batch(21, B=24, k_max=4, V=9000, dtype="bf16", greedy_frac=0.0)
    w.top_k[:12] = 3000
    w.top_p[:12] = 0.7
    w.top_k[12:] = 0
    w.top_p[12:] = np.linspace(0.05, 0.99, 12).astype(np.float32)
    full_compare(oracle_lib, w)


def test_candidate_overflow_falls_back(sv, oracle_lib):
    """All-equal rows: every token ties for the top-k set, overflowing the candidate buffer."""
    w = W.random_batch(22, B=6, k_max=3, V=5000, dtype="bf16", greedy_frac=0.0)
    w.target_logits[:] = W.f32_to_bf16_bits(np.full((w.total_rows, w.V), 0.5, np.float32))
    w.top_k[:] = 10
    w.top_p[:] = np.array([1.0, 0.5, 0.999, 1.0, 0.1, 0.9], np.float32)
    full_compare(oracle_lib, w)


@pytest.mark.parametrize("B", [6, 400])
def test_overflow_residuals_with_list_rows_only(sv, oracle_lib, B):
    """Every sampled row asks for a small top-k, so the stream kernel counts no row whose kept
    set is built otherwise than as a candidate list, and all residual workers but the first
    leave at once; all-equal rows overflow the candidate buffer all the same, and their
    rejections queue whole-row residual jobs that the one remaining worker must draw.  B=400
    (1600 rows) takes per-row selection, B=6 whole-grid selection."""
    w = W.random_batch(24, B=B, k_max=3, V=2048, dtype="bf16", greedy_frac=0.25)
    w.target_logits[:] = W.f32_to_bf16_bits(np.full((w.total_rows, w.V), 0.25, np.float32))
    w.top_k[:] = 12
    w.top_p[:] = 1.0
    s, g, o, _ = full_compare(oracle_lib, w)
    sampled = ~w.greedy.astype(bool)
    # rejections happened among sampled requests (so residual jobs were drawn)
    assert ((g["accept_len"] < w.num_drafts) & sampled).any()


def test_zero_drafts_and_padding_rows(sv, oracle_lib):
    w = W.random_batch(23, B=30, k_max=5, V=2000, dtype="bf16", greedy_frac=0.3)
    w.num_drafts[::3] = 0          # uniform layout with unused (padding) rows
    w.num_drafts[1::3] = 2
    full_compare(oracle_lib, w)


def test_empty_requests_in_ragged_layout(sv, oracle_lib):
    """Requests that own no rows in row_offsets get -1 and a layout error, the others verify."""
    w = W.random_batch(71, B=12, k_max=4, V=3000, dtype="bf16", varlen=True, greedy_frac=0.3)
    ro = w.row_offsets.copy()
    ro[6] = ro[5]                  # request 5 owns no rows: its rows go to the front of request 6
    w.row_offsets = ro
    w.num_drafts[6] = min(w.k_max, int(ro[7] - ro[6]) - 1)
    # request 6's draft rows now start one slot early, on the last draft slot of the requests
    # before it: those leave that slot unused
    for b in range(5):
        w.num_drafts[b] = min(int(w.num_drafts[b]), max(0, int(ro[6]) - 6 - (int(ro[b]) - b)))
    s, g, o, db = full_compare(oracle_lib, w)
    assert g["accept_len"][5] == -1 and (g["out_tokens"][5] == -1).all() and o["error"][5] == 1
    assert sv.sv_read_device_error(db.workspace)[0] == 1


@pytest.mark.parametrize("pattern", ["all_sampled", "all_greedy", "alternate", "greedy_first_half"])
def test_streaming_order_mixes(sv, oracle_lib, pattern):
    """With more rows than the select kernel holds at once (about 1600 here, against 9 per SM on
    152 SMs), sampled requests stream first and greedy ones last, and each row is selected once its
    own statistics are complete: every mix of the two (none, all, interleaved, in blocks), over
    more requests than one block of the order builder takes at a time, ragged and uniform."""
    for varlen in (True, False):
        w = W.random_batch(80, B=700 if varlen else 400, k_max=3, V=2048, dtype="bf16", varlen=varlen,
                           greedy_frac=0.0)
        assert w.total_rows > 1368
        idx = np.arange(w.B)
        w.greedy[:] = {"all_sampled": 0 * idx, "all_greedy": 0 * idx + 1, "alternate": idx % 2,
                       "greedy_first_half": (idx < w.B // 2)}[pattern].astype(np.uint8)
        full_compare(oracle_lib, w)


@pytest.mark.parametrize("mode", ["u_zero", "u_top", "t_small", "t_large"])
def test_extreme_uniforms_and_temperatures(sv, oracle_lib, mode):
    """Uniforms at both ends of [0, 1) (u = 0 keeps every draft with p > 0 and draws the first
    token of positive weight; u just below 1 draws from the top of the CDF) and temperatures of
    1e-3 (nearly one-hot rows) and 50 (nearly flat rows)."""
    w = W.random_batch(31, B=24, k_max=4, V=5000, dtype="bf16", varlen=True, greedy_frac=0.2)
    if mode == "u_zero":
        w.uniforms[:] = 0.0
    elif mode == "u_top":
        w.uniforms[:] = np.nextafter(np.float32(1), np.float32(0))
    elif mode == "t_small":
        w.temperature[:] = np.float32(1e-3)
    else:
        w.temperature[:] = np.float32(50.0)
    full_compare(oracle_lib, w)


def test_q_equals_p_and_disjoint_supports(sv, oracle_lib):
    V, k, B = 64, 4, 40
    g = np.random.default_rng(5)
    logits = np.zeros((k + 1, V), np.float32)
    q = np.full((k, V), 1.0 / V, np.float32)
    w = W.from_rows(V, logits, q, g.integers(0, V, (B, k)).astype(np.int32),
                    g.random((B, k + 1, 2), dtype=np.float32))
    s, gg, o, _ = full_compare(oracle_lib, w)
    assert (gg["accept_len"] == k).all()
    z = np.full(V, -30.0, np.float32)
    z[:2] = [5.0, 4.0]
    qd = np.zeros(V, np.float32)
    qd[2:] = 1.0 / (V - 2)
    w = W.from_rows(V, np.tile(z, (k + 1, 1)), np.tile(qd, (k, 1)), g.integers(2, V, (B, k)).astype(np.int32),
                    g.random((B, k + 1, 2), dtype=np.float32), top_k=2)
    s, gg, o, _ = full_compare(oracle_lib, w)
    assert (gg["accept_len"] == 0).all()


def test_device_data_errors(sv, oracle_lib):
    w = W.random_batch(24, B=10, k_max=3, V=500, dtype="f32", greedy_frac=0.0)
    w.draft_tokens[1] = 500
    w.temperature[1] = -1.0
    w.top_p[2] = 0.0
    w.uniforms[3 * 4 + 2, 1] = 1.0
    w.num_drafts[4] = 9
    s, g, o, db = full_compare(oracle_lib, w)
    code, bad = sv.sv_read_device_error(db.workspace)
    assert code != 0 and bad == 0
    assert (g["accept_len"][:5] == -1).all() and (g["accept_len"][5:] >= 0).all()


def test_device_data_errors_per_row_selection(sv, oracle_lib):
    """The same device-data errors, and a request that owns no rows, in a batch of more rows
    than the select kernel holds at once (per-row selection, streamed in the built order)."""
    w = W.random_batch(26, B=700, k_max=3, V=2048, dtype="bf16", varlen=True, greedy_frac=0.3)
    assert w.total_rows > 1368
    d1 = w.draft_start(1)
    if w.num_drafts[1] == 0:
        w.num_drafts[1] = 1
    w.draft_tokens[d1] = 2048                 # a draft outside the vocabulary
    w.temperature[2] = -1.0
    w.greedy[2] = 0
    w.top_p[3] = 0.0
    w.greedy[3] = 0
    w.num_drafts[4] = 9                       # beyond k_max
    ro = w.row_offsets.copy()
    ro[301] = ro[300]                         # request 300 owns no rows: request 301 takes them
    w.row_offsets = ro
    w.num_drafts[301] = min(w.k_max, int(ro[302] - ro[301]) - 1)
    for b in range(300):                      # (the draft slot request 301 now starts on)
        w.num_drafts[b] = min(int(w.num_drafts[b]), max(0, int(ro[301]) - 301 - (int(ro[b]) - b)))
    s, g, o, db = full_compare(oracle_lib, w)
    code, bad = sv.sv_read_device_error(db.workspace)
    assert code != 0
    assert g["accept_len"][300] == -1 and o["error"][300] != 0
    assert (g["accept_len"][[2, 3, 4]] == -1).all()


def test_deterministic_repeat(sv):
    w = W.random_batch(25, B=40, k_max=6, V=30000, dtype="bf16", varlen=True)
    g1, db = run_gpu(w)
    db.run()
    g2 = db.results()
    for key in g1:
        assert np.array_equal(g1[key], g2[key], equal_nan=True), key


@pytest.mark.parametrize("rows", ["one_wave", "many_rows"])
def test_back_to_back_calls_share_a_workspace(sv, rows):
    """Calls queued back to back on one stream, sharing one workspace, with no synchronisation
    between them: one-pass, lazy, one-pass, one-pass again.  Each gives what it gives alone: a
    call's clearing kernel waits for the call before it, and its stream kernel for the clearing
    kernel, whether that kernel lets it in before or after its own wait (per-row selection
    above 9 rows per SM, whole-grid selection below; the lazy call's clear always after)."""
    from speculative_decoding_verification_12_gb300.batch import DeviceBatch
    B = 60 if rows == "one_wave" else 400
    ws = [W.random_batch(90 + i, B=B, k_max=4, V=4096, dtype="bf16", varlen=False, greedy_frac=0.3)
          for i in range(3)]
    assert (ws[0].total_rows > 9 * 152) == (rows == "many_rows")
    dbs = [DeviceBatch.from_host(w, "cuda") for w in ws]
    solo = []
    for j, db in enumerate(dbs):
        db.run(lazy=(j == 1))
        solo.append(db.results())
    shared = dbs[0].workspace
    for db in dbs:
        db.workspace = shared
        db.out_tokens.fill_(-7)
        db.accept_len.fill_(-7)
        db.out_pq.fill_(-7.0)
    dbs[0].run()
    dbs[1].run(lazy=True)
    dbs[2].run()
    dbs[0].run()
    for j, db in enumerate(dbs):
        got = db.results()
        for key in solo[j]:
            assert np.array_equal(got[key], solo[j][key], equal_nan=True), (j, key)


def test_unaligned_pointers(sv, oracle_lib):
    """Logit and draft rows that start off a 16-byte boundary take the scalar-load path."""
    from speculative_decoding_verification_12_gb300.batch import DeviceBatch
    w = W.random_batch(26, B=8, k_max=3, V=1024, dtype="bf16", greedy_frac=0.2)
    db = DeviceBatch.from_host(w, "cuda")
    tl = torch.empty(db.target_logits.numel() + 1, dtype=torch.bfloat16, device="cuda")
    tl[1:] = db.target_logits.reshape(-1)
    dp = torch.empty(db.draft_probs.numel() + 1, dtype=torch.float32, device="cuda")
    dp[1:] = db.draft_probs.reshape(-1)
    db.run(target_logits=tl[1:].view(w.total_rows, w.V), draft_probs=dp[1:].view(-1, w.V))
    g = db.results()
    compare(w, g, oracle_lib.verify(w))


def test_rollback_matches_closed_form(sv, oracle_lib):
    g = np.random.default_rng(3)
    B = 1000
    k = g.integers(0, 9, B).astype(np.int32)
    a = np.minimum(g.integers(0, 9, B), k).astype(np.int32)
    L = g.integers(10, 5000, B).astype(np.int32)
    a[5] = k[5] + 1          # accept_len beyond k: rejected, length kept
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    kv = torch.from_numpy(L).cuda()
    sv.spec_rollback(kv, torch.from_numpy(a).cuda(), torch.from_numpy(k).cuda(), ws)
    ref, nerr = oracle_lib.rollback(L, a, k)
    got = kv.cpu().numpy()
    ok = ref >= 0
    assert np.array_equal(got[ok], ref[ok]) and got[5] == L[5] and nerr == 1
    assert sv.sv_read_device_error(ws)[0] == 1


def test_rollback_of_draft_cache_lengths(sv, oracle_lib):
    """spec_rollback on the draft cache's lengths (k drafts appended, accepted ones kept)."""
    import json
    import os
    here = os.path.dirname(os.path.abspath(__file__))
    cs = json.load(open(os.path.join(here, "golden", "worked_examples.json")))["rollback_draft"]["cases"]
    L = np.array([c["current_len"] for c in cs], np.int32)
    k = np.array([c["k"] for c in cs], np.int32)
    a = np.array([c["accepted"] for c in cs], np.int32)
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    kv = torch.from_numpy(L).cuda()
    sv.spec_rollback(kv, torch.from_numpy(a).cuda(), torch.from_numpy(k).cuda(), ws)
    assert list(kv.cpu().numpy()) == [c["committed"] for c in cs]


# ------------------------------------------------------------------------------------------
# the measured workloads at full size, every request against the oracle
# ------------------------------------------------------------------------------------------

def _full_workload(oracle_lib, name):
    w = W.make(name)
    g, _ = run_gpu(w)
    check_invariants(w, g)
    o = oracle_lib.verify(w, threads=16)
    s = compare(w, g, o, check_share=True)
    print(name, s)
    assert s["requests"] == w.B
    return s, g, w


def test_peaks_b64_k5_v32000_full(sv, oracle_lib):
    s, g, w = _full_workload(oracle_lib, "peaks")
    acc = g["accept_len"].mean() / 5
    assert 0.2 < acc < 1.0


def test_zipf_b256_k4_v128256_full(sv, oracle_lib):
    _full_workload(oracle_lib, "zipf")


def test_ragged_b512_v151936_full(sv, oracle_lib):
    _full_workload(oracle_lib, "ragged")


def test_stream_b1024_k7_v128256_full(sv, oracle_lib):
    _full_workload(oracle_lib, "stream")


def test_max_vocabulary(sv, oracle_lib):
    """V = 2^21 (the largest supported): 8192 segments per row, beyond the select kernel's
    one-pass bound (1024 segments), so top-k rows take the general radix bound; the select
    kernel then holds 168 KB of statistics and scratch per row."""
    w = W.random_batch(27, B=3, k_max=2, V=1 << 21, dtype="bf16", greedy_frac=0.3, penalties=True)
    w.top_k[:] = [0, 40, 3000]
    w.top_p[:] = [1.0, 0.9, 0.5]
    full_compare(oracle_lib, w)


def test_many_rows_few_ctas(sv, oracle_lib):
    """More rows than resident CTAs with mixed greedy / sampled / ragged requests: rows are
    claimed dynamically and requests finalised by whichever CTA completes them."""
    w = W.random_batch(28, B=300, k_max=8, V=4096, dtype="bf16", varlen=True, greedy_frac=0.3)
    full_compare(oracle_lib, w)


def test_phase_events_time_the_stream_kernel(sv):
    """sv_set_phase_events: the library records the caller's two events around the stream
    kernel; the interval is positive and shorter than the whole call, and results match a call
    made without the events."""
    from speculative_decoding_verification_12_gb300.batch import DeviceBatch
    w = W.random_batch(11, B=32, k_max=4, V=20000, dtype="bf16", varlen=False, greedy_frac=0.3)
    db = DeviceBatch.from_host(w, "cuda", want_pq=True)
    db.run()
    torch.cuda.synchronize()
    ref = (db.out_tokens.cpu().numpy().copy(), db.accept_len.cpu().numpy().copy())
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    b.record()
    torch.cuda.synchronize()
    assert sv.lib().sv_set_phase_events(a.cuda_event, b.cuda_event) == sv.SV_OK
    try:
        c0.record()
        db.run()
        c1.record()
    finally:
        sv.lib().sv_set_phase_events(None, None)
    torch.cuda.synchronize()
    stream_ms, call_ms = a.elapsed_time(b), c0.elapsed_time(c1)
    assert 0.0 < stream_ms <= call_ms
    np.testing.assert_array_equal(db.out_tokens.cpu().numpy(), ref[0])
    np.testing.assert_array_equal(db.accept_len.cpu().numpy(), ref[1])
