"""Target rows with masked tokens (logits of -inf, as a constrained-decoding mask leaves them)
against the float64 oracle, element by element, through the C ABI.  A masked token has weight
exp(-inf) = 0 under every filter: it is never kept with mass, never accepted (p = 0), never
drawn.  Covers scattered and whole-segment masks, drafts on masked tokens, rows with fewer
finite tokens than top-k (the k-th largest is then -inf), both dtypes, both selection schemes
and the lazy call."""
import numpy as np
import pytest

import sv_workloads as W
from sv_parity import compare

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_12_gb300 as sv
    sv.lib()
    return sv


def run(w, lazy=False):
    from speculative_decoding_verification_12_gb300.batch import DeviceBatch
    db = DeviceBatch.from_host(w, "cuda", want_pq=True)
    db.run(lazy=lazy)
    return db.results()


def no_masked_output(w, g, m):
    for b in range(w.B):
        a = int(g["accept_len"][b])
        r0 = w.row_start(b)
        for i in range(a + 1 if a >= 0 else 0):
            t = int(g["out_tokens"][b][i])
            assert 0 <= t < w.V and not m[r0 + i, t], (b, i, t)


CASES = [
    # seed, B, k_max, V, dtype, varlen, masked share, lazy
    (1, 30, 4, 3000, "bf16", True, 0.5, False),
    (2, 20, 5, 9000, "f32", False, 0.3, False),
    (3, 16, 3, 1000, "bf16", True, 0.9, False),
    (1, 30, 4, 3000, "bf16", True, 0.5, True),
    (5, 400, 4, 2048, "bf16", False, 0.5, False),    # per-row selection (2000 rows)
    (5, 400, 4, 2048, "bf16", False, 0.5, True),
]


@pytest.mark.parametrize("case", CASES, ids=[f"seed{c[0]}_V{c[3]}_{c[4]}_{'lazy' if c[7] else 'onepass'}" for c in CASES])
def test_masked_vocabulary(sv, oracle_lib, case):
    seed, B, k, V, dt, varlen, frac, lazy = case
    w = W.random_batch(seed, B=B, k_max=k, V=V, dtype=dt, varlen=varlen, greedy_frac=0.3)
    m = W.with_masked_vocab(w, seed, frac)
    g = run(w, lazy)
    o = oracle_lib.verify(w, threads=16)
    compare(w, g, o, pq_on_path=lazy)
    no_masked_output(w, g, m)


def test_fewer_finite_tokens_than_top_k(sv, oracle_lib):
    """Three finite tokens per row and top-k 50 on half the requests: every token is at or above
    the k-th largest (-inf), so the kept set is the whole row, with mass on three tokens."""
    w = W.random_batch(4, B=12, k_max=4, V=20000, dtype="bf16", greedy_frac=0.25)
    m = W.with_masked_vocab(w, 4, 1.0)
    w.top_k[::2] = 50
    g = run(w)
    o = oracle_lib.verify(w, threads=16)
    compare(w, g, o)
    no_masked_output(w, g, m)
    assert (g["accept_len"] >= 1).any()
