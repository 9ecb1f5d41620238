"""bench.py's algorithmic byte count (the numerator of the roofline figures), checked against
hand counts on small batches: every target row once, one 32-byte q sector per sampled draft,
and at a sampled rejection the residual's support of q (top-k sectors, or the whole q row plus
a re-read of the target row when nothing is filtered); the one-hot scheme reads no q."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import sv_workloads as W  # noqa: E402


def _batch():
    w = W.random_batch(5, B=4, k_max=3, V=1000, dtype="bf16", greedy_frac=0.0)
    w.greedy[:] = [0, 0, 1, 0]
    w.top_k[:] = [10, 0, 0, 2000]          # request 3: top-k >= V is no filter
    w.num_drafts[:] = [3, 3, 3, 2]
    return w


def test_accept_test_scheme_bytes():
    w = _batch()
    acc = np.array([1, 3, 0, 0], np.int32)  # requests 0 and 3 rejected; request 2 is greedy
    nb = bench.algorithmic_bytes(w, acc)
    rows = (3 + 1) * 3 + (2 + 1)
    assert nb["rows"] == rows * 1000 * 2
    assert nb["q_sectors"] == (3 + 3 + 2) * 32                  # sampled drafts only
    assert nb["rejected"] == 10 * 32 + (1000 * 2 + 1000 * 4)    # top-k list; unfiltered row
    assert nb["total"] == nb["rows"] + nb["q_sectors"] + nb["rejected"] + nb["io"]


def test_one_hot_scheme_reads_no_q():
    w = _batch()
    acc = np.array([1, 3, 0, 0], np.int32)
    nb = bench.algorithmic_bytes(w, acc, onehot=True)
    assert nb["q_sectors"] == 0 and nb["rejected"] == 0
    assert nb["total"] == nb["rows"] + nb["io"]


def test_invalid_requests_add_no_rejection_bytes():
    w = _batch()
    nb = bench.algorithmic_bytes(w, np.array([-1, -1, -1, -1], np.int32))
    assert nb["rejected"] == 0
