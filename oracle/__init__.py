"""ctypes loader for the float64 verification oracle (oracle/sv_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, by __graft_entry__.smoke() and by the
benchmark's CPU-baseline leg.  The CUDA library and its binding never import this.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sv_oracle.c")
_LIB = os.path.join(_HERE, "libsvoracle.so")

ERR_LAYOUT, ERR_TOKEN, ERR_TEMP, ERR_TOPP, ERR_UNIFORM, ERR_PENALTY = 1, 2, 3, 4, 5, 6
ERR_HISTORY = 8


def build(force: bool = False) -> str:
    """Compile the oracle with plain IEEE double arithmetic (no fused multiply-add)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Batch(C.Structure):
    _fields_ = [("B", C.c_int32), ("k_max", C.c_int32), ("V", C.c_int32), ("total_rows", C.c_int32),
                ("logits_bf16", C.c_int32),
                ("target_logits", C.c_void_p), ("draft_probs", C.c_void_p), ("draft_tokens", C.c_void_p),
                ("num_drafts", C.c_void_p), ("row_offsets", C.c_void_p), ("temperature", C.c_void_p),
                ("top_k", C.c_void_p), ("top_p", C.c_void_p), ("presence", C.c_void_p),
                ("frequency", C.c_void_p), ("greedy", C.c_void_p), ("uniforms", C.c_void_p),
                ("prior_offsets", C.c_void_p), ("prior_tokens", C.c_void_p), ("prior_counts", C.c_void_p),
                ("prior_len", C.c_int32)]


DIAG_FIELDS = ("decisions", "near_ties", "error", "near_accept", "near_cdf", "near_filter", "near_argmax",
               "near_w", "near_rows_lo", "near_rows_hi", "near_final")


class _Diag(C.Structure):
    _fields_ = [(f, C.c_int32) for f in DIAG_FIELDS]


_lib = None


def load(path: str):
    """Load a compiled oracle shared object and declare its entry points."""
    l = C.CDLL(path)
    l.sv_oracle_verify.restype = C.c_int
    l.sv_oracle_verify.argtypes = [C.POINTER(_Batch), C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                   C.c_void_p, C.c_void_p, C.c_void_p]
    l.sv_oracle_verify_onehot.restype = C.c_int
    l.sv_oracle_verify_onehot.argtypes = l.sv_oracle_verify.argtypes
    l.sv_oracle_row_probs.restype = C.c_int32
    l.sv_oracle_row_probs.argtypes = [C.POINTER(_Batch), C.c_int32, C.c_int32, C.c_void_p]
    l.sv_oracle_residual.restype = C.c_int32
    l.sv_oracle_residual.argtypes = [C.POINTER(_Batch), C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]
    l.sv_oracle_rollback.restype = C.c_int32
    l.sv_oracle_rollback.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p]
    return l


def lib():
    global _lib
    if _lib is None:
        _lib = load(build())
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


class _Held:
    """Keeps contiguous copies of a workload's arrays alive while the C side reads them."""

    def __init__(self, w):
        c = np.ascontiguousarray
        self.arrays = dict(
            tl=c(w.target_logits), dp=c(w.draft_probs, dtype=np.float32), dt=c(w.draft_tokens, dtype=np.int32),
            nd=c(w.num_drafts, dtype=np.int32),
            ro=None if w.row_offsets is None else c(w.row_offsets, dtype=np.int32),
            T=c(w.temperature, dtype=np.float32), tk=c(w.top_k, dtype=np.int32), tp=c(w.top_p, dtype=np.float32),
            pr=None if w.presence is None else c(w.presence, dtype=np.float32),
            fr=None if w.frequency is None else c(w.frequency, dtype=np.float32),
            g=c(w.greedy, dtype=np.uint8), u=c(w.uniforms, dtype=np.float32),
            ho=None if getattr(w, "prior_offsets", None) is None else c(w.prior_offsets, dtype=np.int32),
            ht=None if getattr(w, "prior_offsets", None) is None else c(w.prior_tokens, dtype=np.int32),
            hc=None if getattr(w, "prior_offsets", None) is None else c(w.prior_counts, dtype=np.int32))
        a = self.arrays
        if w.dtype == "bf16":
            assert a["tl"].dtype == np.uint16
        else:
            assert a["tl"].dtype == np.float32
        self.batch = _Batch(w.B, w.k_max, w.V, w.total_rows, 1 if w.dtype == "bf16" else 0,
                            _ptr(a["tl"]), _ptr(a["dp"]), _ptr(a["dt"]), _ptr(a["nd"]), _ptr(a["ro"]),
                            _ptr(a["T"]), _ptr(a["tk"]), _ptr(a["tp"]), _ptr(a["pr"]), _ptr(a["fr"]),
                            _ptr(a["g"]), _ptr(a["u"]), _ptr(a["ho"]), _ptr(a["ht"]), _ptr(a["hc"]),
                            0 if a["ht"] is None else int(a["ht"].shape[0]))


def verify(w, requests: Optional[Sequence[int]] = None, threads: int = 1, onehot: bool = False):
    """Run the oracle on a workload (all requests or a subset); returns a dict of arrays.

    out_tokens [B, k_max+1] int32 (-1 padded), accept_len [B] int32, pq [D, 2] float64
    (p(x_i), q(x_i); NaN for greedy requests), pq_near [D] uint8 (p(x_i) sits on a near-tie
    of the row's kept set), decisions / near_ties / error [B] int32 and the near-ties by
    kind; near_rows [B] uint64 (bit i: row i's decision whether to keep draft i is a
    near-tie) and near_final [B] int32 (the final token's draw or argmax is one).  Requests
    not in `requests` are left at -1 / NaN.

    onehot=True runs the one-hot-draft scheme: every row is sampled with its draw uniform
    and the drafts are accepted while they match those samples; draft_probs is not read and
    pq's second column is 1.
    """
    h = _Held(w)
    B, D = w.B, w.total_drafts
    out = np.full((B, w.k_max + 1), -1, np.int32)
    acc = np.full(B, -1, np.int32)
    pq = np.full((max(D, 1), 2), np.nan, np.float64)
    near = np.zeros(max(D, 1), np.uint8)
    diag = (_Diag * max(B, 1))()
    l = lib()
    if requests is None:
        ranges = []
        n = max(1, threads)
        step = max(1, -(-B // (n * 4)))
        ranges = [(lo, min(B, lo + step)) for lo in range(0, B, step)]
    else:
        ranges = [(int(b), int(b) + 1) for b in requests]

    fn = l.sv_oracle_verify_onehot if onehot else l.sv_oracle_verify

    def run(rg):
        rc = fn(C.byref(h.batch), rg[0], rg[1], out.ctypes.data, acc.ctypes.data,
                                pq.ctypes.data, near.ctypes.data, diag)
        if rc != 0:
            raise RuntimeError(f"oracle failed rc={rc}")

    if threads > 1 and len(ranges) > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(run, ranges))
    else:
        for rg in ranges:
            run(rg)
    dg = np.frombuffer(diag, dtype=np.int32).reshape(-1, len(DIAG_FIELDS))[:B]
    res = dict(out_tokens=out, accept_len=acc, pq=pq[:D], pq_near=near[:D])
    for j, f in enumerate(DIAG_FIELDS):
        res[f] = dg[:, j].copy()
    # bit i: the decision of row i whether to keep draft i is a near-tie
    res["near_rows"] = (res.pop("near_rows_lo").view(np.uint32).astype(np.uint64)
                        | (res.pop("near_rows_hi").view(np.uint32).astype(np.uint64) << np.uint64(32)))
    return res


def row_probs(w, b: int, i: int) -> np.ndarray:
    """The distribution row i of request b is sampled from (float64, length V)."""
    h = _Held(w)
    p = np.zeros(w.V, np.float64)
    rc = lib().sv_oracle_row_probs(C.byref(h.batch), b, i, p.ctypes.data)
    if rc < 0:
        raise ValueError(f"row_probs({b}, {i}) rc={rc}")
    return p


def residual(w, b: int, i: int):
    """(normalised residual max(0, p - q)/W at draft row i of request b, W)."""
    h = _Held(w)
    r = np.zeros(w.V, np.float64)
    W = C.c_double(0.0)
    rc = lib().sv_oracle_residual(C.byref(h.batch), b, i, r.ctypes.data, C.byref(W))
    if rc < 0:
        raise ValueError(f"residual({b}, {i}) rc={rc}")
    return r, W.value


def rollback(kv_seq_len, accept_len, num_drafts):
    """Committed KV length per request (and the error count): L - (k+1) + 1 + a."""
    L = np.ascontiguousarray(kv_seq_len, dtype=np.int32)
    a = np.ascontiguousarray(accept_len, dtype=np.int32)
    k = np.ascontiguousarray(num_drafts, dtype=np.int32)
    out = np.zeros_like(L)
    n = lib().sv_oracle_rollback(L.ctypes.data, a.ctypes.data, k.ctypes.data, L.shape[0], out.ctypes.data)
    return out, int(n)
