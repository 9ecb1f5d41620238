"""Seeded synthetic inputs for batched speculative-decoding verification.

This module draws inputs only: target logits, the draft model's distributions q and the
draft tokens sampled from them, the accept/resample uniforms and the per-request sampling
parameters.  It holds none of the verification arithmetic; the CUDA path and the float64
oracle both consume exactly the arrays produced here.  (The draft side's softmax below
makes the draft model's *input* distribution q, as the draft proposer would; the
verification method itself takes q as given.)

Every random stream is a counter-based Philox generator keyed by (stream seed, request
index), so any single request can be regenerated on its own and a large batch can be made
in parallel chunks.  Streams per workload with base seed s = 1000*c:
  s+0  target logits            s+1  draft noise
  (s+2) ^ (1<<30)  draft-token sampling (salted, mirroring the separate draft RNG stream
                   of "Adding Speculative Decoding", Verification and sampling item 4)
  s+3  per-request scalars      key (0, b)  uniforms, fp32 U[0,1)

Layouts follow the verification call: target logits packed [R, V] (bf16 stored as uint16
bit patterns, or float32), draft probs packed [D, V] float32, draft tokens [D] int32,
uniforms [R, 2] float32, num_drafts [B] int32 and, for ragged batches, row_offsets [B+1].
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Callable, Dict, Optional, Sequence

import numpy as np

DRAFT_SALT = 1 << 30


def _rng(stream: int, b: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=np.array([stream, b], dtype=np.uint64)))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest-even), returned as uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Workload:
    """One packed batch.  Arrays are host numpy arrays in the call's layout."""
    name: str
    V: int
    k_max: int
    dtype: str                      # "bf16" (uint16 bits) or "f32"
    num_drafts: np.ndarray          # [B] int32
    row_offsets: Optional[np.ndarray]  # [B+1] int32, or None for the uniform [B, k_max+1] layout
    target_logits: np.ndarray       # [R, V] uint16 or float32
    draft_probs: np.ndarray         # [D, V] float32
    draft_tokens: np.ndarray        # [D] int32
    uniforms: np.ndarray            # [R, 2] float32
    temperature: np.ndarray         # [B] float32
    top_k: np.ndarray               # [B] int32
    top_p: np.ndarray               # [B] float32
    presence: Optional[np.ndarray]  # [B] float32 or None
    frequency: Optional[np.ndarray]  # [B] float32 or None
    greedy: np.ndarray              # [B] uint8
    # the requests' prior history for the penalties, or None: request b generated the tokens
    # prior_tokens[o_b:o_{b+1}] (distinct, ascending) prior_counts[...] times each
    prior_offsets: Optional[np.ndarray] = None   # [B+1] int32
    prior_tokens: Optional[np.ndarray] = None    # [H] int32
    prior_counts: Optional[np.ndarray] = None    # [H] int32

    @property
    def B(self) -> int:
        return int(self.num_drafts.shape[0])

    @property
    def total_rows(self) -> int:
        return int(self.target_logits.shape[0])

    @property
    def total_drafts(self) -> int:
        return int(self.draft_tokens.shape[0])

    def row_start(self, b: int) -> int:
        if self.row_offsets is None:
            return b * (self.k_max + 1)
        return int(self.row_offsets[b])

    def draft_start(self, b: int) -> int:
        return self.row_start(b) - b

    def logits_f32(self) -> np.ndarray:
        if self.dtype == "bf16":
            return bf16_bits_to_f32(self.target_logits)
        return self.target_logits

    def copy(self) -> "Workload":
        return dataclasses.replace(self, **{f.name: (getattr(self, f.name).copy()
                                                     if isinstance(getattr(self, f.name), np.ndarray)
                                                     else getattr(self, f.name))
                                            for f in dataclasses.fields(self)})


@dataclasses.dataclass
class Spec:
    """A workload recipe: per-request scalars plus a per-request row generator."""
    name: str
    seed: int
    B: int
    V: int
    k_max: int
    dtype: str
    varlen: bool
    scalars: Callable[["Spec"], Dict[str, np.ndarray]]
    target_rows: Callable[["Spec", int, int, float], tuple]  # (b, n_rows, T) -> (fp32 target, fp32 draft logits)


# --------------------------------------------------------------------------------------
# recipes (shapes and value distributions of the workloads the method is measured on)
# --------------------------------------------------------------------------------------

def _scalars_const(temperature=1.0, top_k=0, top_p=1.0, presence=None, frequency=None,
                   greedy_frac=0.0, ragged_k=None):
    def f(spec: Spec) -> Dict[str, np.ndarray]:
        B = spec.B
        r = _rng(spec.seed + 3, 0)
        if ragged_k is None:
            nd = np.full(B, spec.k_max, np.int32)
        else:
            nd = r.integers(ragged_k[0], ragged_k[1] + 1, size=B).astype(np.int32)
        if callable(temperature):
            T = temperature(r, B).astype(np.float32)
        else:
            T = np.full(B, temperature, np.float32)
        if greedy_frac == "bernoulli":
            g = (r.random(B) < 0.5).astype(np.uint8)
        elif greedy_frac > 0:
            g = np.zeros(B, np.uint8)
            g[r.permutation(B)[: int(round(greedy_frac * B))]] = 1
        else:
            g = np.zeros(B, np.uint8)
        out = dict(num_drafts=nd, temperature=T, top_k=np.full(B, top_k, np.int32),
                   top_p=np.full(B, top_p, np.float32), greedy=g)
        out["presence"] = None if presence is None else np.full(B, presence, np.float32)
        out["frequency"] = None if frequency is None else np.full(B, frequency, np.float32)
        return out
    return f


def _rows_gauss(sigma, draft_sigma, peaks=0, peak_height=0.0, independent_half=None):
    def f(spec: Spec, b: int, n: int, T: float):
        r = _rng(spec.seed + 0, b)
        x = (r.standard_normal((n, spec.V), dtype=np.float32) * np.float32(sigma))
        if peaks:
            for i in range(n):
                idx = r.choice(spec.V, size=peaks, replace=False)
                x[i, idx] += np.float32(peak_height)
        rd = _rng(spec.seed + 1, b)
        if independent_half is not None and independent_half(b):
            d = rd.standard_normal((max(n - 1, 0), spec.V), dtype=np.float32) * np.float32(sigma)
        else:
            d = x[: max(n - 1, 0)] + rd.standard_normal((max(n - 1, 0), spec.V), dtype=np.float32) * np.float32(draft_sigma)
        return x, d
    return f


def _rows_zipf(slope, noise, draft_sigma):
    def f(spec: Spec, b: int, n: int, T: float):
        r = _rng(spec.seed + 0, b)
        ranks = np.arange(1, spec.V + 1, dtype=np.float64)
        base = (-slope * np.log(ranks)).astype(np.float32)
        x = np.empty((n, spec.V), np.float32)
        for i in range(n):
            vals = base + r.standard_normal(spec.V, dtype=np.float32) * np.float32(noise)
            perm = r.permutation(spec.V)
            x[i, perm] = vals           # token perm[j] has rank j+1
        rd = _rng(spec.seed + 1, b)
        d = x[: max(n - 1, 0)] + rd.standard_normal((max(n - 1, 0), spec.V), dtype=np.float32) * np.float32(draft_sigma)
        return x, d
    return f


def _half_indep(spec_seed):
    def pick(b):
        return bool(_rng(spec_seed + 5, b).random() < 0.5)
    return pick


SPECS: Dict[str, Spec] = {}


def _add(spec: Spec):
    SPECS[spec.name] = spec


# Tiny correctness case: B=1, k=4, V=1000, fp32 N(0, 2^2); draft = target + N(0, 0.5^2); T=1.
_add(Spec("tiny_b1_k4_v1000_f32", 1000, 1, 1000, 4, "f32", False,
          _scalars_const(), _rows_gauss(2.0, 0.5)))
_add(Spec("tiny_b1_k4_v1000_f32_greedy", 1000, 1, 1000, 4, "f32", False,
          _scalars_const(greedy_frac=1.0), _rows_gauss(2.0, 0.5)))
# B=64, k=5, V=32000 bf16 N(0, 3^2) with 20 peak tokens per row raised by +8; draft noise 1.0; T=0.8.
_add(Spec("b64_k5_v32000_bf16_peaks", 2000, 64, 32000, 5, "bf16", False,
          _scalars_const(temperature=0.8), _rows_gauss(3.0, 1.0, peaks=20, peak_height=8.0)))
# B=256, k=4, V=128256 bf16 Zipf ranks (-1.1 ln r + N(0, 0.3^2)), draft noise 0.8,
# T ~ U(0.5, 1.2), top-k 50, top-p 0.9, a quarter greedy.
_add(Spec("b256_k4_v128256_bf16_zipf", 3000, 256, 128256, 4, "bf16", False,
          _scalars_const(temperature=lambda r, B: r.uniform(0.5, 1.2, size=B), top_k=50,
                         top_p=0.9, greedy_frac=0.25),
          _rows_zipf(1.1, 0.3, 0.8)))
# Ragged B=512, k ~ U{0..8}, V=151936 bf16 N(0, 2.5^2); half close drafts (noise 0.4), half
# independent N(0, 2.5^2); presence 0.5, frequency 0.3; greedy Bernoulli(0.5); T=1.
_add(Spec("ragged_b512_k0to8_v151936_bf16_pen", 4000, 512, 151936, 8, "bf16", True,
          _scalars_const(presence=0.5, frequency=0.3, greedy_frac="bernoulli", ragged_k=(0, 8)),
          _rows_gauss(2.5, 0.4, independent_half=_half_indep(4000))))
# Large streaming case: B=1024, k=7, V=128256 fp32 N(0, 2^2); draft noise 0.6; T=1, top-p 0.95.
_add(Spec("b1024_k7_v128256_f32_topp095", 5000, 1024, 128256, 7, "f32", False,
          _scalars_const(top_p=0.95), _rows_gauss(2.0, 0.6)))

# Short aliases used by tests and the bench CLI.
ALIASES = {
    "tiny": "tiny_b1_k4_v1000_f32",
    "tiny_greedy": "tiny_b1_k4_v1000_f32_greedy",
    "peaks": "b64_k5_v32000_bf16_peaks",
    "zipf": "b256_k4_v128256_bf16_zipf",
    "ragged": "ragged_b512_k0to8_v151936_bf16_pen",
    "stream": "b1024_k7_v128256_f32_topp095",
}


def spec(name: str) -> Spec:
    return SPECS[ALIASES.get(name, name)]


# --------------------------------------------------------------------------------------
# per-request generation and packing
# --------------------------------------------------------------------------------------

def _softmax_rows_f32(logits: np.ndarray, T: float) -> np.ndarray:
    """The draft model's output distribution q = softmax(draft_logits / T), stored fp32."""
    if logits.shape[0] == 0:
        return np.zeros((0, logits.shape[1]), np.float32)
    z = logits.astype(np.float64) / float(T)
    z -= z.max(axis=1, keepdims=True)
    np.exp(z, out=z)
    z /= z.sum(axis=1, keepdims=True)
    return z.astype(np.float32)


def _sample_rows(q: np.ndarray, u: np.ndarray) -> np.ndarray:
    """Draft tokens drawn from q by inverse CDF (the draft proposer's own sampling)."""
    out = np.empty(q.shape[0], np.int32)
    for i in range(q.shape[0]):
        c = np.cumsum(q[i].astype(np.float64))
        t = u[i] * c[-1]
        j = int(np.searchsorted(c, t, side="right"))
        out[i] = min(j, q.shape[1] - 1)
    return out


def _gen_request(sp: Spec, sc: Dict[str, np.ndarray], b: int, cap_rows: int):
    k = int(sc["num_drafts"][b])
    T = float(sc["temperature"][b])
    x, d = sp.target_rows(sp, b, k + 1, T)
    q = _softmax_rows_f32(d, T)
    ud = _rng((sp.seed + 2) ^ DRAFT_SALT, b).random(k)
    toks = _sample_rows(q, ud)
    uni = _rng(0, b).random((cap_rows, 2), dtype=np.float32)
    if sp.dtype == "bf16":
        tl = f32_to_bf16_bits(x)
    else:
        tl = x.astype(np.float32)
    return k, tl, q, toks, uni


def _threads(n_jobs: int) -> int:
    return max(1, min(n_jobs, os.cpu_count() or 1, 32))


def make(name: str, requests: Optional[Sequence[int]] = None, threads: Optional[int] = None) -> Workload:
    """Generate a workload (all requests, or only the listed request indices, packed in order).

    A subset keeps every request's own values (each request has its own random streams),
    so oracle results on a subset line up one-to-one with the full batch.
    """
    sp = spec(name)
    sc = sp.scalars(sp)
    idx = list(range(sp.B)) if requests is None else [int(b) for b in requests]
    cap = (lambda b: int(sc["num_drafts"][b]) + 1) if sp.varlen else (lambda b: sp.k_max + 1)
    with ThreadPoolExecutor(threads or _threads(len(idx))) as ex:
        parts = list(ex.map(lambda b: _gen_request(sp, sc, b, cap(b)), idx))
    return _pack(sp.name, sp.V, sp.k_max, sp.dtype, sp.varlen, idx, sc, parts)


def _pack(name, V, k_max, dtype, varlen, idx, sc, parts) -> Workload:
    B = len(idx)
    nd = np.array([p[0] for p in parts], np.int32)
    caps = [(int(nd[j]) + 1) if varlen else (k_max + 1) for j in range(B)]
    R = int(sum(caps))
    D = R - B
    tl = np.zeros((R, V), np.uint16 if dtype == "bf16" else np.float32)
    dp = np.zeros((D, V), np.float32)
    dt = np.zeros(D, np.int32)
    un = np.zeros((R, 2), np.float32)
    r0 = 0
    for j, (k, t, q, toks, uni) in enumerate(parts):
        d0 = r0 - j
        tl[r0: r0 + k + 1] = t
        dp[d0: d0 + k] = q
        dt[d0: d0 + k] = toks
        un[r0: r0 + caps[j]] = uni[: caps[j]]
        r0 += caps[j]
    ro = None
    if varlen:
        ro = np.zeros(B + 1, np.int32)
        ro[1:] = np.cumsum(caps)
    pick = lambda a: None if a is None else np.ascontiguousarray(a[idx])
    return Workload(name=name, V=V, k_max=k_max, dtype=dtype, num_drafts=nd, row_offsets=ro,
                    target_logits=tl, draft_probs=dp, draft_tokens=dt, uniforms=un,
                    temperature=pick(sc["temperature"]), top_k=pick(sc["top_k"]),
                    top_p=pick(sc["top_p"]), presence=pick(sc["presence"]),
                    frequency=pick(sc["frequency"]), greedy=pick(sc["greedy"]))


def with_history(w: Workload, seed: int, max_len: int, top_share: float = 0.5) -> Workload:
    """Attach a seeded prior history to every request (in place): up to max_len distinct
    tokens, about `top_share` of them among the largest logits of the request's first row (so
    that they meet the kept sets and the drafts) and the rest uniform over the vocabulary,
    each with a count of 1 + Geometric(0.5).  Some requests get an empty history."""
    offs = np.zeros(w.B + 1, np.int32)
    toks, cnts = [], []
    lg = w.logits_f32()
    for b in range(w.B):
        r = _rng(7_400_000 + seed, b)
        n = int(r.integers(0, max_len + 1)) if r.random() < 0.85 else 0
        n = min(n, w.V)
        n_top = min(int(round(n * top_share)), w.V)
        top = np.argsort(-lg[w.row_start(b)], kind="stable")[: max(n_top * 2, 1)]
        pick = set(r.choice(top, size=min(n_top, top.size), replace=False).tolist()) if n_top else set()
        d0 = w.draft_start(b)
        k = int(w.num_drafts[b])
        if k and r.random() < 0.5:
            pick.add(int(w.draft_tokens[d0 + int(r.integers(0, k))]))   # a drafted token too
        while len(pick) < n:
            pick.add(int(r.integers(0, w.V)))
        t = np.array(sorted(pick), np.int32)
        toks.append(t)
        cnts.append((1 + r.geometric(0.5, size=t.size) - 1).astype(np.int32).clip(1, None))
        offs[b + 1] = offs[b] + t.size
    w.prior_offsets = offs
    w.prior_tokens = np.concatenate(toks).astype(np.int32) if toks else np.zeros(0, np.int32)
    w.prior_counts = np.concatenate(cnts).astype(np.int32) if cnts else np.zeros(0, np.int32)
    return w


def with_argmax_drafts(w: Workload) -> Workload:
    """The same batch with every draft token replaced by the argmax of its draft row's q: the
    draft proposer proposing its most likely token, which is the input of the one-hot-draft
    scheme (that scheme then reads no q).  Ties go to the lowest id.  Modifies w in place."""
    if w.draft_tokens.size:
        w.draft_tokens[:] = np.argmax(w.draft_probs, axis=1).astype(np.int32)
    return w


def with_masked_vocab(w: Workload, seed: int, frac: float, keep: int = 3) -> np.ndarray:
    """Masks tokens out of the target rows, as a constrained-decoding mask does: each logit is
    set to -inf with probability frac, and each 256-token segment wholly with probability
    frac / 2; `keep` random tokens of every row stay finite.  A third of the drafts are moved
    onto masked tokens of their row, and half of the rest onto finite ones.  Modifies w in
    place; returns the mask [R, V] (True: masked)."""
    r = np.random.default_rng(np.random.Philox(key=np.array([8_000_000 + seed, 0], dtype=np.uint64)))
    R, V = w.total_rows, w.V
    m = r.random((R, V)) < frac
    nseg = (V + 255) // 256
    for row in range(R):
        for sg in np.nonzero(r.random(nseg) < frac / 2)[0]:
            m[row, sg * 256:(sg + 1) * 256] = True
        m[row, r.choice(V, size=min(keep, V), replace=False)] = False
    if w.dtype == "bf16":
        w.target_logits[m] = np.uint16(0xFF80)
    else:
        w.target_logits[m] = -np.inf
    for b in range(w.B):
        r0, d0 = w.row_start(b), w.draft_start(b)
        for i in range(int(w.num_drafts[b])):
            x = r.random()
            pool = np.nonzero(m[r0 + i])[0] if x < 1 / 3 else (np.nonzero(~m[r0 + i])[0] if x < 2 / 3 else None)
            if pool is not None and len(pool):
                w.draft_tokens[d0 + i] = int(r.choice(pool))
    return m


def layout(name: str):
    """(num_drafts, row_offsets or None, total_rows, total_drafts) of a full workload, cheaply."""
    sp = spec(name)
    sc = sp.scalars(sp)
    nd = sc["num_drafts"]
    if sp.varlen:
        ro = np.zeros(sp.B + 1, np.int32)
        ro[1:] = np.cumsum(nd.astype(np.int64) + 1)
        return nd, ro, int(ro[-1]), int(ro[-1]) - sp.B
    R = sp.B * (sp.k_max + 1)
    return nd, None, R, R - sp.B


def iter_chunks(name: str, chunk: int = 64, threads: Optional[int] = None):
    """Yield (b_lo, b_hi, row_lo, draft_lo, Workload-of-that-range) over a full workload."""
    sp = spec(name)
    _, ro, _, _ = layout(name)
    for lo in range(0, sp.B, chunk):
        hi = min(sp.B, lo + chunk)
        w = make(name, range(lo, hi), threads=threads)
        r0 = int(ro[lo]) if ro is not None else lo * (sp.k_max + 1)
        yield lo, hi, r0, r0 - lo, w


# --------------------------------------------------------------------------------------
# small random batches for parity tests (edge cases, ties, mixed parameters)
# --------------------------------------------------------------------------------------

def random_batch(seed: int, B: int, k_max: int, V: int, dtype: str = "bf16", varlen: bool = False,
                 greedy_frac: float = 0.3, penalties: bool = True, tie_step: float = 0.0,
                 sigma: float = 2.0, draft_sigma: float = 0.7, name: str = "random") -> Workload:
    """A mixed batch: per-request k, temperature, top-k, top-p, penalties and greedy flags.

    tie_step > 0 quantises the target logits to multiples of tie_step, which forces exact
    ties (as bf16 rows have) at top-k/top-p boundaries and at the argmax.
    """
    r = _rng(7_000_000 + seed, 0)
    nd = (r.integers(0, k_max + 1, size=B) if varlen else np.full(B, k_max)).astype(np.int32)
    T = r.uniform(0.3, 1.7, size=B).astype(np.float32)
    tk = np.where(r.random(B) < 0.5, r.integers(1, max(2, min(V, 64)), size=B), 0).astype(np.int32)
    tk = np.where(r.random(B) < 0.1, V + 3, tk).astype(np.int32)     # >= V: disabled
    tp = np.where(r.random(B) < 0.5, r.uniform(0.05, 0.999, size=B), 1.0).astype(np.float32)
    g = (r.random(B) < greedy_frac).astype(np.uint8)
    pres = np.where(r.random(B) < 0.5, r.uniform(0.0, 1.5, size=B), 0.0).astype(np.float32) if penalties else None
    freq = np.where(r.random(B) < 0.5, r.uniform(0.0, 1.0, size=B), 0.0).astype(np.float32) if penalties else None
    parts = []
    caps = [(int(nd[b]) + 1) if varlen else (k_max + 1) for b in range(B)]
    for b in range(B):
        k = int(nd[b])
        rr = _rng(7_100_000 + seed, b)
        x = rr.standard_normal((k + 1, V)).astype(np.float32) * np.float32(sigma)
        if tie_step > 0:
            x = (np.round(x / tie_step) * tie_step).astype(np.float32)
        dl = x[:k] + rr.standard_normal((k, V)).astype(np.float32) * np.float32(draft_sigma)
        q = _softmax_rows_f32(dl, float(T[b]))
        toks = _sample_rows(q, _rng((7_200_000 + seed) ^ DRAFT_SALT, b).random(k))
        uni = _rng(7_300_000 + seed, b).random((caps[b], 2), dtype=np.float32)
        tl = f32_to_bf16_bits(x) if dtype == "bf16" else x
        parts.append((k, tl, q, toks, uni))
    sc = dict(temperature=T, top_k=tk, top_p=tp, greedy=g, presence=pres, frequency=freq)
    return _pack(name, V, k_max, dtype, varlen, list(range(B)), sc, parts)


def from_rows(V: int, logits: np.ndarray, q: np.ndarray, drafts: np.ndarray, uniforms: np.ndarray,
              temperature=1.0, top_k=0, top_p=1.0, presence=None, frequency=None, greedy=0,
              dtype: str = "f32", name: str = "explicit") -> Workload:
    """Pack B requests that share k drafts in the uniform layout from explicit arrays.

    logits [B, k+1, V] (float32, or uint16 bf16 bits when dtype == "bf16") or [k+1, V] to
    repeat one set of rows for every request; q [B, k, V] or [k, V]; drafts [B, k];
    uniforms [B, k+1, 2].  Scalar parameters broadcast over the batch.
    """
    drafts = np.asarray(drafts, np.int32)
    B, k = drafts.shape
    lg = np.asarray(logits)
    if lg.ndim == 2:
        lg = np.broadcast_to(lg, (B,) + lg.shape)
    qq = np.asarray(q, np.float32)
    if qq.ndim == 2:
        qq = np.broadcast_to(qq, (B,) + qq.shape)
    bc = lambda x, dt: None if x is None else np.ascontiguousarray(np.broadcast_to(np.asarray(x, dt), (B,)))
    return Workload(name=name, V=V, k_max=k, dtype=dtype, num_drafts=np.full(B, k, np.int32),
                    row_offsets=None,
                    target_logits=np.ascontiguousarray(lg.reshape(B * (k + 1), V)),
                    draft_probs=np.ascontiguousarray(qq.reshape(B * k, V)),
                    draft_tokens=np.ascontiguousarray(drafts.reshape(-1)),
                    uniforms=np.ascontiguousarray(np.asarray(uniforms, np.float32).reshape(B * (k + 1), 2)),
                    temperature=bc(temperature, np.float32), top_k=bc(top_k, np.int32),
                    top_p=bc(top_p, np.float32), presence=bc(presence, np.float32),
                    frequency=bc(frequency, np.float32), greedy=bc(greedy, np.uint8))
